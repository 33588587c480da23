// C ABI of libvcattn.so (declared in include/vcattn.h): argument checks,
// workspace carving and kernel launches.  Nothing here allocates device
// memory; the caller owns every buffer.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/vcattn.h"
#include "internal.h"

namespace vc {
// The CUDA error behind the calling thread's last VCATTN_ERR_CUDA.
thread_local cudaError_t g_last_cuda = cudaSuccess;

vcattn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return VCATTN_OK;
  g_last_cuda = e;
  return VCATTN_ERR_CUDA;
}
}  // namespace vc
using vc::from_cuda;

namespace {
uint32_t* err_word(vcattn_status* st);
}  // namespace

namespace vc {
// The device error word of the current device (for the other translation
// units of the library).
uint32_t* device_error_word(vcattn_status* st) { return err_word(st); }
}  // namespace vc

namespace {

using vc::D;

// Per-device error word.  Kernels OR bits into it; vcattn_last_device_error
// reads and clears it.  Host code needs its device address, obtained once per
// device with cudaGetSymbolAddress (no allocation).
__device__ uint32_t g_err_word;

constexpr int MAX_DEV = 64;
uint32_t* g_err_ptr[MAX_DEV];
std::mutex g_mu;

uint32_t* err_word(vcattn_status* st) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= MAX_DEV) {
    *st = e != cudaSuccess ? from_cuda(e) : VCATTN_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e2 = cudaGetSymbolAddress(&p, g_err_word);
    if (e2 != cudaSuccess || !p) {
      *st = from_cuda(e2 != cudaSuccess ? e2 : cudaErrorInvalidSymbol);
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vcattn_status check_shape(const vcattn_shape* s) {
  if (!s) return VCATTN_ERR_INVALID_ARG;
  if (s->D != D) return VCATTN_ERR_UNSUPPORTED;
  if (s->B < 1 || s->H < 1 || s->N < 1) return VCATTN_ERR_INVALID_ARG;
  if (s->N > (int64_t(1) << 30) || s->B * s->H > 65535) return VCATTN_ERR_UNSUPPORTED;
  return VCATTN_OK;
}


// Row layout of a [B, H, N, D] tensor from caller strides (nullptr = contiguous).
// Strides must be positive multiples of 8 elements (every row 16-byte aligned).
bool rows_of(const vcattn_shape* s, const vcattn_strides* st, vc::RowLayout* out) {
  if (!st) {
    *out = vc::contiguous_rows(s->H, s->N);
    return true;
  }
  const int64_t v[3] = {st->b, st->h, st->n};
  for (int64_t x : v)
    if (x <= 0 || (x & 7) != 0 || x > (int64_t(1) << 38)) return false;
  if (st->n >= (int64_t(1) << 31)) return false;
  *out = vc::RowLayout{st->b, st->h, s->H, static_cast<int32_t>(st->n), 0};
  return true;
}

// Layout of the prepped tensors inside one buffer (256-byte aligned parts).
size_t prepped_layout(const vcattn_shape* s, void* base, vcattn_prepped* out) {
  const int64_t BH = s->B * s->H, N = s->N, Np = vc::npad(N), nbp = Np / vc::BLK;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = vc::align256(off + bytes);
    return base ? static_cast<char*>(base) + o : nullptr;
  };
  vcattn_prepped p{};
  p.q8 = reinterpret_cast<uint8_t*>(take(size_t(BH) * Np * D));
  p.k8 = reinterpret_cast<uint8_t*>(take(size_t(BH) * Np * D));
  p.r8t = reinterpret_cast<uint8_t*>(take(size_t(BH) * Np * D));
  p.q_scale = reinterpret_cast<float*>(take(size_t(BH) * nbp * 4));
  p.k_scale = reinterpret_cast<float*>(take(size_t(BH) * nbp * 4));
  p.v_scale = reinterpret_cast<float*>(take(size_t(BH) * D * 4));
  p.k_mean = reinterpret_cast<float*>(take(size_t(BH) * D * 4));
  p.v_mean = reinterpret_cast<float*>(take(size_t(BH) * nbp * D * 4));
  p.qmu = reinterpret_cast<float*>(take(size_t(BH) * N * 4));
  p.vmu_op = reinterpret_cast<float*>(take(size_t(BH) * (Np / vc::BLK) * vc::D * 4 * 4));
  if (out) *out = p;
  return off;
}

bool prepped_ok(const vcattn_prepped* p) {
  const void* ptrs[] = {p->q8, p->k8, p->r8t, p->q_scale, p->k_scale, p->v_scale,
                        p->k_mean, p->v_mean, p->qmu, p->vmu_op};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return false;
  return true;
}

vc::PrepOut to_prep_out(const vcattn_prepped* p) {
  return vc::PrepOut{p->q8, p->k8, p->r8t, p->q_scale, p->k_scale, p->v_scale,
                     p->k_mean, p->v_mean, p->qmu, p->vmu_op};
}

}  // namespace

extern "C" {

int64_t vcattn_npad(int64_t N) { return vc::npad(N); }

size_t vcattn_group_workspace_bytes(const vcattn_shape* s, int k) {
  if (check_shape(s) != VCATTN_OK || k < 1 || k > vc::KMAX) return 0;
  return vc::group_ws_layout(s->B * s->H, s->N, k, nullptr, nullptr);
}

}  // extern "C"

namespace {
vcattn_status group_impl(const vcattn_shape* s, const void* V, const vcattn_strides* sv, int k, int iters,
                         const float* init, int32_t* labels, int32_t* perm, float* centroids, void* ws,
                         size_t ws_bytes, void* stream) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  vc::RowLayout lv{};
  if (!rows_of(s, sv, &lv)) return VCATTN_ERR_INVALID_ARG;
  if (k < 1 || k > vc::KMAX) return VCATTN_ERR_UNSUPPORTED;
  if (iters < 1 || !V || !labels || !perm || !ws) return VCATTN_ERR_INVALID_ARG;
  if (!aligned16(V) || !aligned16(labels) || !aligned16(perm) || !aligned16(ws) ||
      (centroids && !aligned16(centroids)) || (init && !aligned16(init)))
    return VCATTN_ERR_INVALID_ARG;
  const int64_t BH = s->B * s->H;
  vc::GroupWs w{};
  if (ws_bytes < vc::group_ws_layout(BH, s->N, k, ws, &w)) return VCATTN_ERR_INVALID_ARG;
  uint32_t* err = err_word(&st);
  if (!err) return st;
  return from_cuda(vc::launch_group(static_cast<const uint16_t*>(V), lv, BH, s->N, k, iters, init, labels,
                                    perm, centroids, w, err, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

vcattn_status vcattn_group(const vcattn_shape* s, const void* V, int k, int iters, int32_t* labels,
                           int32_t* perm, float* centroids, void* ws, size_t ws_bytes,
                           void* stream) {
  return group_impl(s, V, nullptr, k, iters, nullptr, labels, perm, centroids, ws, ws_bytes, stream);
}

vcattn_status vcattn_group_warm(const vcattn_shape* s, const void* V, int k, int iters,
                                const float* init_centroids, int32_t* labels, int32_t* perm,
                                float* centroids, void* ws, size_t ws_bytes, void* stream) {
  if (!init_centroids) return VCATTN_ERR_INVALID_ARG;
  return group_impl(s, V, nullptr, k, iters, init_centroids, labels, perm, centroids, ws, ws_bytes, stream);
}

vcattn_status vcattn_group_strided(const vcattn_shape* s, const void* V, const vcattn_strides* sv, int k,
                                   int iters, const float* init_centroids, int32_t* labels, int32_t* perm,
                                   float* centroids, void* ws, size_t ws_bytes, void* stream) {
  if (!sv) return VCATTN_ERR_INVALID_ARG;
  return group_impl(s, V, sv, k, iters, init_centroids, labels, perm, centroids, ws, ws_bytes, stream);
}

size_t vcattn_prepped_bytes(const vcattn_shape* s) {
  if (check_shape(s) != VCATTN_OK) return 0;
  return prepped_layout(s, nullptr, nullptr);
}

vcattn_status vcattn_prepped_carve(const vcattn_shape* s, void* base, size_t bytes,
                                   vcattn_prepped* out) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  if (!base || !out || !aligned16(base)) return VCATTN_ERR_INVALID_ARG;
  if (bytes < prepped_layout(s, nullptr, nullptr)) return VCATTN_ERR_INVALID_ARG;
  prepped_layout(s, base, out);
  return VCATTN_OK;
}

size_t vcattn_prep_workspace_bytes(const vcattn_shape* s) {
  if (check_shape(s) != VCATTN_OK) return 0;
  return vc::prep_ws_layout(s->B * s->H, s->N, nullptr, nullptr);
}

}  // extern "C"

namespace {
vcattn_status prep_impl(const vcattn_shape* s, const void* Q, const vcattn_strides* sq, const void* K,
                        const vcattn_strides* sk, const void* V, const vcattn_strides* sv, const int32_t* perm,
                        int flags, const vcattn_prepped* out, void* ws, size_t ws_bytes, void* stream) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  if (flags & ~VCATTN_PREP_QK_HADAMARD) return VCATTN_ERR_INVALID_ARG;
  vc::RowLayout lq{}, lk{}, lv{};
  if (!rows_of(s, sq, &lq) || !rows_of(s, sk, &lk) || !rows_of(s, sv, &lv)) return VCATTN_ERR_INVALID_ARG;
  if (!Q || !K || !V || !out || !ws || !prepped_ok(out)) return VCATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws) ||
      (perm && !aligned16(perm)))
    return VCATTN_ERR_INVALID_ARG;
  const int64_t BH = s->B * s->H;
  vc::PrepWs w{};
  if (ws_bytes < vc::prep_ws_layout(BH, s->N, ws, &w)) return VCATTN_ERR_INVALID_ARG;
  uint32_t* err = err_word(&st);
  if (!err) return st;
  return from_cuda(vc::launch_prep(static_cast<const uint16_t*>(Q), lq, static_cast<const uint16_t*>(K), lk,
                                   static_cast<const uint16_t*>(V), lv, perm, BH, s->N,
                                   to_prep_out(out), w, err, flags, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

vcattn_status vcattn_prep(const vcattn_shape* s, const void* Q, const void* K, const void* V,
                          const int32_t* perm, const vcattn_prepped* out, void* ws,
                          size_t ws_bytes, void* stream) {
  return prep_impl(s, Q, nullptr, K, nullptr, V, nullptr, perm, 0, out, ws, ws_bytes, stream);
}

vcattn_status vcattn_prep_strided(const vcattn_shape* s, const void* Q, const vcattn_strides* sq,
                                  const void* K, const vcattn_strides* sk, const void* V,
                                  const vcattn_strides* sv, const int32_t* perm, const vcattn_prepped* out,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (!sq || !sk || !sv) return VCATTN_ERR_INVALID_ARG;
  return prep_impl(s, Q, sq, K, sk, V, sv, perm, 0, out, ws, ws_bytes, stream);
}

vcattn_status vcattn_prep_ex(const vcattn_shape* s, const void* Q, const vcattn_strides* sq, const void* K,
                             const vcattn_strides* sk, const void* V, const vcattn_strides* sv,
                             const int32_t* perm, int flags, const vcattn_prepped* out, void* ws,
                             size_t ws_bytes, void* stream) {
  return prep_impl(s, Q, sq, K, sk, V, sv, perm, flags, out, ws, ws_bytes, stream);
}

namespace {
vcattn_status attn_impl(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale, int off,
                        float tau8, int out_f32, const uint8_t* tile_mask, void* O, const vcattn_strides* so,
                        float* lse2, void* stream, int debug_flags) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  vc::RowLayout lo{};
  if (!rows_of(s, so, &lo)) return VCATTN_ERR_INVALID_ARG;
  if (!in || !prepped_ok(in) || !O || !aligned16(O) || (lse2 && !aligned16(lse2)))
    return VCATTN_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || off < 0 || off > 8 || !(tau8 >= 0.0f) || tau8 > 8.0f * (8.75f - off) ||
      (out_f32 != 0 && out_f32 != 1))
    return VCATTN_ERR_INVALID_ARG;
  uint32_t* err = err_word(&st);
  if (!err) return st;
  vc::AttnArgs a{};
  a.q8 = in->q8;
  a.k8 = in->k8;
  a.r8t = in->r8t;
  a.q_scale = in->q_scale;
  a.k_scale = in->k_scale;
  a.v_scale = in->v_scale;
  a.qmu = in->qmu;
  a.vmu_op = in->vmu_op;
  a.mask = tile_mask;
  a.O = O;
  a.lo = lo;
  a.out_f32 = out_f32;
  a.lse2 = lse2;
  a.BH = s->B * s->H;
  a.N = s->N;
  a.sm_scale = sm_scale;
  a.off = off;
  a.tau8 = tau8;
  a.err = err;
  a.debug_flags = debug_flags;
  return from_cuda(vc::launch_attn(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

vcattn_status vcattn_attn_ex(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale,
                             int off, float tau8, int out_f32, const uint8_t* tile_mask, void* O,
                             float* lse2, void* stream) {
  return attn_impl(s, in, sm_scale, off, tau8, out_f32, tile_mask, O, nullptr, lse2, stream, 0);
}

vcattn_status vcattn_attn_strided(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale,
                                  int off, float tau8, int out_f32, const uint8_t* tile_mask, void* O,
                                  const vcattn_strides* so, float* lse2, void* stream) {
  if (!so) return VCATTN_ERR_INVALID_ARG;
  return attn_impl(s, in, sm_scale, off, tau8, out_f32, tile_mask, O, so, lse2, stream, 0);
}

vcattn_status vcattn_test_attn_stalled(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale,
                                       void* O, float* lse2, void* stream) {
  return attn_impl(s, in, sm_scale, 8, 6.0f, 0, nullptr, O, nullptr, lse2, stream, 1);
}

vcattn_status vcattn_test_attn_stalled_after(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale,
                                             const uint8_t* tile_mask, int steps, void* O, float* lse2,
                                             void* stream) {
  if (steps < 1 || steps > (1 << 20)) return VCATTN_ERR_INVALID_ARG;
  return attn_impl(s, in, sm_scale, 8, 6.0f, 0, tile_mask, O, nullptr, lse2, stream, steps << 8);
}

vcattn_status vcattn_test_km_scores(const vcattn_shape* s, const void* V, int k, const float* centroids,
                                    int32_t* labels, float* scores, void* ws, size_t ws_bytes, void* stream) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  if (k < 1 || k > vc::KMAX) return VCATTN_ERR_UNSUPPORTED;
  if (!V || !centroids || !labels || !scores || !ws || !aligned16(V) || !aligned16(centroids) ||
      !aligned16(labels) || !aligned16(scores) || !aligned16(ws))
    return VCATTN_ERR_INVALID_ARG;
  const int64_t BH = s->B * s->H;
  vc::GroupWs w{};
  if (ws_bytes < vc::group_ws_layout(BH, s->N, k, ws, &w)) return VCATTN_ERR_INVALID_ARG;
  uint32_t* err = err_word(&st);
  if (!err) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(w.amb_count, 0, 2 * sizeof(uint32_t), cs);
  if (e == cudaSuccess)
    e = vc::launch_km_assign_tc(static_cast<const uint16_t*>(V), vc::contiguous_rows(s->H, s->N), BH, s->N, k,
                                centroids, labels, w, 0, err, cs, scores);
  return from_cuda(e);
}

vcattn_status vcattn_test_expcast(const float* x, const float* A, const float* B, uint8_t* codes, int64_t n,
                                  void* stream) {
  if (n < 0 || (n & 3) != 0) return VCATTN_ERR_INVALID_ARG;
  if (n == 0) return VCATTN_OK;
  if (!x || !A || !B || !codes || !aligned16(x) || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))
    return VCATTN_ERR_INVALID_ARG;
  return from_cuda(vc::launch_expcast_probe(x, A, B, codes, n, static_cast<cudaStream_t>(stream)));
}

vcattn_status vcattn_attn(const vcattn_shape* s, const vcattn_prepped* in, float sm_scale,
                          const uint8_t* tile_mask, void* O, float* lse2, void* stream) {
  return vcattn_attn_ex(s, in, sm_scale, 8, 6.0f, 0, tile_mask, O, lse2, stream);
}

size_t vcattn_fwd_workspace_bytes(const vcattn_shape* s) {
  if (check_shape(s) != VCATTN_OK) return 0;
  return vc::align256(prepped_layout(s, nullptr, nullptr)) +
         vc::prep_ws_layout(s->B * s->H, s->N, nullptr, nullptr);
}

vcattn_status vcattn_fwd(const vcattn_shape* s, const void* Q, const void* K, const void* V,
                         const int32_t* perm, float sm_scale, const uint8_t* tile_mask, void* O,
                         float* lse2, void* ws, size_t ws_bytes, void* stream) {
  vcattn_status st = check_shape(s);
  if (st != VCATTN_OK) return st;
  if (!ws || !aligned16(ws)) return VCATTN_ERR_INVALID_ARG;
  if (ws_bytes < vcattn_fwd_workspace_bytes(s)) return VCATTN_ERR_INVALID_ARG;
  vcattn_prepped pp{};
  const size_t pb = vc::align256(prepped_layout(s, ws, &pp));
  st = vcattn_prep(s, Q, K, V, perm, &pp, static_cast<char*>(ws) + pb, ws_bytes - pb, stream);
  if (st != VCATTN_OK) return st;
  return vcattn_attn(s, &pp, sm_scale, tile_mask, O, lse2, stream);
}

vcattn_status vcattn_last_device_error(void* stream) {
  vcattn_status st = VCATTN_OK;
  uint32_t* err = err_word(&st);
  if (!err) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  uint32_t h = 0;
  if ((e = cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) return from_cuda(e);
  if (h) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(err, &zero, 4, cudaMemcpyHostToDevice)) != cudaSuccess) return from_cuda(e);
  }
  if (h & vc::ERR_TIMEOUT) return VCATTN_ERR_TIMEOUT;
  if (h) return VCATTN_ERR_DEVICE;
  return VCATTN_OK;
}

const char* vcattn_last_cuda_error(void) {
  return vc::g_last_cuda == cudaSuccess ? "no error" : cudaGetErrorString(vc::g_last_cuda);
}

const char* vcattn_status_string(vcattn_status s) {
  switch (s) {
    case VCATTN_OK: return "ok";
    case VCATTN_ERR_INVALID_ARG: return "invalid argument";
    case VCATTN_ERR_UNSUPPORTED: return "unsupported shape or device";
    case VCATTN_ERR_CUDA: return "CUDA error";
    case VCATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case VCATTN_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

}  // extern "C"
