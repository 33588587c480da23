// vcattn_fwd_host: grouping, preprocessing and attention for Q, K, V and O in
// host memory, with the host<->device copies overlapped with the computation.
//
// The method is independent per (b, h): k-means, the permutation, the
// quantisers and the attention of one head never read another head.  The
// flattened B*H heads therefore go through the device in chunks, and two
// device slots alternate:
//
//   copy-in stream     in(0)  in(1)  in(2) ...             (waits: slot free)
//   compute stream 0          grp+prep(0) attn(0)   grp+prep(2) attn(2) ...
//   compute stream 1                 grp+prep(1) attn(1)   grp+prep(3) ...
//   copy-out stream                          out(0)    out(1) ...
//
// The first two chunks have an eighth and three eighths of the heads of the
// others, so that the device starts computing after a short copy and each
// copy in hides behind the computation before it; V of each chunk is copied
// first, so the k-means (which reads only V) overlaps the copy of Q and K.
// Slot s = c % 2 holds chunk c's Q, K, V, labels, perm, workspaces and O, and
// chunk c computes on compute stream s.  With two distinct compute streams
// the launch-bound k-means of one chunk runs beside the attention of the
// other; with one, the chunks compute in turn.  Events per slot order the
// reuse: in(c) waits until the preprocessing of chunk c-2 has read the
// slot's Q, K, V; attn(c) waits until out(c-2) has read the slot's O.
// Everything is enqueued on the caller's streams.  A call starts after the
// work already on compute stream 0 (the other streams wait for it), and
// compute stream 0 finally waits for the last copies out: synchronising it
// completes the call, and consecutive calls can share one workspace.  No
// device memory is allocated; the eleven events are created and released
// (released once complete) inside the call.
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/vcattn.h"
#include "internal.h"

namespace {

constexpr int DEFAULT_CHUNK = 8;

struct Slot {
  void *Q, *K, *V, *O;
  float* lse2;
  int32_t *labels, *perm;
  void* gws;  // grouping workspace
  void* fws;  // prepped tensors + preprocessing workspace (vcattn_fwd layout)
};

// Byte layout of one slot for `ch` heads (256-byte aligned parts).
size_t slot_layout(const vcattn_shape* cs, int k, bool with_lse, char* base, Slot* out,
                   size_t* gws_bytes, size_t* fws_bytes) {
  const size_t BH = size_t(cs->B * cs->H), N = size_t(cs->N);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = vc::align256(off + bytes);
    return p;
  };
  const size_t qkv = BH * N * vc::D * 2;
  Slot s{};
  s.Q = take(qkv);
  s.K = take(qkv);
  s.V = take(qkv);
  s.O = take(qkv);
  s.lse2 = with_lse ? reinterpret_cast<float*>(take(BH * N * 4)) : nullptr;
  s.labels = reinterpret_cast<int32_t*>(take(BH * N * 4));
  s.perm = reinterpret_cast<int32_t*>(take(BH * N * 4));
  const size_t g = vcattn_group_workspace_bytes(cs, k);
  const size_t f = vcattn_fwd_workspace_bytes(cs);
  s.gws = take(g);
  s.fws = take(f);
  if (out) *out = s;
  if (gws_bytes) *gws_bytes = g;
  if (fws_bytes) *fws_bytes = f;
  return (g && f) ? off : 0;
}

int chunk_of(const vcattn_shape* s, int chunk_heads) {
  const int64_t BH = s->B * s->H;
  const int64_t c = chunk_heads > 0 ? chunk_heads : DEFAULT_CHUNK;
  return static_cast<int>(c < BH ? c : BH);
}

vcattn_shape chunk_shape(const vcattn_shape* s, int heads) { return vcattn_shape{1, heads, s->N, s->D}; }

// Events of one call, released when the call returns (each once complete).
struct Events {
  cudaEvent_t e[11] = {};
  cudaError_t init() {
    for (auto& x : e) {
      const cudaError_t r = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
  ~Events() {
    for (auto x : e)
      if (x) cudaEventDestroy(x);
  }
};

}  // namespace

namespace vc {
vcattn_status from_cuda(cudaError_t e);
}

extern "C" {

size_t vcattn_fwd_host_workspace_bytes(const vcattn_shape* s, int k, int chunk_heads) {
  if (!s || s->D != vc::D || s->B < 1 || s->H < 1 || s->N < 1 || chunk_heads < 0) return 0;
  const vcattn_shape cs = chunk_shape(s, chunk_of(s, chunk_heads));
  const size_t one = slot_layout(&cs, k, true, nullptr, nullptr, nullptr, nullptr);
  return one ? 2 * one : 0;
}

vcattn_status vcattn_fwd_host(const vcattn_shape* s, const void* hQ, const void* hK, const void* hV,
                              int k, int iters, float sm_scale, const uint8_t* tile_mask, void* hO,
                              float* hlse2, int chunk_heads, void* ws, size_t ws_bytes,
                              void* const streams[4]) {
  if (!s || !hQ || !hK || !hV || !hO || !ws || !streams) return VCATTN_ERR_INVALID_ARG;
  if (s->D != vc::D) return VCATTN_ERR_UNSUPPORTED;
  if (s->B < 1 || s->H < 1 || s->N < 1 || chunk_heads < 0 || iters < 1) return VCATTN_ERR_INVALID_ARG;
  if (k < 1 || k > vc::KMAX) return VCATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return VCATTN_ERR_INVALID_ARG;
  cudaStream_t scs[2] = {static_cast<cudaStream_t>(streams[0]), static_cast<cudaStream_t>(streams[1])};
  cudaStream_t si = static_cast<cudaStream_t>(streams[2]);
  cudaStream_t so = static_cast<cudaStream_t>(streams[3]);
  if (si == so || si == scs[0] || si == scs[1] || so == scs[0] || so == scs[1]) return VCATTN_ERR_INVALID_ARG;
  const int64_t BH = s->B * s->H, N = s->N;
  const int ch = chunk_of(s, chunk_heads);
  const vcattn_shape cs = chunk_shape(s, ch);
  size_t gb = 0, fb = 0;
  const size_t one = slot_layout(&cs, k, true, nullptr, nullptr, &gb, &fb);
  if (!one || ws_bytes < 2 * one) return VCATTN_ERR_INVALID_ARG;
  Slot slot[2];
  slot_layout(&cs, k, true, static_cast<char*>(ws), &slot[0], nullptr, nullptr);
  slot_layout(&cs, k, true, static_cast<char*>(ws) + one, &slot[1], nullptr, nullptr);
  if (!hlse2) slot[0].lse2 = slot[1].lse2 = nullptr;

  Events ev;
  cudaError_t ce = ev.init();
  if (ce != cudaSuccess) return vc::from_cuda(ce);
  cudaEvent_t* ev_in = ev.e;        // copy-in of the slot finished
  cudaEvent_t* ev_free = ev.e + 2;  // preprocessing has read the slot's Q, K, V
  cudaEvent_t* ev_comp = ev.e + 4;  // the slot's O is written
  cudaEvent_t* ev_out = ev.e + 6;   // the slot's O has been copied out
  cudaEvent_t ev_start = ev.e[8];   // everything before the call on compute stream 0
  cudaEvent_t* ev_inv = ev.e + 9;   // V of the slot is in

  const size_t row = size_t(N) * vc::D * 2;  // bytes of one head of Q, K, V or O
  const int64_t nq64 = (N + vc::BLK - 1) / vc::BLK, nbp = vc::npad(N) / vc::BLK;
  // chunk c covers heads [h0(c), h0(c) + heads(c)): ramp-up chunks of ch/8 and
  // 3ch/8 heads (rounded up; while the first computes, the second is copied
  // in, and so on), then ch
  const int r0 = (ch + 7) / 8, r1 = (3 * ch + 7) / 8;
  auto chunk_at = [&](int64_t c, int64_t* h0, int64_t* want) {
    if (c == 0) { *h0 = 0; *want = r0; }
    else if (c == 1) { *h0 = r0; *want = r1; }
    else { *h0 = r0 + r1 + (c - 2) * ch; *want = ch; }
  };
  int64_t nchunks = 0;
  for (int64_t h = 0; h < BH; ++nchunks) {
    int64_t a, b;
    chunk_at(nchunks, &a, &b);
    h = a + b;
  }
  auto cu = [](cudaError_t e) { return e == cudaSuccess ? VCATTN_OK : vc::from_cuda(e); };
  vcattn_status st = cu(cudaEventRecord(ev_start, scs[0]));
  if (st == VCATTN_OK) st = cu(cudaStreamWaitEvent(si, ev_start, 0));
  if (st == VCATTN_OK) st = cu(cudaStreamWaitEvent(so, ev_start, 0));
  if (st == VCATTN_OK && scs[1] != scs[0]) st = cu(cudaStreamWaitEvent(scs[1], ev_start, 0));
  for (int64_t c = 0; c < nchunks && st == VCATTN_OK; ++c) {
    const int b = static_cast<int>(c & 1);
    const Slot& sl = slot[b];
    cudaStream_t sc = scs[b];
    int64_t h0 = 0, want = 0;
    chunk_at(c, &h0, &want);
    const int heads = static_cast<int>(BH - h0 < want ? BH - h0 : want);
    const vcattn_shape hs = chunk_shape(s, heads);
    const size_t bytes = size_t(heads) * row;
    // copy in
    if ((st = cu(cudaStreamWaitEvent(si, ev_free[b], 0))) != VCATTN_OK) break;
    if ((st = cu(cudaMemcpyAsync(sl.V, static_cast<const char*>(hV) + h0 * row, bytes,
                                 cudaMemcpyHostToDevice, si))) != VCATTN_OK) break;
    if ((st = cu(cudaEventRecord(ev_inv[b], si))) != VCATTN_OK) break;
    if ((st = cu(cudaMemcpyAsync(sl.Q, static_cast<const char*>(hQ) + h0 * row, bytes,
                                 cudaMemcpyHostToDevice, si))) != VCATTN_OK) break;
    if ((st = cu(cudaMemcpyAsync(sl.K, static_cast<const char*>(hK) + h0 * row, bytes,
                                 cudaMemcpyHostToDevice, si))) != VCATTN_OK) break;
    if ((st = cu(cudaEventRecord(ev_in[b], si))) != VCATTN_OK) break;
    // compute: grouping once V is in, preprocessing once Q and K are, then
    // (once the slot's O is free) attention
    if ((st = cu(cudaStreamWaitEvent(sc, ev_inv[b], 0))) != VCATTN_OK) break;
    if ((st = vcattn_group(&hs, sl.V, k, iters, sl.labels, sl.perm, nullptr, sl.gws, gb, sc)) != VCATTN_OK) break;
    if ((st = cu(cudaStreamWaitEvent(sc, ev_in[b], 0))) != VCATTN_OK) break;
    vcattn_prepped pp{};
    const size_t pb = vc::align256(vcattn_prepped_bytes(&hs));
    if ((st = vcattn_prepped_carve(&hs, sl.fws, pb, &pp)) != VCATTN_OK) break;
    if ((st = vcattn_prep(&hs, sl.Q, sl.K, sl.V, sl.perm, &pp, static_cast<char*>(sl.fws) + pb, fb - pb,
                          sc)) != VCATTN_OK)
      break;
    if ((st = cu(cudaEventRecord(ev_free[b], sc))) != VCATTN_OK) break;
    if ((st = cu(cudaStreamWaitEvent(sc, ev_out[b], 0))) != VCATTN_OK) break;
    const uint8_t* mask = tile_mask ? tile_mask + h0 * nq64 * nbp : nullptr;
    if ((st = vcattn_attn(&hs, &pp, sm_scale, mask, sl.O, sl.lse2, sc)) != VCATTN_OK) break;
    if ((st = cu(cudaEventRecord(ev_comp[b], sc))) != VCATTN_OK) break;
    // copy out
    if ((st = cu(cudaStreamWaitEvent(so, ev_comp[b], 0))) != VCATTN_OK) break;
    if ((st = cu(cudaMemcpyAsync(static_cast<char*>(hO) + h0 * row, sl.O, bytes, cudaMemcpyDeviceToHost,
                                 so))) != VCATTN_OK)
      break;
    if (hlse2 && (st = cu(cudaMemcpyAsync(hlse2 + h0 * N, sl.lse2, size_t(heads) * N * 4,
                                          cudaMemcpyDeviceToHost, so))) != VCATTN_OK)
      break;
    if ((st = cu(cudaEventRecord(ev_out[b], so))) != VCATTN_OK) break;
  }
  // The compute stream completes only after every copy out (a wait on an
  // event that was never recorded is a no-op).
  for (int b = 0; b < 2 && st == VCATTN_OK; ++b) st = cu(cudaStreamWaitEvent(scs[0], ev_out[b], 0));
  return st;
}

}  // extern "C"
