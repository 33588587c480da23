// Internal declarations shared by the translation units of libvcattn.so.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace vc {

constexpr int D = 128;          // head dimension
constexpr int BLK = 64;         // quantisation / mean block (tokens)
constexpr int TILE = 128;       // KV tile and padding granule
constexpr int UPD_CHUNK = 512;  // token chunk of the centroid sums
constexpr int KMAX = 64;        // largest k-means k
constexpr float AMAX_FLOOR = 7.888609052210118e-31f;  // 2^-100

// Device error word codes (bit flags, OR-ed by kernels).
constexpr uint32_t ERR_TIMEOUT = 1u;
constexpr uint32_t ERR_BAD_LABEL = 2u;
constexpr uint32_t ERR_BAD_PERM = 4u;   // a permutation entry outside [0, N)

__host__ __device__ inline int64_t npad(int64_t n) { return ((n + TILE - 1) / TILE) * TILE; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Where the rows of a bf16 [B, H, N, D] tensor live: element strides of the
// batch, head and token dimensions (channels contiguous).  Row (bh, n) starts
// at head(bh) + row(n), bh = b * H + h.  The token stride is below 2^31 and
// n below 2^30, so row(n) is one 32 x 32 -> 64-bit multiply.
struct RowLayout {
  int64_t sb, sh, H;
  int32_t sn, pad;
  __host__ __device__ int64_t head(int64_t bh) const { return (bh / H) * sb + (bh % H) * sh; }
  __host__ __device__ int64_t row(int64_t n) const {
    return static_cast<int64_t>(static_cast<int32_t>(n)) * static_cast<int64_t>(sn);
  }
};
inline RowLayout contiguous_rows(int64_t H, int64_t N) { return RowLayout{H * N * D, N * D, H, D, 0}; }

// The current device, for per-device host state (function attributes and
// SM counts are per device); false when it is not one of the first 64.
constexpr int MAX_DEVICES = 64;
inline bool current_device(int* dev) {
  return cudaGetDevice(dev) == cudaSuccess && *dev >= 0 && *dev < MAX_DEVICES;
}

// Per-device host state (kernel attributes, SM counts) set up by the first
// call on each device.  `setup(dev)` returns a cudaError_t; it runs under a
// lock, so first calls from several host threads at once do not race, and a
// failure is returned and retried by the next call.
struct PerDevice {
  std::mutex mu;
  bool done[MAX_DEVICES] = {};
  int value[MAX_DEVICES] = {};
};
template <class F>
cudaError_t per_device_setup(PerDevice& pd, int* dev, F&& setup) {
  if (!current_device(dev)) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(pd.mu);
  if (pd.done[*dev]) return cudaSuccess;
  const cudaError_t e = setup(*dev, &pd.value[*dev]);
  if (e == cudaSuccess) pd.done[*dev] = true;
  return e;
}

// ---- grouping (group.cu) ----
// A token whose assignment the tensor-core filter left open: its flat index
// b*H*N + h*N + j, the candidate clusters and its |v| bound.
struct KmAmb {
  int64_t tok;
  uint64_t cand;
  float vn;
  float pad;
};
struct GroupWs {
  float* cent;         // [BH, k, D]
  float* part;         // [BH, k, nchunk, D]
  int32_t* cnt;        // [BH, nchunk, k]
  int32_t* offs;       // [BH, nchunk, k]
  KmAmb* amb;          // [BH * N] open assignments of one iteration
  uint32_t* amb_count; // [2]: how many, for even and odd iterations
  float* head_cn;      // [BH, 2]: max |c| and max |h| bounds of each head
  float* head_h;       // [BH, 64]: h_c of each head
  float* vnorm;        // [BH, N]: |v| bound of each token (stored by the first iteration)
};
size_t group_ws_layout(int64_t BH, int64_t N, int k, void* base, GroupWs* ws);
// Tensor-core k-means assignment with an exact FP32 fallback (km_tc.cu);
// 1 <= k <= 64.
// Iteration `iter` = 0 computes the tokens' |v| bounds into ws.vnorm, later
// iterations read them.
// tdump (test hook, nullable): [BH, N, 65] f32, the tensor-core scores T_c
// (c < 64) and the token's filter bound E, written for every token.
cudaError_t launch_km_assign_tc(const uint16_t* V, const RowLayout& lv, int64_t BH, int64_t N, int k,
                                const float* cent, int32_t* labels, const GroupWs& ws, int iter,
                                uint32_t* err, cudaStream_t s, float* tdump = nullptr);
cudaError_t launch_group(const uint16_t* V, const RowLayout& lv, int64_t BH, int64_t N, int k, int iters,
                         const float* init, int32_t* labels, int32_t* perm, float* centroids_out,
                         const GroupWs& ws, uint32_t* err, cudaStream_t s);

// ---- preprocessing (prep.cu) ----
struct PrepOut {
  uint8_t *q8, *k8, *r8t;
  float *q_scale, *k_scale, *v_scale, *k_mean, *v_mean, *qmu, *vmu_op;
};
struct PrepWs {
  float* kbs;       // [BH, nbp, D] K block sums (original order)
  uint32_t* vamax;  // [BH, D] V residual amax (float bits)
};
size_t prep_ws_layout(int64_t BH, int64_t N, void* base, PrepWs* ws);
// A perm entry outside [0, N) gathers a zero row and sets ERR_BAD_PERM in *err.
// flags: PREP_QK_HADAMARD rotates Q and centred K before their quantisers.
constexpr int PREP_QK_HADAMARD = 1;
cudaError_t launch_prep(const uint16_t* Q, const RowLayout& lq, const uint16_t* K, const RowLayout& lk,
                        const uint16_t* V, const RowLayout& lv, const int32_t* perm, int64_t BH, int64_t N,
                        const PrepOut& out, const PrepWs& ws, uint32_t* err, int flags, cudaStream_t s);

// ---- attention (attn.cu) ----
struct AttnArgs {
  const uint8_t *q8, *k8, *r8t;
  const float *q_scale, *k_scale, *v_scale, *qmu, *vmu_op;
  const uint8_t* mask;  // nullable
  void* O;              // bf16, or f32 when out_f32
  RowLayout lo;         // rows of O (in elements of O's type)
  int out_f32;
  float* lse2;          // nullable
  int64_t BH, N;
  float sm_scale;
  int off;
  float tau8;
  uint32_t* err;
  int debug_flags;  // test hook: bit 0 = the TMA producer issues nothing;
                    // bits 8.. = n > 0: it stops after n steps
};
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);
// Test hook: the attention kernel's ExpCast bytes for given scores (n a
// multiple of 4; four consecutive scores share A[i/4] and B[i/4]).
cudaError_t launch_expcast_probe(const float* x, const float* A, const float* B, uint8_t* codes, int64_t n,
                                 cudaStream_t s);

}  // namespace vc
