// Fused preprocessing of the smoothed FP8 attention forward:
//  - K centring ("Feat: Attention Smoothing to Improve Generation Quality",
//    Changes: K centred by its FP32 sequence mean before E4M3 quantisation);
//  - V-Smooth ("VC-Attention: Value Smoothing and Softmax Casting for Low-bit
//    Attention", Key Contributions 1 and 3): K and V gathered by the grouping
//    permutation, each 64-token block of V demeaned, only the residual
//    quantised; the gather happens on the fly so the permuted bf16 tensors
//    never make an HBM round trip.
//
// Thread mapping of the block kernels (256 threads per 64-token block):
// lane bits 0..3 pick a group of 4 consecutive tokens, lane bit 4 and the
// warp pick a chunk of 8 channels; each thread loads 4 x 16 bytes.  Block
// sums are the adjacent-pairing tree: the 4 tokens of a thread first, then a
// shuffle butterfly over the token-group lanes (xor 1, 2, 4, 8).
// Quantiser: amax = max|x|; amax < 2^-100 -> bytes 0, scale 1; inv =
// fl(448/amax); byte = E4M3_rne_satfinite(fl(x*inv)); scale = fl(amax/448).
// Compiled with --fmad=false: only explicit __fmaf_rn calls fuse.
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace vc {
namespace {

__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Two FP32 values -> two E4M3 bytes (round to nearest even, saturating to
// +-448), `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint2 e4m3x8(const float (&x)[8]) {
  uint2 o;
  o.x = e4m3x2(x[0], x[1]) | (e4m3x2(x[2], x[3]) << 16);
  o.y = e4m3x2(x[4], x[5]) | (e4m3x2(x[6], x[7]) << 16);
  return o;
}

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

struct Map {
  int warp, lane, g, cc;
};
__device__ __forceinline__ Map thread_map() {
  Map m;
  m.warp = threadIdx.x >> 5;
  m.lane = threadIdx.x & 31;
  m.g = m.lane & 15;                     // token group (4 tokens)
  m.cc = 2 * m.warp + (m.lane >> 4);     // channel chunk (8 channels)
  return m;
}
// The quantisers' mapping: the 16 lanes of a half-warp take the 16 channel
// chunks of the same 4 rows, so each of their 8-byte stores of a row is one
// contiguous 128-byte line.
__device__ __forceinline__ Map quant_map() {
  Map m;
  m.warp = threadIdx.x >> 5;
  m.lane = threadIdx.x & 31;
  m.cc = m.lane & 15;                    // channel chunk (8 channels)
  m.g = 2 * m.warp + (m.lane >> 4);      // token group (4 tokens)
  return m;
}

// A block's 64 rows are staged in shared memory with cp.async (all loads in
// flight at once): [64 rows][16 chunks of 16 bytes], the chunk index XOR-ed
// with (row / 4) so that the compute mapping (lanes = 4-row groups) reads
// without bank conflicts.  Rows past N are zero.  `perm` maps a sorted
// position to its source token (nullptr = identity).
constexpr int TILE_SMEM = BLK * D * 2;  // 16 KiB
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 256 + ((chunk ^ ((row >> 2) & 15)) * 16));
}
// The source rows of the 4 pieces a thread stages for the block starting at
// r0 (rows r0 + threadIdx.x / 16 + 16 u); loaded one block ahead so that the
// gather index is in a register when the copy is issued.
struct Src4 {
  int32_t r[4];
};
// A perm entry outside [0, N) is never dereferenced: its row is staged as
// zeros and `bad` is set (the kernel reports it once, at its end, through
// report_bad_perm; an atomic here would slow every load).
__device__ __forceinline__ Src4 load_src(const int32_t* perm, int64_t r0, int64_t N, bool& bad) {
  Src4 s;
  const int32_t n32 = static_cast<int32_t>(N);  // N < 2^30
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int32_t r = static_cast<int32_t>(r0) + u * 16 + (static_cast<int>(threadIdx.x) >> 4);
    const int32_t src = r < n32 ? (perm ? perm[r] : r) : -1;
    const bool out = r < n32 && static_cast<uint32_t>(src) >= static_cast<uint32_t>(n32);
    bad |= out;
    s.r[u] = out ? -1 : src;
  }
  return s;
}
__device__ __forceinline__ void report_bad_perm(bool bad, uint32_t* err) {
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(err, ERR_BAD_PERM);
}
// rows src of the head at `base`, `sn` elements apart
__device__ __forceinline__ void stage_rows(uint8_t* tile, const uint16_t* base, int32_t sn, const Src4& src4) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int piece = u * 256 + static_cast<int>(threadIdx.x);
    const int row = piece >> 4, chunk = piece & 15;
    uint8_t* dst = tile + swz(row, chunk);
    if (src4.r[u] >= 0) {
      const int32_t src = src4.r[u];
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                   "l"(base + static_cast<int64_t>(static_cast<int32_t>(src)) * sn + chunk * 8)
                   : "memory");
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}
// The 4 rows x 8 channels of thread (g, cc) from a staged tile.
__device__ __forceinline__ void read_rows(const uint8_t* tile, int g, int cc, float (&x)[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack8(*reinterpret_cast<const uint4*>(tile + swz(4 * g + i, cc)), x[i]);
}

// Adjacent-pairing tree over the 64 tokens of the block (per channel).
__device__ __forceinline__ void block_tree(const float (&x)[4][8], float (&s)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) s[c] = (x[0][c] + x[1][c]) + (x[2][c] + x[3][c]);
#pragma unroll
  for (int m = 1; m < 16; m <<= 1)
#pragma unroll
    for (int c = 0; c < 8; ++c) s[c] = s[c] + __shfl_xor_sync(0xffffffffu, s[c], m);
}

__device__ __forceinline__ float max16(float a) {
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  return a;
}

// Block max of two values at once over all 256 threads (one pair of barriers).
__device__ __forceinline__ float2 block_max2(float a, float b, float* red) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, m));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = a;
    red[8 + (threadIdx.x >> 5)] = b;
  }
  __syncthreads();
  float ra = red[0], rb = red[8];
#pragma unroll
  for (int w = 1; w < 8; ++w) {
    ra = fmaxf(ra, red[w]);
    rb = fmaxf(rb, red[8 + w]);
  }
  return make_float2(ra, rb);
}

// The 128-point Hadamard butterfly of one row held by four consecutive lanes,
// 32 channels each (lane & 3 = qq holds channels 32 qq ..): stages
// h = 1, 2, ..., 64 in that order, each pair (x[i], x[i + h]) with i & h == 0
// becoming (x[i] + x[i + h], x[i] - x[i + h]) in FP32.  From h = 2 on, two
// neighbouring pairs go through one packed f32x2 instruction each, and the
// difference is fma(x[i + h], -1, x[i]): one rounding of the same exact
// value.  In the two cross-lane stages the lane holding the upper half takes
// fma(own, -1, partner) = partner - own, the other fma(own, 1, partner).
__device__ __forceinline__ void hadamard_row32(float (&x)[32], int qq) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {  // h = 1
    const float a = x[i], c = x[i + 1];
    x[i] = a + c;
    x[i + 1] = a - c;
  }
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 2; h < 32; h <<= 1)
#pragma unroll
    for (int i = 0; i < 32; i += 2)
      if ((i & h) == 0) {
        const float2 a = make_float2(x[i], x[i + 1]), c = make_float2(x[i + h], x[i + h + 1]);
        const float2 sum = __fadd2_rn(a, c), dif = __ffma2_rn(c, m1, a);
        x[i] = sum.x;
        x[i + 1] = sum.y;
        x[i + h] = dif.x;
        x[i + h + 1] = dif.y;
      }
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int lm = 1 << s;             // h = 32 (lane ^ 1), then h = 64 (lane ^ 2)
    const float sg = (qq & lm) != 0 ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, x[i], lm), __shfl_xor_sync(0xffffffffu, x[i + 1], lm));
      const float2 r = __ffma2_rn(make_float2(x[i], x[i + 1]), sg2, o);
      x[i] = r.x;
      x[i + 1] = r.y;
    }
  }
}

// Stats: K block sums (original order), mean of each permuted V block, and
// the per-channel amax of the V residual.  Each CTA handles STATS_BPC
// consecutive blocks; block b+1 is staged while block b is reduced, and the
// residual amax is kept in registers until one atomicMax per channel at the
// end (max is order-independent).  grid (ceil(nb / STATS_BPC), BH), block
// 256, dynamic shared memory STATS_SMEM (two stages of K and V tiles).
constexpr int STATS_BPC = 8;
constexpr int STATS_SMEM = 2 * 2 * TILE_SMEM;
__global__ void __launch_bounds__(256, 3) prep_stats(const uint16_t* __restrict__ K, RowLayout lk,
                                                  const uint16_t* __restrict__ V, RowLayout lv,
                                                  const int32_t* __restrict__ perm, int64_t N,
                                                  int nb, int nbp, float* __restrict__ kbs,
                                                  float* __restrict__ v_mean,
                                                  uint32_t* __restrict__ vamax, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t ssm[];
  const Map m = thread_map();
  const int64_t bh = blockIdx.y;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * STATS_BPC;
  const int64_t b1 = b0 + STATS_BPC < nb ? b0 + STATS_BPC : nb;
  const int32_t* ph = perm ? perm + bh * N : nullptr;
  const uint16_t* Kh = K + lk.head(bh);
  const uint16_t* Vh = V + lv.head(bh);
  // gather indices of the next block to stage (one block ahead)
  bool bad = false;
  Src4 nk = load_src(nullptr, b0 * BLK, N, bad), nv = load_src(ph, b0 * BLK, N, bad);
  auto stage = [&](int64_t b, int buf) {
    stage_rows(ssm + buf * 2 * TILE_SMEM, Kh, lk.sn, nk);
    stage_rows(ssm + buf * 2 * TILE_SMEM + TILE_SMEM, Vh, lv.sn, nv);
    cp_commit();
    if (b + 1 < b1) {
      nk = load_src(nullptr, (b + 1) * BLK, N, bad);
      nv = load_src(ph, (b + 1) * BLK, N, bad);
    }
  };
  stage(b0, 0);
  float am[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) am[c] = 0.0f;
  for (int64_t b = b0; b < b1; ++b) {
    const int buf = static_cast<int>((b - b0) & 1);
    if (b + 1 < b1) {
      stage(b + 1, buf ^ 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const int64_t r0 = b * BLK + 4 * m.g;
    float kx[4][8], vx[4][8];
    read_rows(ssm + buf * 2 * TILE_SMEM, m.g, m.cc, kx);
    read_rows(ssm + buf * 2 * TILE_SMEM + TILE_SMEM, m.g, m.cc, vx);
    float ks[8], vs[8], mu[8];
    block_tree(kx, ks);
    block_tree(vx, vs);
    const int64_t nvalid = N - b * BLK < BLK ? N - b * BLK : BLK;
    const float fn = static_cast<float>(nvalid);
    // x / 64 is x * 2^-6 exactly (both correctly round the same value), so
    // full blocks multiply; only the last, partial block divides.
    if (nvalid == BLK) {
#pragma unroll
      for (int c = 0; c < 8; ++c) mu[c] = vs[c] * 0.015625f;
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) mu[c] = vs[c] / fn;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (r0 + i < N) am[c] = fmaxf(am[c], fabsf(vx[i][c] - mu[c]));
    if (m.g == 0) {
      const int64_t o = (bh * nbp + b) * D + 8 * m.cc;
      *reinterpret_cast<float4*>(kbs + o) = make_float4(ks[0], ks[1], ks[2], ks[3]);
      *reinterpret_cast<float4*>(kbs + o + 4) = make_float4(ks[4], ks[5], ks[6], ks[7]);
      *reinterpret_cast<float4*>(v_mean + o) = make_float4(mu[0], mu[1], mu[2], mu[3]);
      *reinterpret_cast<float4*>(v_mean + o + 4) = make_float4(mu[4], mu[5], mu[6], mu[7]);
    }
    __syncthreads();  // this stage may be restaged next iteration
  }
  report_bad_perm(bad, err);
#pragma unroll
  for (int c = 0; c < 8; ++c) am[c] = max16(am[c]);
  if (m.g == 0)
#pragma unroll
    for (int c = 0; c < 8; ++c) atomicMax(vamax + bh * D + 8 * m.cc + c, __float_as_uint(am[c]));
}

// mu_K = (adjacent-pairing tree over the block sums, padded with +0 to a
// power of two P) / N; v_scale from the residual amax.  The tree over P
// leaves is cut into KM_SEG aligned subtrees of P / KM_SEG leaves (the
// tree's own nodes, so the sums are bit-identical): thread (d, seg) reduces
// subtree seg of channel d with eight independent loads in flight, then the
// KM_SEG subtree sums are combined in tree order.  grid (BH), block
// (D, KM_SEG).
constexpr int KM_SEG = 8;
__global__ void __launch_bounds__(D * KM_SEG) prep_kmean(const float* __restrict__ kbs,
                                                         const uint32_t* __restrict__ vamax, int64_t N,
                                                         int nb, int nbp, float* __restrict__ k_mean,
                                                         float* __restrict__ v_scale) {
  __shared__ float sub[KM_SEG][D];
  const int64_t bh = blockIdx.x;
  const int d = threadIdx.x, seg = threadIdx.y;
  int64_t P = 1;
  while (P < nb) P *= 2;
  const int nseg = P < KM_SEG ? static_cast<int>(P) : KM_SEG;  // a power of two
  const int64_t len = P / nseg;                                 // leaves per subtree
  if (seg < nseg) {
    const int64_t lo = seg * len;
    const float* src = kbs + bh * nbp * D + d;
    float st[40];
    int top = 0;
    for (int64_t b = 0; b < len; b += 8) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t leaf = lo + b + e;
        v[e] = (b + e < len && leaf < nb) ? src[leaf * D] : 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (b + e >= len) break;
        float x = v[e];
        for (int64_t t = b + e; t & 1; t >>= 1) x = st[--top] + x;
        st[top++] = x;
      }
    }
    sub[seg][d] = st[0];
  }
  __syncthreads();
  if (seg == 0) {
    float st[4];
    int top = 0;
    for (int i = 0; i < nseg; ++i) {
      float x = sub[i][d];
      for (int t = i; t & 1; t >>= 1) x = st[--top] + x;
      st[top++] = x;
    }
    k_mean[bh * D + d] = st[0] / static_cast<float>(N);
    const float a = __uint_as_float(vamax[bh * D + d]);
    v_scale[bh * D + d] = a >= AMAX_FLOOR ? a / 448.0f : 1.0f;
  }
}

// Quantisers, one tensor per CTA (blockIdx.y: 0 = Q, 1 = K, 2 = V).  Each CTA
// handles QUANT_BPC consecutive 64-token blocks of one (b, h) through a ring
// of QUANT_NST staged tiles (16 KiB each, all rows of a tile in flight at
// once), so QUANT_NST - 1 blocks load while one is quantised.  One tensor per
// CTA keeps the per-thread state small (32 values), so three CTAs fit on an
// SM, and lets each path do only its own arithmetic:
//   Q: block amax from the bf16 bits (|x| as an integer max of the bit
//      patterns, exact), q8 = E4M3(fl(x * inv)), q_scale, and qmu (one fmaf
//      chain per row, warps 0-1);
//   K: gathered, centred (fl(k - mu_K)), block amax, k8, k_scale;
//   V: gathered, fl(fl(v - mu_b) * vinv_d) transposed to r8t, the mean
//      operand of the block, zero means for padding blocks.
// The FP32 operations and their order are those of the per-element
// definition (packed f32x2 instructions round each lane as the scalar ones
// do).  With the QK Hadamard flag the Q and K paths rotate first (four lanes
// per row, as in hadamard_row32).  grid (ceil(nbp / QUANT_BPC), 3, BH),
// block 256, dynamic shared memory QUANT_SMEM: the heads in reverse order
// with the three tensors of a head together, so that the first heads
// quantised are the last ones prep_stats read, whose K and V are still in
// L2.
constexpr int QUANT_BPC = 8;
constexpr int QUANT_NST = 3;
constexpr int QUANT_SMEM = QUANT_NST * TILE_SMEM + D * (BLK + 16) + D * 4 + 64;

__device__ __forceinline__ float2 bf2f(uint32_t w) {  // (low, high) bf16 of a word as floats
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t e4m3x4(float2 a, float2 b) {
  return e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
}
// Block max over all 256 threads (one barrier; `red` is reused after the
// caller's next barrier).
__device__ __forceinline__ float block_max1(float a, float* red) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
  return r;
}

__global__ void __launch_bounds__(256, 3) prep_quant(
    const uint16_t* __restrict__ Q, RowLayout lq, const uint16_t* __restrict__ K, RowLayout lk,
    const uint16_t* __restrict__ V, RowLayout lv,
    const int32_t* __restrict__ perm, int64_t N, int64_t Npad, int nbp,
    const uint32_t* __restrict__ vamax, const float* __restrict__ k_mean,
    const float* __restrict__ v_scale, float* __restrict__ v_mean, uint8_t* __restrict__ q8,
    uint8_t* __restrict__ k8, uint8_t* __restrict__ r8t, float* __restrict__ q_scale,
    float* __restrict__ k_scale, float* __restrict__ qmu, float* __restrict__ vmu_op, uint32_t* err,
    int rot) {
  extern __shared__ __align__(128) uint8_t qsm[];
  uint8_t (*tb)[BLK + 16] = reinterpret_cast<uint8_t (*)[BLK + 16]>(qsm + QUANT_NST * TILE_SMEM);
  float* kmu = reinterpret_cast<float*>(qsm + QUANT_NST * TILE_SMEM + D * (BLK + 16));
  float* red = kmu + D;
  const int z = blockIdx.y;  // 0 = Q, 1 = K, 2 = V
  // V keeps the token-group lanes (its transposed bytes go to shared memory
  // without bank conflicts); Q and K take the coalescing mapping
  const Map m = z == 2 ? thread_map() : quant_map();
  const int64_t bh = gridDim.z - 1 - blockIdx.z;  // heads in reverse order
  const int64_t nb = ceil_div(N, BLK);
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * QUANT_BPC;
  const int64_t b1 = b0 + QUANT_BPC < nbp ? b0 + QUANT_BPC : nbp;
  const int32_t* ph = (perm && z > 0) ? perm + bh * N : nullptr;
  const uint16_t* src = z == 0 ? Q + lq.head(bh) : z == 1 ? K + lk.head(bh) : V + lv.head(bh);
  const int32_t sn = z == 0 ? lq.sn : z == 1 ? lk.sn : lv.sn;
  // the ring: block b in stage (b - b0) % QUANT_NST; the gather indices of
  // the next block to stage are loaded one staging ahead
  bool bad = false;
  Src4 nxt = load_src(ph, b0 * BLK, N, bad);
  int64_t bs = b0;  // next block to stage
  auto stage_next = [&]() {
    if (bs < b1) {
      stage_rows(qsm + ((bs - b0) % QUANT_NST) * TILE_SMEM, src, sn, nxt);
      ++bs;
      if (bs < b1) nxt = load_src(ph, bs * BLK, N, bad);
    }
    cp_commit();  // one group per call, empty past the last block
  };
#pragma unroll
  for (int u = 0; u < QUANT_NST - 1; ++u) stage_next();
  if (z < 2 && threadIdx.x < D) kmu[threadIdx.x] = k_mean[bh * D + threadIdx.x];
  float vinv[8];
  if (z == 2) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float am = __uint_as_float(vamax[bh * D + 8 * m.cc + c]);
      vinv[c] = am >= AMAX_FLOOR ? 448.0f / am : 0.0f;
    }
  }

  for (int64_t b = b0; b < b1; ++b) {
    cp_wait<QUANT_NST - 2>();
    __syncthreads();  // block b has landed everywhere; the stage of b - 1 is free
    stage_next();
    const uint8_t* t = qsm + ((b - b0) % QUANT_NST) * TILE_SMEM;
    const int64_t r0 = b * BLK + 4 * m.g;
    const bool tail = b * BLK + BLK > N;  // the block holds rows past N
    const bool pad_block = b >= nb;

    if (z == 2) {
      // ---- V: gathered, block-demeaned residual, per-channel scale, transposed ----
      const int64_t mo = (bh * nbp + b) * D + 8 * m.cc;
      float mu[8];
      if (pad_block) {
#pragma unroll
        for (int c = 0; c < 8; ++c) mu[c] = 0.0f;
      } else {
        const float4 a0 = *reinterpret_cast<const float4*>(v_mean + mo);
        const float4 a1 = *reinterpret_cast<const float4*>(v_mean + mo + 4);
        mu[0] = a0.x; mu[1] = a0.y; mu[2] = a0.z; mu[3] = a0.w;
        mu[4] = a1.x; mu[5] = a1.y; mu[6] = a1.z; mu[7] = a1.w;
      }
      const float2 nmu[4] = {make_float2(-mu[0], -mu[1]), make_float2(-mu[2], -mu[3]),
                             make_float2(-mu[4], -mu[5]), make_float2(-mu[6], -mu[7])};
      const float2 vi[4] = {make_float2(vinv[0], vinv[1]), make_float2(vinv[2], vinv[3]),
                            make_float2(vinv[4], vinv[5]), make_float2(vinv[6], vinv[7])};
      uint2 by[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = *reinterpret_cast<const uint4*>(t + swz(4 * m.g + i, m.cc));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float2 y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = __fmul2_rn(__fadd2_rn(bf2f(w[e]), nmu[e]), vi[e]);
        if (tail && r0 + i >= N) {
#pragma unroll
          for (int e = 0; e < 4; ++e) y[e] = make_float2(0.0f, 0.0f);
        }
        by[i] = make_uint2(e4m3x4(y[0], y[1]), e4m3x4(y[2], y[3]));
      }
      // channel c's bytes of the thread's 4 rows -> one 32-bit word of tb[d][4g..4g+3]
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t sel = static_cast<uint32_t>((c & 3) | ((4 + (c & 3)) << 4));
        const uint32_t w01 = c < 4 ? __byte_perm(by[0].x, by[1].x, sel) : __byte_perm(by[0].y, by[1].y, sel);
        const uint32_t w23 = c < 4 ? __byte_perm(by[2].x, by[3].x, sel) : __byte_perm(by[2].y, by[3].y, sel);
        *reinterpret_cast<uint32_t*>(&tb[8 * m.cc + c][4 * m.g]) = __byte_perm(w01, w23, 0x5410);
      }
      if (pad_block && m.g == 0) {
        *reinterpret_cast<float4*>(v_mean + mo) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(v_mean + mo + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // the mean operand of the rank-one restoration MMA: one 16-byte row
      // per channel d, (hi, hi, lo, 0) of mu_b[d] / v_scale[d] (2 KiB per
      // block, so the mean tile of any two blocks is two contiguous copies)
      if (threadIdx.x < D) {
        const int d = threadIdx.x;
        const float mud = pad_block ? 0.0f : v_mean[(bh * nbp + b) * D + d];
        const float uq = mud / v_scale[bh * D + d];
        const float hi = to_tf32(uq);
        const float lo = to_tf32(uq - hi);
        reinterpret_cast<float4*>(vmu_op + (bh * nbp + b) * (4 * D))[d] = make_float4(hi, hi, lo, 0.0f);
      }
      __syncthreads();
      {
        const int d = threadIdx.x >> 1, h = threadIdx.x & 1;
        const uint4* s4 = reinterpret_cast<const uint4*>(&tb[d][32 * h]);
        uint4* dst = reinterpret_cast<uint4*>(r8t + (bh * D + d) * Npad + b * BLK + 32 * h);
        dst[0] = s4[0];
        dst[1] = s4[1];
      }
    } else if (!rot) {
      // ---- Q (original order) or K (gathered, centred): per 64-row block ----
      uint8_t* out = z == 0 ? q8 : k8;
      uint32_t w[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = *reinterpret_cast<const uint4*>(t + swz(4 * m.g + i, m.cc));
        w[i][0] = u.x; w[i][1] = u.y; w[i][2] = u.z; w[i][3] = u.w;
      }
      float2 x[4][4];
      float a;
      if (z == 0) {
        // |x| of bf16 as the integer max of the sign-cleared bit patterns
        uint32_t mb = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) mb = __vmaxu2(mb, w[i][e] & 0x7FFF7FFFu);
        a = __uint_as_float(((mb >> 16) > (mb & 0xFFFFu) ? (mb >> 16) : (mb & 0xFFFFu)) << 16);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) x[i][e] = bf2f(w[i][e]);  // rows past N are staged as +0
      } else {
        const float* km = kmu + 8 * m.cc;
        const float2 nk[4] = {make_float2(-km[0], -km[1]), make_float2(-km[2], -km[3]),
                              make_float2(-km[4], -km[5]), make_float2(-km[6], -km[7])};
        a = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[i][e] = __fadd2_rn(bf2f(w[i][e]), nk[e]);
          if (tail && r0 + i >= N) {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[i][e] = make_float2(0.0f, 0.0f);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) a = fmaxf(a, fmaxf(fabsf(x[i][e].x), fabsf(x[i][e].y)));
        }
      }
      const float amax = block_max1(a, red);
      const bool live = amax >= AMAX_FLOOR;
      const float inv = live ? 448.0f / amax : 0.0f;
      const float2 iv = make_float2(inv, inv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint2 o = make_uint2(0u, 0u);
        if (live) {
          float2 y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) y[e] = __fmul2_rn(x[i][e], iv);
          o = make_uint2(e4m3x4(y[0], y[1]), e4m3x4(y[2], y[3]));
        }
        *reinterpret_cast<uint2*>(out + (bh * Npad + r0 + i) * D + 8 * m.cc) = o;
      }
      if (threadIdx.x == 0) (z == 0 ? q_scale : k_scale)[bh * nbp + b] = live ? amax / 448.0f : 1.0f;
    } else {
      // ---- Q or centred K with the Hadamard rotation: thread (row rr,
      // quarter qq) holds channels 32 qq .. 32 qq + 31 of one row ----
      uint8_t* out = z == 0 ? q8 : k8;
      const int rr = threadIdx.x >> 2, qq = threadIdx.x & 3;
      const bool valid = b * BLK + rr < N;
      float hx[32];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float tv[8];
        unpack8(*reinterpret_cast<const uint4*>(t + swz(rr, 4 * qq + c4)), tv);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          hx[8 * c4 + e] = z == 0 ? tv[e] : (valid ? tv[e] - kmu[32 * qq + 8 * c4 + e] : 0.0f);
      }
      hadamard_row32(hx, qq);
      const float sc = z == 0 ? 0.0625f : 0.125f;
      float a = 0.0f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        hx[e] *= sc;
        a = fmaxf(a, fabsf(hx[e]));
      }
      const float amax = block_max1(a, red);
      const bool live = amax >= AMAX_FLOOR;
      const float inv = live ? 448.0f / amax : 0.0f;
      uint2 o4[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = (live && valid) ? hx[8 * c4 + e] * inv : 0.0f;
        o4[c4] = e4m3x8(y);
      }
      uint4* dst = reinterpret_cast<uint4*>(out + (bh * Npad + b * BLK + rr) * D + 32 * qq);
      dst[0] = make_uint4(o4[0].x, o4[0].y, o4[1].x, o4[1].y);
      dst[1] = make_uint4(o4[2].x, o4[2].y, o4[3].x, o4[3].y);
      if (threadIdx.x == 0) (z == 0 ? q_scale : k_scale)[bh * nbp + b] = live ? amax / 448.0f : 1.0f;
    }
    if (z == 0 && threadIdx.x < BLK) {
      // qmu = q . mu_K (the unrotated q): one fmaf chain over d ascending
      const int rr = threadIdx.x;
      const int64_t r = b * BLK + rr;
      if (r < N) {
        float acc = 0.0f;
        for (int cc = 0; cc < 16; ++cc) {
          float qv[8];
          unpack8(*reinterpret_cast<const uint4*>(t + swz(rr, cc)), qv);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = __fmaf_rn(qv[e], kmu[8 * cc + e], acc);
        }
        qmu[bh * N + r] = acc;
      }
    }
  }
  report_bad_perm(bad, err);
}

}  // namespace

size_t prep_ws_layout(int64_t BH, int64_t N, void* base, PrepWs* ws) {
  const int64_t nbp = npad(N) / BLK;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return base ? static_cast<char*>(base) + o : nullptr;
  };
  PrepWs w{};
  w.kbs = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * nbp * D * 4));
  w.vamax = reinterpret_cast<uint32_t*>(take(static_cast<size_t>(BH) * D * 4));
  if (ws) *ws = w;
  return off;
}

cudaError_t launch_prep(const uint16_t* Q, const RowLayout& lq, const uint16_t* K, const RowLayout& lk,
                        const uint16_t* V, const RowLayout& lv, const int32_t* perm, int64_t BH, int64_t N,
                        const PrepOut& o, const PrepWs& ws, uint32_t* err, int flags, cudaStream_t s) {
  const int64_t Np = npad(N);
  const int nbp = static_cast<int>(Np / BLK);
  const int nb = static_cast<int>(ceil_div(N, BLK));
  cudaError_t e = cudaMemsetAsync(ws.vamax, 0, static_cast<size_t>(BH) * D * 4, s);
  if (e != cudaSuccess) return e;
  // the shared-memory limit is a per-device attribute of each kernel
  static PerDevice attr;
  int dev = 0;
  e = per_device_setup(attr, &dev, [](int, int*) {
    cudaError_t r = cudaFuncSetAttribute(prep_stats, cudaFuncAttributeMaxDynamicSharedMemorySize, STATS_SMEM);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(prep_quant, cudaFuncAttributeMaxDynamicSharedMemorySize, QUANT_SMEM);
    return r;
  });
  if (e != cudaSuccess) return e;
  prep_stats<<<dim3(static_cast<unsigned>(ceil_div(nb, STATS_BPC)), static_cast<unsigned>(BH)), 256,
               STATS_SMEM, s>>>(K, lk, V, lv, perm, N, nb, nbp, ws.kbs, o.v_mean, ws.vamax, err);
  prep_kmean<<<static_cast<unsigned>(BH), dim3(D, KM_SEG), 0, s>>>(ws.kbs, ws.vamax, N, nb, nbp,
                                                                   o.k_mean, o.v_scale);
  prep_quant<<<dim3(static_cast<unsigned>(ceil_div(nbp, QUANT_BPC)), 3, static_cast<unsigned>(BH)), 256,
               QUANT_SMEM, s>>>(
      Q, lq, K, lk, V, lv, perm, N, Np, nbp, ws.vamax, o.k_mean, o.v_scale, o.v_mean, o.q8, o.k8, o.r8t,
      o.q_scale, o.k_scale, o.qmu, o.vmu_op, err, (flags & PREP_QK_HADAMARD) != 0);
  return cudaGetLastError();
}

}  // namespace vc
