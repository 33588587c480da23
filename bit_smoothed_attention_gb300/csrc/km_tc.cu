// k-means assignment on the tensor core, with an exact fallback
// ("VC-Attention: Value Smoothing and Softmax Casting for Low-bit
// Attention", Key Contribution 1: the online k-means of V-Smooth).
//
// The label of token j is the lowest cluster c with the largest
//   score_c = fl(chain_c - h_c),  chain_c = fmaf chain over d = 0..127 of
//   v_d c_{c,d} from +0,  h_c = 0.5f * (fmaf chain of c_{c,d}^2),
// the same definition as the FP32-core assign.  Here the tensor core first
// computes an approximation T_c of every score:
//   c = hi + lo (two bf16 parts, |c - hi - lo| <= 2^-18 |c|), v exact in
//   bf16, h = h1 + h2 + h3 (three bf16 parts, exact to 2^-24 |h|);
//   T = v . hi + v . lo - (h1 + h2 + h3) as one kind::f16 MMA chain with
//   FP32 accumulation (M = 128 tokens, N = 64 clusters, K = 2 x 128 + 16,
//   the last K step a constant operand of ones against -h).
// |T_c - score_c| <= 2^-14 (|v| |c| + |h_c|) + 2^-23 |T_c|: the products
// are exact; the accumulation of 272 terms, even with every add truncating,
// errs by at most 272 x 2^-23 < 2^-14.9 of the sum of their magnitudes; the
// FP32 chain and the split add 2^-17 and 2^-18 of |v| |c|, the final
// subtraction 2^-24 |score|; and sum_d |v_d c_d| <= |v| |c|.  With the
// token's E = (2^-13 + 2^-21) (|v| max|c| + max|h|), at least twice that,
// and m = max_c T_c, the winner w has T_w >= score_w - E/2 >= score_c* -
// E/2 >= m - E (c* the argmax of T).  So clusters with T_c < m - E cannot
// win.
// When one cluster is left it is the label.  Otherwise (0.6% of the tokens
// on the live workload) the token goes on a list, and km_fixup, launched
// right after, resolves every listed token with one warp: a second filter
// computes the candidates' FP32 dot products (lanes over candidates and
// channel groups) and drops those more than E2 = 2^-15 (|v| max|c| +
// max|h|) below the best of them (the same argument with a tighter bound);
// the exact chains of what is left decide, lowest index first on ties.
// (Done in place, these few tokens held their whole warp on a chain of
// global loads: a third of the assignment time.)  The labels are those of
// the FP32 definition, bit for bit, whatever the data.
//
// CTA: a run of consecutive 128-token tiles of one (b, h).  Warps 0-3:
// one thread per token (= TMEM lane) for the selection; warp 4: TMA; warp 5:
// MMA lane.  V tiles (bf16, two 64-channel K chunks, 128B swizzle) through a
// ring of KT_NS stages; the scores T in two TMEM buffers of 64 columns.
// Compiled with --fmad=false: only the explicit __fmaf_rn calls fuse.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace vc {
namespace {

constexpr int KT_NS = 2;            // V stages
constexpr int KT_THREADS = 192;     // 4 selection warps, TMA warp, MMA warp
constexpr int KT_WARP_TMA = 4;
constexpr int KT_WARP_MMA = 5;
constexpr uint32_t V_HALF = 128 * 128;       // 128 tokens x 64 bf16 channels
constexpr uint32_t V_STAGE = 2 * V_HALF;     // one 128-token tile
constexpr uint32_t CP_CHUNK = 64 * 128;      // 64 clusters x 64 bf16 channels
constexpr uint32_t SM_V = 0;
constexpr uint32_t SM_CP = SM_V + KT_NS * V_STAGE;  // [part][K chunk]
constexpr uint32_t SM_AB = SM_CP + 4 * CP_CHUNK;    // A of the bias step: 128 rows of (1, 1, 1, 0, ...)
constexpr uint32_t SM_BB = SM_AB + 128 * 32;        // B of the bias step: 64 rows of (-h1, -h2, -h3, 0, ...)
constexpr uint32_t SM_H = SM_BB + 64 * 32;          // h_c
constexpr uint32_t SM_CN = SM_H + 64 * 4;           // [0]: max |c|, [1]: max |h|
enum { KB_FULL = 0, KB_EMPTY = KT_NS, KB_DFULL = 2 * KT_NS, KB_DEMPTY = 2 * KT_NS + 2, KB_FIN = 2 * KT_NS + 4, KB_N };
constexpr uint32_t SM_BAR = SM_CN + 64 * 4;
constexpr uint32_t SM_TSLOT = SM_BAR + KB_N * 8;
constexpr uint32_t SM_ABORT = SM_TSLOT + 8;
constexpr uint32_t KT_SMEM = SM_ABORT + 8 + 1024;  // slack for 1024-byte alignment
constexpr uint32_t IDESC_KM = idesc(FMT_BF16, FMT_BF16, 128, 64);
constexpr uint64_t KT_WAIT_NS = 2000000000ull;

// Byte offset of element e (0..63) of row r in a 128-byte-row, 128B-swizzled
// K-major tile: 8-row atoms of 1 KiB, 16-byte chunk q stored at q ^ (r & 7).
__device__ __forceinline__ uint32_t sw128(int r, int e) {
  const int byte = 2 * e;
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

// Byte offset of element e (0..15) of row r in a K = 16 bf16 operand in the
// interleaved no-swizzle layout (core matrices of 8 rows x 16 bytes, the
// two K halves 128 bytes apart, 8-row groups 256 bytes apart).
__device__ __forceinline__ uint32_t k16(int r, int e) {
  return static_cast<uint32_t>((r >> 3) * 256 + (e >> 3) * 128 + (r & 7) * 16 + (e & 7) * 2);
}

__global__ void __launch_bounds__(KT_THREADS, 2)
    km_assign_tc(const __grid_constant__ CUtensorMap tmv, int64_t N, int64_t H, int k, int tpc,
                 const float* __restrict__ cent,
                 int32_t* __restrict__ labels, KmAmb* __restrict__ amb, uint32_t* __restrict__ amb_count,
                 float* __restrict__ head_cn, float* __restrict__ head_h, float* __restrict__ vnorm,
                 int vnorm_ready, uint32_t* __restrict__ err, float* __restrict__ tdump) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, derived from the shared array itself so that the
  // compiler keeps every access through it in the shared state space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * static_cast<uint32_t>(i); };
  volatile int* abort = reinterpret_cast<volatile int*>(sm + SM_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = blockIdx.y;
  const int64_t ntile_all = (N + 127) / 128;
  const int64_t tile0 = static_cast<int64_t>(blockIdx.x) * tpc;
  const int ntl = static_cast<int>(ntile_all - tile0 < tpc ? ntile_all - tile0 : tpc);
  const float* cb = cent + bh * k * D;
  float* hs = reinterpret_cast<float*>(sm + SM_H);
  float* cn = reinterpret_cast<float*>(sm + SM_CN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < KT_NS; ++s) {
      mbar_init(bar(KB_FULL + s), 1);
      mbar_init(bar(KB_EMPTY + s), 5);  // the MMA lane's commit + the 4 selection warps (after |v|)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(KB_DFULL + b), 1);
      mbar_init(bar(KB_DEMPTY + b), 4);
    }
    mbar_init(bar(KB_FIN), 1);
    *abort = 0;
    mbar_fence_init();
  }
  // The FP32 centroids, staged in the V stages (not yet in use) with
  // 16-byte loads, all in flight at once; rows CS floats apart, so that the
  // h_c chains below (thread c reads row c) spread over the banks.
  constexpr int CS = D + 4;
  static_assert(64 * CS * 4 <= KT_NS * V_STAGE, "centroid staging");
  float* cs = reinterpret_cast<float*>(sm + SM_V);
  for (int i = threadIdx.x; i < 64 * D / 4; i += KT_THREADS) {
    const int c = i >> 5;
    *reinterpret_cast<float4*>(cs + c * CS + 4 * (i & 31)) =
        c < k ? *reinterpret_cast<const float4*>(cb + 4 * i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  __syncthreads();
  // B operand: the centroids as bf16 high and low parts (clusters >= k are 0)
  for (int i = threadIdx.x; i < 64 * D; i += KT_THREADS) {
    const int c = i >> 7, d = i & (D - 1);
    const float x = cs[c * CS + d];
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    const int kc = d >> 6, e = d & 63;
    *reinterpret_cast<__nv_bfloat16*>(sm + SM_CP + (0 * 2 + kc) * CP_CHUNK + sw128(c, e)) = hi;
    *reinterpret_cast<__nv_bfloat16*>(sm + SM_CP + (1 * 2 + kc) * CP_CHUNK + sw128(c, e)) = lo;
  }
  // the constant A of the bias step
  for (int i = threadIdx.x; i < 128 * 16; i += KT_THREADS) {
    const int r = i >> 4, e = i & 15;
    *reinterpret_cast<__nv_bfloat16*>(sm + SM_AB + k16(r, e)) = __float2bfloat16_rn(e < 3 ? 1.0f : 0.0f);
  }
  if (threadIdx.x < 64) {
    const int c = threadIdx.x;
    float acc = 0.0f;
    if (c < k)
#pragma unroll 16
      for (int d = 0; d < D; ++d) acc = __fmaf_rn(cs[c * CS + d], cs[c * CS + d], acc);
    const float h = 0.5f * acc;
    hs[c] = h;
    // B of the bias step: -h in three bf16 parts; clusters >= k get -inf
    // (their T is -inf and they never become candidates)
    float hp[3];
    hp[0] = c < k ? h : __int_as_float(0x7f800000);
    hp[1] = c < k ? h - __bfloat162float(__float2bfloat16_rn(hp[0])) : 0.0f;
    hp[2] = c < k ? hp[1] - __bfloat162float(__float2bfloat16_rn(hp[1])) : 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      *reinterpret_cast<__nv_bfloat16*>(sm + SM_BB + k16(c, e)) =
          __float2bfloat16_rn(e < 3 ? -hp[e] : 0.0f);
    // max |c| (sqrt(acc) (1 + 2^-16) >= |c|) and max |h| over the k clusters
    float cm = c < k ? sqrtf(acc) * 1.0000153f : 0.0f, hm = c < k ? fabsf(h) : 0.0f;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, m));
      hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, m));
    }
    if (lane == 0) {
      cn[2 + warp * 2] = cm;
      cn[3 + warp * 2] = hm;
    }
  }
  fence_proxy_async_smem();
  if (warp == KT_WARP_MMA) tmem_alloc(sb + SM_TSLOT, 128);
  // (the V stages are overwritten by TMA only after this barrier)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + SM_TSLOT);

  if (warp == KT_WARP_TMA) {
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < ntl && !*abort; ++t) {
        const int s = t % KT_NS;
        if (t >= KT_NS && !mbar_wait(bar(KB_EMPTY + s), ((t / KT_NS) - 1) & 1, abort, KT_WAIT_NS)) {
          *abort = 1;
          atomicOr(err, ERR_TIMEOUT);
          break;
        }
        const int row = static_cast<int>((tile0 + t) * 128);
        mbar_arrive_expect_tx(bar(KB_FULL + s), V_STAGE);
        const int hh = static_cast<int>(bh % H), bb = static_cast<int>(bh / H);
        tma_load_4d(sb + SM_V + s * V_STAGE, &tmv, 0, row, hh, bb, bar(KB_FULL + s));
        tma_load_4d(sb + SM_V + s * V_STAGE + V_HALF, &tmv, 64, row, hh, bb, bar(KB_FULL + s));
        issued = t + 1;
      }
      // Copies still in flight land before the CTA exits (possible only after
      // an abort; otherwise the consumers have waited for every one).  The
      // wait is bounded by time alone.
      for (int t = issued > KT_NS ? issued - KT_NS : 0; t < issued; ++t)
        if (!mbar_wait_time(bar(KB_FULL + t % KT_NS), (t / KT_NS) & 1, KT_WAIT_NS)) atomicOr(err, ERR_TIMEOUT);
    }
  } else if (warp == KT_WARP_MMA) {
    if (lane == 0) {
      bool ok = true;
      const uint64_t dV = sdesc_sw128(sb + SM_V), dC = sdesc_sw128(sb + SM_CP);
      const uint64_t dAB = sdesc_k8_tf32(sb + SM_AB), dBB = sdesc_k8_tf32(sb + SM_BB);  // 32-byte rows, no swizzle
      for (int t = 0; t < ntl && ok; ++t) {
        const int s = t % KT_NS, b = t & 1;
        ok = mbar_wait(bar(KB_FULL + s), (t / KT_NS) & 1, abort, KT_WAIT_NS);
        if (ok && t >= 2) ok = mbar_wait(bar(KB_DEMPTY + b), ((t >> 1) - 1) & 1, abort, KT_WAIT_NS);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16(tmem + 64 * b, dV + ((s * V_STAGE + kc * V_HALF + 32 * ks) >> 4),
                       dC + (((part * 2 + kc) * CP_CHUNK + 32 * ks) >> 4), IDESC_KM,
                       (part | kc | ks) != 0 ? 1u : 0u);
        mma_bf16(tmem + 64 * b, dAB, dBB, IDESC_KM, 1u);  // - h_c
        mma_commit(bar(KB_DFULL + b));
        mma_commit(bar(KB_EMPTY + s));  // this V stage has been read by the tensor core
      }
      if (!ok) {
        *abort = 1;
        atomicOr(err, ERR_TIMEOUT);
      }
      // every MMA of this lane completes before TMEM is released, also after
      // an abort (the wait ignores the abort flag)
      mma_commit(bar(KB_FIN));
      if (!mbar_wait_time(bar(KB_FIN), 0, KT_WAIT_NS)) atomicOr(err, ERR_TIMEOUT);
    }
  } else {
    // ---------------------------------------------------- selection warps
    const int r = warp * 32 + lane;  // token within the tile = TMEM lane
    // E = EA |v| + EB, with EA = (2^-13 + 2^-21) max|c|, EB = (2^-13 + 2^-21) max|h|
    const float CM = fmaxf(cn[2], cn[4]), HM = fmaxf(cn[3], cn[5]);
    if (blockIdx.x == 0) {  // the same in every CTA of the head
      if (threadIdx.x == 0) {
        head_cn[2 * bh] = CM;
        head_cn[2 * bh + 1] = HM;
      }
      if (threadIdx.x < 64) head_h[bh * 64 + threadIdx.x] = hs[threadIdx.x];
    }
    const float EA = (1.220703125e-4f + 4.76837158e-7f) * CM;
    const float EB = (1.220703125e-4f + 4.76837158e-7f) * HM;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t FULLM = 0xffffffffu;
    // |v| of this thread's token in the next tile, loaded a tile ahead (once
    // the first iteration has stored them)
    float vn_next = 0.0f;
    if (vnorm_ready && tile0 * 128 + r < N) vn_next = vnorm[bh * N + tile0 * 128 + r];
    for (int t = 0; t < ntl; ++t) {
      const int s = t % KT_NS, b = t & 1;
      bool ok = __all_sync(FULLM, mbar_wait(bar(KB_FULL + s), (t / KT_NS) & 1, abort, KT_WAIT_NS));
      const uint8_t* vt = sm + SM_V + s * V_STAGE;
      const int64_t j = (tile0 + t) * 128 + r;
      // |v|: an upper bound (the sum's relative error is far below the
      // factor); it depends on V alone, so the first iteration stores it and
      // the others read it back
      float vn = vn_next;
      if (vnorm_ready && t + 1 < ntl && j + 128 < N) vn_next = vnorm[bh * N + j + 128];  // the next tile's
      if (ok && j < N) {
        if (!vnorm_ready) {
          float2 q2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 u = *reinterpret_cast<const uint4*>(vt + kc * V_HALF + sw128(r, 8 * ch));
              const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 v2 = make_float2(__uint_as_float(w4[e] << 16), __uint_as_float(w4[e] & 0xFFFF0000u));
                q2 = __ffma2_rn(v2, v2, q2);
              }
            }
          vn = sqrtf(q2.x + q2.y) * 1.0000153f;
          vnorm[bh * N + j] = vn;
        }
      }
      // The selection reads nothing else from the V stage: it is free once
      // the tensor core is done with it.  (Waiting for FULL first keeps this
      // arrival in the stage's current phase.)
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar(KB_EMPTY + s));
      ok = ok && __all_sync(FULLM, mbar_wait(bar(KB_DFULL + b), (t >> 1) & 1, abort, KT_WAIT_NS));
      if (!ok) {
        if (lane == 0) atomicOr(err, ERR_TIMEOUT);
        *abort = 1;
        break;
      }
      tc_fence_after();
      float T[64];
      tmem_ld64(tmem + lane_addr + 64 * b, *reinterpret_cast<uint32_t(*)[64]>(&T[0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_DEMPTY + b));

      if (j < N) {
        const float E = EA * vn + EB;
        // m = max_c T_c (eight independent chains), then the candidates
        float m8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) m8[q] = T[q];
#pragma unroll
        for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], T[c]);
        const float m = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                              fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float thr = m - E;
        uint32_t cm8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) cm8[q] = 0u;
#pragma unroll
        for (int c = 0; c < 64; ++c) cm8[c >> 3] |= (T[c] >= thr ? 1u : 0u) << (c & 7);
        uint64_t cand = 0;  // bit c: cluster c can still win
#pragma unroll
        for (int q = 0; q < 8; ++q) cand |= static_cast<uint64_t>(cm8[q]) << (8 * q);
        if (tdump) {  // test hook: the tensor-core scores T_c and the token's bound E
          float* td = tdump + (bh * N + j) * 65;
#pragma unroll
          for (int c = 0; c < 64; ++c) td[c] = T[c];
          td[64] = E;
        }
        const int best = __ffsll(static_cast<long long>(cand)) - 1;
        if (cand & (cand - 1)) {  // left open: km_fixup decides
          const uint32_t slot = atomicAdd(amb_count, 1u);
          amb[slot] = KmAmb{bh * N + j, cand, vn, 0.0f};
        }
        labels[bh * N + j] = best;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == KT_WARP_MMA) tmem_dealloc(tmem, 128);
}

// The assignments the tensor-core filter left open, one warp each.  v comes
// from the bf16 row in global memory, h_c as km_assign_tc computed it.
//  - Second filter (at most four candidates): lanes (q, g) = (lane >> 3,
//    lane & 7) form candidate q's dot product over channels 16g .. 16g+15
//    (an fmaf chain), then a three-level tree over g.  Against the exact
//    chain this errs by at most (128 + 16 + 3) 2^-24 |v| |c| < 2^-16.7 |v| |c|,
//    so E2 = 2^-15 (|v| max|c| + max|h|) is again at least twice the
//    difference of the scores, and candidates more than E2 below the best
//    cannot win.
//  - If two or more are left: lane i runs the exact chain of the i-th
//    candidate; the best score wins, the lower cluster on ties.
__global__ void __launch_bounds__(256) km_fixup(const uint16_t* __restrict__ V, RowLayout lv, int64_t N, int k,
                                                const float* __restrict__ cent, int32_t* __restrict__ labels,
                                                const KmAmb* __restrict__ amb, const uint32_t* __restrict__ count,
                                                uint32_t* __restrict__ next_count,
                                                const float* __restrict__ head_cn,
                                                const float* __restrict__ head_h) {
  const uint32_t n = *count;
  if (blockIdx.x == 0 && threadIdx.x == 0) *next_count = 0;  // for the next iteration's assign
  const int lane = threadIdx.x & 31;
  const uint32_t FULLM = 0xffffffffu;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nwarps) {
    const KmAmb a = amb[i];
    const int64_t bh = a.tok / N;
    const uint16_t* vrow = V + lv.head(bh) + lv.row(a.tok - bh * N);
    const float* cb = cent + bh * k * D;
    const float* hh = head_h + bh * 64;
    uint64_t cand = a.cand;
    if (__popcll(cand) <= 4) {
      const int q = lane >> 3, g = lane & 7;
      // the q-th candidate (or none)
      uint64_t rest = cand;
      for (int x = 0; x < q && rest; ++x) rest &= rest - 1;
      const int cl = rest ? __ffsll(static_cast<long long>(rest)) - 1 : -1;
      float part = 0.0f;
      if (cl >= 0) {
        const uint4 u0 = *reinterpret_cast<const uint4*>(vrow + 16 * g);
        const uint4 u1 = *reinterpret_cast<const uint4*>(vrow + 16 * g + 8);
        const float4* c4 = reinterpret_cast<const float4*>(cb + cl * D + 16 * g);
        const float4 c0 = c4[0], c1 = c4[1], c2 = c4[2], c3 = c4[3];
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float cc[16] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w,
                              c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          part = __fmaf_rn(__uint_as_float(w[e] << 16), cc[2 * e], part);
          part = __fmaf_rn(__uint_as_float(w[e] & 0xFFFF0000u), cc[2 * e + 1], part);
        }
      }
#pragma unroll
      for (int m = 4; m >= 1; m >>= 1) part = part + __shfl_xor_sync(FULLM, part, m);
      const float st = cl >= 0 ? part - hh[cl] : -__int_as_float(0x7f800000);
      float m2 = st;
      m2 = fmaxf(m2, __shfl_xor_sync(FULLM, m2, 8));
      m2 = fmaxf(m2, __shfl_xor_sync(FULLM, m2, 16));
      const float thr2 = m2 - 3.0517578125e-5f * (a.vn * head_cn[2 * bh] + head_cn[2 * bh + 1]);
      const bool keep = g == 0 && cl >= 0 && st >= thr2;
      uint64_t c2 = 0;
      const uint32_t kb = __ballot_sync(FULLM, keep);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        if ((kb >> (8 * qq)) & 1u) c2 |= 1ull << __shfl_sync(FULLM, cl, 8 * qq);
      cand = c2;
    }
    int best = __ffsll(static_cast<long long>(cand)) - 1;
    if (cand & (cand - 1)) {
      // exact chains: lane l takes the l-th, (l+32)-th, ... candidate
      float bs = -__int_as_float(0x7f800000);
      int bc = 64;
      uint64_t rest = cand;
      while (rest) {
        uint64_t mine = rest;
        for (int x = 0; x < lane && mine; ++x) mine &= mine - 1;
        if (mine) {
          const int c = __ffsll(static_cast<long long>(mine)) - 1;
          const float* crow = cb + c * D;
          float acc = 0.0f;
#pragma unroll 4
          for (int ch = 0; ch < 16; ++ch) {  // d = 8 ch .. 8 ch + 7, in order
            const uint4 u = *reinterpret_cast<const uint4*>(vrow + 8 * ch);
            const float4 c0 = *reinterpret_cast<const float4*>(crow + 8 * ch);
            const float4 c1 = *reinterpret_cast<const float4*>(crow + 8 * ch + 4);
            acc = __fmaf_rn(__uint_as_float(u.x << 16), c0.x, acc);
            acc = __fmaf_rn(__uint_as_float(u.x & 0xFFFF0000u), c0.y, acc);
            acc = __fmaf_rn(__uint_as_float(u.y << 16), c0.z, acc);
            acc = __fmaf_rn(__uint_as_float(u.y & 0xFFFF0000u), c0.w, acc);
            acc = __fmaf_rn(__uint_as_float(u.z << 16), c1.x, acc);
            acc = __fmaf_rn(__uint_as_float(u.z & 0xFFFF0000u), c1.y, acc);
            acc = __fmaf_rn(__uint_as_float(u.w << 16), c1.z, acc);
            acc = __fmaf_rn(__uint_as_float(u.w & 0xFFFF0000u), c1.w, acc);
          }
          const float e = acc - hh[c];
          if (e > bs || (e == bs && c < bc)) {
            bs = e;
            bc = c;
          }
        }
        for (int x = 0; x < 32 && rest; ++x) rest &= rest - 1;
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const float os = __shfl_xor_sync(FULLM, bs, m);
        const int oc = __shfl_xor_sync(FULLM, bc, m);
        if (os > bs || (os == bs && oc < bc)) {
          bs = os;
          bc = oc;
        }
      }
      // (bc = 64 only if every score is NaN: the first candidate then)
      best = bc < 64 ? bc : best;
    }
    if (lane == 0) labels[a.tok] = best;
  }
}

// The driver's tensor-map encoder (looked up once; a function-local static is
// initialised thread-safely).
PFN_cuTensorMapEncodeTiled_v12000 km_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace

// V as a 4-D tensor map (channels, tokens, heads, batches; strides from the
// row layout) with 64 x 128 boxes, 128B swizzle.
cudaError_t launch_km_assign_tc(const uint16_t* V, const RowLayout& lv, int64_t BH, int64_t N, int k,
                                const float* cent,
                                int32_t* labels, const GroupWs& ws, int iter, uint32_t* err,
                                cudaStream_t s, float* tdump) {
  if (k < 1 || k > 64) return cudaErrorInvalidValue;
  auto enc = km_encoder();
  if (!enc) return cudaErrorInvalidValue;
  CUtensorMap m;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(lv.H), static_cast<cuuint64_t>(BH / lv.H)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(lv.sn) * 2, static_cast<cuuint64_t>(lv.sh) * 2,
                                 static_cast<cuuint64_t>(lv.sb) * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(V), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // per device: the kernel's shared-memory limit and the SM count (two CTA
  // slots per SM)
  static PerDevice setup;
  int dev = 0;
  const cudaError_t est = per_device_setup(setup, &dev, [](int d, int* slots_out) {
    cudaError_t e = cudaFuncSetAttribute(km_assign_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, KT_SMEM);
    int sms = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    if (e == cudaSuccess) *slots_out = 2 * (sms > 0 ? sms : 1);
    return e;
  });
  if (est != cudaSuccess) return est;
  // Tiles per CTA (all of one head): the count that minimises the waves of
  // two CTAs per SM times the tiles of a CTA plus its set-up (about six
  // tiles' worth: the centroid operands and the h_c chains).
  const int slots = setup.value[dev];
  const int64_t ntile = (N + 127) / 128;
  int64_t tpc = 1, best_cost = -1;
  for (int64_t c = 1; c <= ntile; ++c) {
    const int64_t waves = ceil_div(BH * ceil_div(ntile, c), slots);
    const int64_t cost = waves * (c + 6);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      tpc = c;
    }
  }
  const dim3 grid(static_cast<unsigned>((ntile + tpc - 1) / tpc), static_cast<unsigned>(BH));
  // The open-assignment counter of this iteration starts at 0 (cleared
  // before the first iteration, then by the previous fix-up).
  uint32_t* cnt = ws.amb_count + (iter & 1);
  km_assign_tc<<<grid, KT_THREADS, KT_SMEM, s>>>(m, N, lv.H, k, static_cast<int>(tpc), cent, labels, ws.amb, cnt,
                                                 ws.head_cn, ws.head_h, ws.vnorm, iter > 0 ? 1 : 0, err, tdump);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  km_fixup<<<static_cast<unsigned>(slots * 2), 256, 0, s>>>(V, lv, N, k, cent, labels, ws.amb, cnt,
                                                            ws.amb_count + ((iter + 1) & 1), ws.head_cn,
                                                            ws.head_h);
  return cudaGetLastError();
}

}  // namespace vc
