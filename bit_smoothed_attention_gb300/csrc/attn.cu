// FP8 attention forward with ExpCast-FP8 and the V-Smooth rank-one mean
// restoration, on tcgen05 tensor cores (sm_103a).
//
// Method ("VC-Attention: Value Smoothing and Softmax Casting for Low-bit
// Attention", Key Contributions 1-2 and Methodology; block-sparse mask,
// partial tiles, empty selections and log2-LSE from "[perf] Add opt-in SM120
// sparse attention forward kernel for MiniMax-H3", Changes):
//   S = Q8 K8^T (E4M3 x E4M3 -> FP32 in TMEM);
//   the softmax warps turn S into E4M3 probability bytes with ExpCast
//   (byte = rint(fmaf(x, A, C - m)), bytes below 8 flush to 0) on the FMA
//   pipe: no exp2, no conversion instruction;
//   the bytes P8 go to shared memory and feed, as the A operand,
//   [O | l] += P8 [R8 ; 1_b0 ; 1_b1] (E4M3, N = 144): the 128 output
//   channels plus the per-64-key-block row sums of the decoded bytes, from
//   the same MMA;
//   the block means are restored in the same accumulator as
//   sum_b l_b mu_b / v_scale by one tf32 MMA whose A operand is the row sums
//   split into tf32 high and low parts and whose B operand is the prepared
//   mean tile.
//
// Dense kernel (attn_fwd).  CTA = 256 query rows (two 128-row slots) of one
// (b, h).  Warps 0 and 1 issue the MMAs of slot 0 and slot 1 from one lane
// each (warp 0 also allocates TMEM), warp 2 issues the TMA loads (warp 3 is
// idle), warps 4-7 run
// the softmax of slot 0 (thread = row = TMEM lane quarter warp & 3) and warps
// 8-11 that of slot 1.  The issuing warps have the lowest warp numbers so that
// the warp schedulers favour them over the softmax warps sharing their
// sub-partitions: the kernel's critical path runs through the MMA lanes.
// TMEM columns: S [0,128) shared by the slots, O0 [192,336), O1 [352,496);
// columns 128 and 129 of O_s hold the tile's row sums, which the softmax
// reads and clears after each PV.  P of each slot is a 128B-swizzled tile in
// shared memory (an A operand read from shared memory issues faster than one
// read from TMEM).  K tiles and V/mean tiles come through separate rings of
// NS stages: a K stage is released once both slots' QK have read it, a V
// stage only after both mean terms of its tile.
//
// S is a single TMEM buffer that the two slots take in turn (S0(t), S1(t),
// S0(t+1), ...).  Per KV tile t the two MMA lanes (slot 0's, slot 1's) issue
//   QK_0(t+1) | MEAN_0(t-1) PV_0(t) | QK_1(t+1) | MEAN_1(t-1) PV_1(t)
// each QK as soon as the other slot holds its S in registers, so the next S
// is computed while the softmax of the current one runs, and the softmax of
// slot s does
//   wait S(t), load it, release S -> max -> ExpCast -> wait PV(t-1) ->
//   P(t) to shared memory, read and clear the row sums of t-1, (rare) rescale O,
//   write the mean operand of t-1 -> release P(t) and the mean operand.
// The row sums of tile t-1 are read one tile late, so no softmax waits for
// its own PV; when the running maximum moves at tile t, O (which then holds
// PV up to t-1 and the mean terms up to t-2) is rescaled in place and the
// mean operand of t-1 is written already multiplied by the factor.
// tcgen05 operations of one thread complete in issue order, so "PV(t-1)
// done" implies that MEAN(t-2) is done.
//
// A KV tile is two 64-key blocks, one per 64-column half of S and P: tile t
// holds blocks 2t and 2t+1 (one 128-row TMA box of K and of V) for both
// slots, through one ring of NS stages.  With a tile mask the block-sparse
// kernel (attn_sparse, below) runs instead.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace vc {
namespace {

constexpr int NS = 4;          // K/V/mean pipeline stages
constexpr int NTHREADS = 384;  // one MMA warp per slot, one TMA warp, one idle, 8 softmax warps
constexpr int WARP_MMA = 0;    // + slot
constexpr int WARP_TMA = 2;
constexpr int WARP_SOFTMAX = 4;
constexpr int CTA_ROWS = 256;

// TMEM columns
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_O = 192;    // + 160 * slot; 144 columns each
constexpr uint32_t COL_L = 128;    // row sums inside O_s

constexpr uint32_t TILE_BYTES = 16384;    // 128 x 128 E4M3
constexpr uint32_t V_STAGE = 18432;       // V tile + 16 indicator rows
constexpr uint32_t MU_BYTES = 4096;       // 128 x 8 tf32
constexpr uint32_t SM_Q = 0;
constexpr uint32_t SM_K = SM_Q + 2 * TILE_BYTES;
constexpr uint32_t SM_V = SM_K + NS * TILE_BYTES;
constexpr uint32_t SM_MU = SM_V + NS * V_STAGE;
constexpr uint32_t SM_L = SM_MU + NS * MU_BYTES;
constexpr uint32_t SM_P = SM_L + 2 * MU_BYTES;  // P of each slot, A operand of the PV MMA
constexpr uint32_t SM_BAR = SM_P + 2 * TILE_BYTES;
enum {
  B_QFULL = 0,  // both Q tiles and K(0)
  B_FULL = 1,   // V(j) and its mean tile in stage j's, plus K(j+1)
  B_KEMPTY = B_FULL + NS,
  B_VEMPTY = B_KEMPTY + NS,
  B_SFULL = B_VEMPTY + NS,
  B_STAKEN = B_SFULL + 2,
  B_PFULL = B_STAKEN + 2,  // P(j) and the mean operand of tile j-1
  B_ODONE = B_PFULL + 2,
  B_MDONE = B_ODONE + 2,
  B_FIN = B_MDONE + 2,
  NBAR = B_FIN + 2
};
constexpr uint32_t SM_TSLOT = SM_BAR + NBAR * 8;
constexpr uint32_t SM_ABORT = SM_TSLOT + 8;
constexpr uint32_t SM_END = SM_ABORT + 8;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
// Block-sparse kernel: per query 64-tile of the CTA, one bit per 64-key
// block, set when the tile keeps it (the first 32 * KEPT_WORDS blocks; later
// ones are looked up in the mask itself).
constexpr int KEPT_WORDS = 112;  // per query tile

constexpr uint32_t IDESC_QK = idesc(FMT_E4M3, FMT_E4M3, 128, 128);
constexpr uint32_t IDESC_PV = idesc(FMT_E4M3, FMT_E4M3, 128, 144);
constexpr uint32_t IDESC_TF32 = idesc(FMT_TF32, FMT_TF32, 128, 128);
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s per wait

struct Params {
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const float* qmu;
  const float* vmu_op;
  const uint8_t* mask;
  void* O;
  RowLayout lo;  // rows of O, in elements of O's type
  float* lse2;
  int64_t N;
  int out_f32;
  int npad, nbp, ntile, nq64;
  float c0;          // fl(8 log2(e) sm_scale)
  float C;           // fl(56 + 8 off - 8 c*)
  float lse_qmu;     // sm_scale * log2(e)
  float tau8;
  float off;
  uint32_t* err;
  int debug_flags;
};

// Does query 64-tile qt keep 64-key block b?
__device__ __forceinline__ bool block_kept(const Params& p, int64_t bh, int qt, int b) {
  return qt < p.nq64 && p.mask[(bh * p.nq64 + qt) * p.nbp + b] != 0;
}

// The first block at or after u that query tile qt keeps, read from the mask
// itself (blocks beyond the shared-memory bitmask; out of line, it is never
// hot), or -1.
__device__ __noinline__ int next_kept_slow(const Params& p, int64_t bh, int qt, int u) {
  for (; u < p.nbp; ++u)
    if (block_kept(p, bh, qt, u)) return u;
  return -1;
}

__device__ __forceinline__ void record_timeout(const Params& p, volatile int* abort) {
  *abort = 1;
  atomicOr(p.err, ERR_TIMEOUT);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float set_ge(float a, float b) {
  float d;
  asm("set.ge.f32.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// ExpCast of four scores sharing A' = A/256 and B' = (C - m)/256, packed into
// one little-endian word of E4M3 bytes:
//   t' = fma(x, A', B')              = t/256 exactly, t = fmaf(x, A, C - m);
//   u  = sat(t' 2^29 + 1 - 7.5 2^21) = 1 iff t >= 7.5 (iff rint(t) >= 8),
//        else 0 (t' 2^29 is an integer whenever t is near 7.5); for the
//        odd scores the same u comes from set.ge(t', 7.5/256), a compare on
//        the ALU pipe, so that the FMA and ALU pipes carry about the same
//        work per four scores (10 issue cycles each);
//   f  = fma(t', u, 49152)           = 49152 + rint(t)/256 (ulp 2^-8, ties
//        to even) or 49152 when u = 0, so the low byte of f's bits is the
//        code.
// The clip at 126 never binds: t <= C + tau8 <= 125.66 by construction.
__device__ __forceinline__ uint32_t expcast4(float x0, float x1, float x2, float x3, float A,
                                             float B) {
  constexpr float S29 = 536870912.0f;  // 2^29
  constexpr float K29 = -15728639.0f;  // 1 - 7.5 * 2^21
  const float2 A2 = make_float2(A, A), B2 = make_float2(B, B);
  const float2 t01 = __ffma2_rn(make_float2(x0, x1), A2, B2);
  const float2 t23 = __ffma2_rn(make_float2(x2, x3), A2, B2);
  constexpr float T75 = 0.029296875f;  // 7.5 / 256
  const float2 u01 = make_float2(fma_sat(t01.x, S29, K29), set_ge(t01.y, T75));
  const float2 u23 = make_float2(fma_sat(t23.x, S29, K29), set_ge(t23.y, T75));
  const float2 M = make_float2(49152.0f, 49152.0f);
  const float2 f01 = __ffma2_rn(t01, u01, M);
  const float2 f23 = __ffma2_rn(t23, u23, M);
  return prmt(prmt(__float_as_uint(f01.x), __float_as_uint(f01.y), 0x0040u),
              prmt(__float_as_uint(f23.x), __float_as_uint(f23.y), 0x0040u), 0x5410u);
}

// Test hook for the byte-level check of ExpCast: the bytes the attention
// kernel writes for scores x with ExpCast coefficients A (per tile half) and
// B = C - m (per tile), through the same expcast4 and the same treatment of
// a key the kernel excludes (score -inf: cast as 0, byte cleared).  Thread g
// casts the four scores x[4g..4g+3], which share A[g] and B[g].
__global__ void expcast_probe(const float4* __restrict__ x, const float* __restrict__ A,
                              const float* __restrict__ B, uint32_t* __restrict__ out, int64_t ngroups) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= ngroups) return;
  const float4 v = x[g];
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float e[4] = {v.x, v.y, v.z, v.w};
  float f[4];
  uint32_t keep = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[i] = e[i] == NEG_INF ? 0.0f : e[i];
    if (e[i] != NEG_INF) keep |= 0xFFu << (8 * i);
  }
  out[g] = expcast4(f[0], f[1], f[2], f[3], A[g] * 0.00390625f, B[g] * 0.00390625f) & keep;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
             const __grid_constant__ CUtensorMap tmv, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, derived from the shared array itself so that the
  // compiler keeps every access through it in the shared state space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * static_cast<uint32_t>(i); };
  volatile int* abort = reinterpret_cast<volatile int*>(sm + SM_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = blockIdx.y;
  const int q0 = blockIdx.x * CTA_ROWS;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      // both slots' MMA lanes release a stage
      mbar_init(bar(B_KEMPTY + s), 2);
      mbar_init(bar(B_VEMPTY + s), 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_STAKEN + s), 4);
      mbar_init(bar(B_PFULL + s), 4);
      mbar_init(bar(B_ODONE + s), 1);
      mbar_init(bar(B_MDONE + s), 1);
    }
    mbar_init(bar(B_FIN + 0), 1);
    mbar_init(bar(B_FIN + 1), 1);
    *abort = 0;
    mbar_fence_init();
  }
  // Indicator rows 128..143 of every V stage (B operand rows of the PV MMA,
  // K-major, 128B-swizzled): row 128 = 1.0 on keys 0..63, row 129 = 1.0 on
  // keys 64..127, rows 130..143 = 0.  TMA writes only rows 0..127.
  const uint32_t one4 = 0x38383838u;  // four E4M3 1.0 bytes
  for (int c = threadIdx.x; c < NS * 16 * 8; c += NTHREADS) {
    const int st = c >> 7, n = (c >> 3) & 15, k = c & 7;  // stage, row, 16-key chunk
    const uint32_t v = ((n == 0 && k < 4) || (n == 1 && k >= 4)) ? one4 : 0u;
    *reinterpret_cast<uint4*>(sm + SM_V + st * V_STAGE + TILE_BYTES + n * 128 + ((k ^ (n & 7)) * 16)) =
        make_uint4(v, v, v, v);
  }
  fence_proxy_async_smem();
  if (warp == WARP_MMA) tmem_alloc(sb + SM_TSLOT, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + SM_TSLOT);

  // KV tile t = blocks (2t, 2t + 1), for both slots and all their rows;
  // x = -1 past the last tile.
  const int ntiles = p.ntile;
  auto tile_of = [&](int t) { return t < ntiles ? make_int2(2 * t, 2 * t + 1) : make_int2(-1, -1); };

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    // Warp 2 loads both Q tiles and the K/V ring that both slots share.
    if (lane == 0 && !(p.debug_flags & 1) && ntiles > 0) {
      const int h3 = static_cast<int>(bh);
      const float* mu = p.vmu_op + bh * p.nbp * (4 * D);  // 2 KiB per block
      // K of a tile: one 128-row box
      auto load_k = [&](uint32_t dst, int2 pr, uint32_t b) { tma_load_3d(dst, &tmk, 0, pr.x * BLK, h3, b); };
      // V and the mean tile (blocks 2t and 2t+1 are adjacent) of a tile
      auto load_v = [&](int st, int2 pr, uint32_t b) {
        const uint32_t dv = sb + SM_V + st * V_STAGE, dm = sb + SM_MU + st * MU_BYTES;
        tma_load_3d(dv, &tmv, pr.x * BLK, 0, h3, b);
        bulk_load(dm, mu + pr.x * (4 * D), MU_BYTES, b);
      };
      // Q and the first K tile
      int2 pr = tile_of(0);
      const uint32_t qb = bar(B_QFULL);
      mbar_arrive_expect_tx(qb, 3 * TILE_BYTES);
      tma_load_3d(sb + SM_Q, &tmq, 0, q0, h3, qb);
      tma_load_3d(sb + SM_Q + TILE_BYTES, &tmq, 0, q0 + 128, h3, qb);
      load_k(sb + SM_K, pr, qb);
      // Test hook: with debug_flags >> 8 = n > 0 the producer stops after n
      // steps, as if its loads had stalled mid-stream.
      const int stop_after = p.debug_flags >> 8;
      // the last step that armed each stage (-1: none)
      int armed[NS];
#pragma unroll
      for (int u = 0; u < NS; ++u) armed[u] = -1;
      // Step j brings V(j) and its mean tile into stage j % NS and K(j+1)
      // into K stage (j+1) % NS, all on one barrier.  A K stage is free again
      // once both slots' QKs that read it were done, a V stage once both
      // slots' mean terms of its tile were issued.
      for (int j = 0; pr.x >= 0 && !*abort && !(stop_after > 0 && j >= stop_after); ++j) {
        const int st = j % NS, stk = (j + 1) % NS;
        const int2 pn = tile_of(j + 1);
        if (j >= NS && !mbar_wait(bar(B_VEMPTY + st), ((j / NS) - 1) & 1, abort, WAIT_NS)) {
          record_timeout(p, abort);
          break;
        }
        if (pn.x >= 0 && j + 1 >= NS &&
            !mbar_wait(bar(B_KEMPTY + stk), (((j + 1) / NS) - 1) & 1, abort, WAIT_NS)) {
          record_timeout(p, abort);
          break;
        }
        mbar_arrive_expect_tx(bar(B_FULL + st), TILE_BYTES + MU_BYTES + (pn.x >= 0 ? TILE_BYTES : 0));
        load_v(st, pr, bar(B_FULL + st));
        if (pn.x >= 0) load_k(sb + SM_K + stk * TILE_BYTES, pn, bar(B_FULL + st));
        armed[j % NS] = j;
        pr = pn;
      }
      // Drain: every copy this producer issued has landed before the CTA can
      // exit, also when a consumer gave up and never waited for it.  A stage
      // is re-armed only after its previous fill was consumed, so waiting
      // for the parity of its last fill is enough (time-bounded, ignoring
      // the abort flag).
      bool drained = mbar_wait_time(qb, 0, WAIT_NS);
#pragma unroll
      for (int u = 0; u < NS; ++u)
        if (armed[u] >= 0) drained &= mbar_wait_time(bar(B_FULL + u), (armed[u] / NS) & 1, WAIT_NS);
      if (!drained) record_timeout(p, abort);
    }
  } else if (warp == WARP_MMA || warp == WARP_MMA + 1) {
    // ----------------------------------------------------------- MMA issue
    // One issuing lane per slot, so that one slot's waits never hold back
    // the other slot's MMAs; tcgen05.commit tracks each lane's own MMAs.
    const int s = warp - WARP_MMA;
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(bar(B_QFULL), 0, abort, WAIT_NS);
      tc_fence_after();
      // Descriptors are built once; a byte offset o advances them by o >> 4
      // in the start-address field (all of shared memory is below 256 KiB).
      const uint64_t dQ = sdesc_sw128(sb + SM_Q + s * TILE_BYTES), dK = sdesc_sw128(sb + SM_K);
      const uint64_t dV = sdesc_sw128(sb + SM_V);
      const uint64_t dL = sdesc_k8_tf32(sb + SM_L + s * MU_BYTES);
      // mean tile: K-slots 0..3 (block of the first half) and 4..7 (second
      // half) are two 2 KiB parts of 16-byte rows, one row per channel
      const uint64_t dMu = sdesc(sb + SM_MU, MU_BYTES / 2, 128, 0);
      const uint64_t dP = sdesc_sw128(sb + SM_P + s * TILE_BYTES);
      const uint32_t dO = tmem + COL_O + 160 * s;
      auto adv = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      auto wt = [&](int b, uint32_t par) {
        if (!ok) return;
        ok = mbar_wait(bar(b), par, abort, WAIT_NS);
        tc_fence_after();
      };
      auto stg = [](int j) { return j % NS; };
      // S of this slot for its j-th tile
      auto qk = [&](int j) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8(tmem + COL_S, adv(dQ, 32 * kk), adv(dK, stg(j) * TILE_BYTES + 32 * kk), IDESC_QK, kk > 0);
        mma_commit(bar(B_SFULL + s));
        mma_commit(bar(B_KEMPTY + stg(j)));  // this slot has read K(j)
      };
      // The single S buffer is taken in turn: S0(0) S1(0) S0(1) S1(1) ...
      // QK of slot 0 for tile i waits until slot 1 holds S(i-1); QK of slot 1
      // until slot 0 holds S(i).  Each QK goes ahead of the PV that the same
      // slot's softmax releases later.
      auto pv = [&](int j) {  // mean term of tile j-1, then [O | l] += P(j) [V ; 1_b0 ; 1_b1]
        wt(B_PFULL + s, j & 1);  // P(j), and for j > 0 the mean operand of j-1
        if (!ok) return;
        if (j > 0) {
          mma_tf32(dO, dL, adv(dMu, stg(j - 1) * MU_BYTES), IDESC_TF32, 1);
          mma_commit(bar(B_VEMPTY + stg(j - 1)));  // this slot is done with V(j-1)
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8(dO, adv(dP, 32 * kk), adv(dV, stg(j) * V_STAGE + 32 * kk), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_ODONE + s));
      };
      for (int i = 0; ok && i <= ntiles; ++i) {
        if (i < ntiles) {
          // K(i) came with Q (i = 0) or with V(i-1)
          if (i > 0) wt(B_FULL + stg(i - 1), ((i - 1) / NS) & 1);
          if (s == 0) {
            if (i > 0) wt(B_STAKEN + 1, (i - 1) & 1);
          } else {
            wt(B_STAKEN + 0, i & 1);
          }
          if (!ok) break;
          qk(i);
        }
        if (i > 0) {
          if (i == ntiles) wt(B_FULL + stg(i - 1), ((i - 1) / NS) & 1);  // V of the last tile
          pv(i - 1);
        }
      }
      // the last tile's mean term (the softmax's extra p_full arrival)
      wt(B_PFULL + s, ntiles & 1);
      if (ok) {
        mma_tf32(dO, dL, adv(dMu, stg(ntiles - 1) * MU_BYTES), IDESC_TF32, 1);
        mma_commit(bar(B_MDONE + s));
      }
      if (!ok) record_timeout(p, abort);
      // Drain: every MMA of this lane has completed before TMEM is released,
      // also after an abort (the wait ignores the abort flag).
      mma_commit(bar(B_FIN + s));
      if (!mbar_wait_time(bar(B_FIN + s), 0, WAIT_NS)) record_timeout(p, abort);
    }
  } else if (warp >= WARP_SOFTMAX) {
    // ------------------------------------------------------ softmax warps
    const int slot = (warp - WARP_SOFTMAX) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int64_t row = static_cast<int64_t>(q0) + slot * 128 + r;
    const bool row_ok = row < p.N;
    const int qt = static_cast<int>(row >> 6);
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + COL_S;
    // row r of this slot's P tile (128B-swizzled K-major, like Q and K)
    uint8_t* Prow = sm + SM_P + slot * TILE_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
    const uint32_t tO = tmem + lane_addr + COL_O + 160 * slot;
    const float qsc = p.q_scale[bh * p.nbp + (qt < p.nbp ? qt : p.nbp - 1)];
    const float a_i = p.c0 * qsc;
    uint8_t* Lrow = sm + SM_L + slot * MU_BYTES + (r >> 3) * 256 + (r & 7) * 16;
    const float* ksc = p.k_scale + bh * p.nbp;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const uint32_t FULL = 0xffffffffu;
    // the row sums of the two 64-key blocks of the previous tile (columns
    // 128, 129 of O_s)
    auto ld_rowsums = [&](float& l0, float& l1) {
      uint32_t ls0, ls1;
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                   : "=r"(ls0), "=r"(ls1)
                   : "r"(tO + COL_L));
      tmem_wait_ld();
      l0 = __uint_as_float(ls0);
      l1 = __uint_as_float(ls1);
    };
    // tf32 A operand row of the mean restoration, [hi0, lo0, hi0, 0 | hi1, lo1, hi1, 0]
    // against the mean tile's (hi, hi, lo, 0) of each half's block
    auto put_lrow = [&](float v0, float v1) {
      const float h0 = to_tf32(v0), h1 = to_tf32(v1);
      const float g0 = to_tf32(v0 - h0), g1 = to_tf32(v1 - h1);
      *reinterpret_cast<float4*>(Lrow) = make_float4(h0, g0, h0, 0.0f);
      *reinterpret_cast<float4*>(Lrow + 128) = make_float4(h1, g1, h1, 0.0f);
    };
    float m_run = NEG_INF;
    float l = 0.0f;
    bool ok = true;
    int i = 0;
    // block scales of a tile
    auto pair_scales = [&](int2 pr) -> float2 {
      return pr.x < 0 ? make_float2(0.0f, 0.0f) : *reinterpret_cast<const float2*>(ksc + pr.x);
    };
    int2 pr = tile_of(0);
    // loaded one tile ahead
    float2 ks = pair_scales(pr);
    for (; pr.x >= 0; ++i) {
      const int2 pn = tile_of(i + 1);
      const float2 ks_n = pair_scales(pn);
      const bool keep0 = row_ok;
      const bool keep1 = row_ok;
      // Score column j of the tile is a valid key iff j < lim_lo (first
      // half) or j < lim_hi (second half); both are N - 128 t.
      const int n32 = static_cast<int>(p.N);
      const int lim_lo = n32 - pr.x * BLK;
      const int lim_hi = pr.y >= 0 ? BLK + n32 - pr.y * BLK : BLK;
      const float A0 = a_i * ks.x;
      const float A1 = a_i * ks.y;
      // Warp-uniform: does the tile hold keys past N (the last block of the
      // sequence, or an empty second half)?  Only then are keys masked one
      // by one; a row past N keeps no block (no max contribution, code 0).
      const bool partial = !__all_sync(FULL, lim_lo >= BLK && lim_hi >= TILE);

      if (!(ok = __all_sync(FULL, mbar_wait(bar(B_SFULL + slot), i & 1, abort, WAIT_NS)))) break;
      tc_fence_after();
      float x[128];
      uint32_t w[32];  // the row's 128 E4M3 bytes
      float m_new, alpha;
      bool resc;
      {
        tmem_ld128(tS, *reinterpret_cast<uint32_t(*)[128]>(&x[0]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_STAKEN + slot));  // S may be overwritten
        if (partial) {
          // keys past N never contribute: -inf for the max
#pragma unroll
          for (int j = 0; j < 128; ++j) x[j] = j < (j < 64 ? lim_lo : lim_hi) ? x[j] : NEG_INF;
        }
        // four independent max chains (two per 64-key half)
        float ma = fmax3(x[0], x[1], x[2]), mb = fmax3(x[32], x[33], x[34]);
        float mc = fmax3(x[64], x[65], x[66]), md = fmax3(x[96], x[97], x[98]);
#pragma unroll
        for (int j = 3; j < 31; j += 2) {
          ma = fmax3(ma, x[j], x[j + 1]);
          mb = fmax3(mb, x[32 + j], x[33 + j]);
          mc = fmax3(mc, x[64 + j], x[65 + j]);
          md = fmax3(md, x[96 + j], x[97 + j]);
        }
        const float mx0 = fmax3(ma, mb, fmaxf(x[31], x[63]));
        const float mx1 = fmax3(mc, md, fmaxf(x[95], x[127]));
        const float m_tile = fmaxf(keep0 ? A0 * mx0 : NEG_INF, keep1 ? A1 * mx1 : NEG_INF);
        const bool need = m_tile > m_run + p.tau8;
        m_new = need ? m_tile : m_run;
        const bool live = m_new != NEG_INF;
        resc = need && m_run != NEG_INF;
        alpha = resc ? exp2f((m_run - m_new) * 0.125f) : 1.0f;

        // ExpCast -> 32 words of E4M3 bytes.  A row past N, and a row with
        // no key kept so far, cast with A = B = 0: t = 0, every code 0 (the
        // scores are finite).  In the partial tile the -inf scores are
        // replaced by 0 and the bytes of keys past N are cleared after the
        // cast.
        if (partial) {
#pragma unroll
          for (int j = 0; j < 128; ++j) x[j] = x[j] == NEG_INF ? 0.0f : x[j];
        }
        const bool k0 = live && keep0, k1 = live && keep1;
        const float Bq = (p.C - m_new) * 0.00390625f;
        const float A0q = k0 ? A0 * 0.00390625f : 0.0f, B0q = k0 ? Bq : 0.0f;
        const float A1q = k1 ? A1 * 0.00390625f : 0.0f, B1q = k1 ? Bq : 0.0f;
#pragma unroll
        for (int q = 0; q < 32; ++q)
          w[q] = expcast4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3], q < 16 ? A0q : A1q,
                          q < 16 ? B0q : B1q);
        if (partial) {
          const int lim0 = k0 ? (lim_lo < 64 ? lim_lo : 64) : 0;
          const int lim1 = k1 ? (lim_hi < 128 ? lim_hi : 128) : 64;
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            uint32_t keep = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * q + e < (q < 16 ? lim0 : lim1)) keep |= 0xFFu << (8 * e);
            w[q] &= keep;
          }
        }
      }
      m_run = m_new;
      if (i > 0) {
        // PV(i-1) done (and with it the mean term of tile i-2): P may be
        // overwritten and the row sums of tile i-1 are final.
        if (!(ok = __all_sync(FULL, mbar_wait(bar(B_ODONE + slot), (i - 1) & 1, abort, WAIT_NS)))) break;
        tc_fence_after();
      }
      // row r of P_s: 128 bytes, 16-byte chunk c at position c ^ (r & 7)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(Prow + ((c ^ (r & 7)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      if (i > 0) {
        // Row sums of tile i-1: read and cleared, so that PV(i) accumulates
        // its own.  If the maximum moved, O (holding PV up to i-1 and the
        // mean terms up to i-2; the mean term of i-1 is issued only after
        // this slot's l_full) and l move to the new maximum, and the mean
        // operand of tile i-1 is written already scaled by alpha.
        float l0, l1;
        ld_rowsums(l0, l1);
        asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(tO + COL_L), "r"(0u),
                     "r"(0u)
                     : "memory");
        if (__any_sync(FULL, resc)) {
          // all 128 accumulator columns in flight at once (x is dead here)
          uint32_t (&o0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[0]);
          uint32_t (&o1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[32]);
          uint32_t (&o2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[64]);
          uint32_t (&o3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[96]);
          tmem_ld32(tO + 0, o0);
          tmem_ld32(tO + 32, o1);
          tmem_ld32(tO + 64, o2);
          tmem_ld32(tO + 96, o3);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 128; ++e) x[e] *= alpha;
          tmem_st32(tO + 0, o0);
          tmem_st32(tO + 32, o1);
          tmem_st32(tO + 64, o2);
          tmem_st32(tO + 96, o3);
        }
        l = (l + (l0 + l1)) * alpha;
        put_lrow(l0 * alpha, l1 * alpha);
      }
      fence_proxy_async_smem();  // P (and the mean operand) to the tensor core
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + slot));
      pr = pn;
      ks = ks_n;
    }
    // the last tile's row sums, then its mean term
    if (ok && ntiles > 0) {
      ok = __all_sync(FULL, mbar_wait(bar(B_ODONE + slot), (ntiles - 1) & 1, abort, WAIT_NS));
      if (ok) {
        tc_fence_after();
        float l0, l1;
        ld_rowsums(l0, l1);
        l += l0 + l1;
        put_lrow(l0, l1);
        fence_proxy_async_smem();  // the mean operand to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + slot));
        ok = __all_sync(FULL, mbar_wait(bar(B_MDONE + slot), 0, abort, WAIT_NS));
        tc_fence_after();
      }
    }
    if (!ok) record_timeout(p, abort);

    // ------------------------------------------------------------ epilogue
    const bool have = ok && ntiles > 0;
    if (__all_sync(0xffffffffu, have)) {
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        if (row_ok) {
          float y[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            y[e] = __uint_as_float(o[e]) * p.v_scale[bh * D + 32 * c + e] * inv_l;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + p.lo.head(bh) + p.lo.row(row) + 32 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.O) + p.lo.head(bh) + p.lo.row(row) + 32 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
    } else if (row_ok && ntiles == 0) {
      const int nvec = p.out_f32 ? 32 : 16;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.O) +
                                            (p.lo.head(bh) + p.lo.row(row)) * (p.out_f32 ? 4 : 2));
      for (int e = 0; e < nvec; ++e) dst[e] = make_uint4(0, 0, 0, 0);
    }
    if (row_ok && p.lse2) {
      p.lse2[bh * p.N + row] = l > 0.0f
          ? m_run * 0.125f - p.off + log2f(l) + p.qmu[bh * p.N + row] * p.lse_qmu
          : -__int_as_float(0x7f800000);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == WARP_MMA) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- block-sparse
// With a tile mask: one 128-row slot per CTA, its two query 64-tiles A (rows
// 0-63) and B (rows 64-127) each walking their own KV steps (the blocks they
// keep, two per step, in ascending order).  Step t of the slot is A's step t
// and B's step t at once, as one block-diagonal 256-key step:
//   S = Q8 [K_a0; K_a1; K_b0; K_b1]^T (N = 256): A's rows read columns
//       0-127 (their own two blocks), B's rows columns 128-255;
//   [O | l] += [P_A 0; 0 P_B] [R8_a0; R8_a1; R8_b0; R8_b1 | indicators]
//       (K = 256, N = 144): P's off-diagonal quadrants stay zero, so each
//       row accumulates only its own blocks, and the indicator rows give the
//       row sums of the four blocks (A's in columns 128-129 of O, B's in
//       130-131);
//   two tf32 mean MMAs restore A's and B's block means.
// Once one tile has no steps left, the other goes on alone: the finished
// tile's blocks are replaced by a block of the step that is present (finite
// bytes) and its rows cast nothing.  An odd last step has an empty second
// block, filled the same way.  Each row's arithmetic is that of its own
// query tile's steps, done as in the dense kernel; the tensor cores do no
// work for another tile's rows beyond the zero quadrants of P.
//
// Warp 0 issues the QKs from one lane and allocates TMEM (512 columns: S
// [0,256), O [256,400)), warp 2 issues the mean and PV MMAs from one lane,
// warp 1 issues the TMA loads through three rings (K and V of two stages,
// the mean tiles of three, each with barriers of its own), and warps 4-11
// run the softmax, two threads per row (TMEM lane): warps 4-7 take the first
// block of each row's step, warps 8-11 the second.  The single S buffer is
// taken by the next QK as soon as the softmax holds S in registers.
namespace sp {
constexpr int NTHREADS = 384;
constexpr int WARP_MMA = 0, WARP_TMA = 1, WARP_PV = 2, WARP_SOFTMAX = 4;
constexpr int NS = 2;   // K and V stages
constexpr int NM = 3;   // mean-tile stages
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_O = 256;
constexpr uint32_t KBOX = 8192;              // 64 keys x 128 channels, 128B swizzle
constexpr uint32_t K_STAGE = 4 * KBOX;
constexpr uint32_t V_HALF = 9216;            // 144 x 64 keys, 64B swizzle (rows 128-143: indicators)
constexpr uint32_t V_STAGE = 4 * V_HALF;
constexpr uint32_t MU_HALF = 2048;           // mean operand of one block
constexpr uint32_t MU_STAGE = 4 * MU_HALF;
constexpr uint32_t L_BYTES = 4096;           // tf32 A operand of one mean MMA
constexpr uint32_t SM_Q = 0;
constexpr uint32_t SM_K = SM_Q + TILE_BYTES;
constexpr uint32_t SM_V = SM_K + NS * K_STAGE;
constexpr uint32_t SM_MU = SM_V + NS * V_STAGE;
constexpr uint32_t SM_L = SM_MU + NM * MU_STAGE;
constexpr uint32_t SM_P = SM_L + 2 * L_BYTES;      // P tile 0 (keys of A), P tile 1 (keys of B)
constexpr uint32_t SM_KEPT = SM_P + 2 * TILE_BYTES;
constexpr uint32_t SM_XCH = SM_KEPT + 2 * 4 * KEPT_WORDS;  // softmax exchange, [2][2][128] floats
constexpr uint32_t SM_BAR = SM_XCH + 2 * 2 * 128 * 4;
enum {
  B_QFULL = 0,
  B_KFULL,
  B_KEMPTY = B_KFULL + NS,
  B_VFULL = B_KEMPTY + NS,
  B_VEMPTY = B_VFULL + NS,
  B_MFULL = B_VEMPTY + NS,
  B_MEMPTY = B_MFULL + NM,
  B_SFULL = B_MEMPTY + NM,
  B_STAKEN,
  B_PFULL,
  B_ODONE,
  B_MDONE,
  B_FIN,
  B_XCH,  // + 2 * quarter + step parity
  NBAR = B_XCH + 8
};
constexpr uint32_t SM_TSLOT = SM_BAR + NBAR * 8;
constexpr uint32_t SM_ABORT = SM_TSLOT + 8;
constexpr uint32_t SMEM_BYTES = SM_ABORT + 8 + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(SM_K % 1024 == 0 && SM_V % 1024 == 0 && SM_P % 1024 == 0, "swizzle atoms");
constexpr uint32_t IDESC_QK = idesc(FMT_E4M3, FMT_E4M3, 128, 256);

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_sparse(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int i) { return sb + SM_BAR + 8u * static_cast<uint32_t>(i); };
  volatile int* abort = reinterpret_cast<volatile int*>(sm + SM_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = blockIdx.y;
  const int q0 = blockIdx.x * TILE;
  const int qt0 = q0 / BLK;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < NM; ++s) {
      mbar_init(bar(B_MFULL + s), 1);
      mbar_init(bar(B_MEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_STAKEN), 8);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_MDONE), 1);
    mbar_init(bar(B_FIN), 2);  // both issuing lanes
    for (int q = 0; q < 8; ++q) mbar_init(bar(B_XCH + q), 2);  // the two warps of a row quarter
    *abort = 0;
    mbar_fence_init();
  }
  // Indicator rows 128..143 of each 64-key quarter of a V stage: row 128 + h
  // is 1.0 on quarter h's keys (64B swizzle; the rows are uniform, so the
  // swizzle does not move them).
  const uint32_t one4 = 0x38383838u;  // four E4M3 1.0 bytes
  for (int c = threadIdx.x; c < NS * 4 * 16 * 4; c += NTHREADS) {
    const int st = c >> 8, h = (c >> 6) & 3, n = (c >> 2) & 15, k = c & 3;  // stage, quarter, row, chunk
    const uint32_t v = n == h ? one4 : 0u;
    *reinterpret_cast<uint4*>(sm + SM_V + st * V_STAGE + h * V_HALF + 8192 + n * 64 + k * 16) =
        make_uint4(v, v, v, v);
  }
  // The off-diagonal quadrants of P (rows 64-127 of P tile 0, rows 0-63 of
  // P tile 1) and of the mean operand (B's rows of A's, A's rows of B's)
  // stay zero: each row writes only its own tile's part.
  for (int c = threadIdx.x; c < 2 * 512; c += NTHREADS) {  // 16-byte chunks: 2 x 8 KB
    const int t = c >> 9, o = (c & 511) << 4;
    *reinterpret_cast<uint4*>(sm + SM_P + t * TILE_BYTES + (t ? 0 : 8192) + o) = make_uint4(0, 0, 0, 0);
  }
  for (int c = threadIdx.x; c < 2 * 128; c += NTHREADS) {  // 16-byte chunks: 2 x 2 KB
    const int t = c >> 7, o = (c & 127) << 4;
    *reinterpret_cast<uint4*>(sm + SM_L + t * L_BYTES + (t ? 0 : 2048) + o) = make_uint4(0, 0, 0, 0);
  }
  // per query tile of the CTA (two), the bitmask of the blocks it keeps
  uint32_t* kept_w = reinterpret_cast<uint32_t*>(sm + SM_KEPT);
  const int nkw = (p.nbp + 31) >> 5;
  for (int w = warp; w < nkw && w < KEPT_WORDS; w += NTHREADS / 32) {
    const int b = 32 * w + lane;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t m = __ballot_sync(0xffffffffu, b < p.nbp && block_kept(p, bh, qt0 + q, b));
      if (lane == 0) kept_w[q * KEPT_WORDS + w] = m;
    }
  }
  fence_proxy_async_smem();
  if (warp == WARP_MMA) tmem_alloc(sb + SM_TSLOT, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + SM_TSLOT);

  // Each query tile's steps, the same in every role.
  const int kept_lim = p.nbp < 32 * KEPT_WORDS ? p.nbp : 32 * KEPT_WORDS;
  auto next_kept = [&](int q, int b) {  // the next block after b that query tile qt0 + q keeps
    const uint32_t* kw = kept_w + q * KEPT_WORDS;
    int u = b + 1;
    for (; u < kept_lim; u = (u | 31) + 1) {  // bits past nbp are 0
      const uint32_t m = kw[u >> 5] >> (u & 31);
      if (m) return u + __ffs(static_cast<int>(m)) - 1;
    }
    return u < p.nbp ? next_kept_slow(p, bh, qt0 + q, u) : -1;
  };
  auto pair_after = [&](int q, int b) -> int2 {  // the step of query tile q that starts after block b
    const int x = next_kept(q, b);
    return make_int2(x, x >= 0 ? next_kept(q, x) : -1);
  };
  auto next_pair = [&](int q, int2 pr) { return pr.y < 0 ? make_int2(-1, -1) : pair_after(q, pr.y); };
  int nst = 0;  // steps of the slot: the larger of the two tiles' counts
  {
    int nb[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      nb[q] = 0;
      for (int w = 0; w < nkw && w < KEPT_WORDS; ++w) nb[q] += __popc(kept_w[q * KEPT_WORDS + w]);
      for (int u = 32 * KEPT_WORDS; u >= 0 && (u = next_kept_slow(p, bh, qt0 + q, u)) >= 0; ++u) ++nb[q];
    }
    nst = max((nb[0] + 1) >> 1, (nb[1] + 1) >> 1);
  }

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !(p.debug_flags & 1) && nst > 0) {
      const int h3 = static_cast<int>(bh);
      const float* mu = p.vmu_op + bh * p.nbp * (4 * D);  // 2 KiB per block
      // the four blocks of a step (A's two, B's two); an absent one is
      // replaced by a present block of the step, so every byte is finite
      auto quad = [](int2 pa, int2 pb) {
        const int f = pa.x >= 0 ? pa.x : pb.x;
        const int a0 = pa.x >= 0 ? pa.x : f, b0 = pb.x >= 0 ? pb.x : f;
        return make_int4(a0, pa.y >= 0 ? pa.y : a0, b0, pb.y >= 0 ? pb.y : b0);
      };
      auto load_k = [&](int st, int4 q4, uint32_t b) {
        const uint32_t dk = sb + SM_K + st * K_STAGE;
        tma_load_3d(dk, &tmk, 0, q4.x * BLK, h3, b);
        tma_load_3d(dk + KBOX, &tmk, 0, q4.y * BLK, h3, b);
        tma_load_3d(dk + 2 * KBOX, &tmk, 0, q4.z * BLK, h3, b);
        tma_load_3d(dk + 3 * KBOX, &tmk, 0, q4.w * BLK, h3, b);
      };
      auto load_v = [&](int st, int4 q4, uint32_t b) {
        const uint32_t dv = sb + SM_V + st * V_STAGE;
        tma_load_3d(dv, &tmv, q4.x * BLK, 0, h3, b);
        tma_load_3d(dv + V_HALF, &tmv, q4.y * BLK, 0, h3, b);
        tma_load_3d(dv + 2 * V_HALF, &tmv, q4.z * BLK, 0, h3, b);
        tma_load_3d(dv + 3 * V_HALF, &tmv, q4.w * BLK, 0, h3, b);
      };
      auto load_mu = [&](int st, int4 q4, uint32_t b) {
        const uint32_t dm = sb + SM_MU + st * MU_STAGE;
        bulk_load(dm, mu + q4.x * (4 * D), MU_HALF, b);
        bulk_load(dm + MU_HALF, mu + q4.y * (4 * D), MU_HALF, b);
        bulk_load(dm + 2 * MU_HALF, mu + q4.z * (4 * D), MU_HALF, b);
        bulk_load(dm + 3 * MU_HALF, mu + q4.w * (4 * D), MU_HALF, b);
      };
      int2 pa = pair_after(0, -1), pb = pair_after(1, -1);
      const uint32_t qb = bar(B_QFULL);
      mbar_arrive_expect_tx(qb, TILE_BYTES);
      tma_load_3d(sb + SM_Q, &tmq, 0, q0, h3, qb);
      // Test hook: with debug_flags >> 8 = n > 0 the producer stops after n
      // steps, as if its loads had stalled mid-stream.
      const int stop_after = p.debug_flags >> 8;
      // the last step that armed each stage (-1: none)
      int karmed[NS], varmed[NS], marmed[NM];
#pragma unroll
      for (int u = 0; u < NS; ++u) karmed[u] = varmed[u] = -1;
#pragma unroll
      for (int u = 0; u < NM; ++u) marmed[u] = -1;
      // Step j: K(j) once QK(j-2) has read its stage, V(j) once PV(j-2) has,
      // and the mean tiles of j once the mean terms of j-3 are done, each on
      // barriers of its own, so that no load waits for another's stage.
      for (int j = 0; j < nst && !*abort && !(stop_after > 0 && j >= stop_after); ++j) {
        const int sk = j % NS, sm3 = j % NM;
        const int4 q4 = quad(pa, pb);
        if (j >= NS && !mbar_wait(bar(B_KEMPTY + sk), ((j / NS) - 1) & 1, abort, WAIT_NS)) {
          record_timeout(p, abort);
          break;
        }
        mbar_arrive_expect_tx(bar(B_KFULL + sk), K_STAGE);
        load_k(sk, q4, bar(B_KFULL + sk));
        karmed[sk] = j;
        if (j >= NS && !mbar_wait(bar(B_VEMPTY + sk), ((j / NS) - 1) & 1, abort, WAIT_NS)) {
          record_timeout(p, abort);
          break;
        }
        mbar_arrive_expect_tx(bar(B_VFULL + sk), V_STAGE - 4 * 1024);
        load_v(sk, q4, bar(B_VFULL + sk));
        varmed[sk] = j;
        if (j >= NM && !mbar_wait(bar(B_MEMPTY + sm3), ((j / NM) - 1) & 1, abort, WAIT_NS)) {
          record_timeout(p, abort);
          break;
        }
        mbar_arrive_expect_tx(bar(B_MFULL + sm3), MU_STAGE);
        load_mu(sm3, q4, bar(B_MFULL + sm3));
        marmed[sm3] = j;
        if (pa.x >= 0) pa = next_pair(0, pa);
        if (pb.x >= 0) pb = next_pair(1, pb);
      }
      // Drain: every copy issued has landed before the CTA can exit, also
      // when a consumer gave up (time-bounded, ignoring the abort flag).  A
      // stage is re-armed only after its previous fill was consumed, so
      // waiting for the parity of its last fill is enough.
      bool drained = mbar_wait_time(qb, 0, WAIT_NS);
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        if (karmed[u] >= 0) drained &= mbar_wait_time(bar(B_KFULL + u), (karmed[u] / NS) & 1, WAIT_NS);
        if (varmed[u] >= 0) drained &= mbar_wait_time(bar(B_VFULL + u), (varmed[u] / NS) & 1, WAIT_NS);
      }
#pragma unroll
      for (int u = 0; u < NM; ++u)
        if (marmed[u] >= 0) drained &= mbar_wait_time(bar(B_MFULL + u), (marmed[u] / NM) & 1, WAIT_NS);
      if (!drained) record_timeout(p, abort);
    }
  } else if (warp == WARP_MMA || warp == WARP_PV) {
    // ----------------------------------------------------------- MMA issue
    // Two issuing lanes: warp 0 issues the QKs, warp 2 the mean terms and
    // PVs (S and O are disjoint columns; tcgen05.commit tracks each lane's
    // own MMAs).
    if (lane == 0 && nst > 0) {
      bool ok = true;
      const uint64_t dQ = sdesc_sw128(sb + SM_Q), dK = sdesc_sw128(sb + SM_K);
      const uint64_t dV = sdesc_sw64(sb + SM_V), dP = sdesc_sw128(sb + SM_P);
      const uint64_t dL = sdesc_k8_tf32(sb + SM_L);
      // mean operand of one tile: two 2 KiB parts (its two blocks), K-slots
      // 0..3 and 4..7, 16-byte rows, one row per channel
      const uint64_t dMu = sdesc(sb + SM_MU, MU_HALF, 128, 0);
      const uint32_t dO = tmem + COL_O;
      auto adv = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      auto wt = [&](int b, uint32_t par) {
        if (!ok) return;
        ok = mbar_wait(bar(b), par, abort, WAIT_NS);
        tc_fence_after();
      };
      if (warp == WARP_MMA) {
        // QK(i) once K(i) is in and the softmax holds S(i-1)
        wt(B_QFULL, 0);
        for (int i = 0; ok && i < nst; ++i) {
          wt(B_KFULL + i % NS, (i / NS) & 1);
          if (i > 0) wt(B_STAKEN, (i - 1) & 1);
          if (!ok) break;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(tmem + COL_S, adv(dQ, 32 * kk), adv(dK, (i % NS) * K_STAGE + 32 * kk), IDESC_QK, kk > 0);
          mma_commit(bar(B_SFULL));
          mma_commit(bar(B_KEMPTY + i % NS));
        }
      } else {
        auto mean = [&](int j) {  // both tiles' mean terms of step j
#pragma unroll
          for (int t = 0; t < 2; ++t)
            mma_tf32(dO, adv(dL, t * L_BYTES), adv(dMu, (j % NM) * MU_STAGE + t * 2 * MU_HALF), IDESC_TF32, 1);
        };
        // mean terms of step j-1, then [O | l] += P(j) [V ; indicators], once
        // V(j) is in and the softmax has written P(j) (and the mean operand
        // of j-1)
        for (int j = 0; ok && j < nst; ++j) {
          wt(B_VFULL + j % NS, (j / NS) & 1);
          wt(B_PFULL, j & 1);
          if (j > 0) wt(B_MFULL + (j - 1) % NM, ((j - 1) / NM) & 1);
          if (!ok) break;
          if (j > 0) {
            mean(j - 1);
            mma_commit(bar(B_MEMPTY + (j - 1) % NM));
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f8(dO, adv(dP, (kk >> 2) * TILE_BYTES + 32 * (kk & 3)),
                   adv(dV, (j % NS) * V_STAGE + (kk >> 1) * V_HALF + 32 * (kk & 1)), IDESC_PV,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(B_VEMPTY + j % NS));
          mma_commit(bar(B_ODONE));
        }
        // the last step's mean terms (the softmax's extra p_full arrival)
        wt(B_PFULL, nst & 1);
        wt(B_MFULL + (nst - 1) % NM, ((nst - 1) / NM) & 1);
        if (ok) {
          mean(nst - 1);
          mma_commit(bar(B_MDONE));
        }
      }
      if (!ok) record_timeout(p, abort);
      // Drain: every MMA of both lanes has completed before TMEM is
      // released, also after an abort (the wait ignores the abort flag).
      mma_commit(bar(B_FIN));
      if (!mbar_wait_time(bar(B_FIN), 0, WAIT_NS)) record_timeout(p, abort);
    }
  } else if (warp >= WARP_SOFTMAX) {
    // ------------------------------------------------------ softmax warps
    // Two threads per row: warps 4-7 take each row's first block (S columns
    // 0-63 of its tile), warps 8-11 its second (64-127).  The two exchange
    // their block maxima through shared memory (a barrier per quarter and
    // step parity, waited with a time limit), so both take the same running
    // maximum; each casts, writes and sums its own block.
    const int wq = warp & 3;
    const int hf = (warp - WARP_SOFTMAX) >> 2;  // 0: first block of the step, 1: second
    const int r = wq * 32 + lane;
    const int my_tile = r >> 6;  // 0: A, 1: B (warp-uniform)
    const int64_t row = static_cast<int64_t>(q0) + r;
    const bool row_ok = row < p.N;
    const int qt = static_cast<int>(row >> 6);
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + COL_S + 128 * my_tile + 64 * hf;
    const uint32_t tO = tmem + lane_addr + COL_O;
    const uint32_t tL = tO + 128 + 2 * my_tile + hf;  // this block's row-sum column
    uint8_t* Prow = sm + SM_P + my_tile * TILE_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
    uint8_t* Lrow = sm + SM_L + my_tile * L_BYTES + (r >> 3) * 256 + (r & 7) * 16 + 128 * hf;
    float* xch = reinterpret_cast<float*>(sm + SM_XCH);  // [step parity][half][row]
    const float qsc = p.q_scale[bh * p.nbp + (qt < p.nbp ? qt : p.nbp - 1)];
    const float a_i = p.c0 * qsc;
    const float* ksc = p.k_scale + bh * p.nbp;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const uint32_t FULL = 0xffffffffu;
    // the partner thread's value for exchange round k (a step, or nst for l)
    auto exchange = [&](int k, float v, float& other) -> bool {
      xch[((k & 1) * 2 + hf) * 128 + r] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_XCH + 2 * wq + (k & 1)));
      if (!__all_sync(FULL, mbar_wait(bar(B_XCH + 2 * wq + (k & 1)), (k >> 1) & 1, abort, WAIT_NS))) return false;
      other = xch[((k & 1) * 2 + (1 - hf)) * 128 + r];
      return true;
    };
    auto ld_rowsum = [&]() {
      uint32_t ls;
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(ls) : "r"(tL));
      tmem_wait_ld();
      return __uint_as_float(ls);
    };
    // this block's tf32 part of the row of the tile's mean MMA, [hi, lo, hi,
    // 0] against the mean tile's (hi, hi, lo, 0)
    auto put_lrow = [&](float v) {
      const float h = to_tf32(v);
      const float g = to_tf32(v - h);
      *reinterpret_cast<float4*>(Lrow) = make_float4(h, g, h, 0.0f);
    };
    float m_run = NEG_INF;
    float lh = 0.0f;  // this block's share of the row sum
    bool ok = true;
    int2 pr = pair_after(my_tile, -1);  // this row's tile's current step (x = -1: none)
    int i = 0;
    for (; i < nst; ++i) {
      const int2 pn = pr.x >= 0 ? next_pair(my_tile, pr) : pr;
      const int blk = hf ? pr.y : pr.x;
      const bool keep = row_ok && blk >= 0;
      const int n32 = static_cast<int>(p.N);
      const int lim = blk >= 0 ? n32 - blk * BLK : BLK;  // keys of the block before N
      const float A = blk >= 0 ? a_i * ksc[blk] : 0.0f;
      const bool partial = !__all_sync(FULL, lim >= BLK);

      if (!(ok = __all_sync(FULL, mbar_wait(bar(B_SFULL), i & 1, abort, WAIT_NS)))) break;
      tc_fence_after();
      float x[64];
      uint32_t w[16];
      tmem_ld64(tS, *reinterpret_cast<uint32_t(*)[64]>(&x[0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_STAKEN));  // S may be overwritten
      if (partial) {
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = j < lim ? x[j] : NEG_INF;
      }
      float ma = fmax3(x[0], x[1], x[2]), mb = fmax3(x[32], x[33], x[34]);
#pragma unroll
      for (int j = 3; j < 31; j += 2) {
        ma = fmax3(ma, x[j], x[j + 1]);
        mb = fmax3(mb, x[32 + j], x[33 + j]);
      }
      const float mine = keep ? A * fmax3(ma, mb, fmaxf(x[31], x[63])) : NEG_INF;
      float other;
      if (!(ok = exchange(i, mine, other))) break;
      const float m_tile = hf ? fmaxf(other, mine) : fmaxf(mine, other);
      const bool need = m_tile > m_run + p.tau8;
      const float m_new = need ? m_tile : m_run;
      const bool live = m_new != NEG_INF;
      const bool resc = need && m_run != NEG_INF;
      const float alpha = resc ? exp2f((m_run - m_new) * 0.125f) : 1.0f;
      if (partial) {
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = x[j] == NEG_INF ? 0.0f : x[j];
      }
      const bool k = live && keep;
      const float Aq = k ? A * 0.00390625f : 0.0f, Bq = k ? (p.C - m_new) * 0.00390625f : 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) w[q] = expcast4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3], Aq, Bq);
      if (partial) {
        const int lim_k = k ? (lim < 64 ? lim : 64) : 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t keepb = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (4 * q + e < lim_k) keepb |= 0xFFu << (8 * e);
          w[q] &= keepb;
        }
      }
      m_run = m_new;
      if (i > 0) {
        // PV(i-1) done (and with it the mean terms of step i-2): P may be
        // overwritten and the row sums of step i-1 are final.
        if (!(ok = __all_sync(FULL, mbar_wait(bar(B_ODONE), (i - 1) & 1, abort, WAIT_NS)))) break;
        tc_fence_after();
      }
      // this block's 64 bytes of row r of the tile's P: 16-byte chunk c at
      // position c ^ (r & 7)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(Prow + (((4 * hf + c) ^ (r & 7)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      if (i > 0) {
        // The block's row sum of step i-1: read and cleared, so that PV(i)
        // accumulates its own.  If the maximum moved, this thread's half of
        // O and its share of l move to the new maximum, and its part of the
        // mean operand of step i-1 is written already scaled.
        const float ls = ld_rowsum();
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tL), "r"(0u) : "memory");
        if (__any_sync(FULL, resc)) {
          uint32_t (&o)[64] = *reinterpret_cast<uint32_t(*)[64]>(&x[0]);
          tmem_ld64(tO + 64 * hf, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 64; ++e) x[e] *= alpha;
          tmem_st64(tO + 64 * hf, o);
        }
        lh = (lh + ls) * alpha;
        put_lrow(ls * alpha);
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
      pr = pn;
    }
    // the last step's row sums, then its mean terms, then the row sum of
    // both blocks
    float l = 0.0f;
    if (ok && nst > 0) {
      ok = __all_sync(FULL, mbar_wait(bar(B_ODONE), (nst - 1) & 1, abort, WAIT_NS));
      if (ok) {
        tc_fence_after();
        const float ls = ld_rowsum();
        lh += ls;
        put_lrow(ls);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL));
        ok = __all_sync(FULL, mbar_wait(bar(B_MDONE), 0, abort, WAIT_NS));
        tc_fence_after();
      }
      float lo_ = 0.0f;
      if (ok && (ok = exchange(nst, lh, lo_))) l = hf ? lo_ + lh : lh + lo_;
    }
    if (!ok) record_timeout(p, abort);

    // ------------------------------------------------------------ epilogue
    // this thread's 64 output channels, 64 hf .. 64 hf + 63
    const bool have = ok && nst > 0;
    if (__all_sync(0xffffffffu, have)) {
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hf + cc;
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        if (row_ok) {
          float y[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            y[e] = __uint_as_float(o[e]) * p.v_scale[bh * D + 32 * c + e] * inv_l;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + p.lo.head(bh) + p.lo.row(row) + 32 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.O) + p.lo.head(bh) + p.lo.row(row) + 32 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
    } else if (row_ok && nst == 0) {
      // this thread's half of the row: 64 channels
      const int nvec = p.out_f32 ? 16 : 8;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.O) +
                                            (p.lo.head(bh) + p.lo.row(row) + 64 * hf) * (p.out_f32 ? 4 : 2));
      for (int e = 0; e < nvec; ++e) dst[e] = make_uint4(0, 0, 0, 0);
    }
    if (row_ok && p.lse2 && hf == 0) {
      p.lse2[bh * p.N + row] = l > 0.0f
          ? m_run * 0.125f - p.off + log2f(l) + p.qmu[bh * p.N + row] * p.lse_qmu
          : -__int_as_float(0x7f800000);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == WARP_MMA) tmem_dealloc(tmem, 512);
}
}  // namespace sp

// The driver's tensor-map encoder (looked up once; a function-local static is
// initialised thread-safely).
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

// 3-D u8 tensor map with a box of b0 x b1 bytes: 128-byte swizzle for
// 128-byte box rows, 64-byte swizzle for 64-byte rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
              uint32_t b1) {
  auto enc = get_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0, d0 * d1};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, b0 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_expcast_probe(const float* x, const float* A, const float* B, uint8_t* codes, int64_t n,
                                 cudaStream_t s) {
  const int64_t ng = n / 4;
  if (ng == 0) return cudaSuccess;
  expcast_probe<<<static_cast<unsigned>((ng + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(x), A, B, reinterpret_cast<uint32_t*>(codes), ng);
  return cudaGetLastError();
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  const int64_t Np = npad(a.N);
  // Masked, K and V come one 64-key block per box.
  const uint32_t kb = a.mask ? 64 : 128;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q8, D, Np, a.BH, 128, 128) || !make_map(&mk, a.k8, D, Np, a.BH, 128, kb) ||
      !make_map(&mv, a.r8t, Np, D, a.BH, kb, 128))
    return cudaErrorInvalidValue;
  Params p{};
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.qmu = a.qmu;
  p.vmu_op = a.vmu_op;
  p.mask = a.mask;
  p.O = a.O;
  p.lo = a.lo;
  p.lse2 = a.lse2;
  p.out_f32 = a.out_f32;
  p.N = a.N;
  p.npad = static_cast<int>(Np);
  p.nbp = static_cast<int>(Np / BLK);
  p.ntile = static_cast<int>(Np / TILE);
  p.nq64 = static_cast<int>(ceil_div(a.N, BLK));
  p.c0 = static_cast<float>(8.0 * 1.4426950408889634 * static_cast<double>(a.sm_scale));
  const double cstar = (std::log2(1.5) - 0.5) / 2.0;  // minimax centring of the byte
  p.C = static_cast<float>(56.0 + 8.0 * a.off - 8.0 * cstar);
  p.lse_qmu = static_cast<float>(static_cast<double>(a.sm_scale) * 1.4426950408889634);
  p.tau8 = a.tau8;
  p.off = static_cast<float>(a.off);
  p.err = a.err;
  p.debug_flags = a.debug_flags;
  // the shared-memory limit is a per-device attribute of each kernel
  static PerDevice attr;
  int dev = 0;
  const cudaError_t ea = per_device_setup(attr, &dev, [](int, int*) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(sp::attn_sparse, cudaFuncAttributeMaxDynamicSharedMemorySize, sp::SMEM_BYTES);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  if (p.mask) {
    const dim3 grid(static_cast<unsigned>(Np / TILE), static_cast<unsigned>(a.BH));
    sp::attn_sparse<<<grid, sp::NTHREADS, sp::SMEM_BYTES, s>>>(mq, mk, mv, p);
  } else {
    const dim3 grid(static_cast<unsigned>(ceil_div(Np, CTA_ROWS)), static_cast<unsigned>(a.BH));
    attn_fwd<<<grid, NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, p);
  }
  return cudaGetLastError();
}

}  // namespace vc
