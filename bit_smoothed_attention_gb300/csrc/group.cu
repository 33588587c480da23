// V-Smooth grouping ("VC-Attention: Value Smoothing and Softmax Casting for
// Low-bit Attention", Key Contribution 1 and Methodology): online k-means over
// the value tokens of each (batch, head), then a stable sort of the labels
// into the permutation applied jointly to K and V.
//
// Every FP32 result is produced in one fixed order so that labels, centroids
// and the permutation are bit-for-bit reproducible:
//   assign : h_c = 0.5f * (fmaf chain over d of c_c[d]^2); dot = one fmaf
//            chain over d = 0..127 ascending; score = dot - h_c; the lowest
//            cluster with the largest score wins (km_tc.cu: tensor-core
//            scores with an exact fallback).
//   update : per 512-token chunk, the members of each cluster are added in
//            token order to a +0 partial; partials are added in chunk order
//            to a +0 total; centroid = total / (float)count (IEEE division);
//            an empty cluster keeps its centroid.
// This file is compiled with --fmad=false: only the explicit __fmaf_rn calls
// fuse.
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace vc {
namespace {

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Init: c_c = v[floor(c*N/k)].  grid (k, BH), block D.
__global__ void km_init(const uint16_t* __restrict__ V, RowLayout lv, int64_t N, int k,
                        float* __restrict__ cent) {
  const int64_t bh = blockIdx.y;
  const int c = blockIdx.x, d = threadIdx.x;
  const int64_t j = (static_cast<int64_t>(c) * N) / k;
  cent[(bh * k + c) * D + d] = bf16f(V[lv.head(bh) + lv.row(j) + d]);
}

// Chunk partial sums.  The chunk's tokens are first listed cluster by
// cluster, each list in ascending token order (a stable counting sort in
// shared memory: ranks within a warp from __match_any_sync, then a prefix
// over the warps).  Thread (g, q) then owns clusters 4g .. 4g+3 and channels
// 8q .. 8q+7: for each cluster it adds the members' rows in list order to a
// +0 partial, 16-byte loads straight from global memory, several in flight
// (the 16 threads of a cluster group read a whole 256-byte row).  grid
// (nchunk, BH), block 256.
// L2 eviction priorities: the chunk sums stream V through once (evict
// first), and their partials are read back by km_finalize right after
// (evict last).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_l2hint(const void* ptr, uint64_t pol) {
  uint4 r;
  asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr), "l"(pol));
  return r;
}
__device__ __forceinline__ void st_l2hint(void* ptr, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

__global__ void __launch_bounds__(256) km_partial(const uint16_t* __restrict__ V, RowLayout lv,
                                                  const int32_t* __restrict__ labels, int64_t N,
                                                  int k, int nchunk, float* __restrict__ part,
                                                  int32_t* __restrict__ cnt, uint32_t* err) {
  constexpr int NW = UPD_CHUNK / 32;  // 16 warps' worth of tokens, 2 per thread
  __shared__ int wc[NW][KMAX];        // per-warp counts, then per-warp offsets
  __shared__ int cstart[KMAX + 1];
  __shared__ int16_t order[UPD_CHUNK];
  const int64_t bh = blockIdx.y;
  const int g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j0 = static_cast<int64_t>(g) * UPD_CHUNK;
  const int n = static_cast<int>(N - j0 < UPD_CHUNK ? N - j0 : UPD_CHUNK);
  for (int i = tid; i < NW * KMAX; i += 256) wc[i / KMAX][i % KMAX] = 0;
  __syncthreads();
  // each thread takes tokens tid and tid + 256 (warps w and w + 8 of 32 tokens)
  int lab[2], rank[2];
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = tid + 256 * h;
    int c = t < n ? labels[bh * N + j0 + t] : -1;
    if (c >= 0 && static_cast<unsigned>(c) >= static_cast<unsigned>(k)) {
      bad = true;
      c = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, c);
    rank[h] = __popc(same & ((1u << lane) - 1u));
    if (c >= 0 && rank[h] == 0) wc[warp + 8 * h][c] = __popc(same);
    lab[h] = c;
  }
  if (bad) atomicOr(err, ERR_BAD_LABEL);
  __syncthreads();
  if (tid < KMAX) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int t = wc[w][tid];
      wc[w][tid] = run;
      run += t;
    }
    cstart[tid] = run;  // count of cluster tid for now
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int c = 0; c < KMAX; ++c) {
      const int t = cstart[c];
      cstart[c] = run;
      run += t;
    }
    cstart[KMAX] = run;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (lab[h] >= 0) order[cstart[lab[h]] + wc[warp + 8 * h][lab[h]] + rank[h]] = static_cast<int16_t>(tid + 256 * h);
  __syncthreads();
  // sums: clusters 4 cg .. 4 cg + 3, channels 8 q .. 8 q + 7
  const int cg = tid >> 4, q = tid & 15;
  const uint16_t* vb = V + lv.head(bh) + lv.row(j0) + 8 * q;
  // partials [BH, k, nchunk, D]: a cluster's chunks side by side
  float* pg = part + (bh * k * static_cast<int64_t>(nchunk) + g) * D;
  const uint64_t pol_v = l2_evict_first(), pol_p = l2_evict_last();
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * cg + cc;
    if (c >= k) break;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    const int i1 = cstart[c + 1];
    int i = cstart[c];
    for (; i + 8 <= i1; i += 8) {
      uint4 u[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) u[x] = ld_l2hint(vb + lv.row(order[i + x]), pol_v);
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint32_t w4[4] = {u[x].x, u[x].y, u[x].z, u[x].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = acc[2 * e] + __uint_as_float(w4[e] << 16);
          acc[2 * e + 1] = acc[2 * e + 1] + __uint_as_float(w4[e] & 0xFFFF0000u);
        }
      }
    }
    for (; i < i1; ++i) {
      const uint4 u = ld_l2hint(vb + lv.row(order[i]), pol_v);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] = acc[2 * e] + __uint_as_float(w4[e] << 16);
        acc[2 * e + 1] = acc[2 * e + 1] + __uint_as_float(w4[e] & 0xFFFF0000u);
      }
    }
    float* dst = pg + static_cast<int64_t>(c) * nchunk * D + 8 * q;
    st_l2hint(dst, make_float4(acc[0], acc[1], acc[2], acc[3]), pol_p);
    st_l2hint(dst + 4, make_float4(acc[4], acc[5], acc[6], acc[7]), pol_p);
    if (q == 0) cnt[(bh * nchunk + g) * k + c] = i1 - cstart[c];
  }
}

// Centroid = (partials added in chunk order) / count.  grid (k, BH), block D.
__global__ void __launch_bounds__(D) km_finalize(const float* __restrict__ part,
                                                 const int32_t* __restrict__ cnt, int nchunk,
                                                 int k, float* __restrict__ cent) {
  const int64_t bh = blockIdx.y;
  const int c = blockIdx.x;
  const int d = threadIdx.x;
  float total = 0.0f;
  int count = 0;
  const float* pc = part + (bh * k + c) * static_cast<int64_t>(nchunk) * D + d;
  for (int g = 0; g < nchunk; ++g) {
    total = total + pc[static_cast<int64_t>(g) * D];
    count += cnt[(bh * nchunk + g) * k + c];
  }
  if (count > 0) cent[(bh * k + c) * D + d] = total / static_cast<float>(count);
}

// Output offsets of the stable counting sort: offs[g][c] = (tokens with a
// smaller label) + (tokens with label c in earlier chunks).  grid (BH),
// block KMAX.
__global__ void sort_offsets(const int32_t* __restrict__ cnt, int nchunk, int k,
                             int32_t* __restrict__ offs) {
  __shared__ int tot[KMAX];
  const int64_t bh = blockIdx.x;
  const int c = threadIdx.x;
  int t = 0;
  if (c < k)
    for (int g = 0; g < nchunk; ++g) t += cnt[(bh * nchunk + g) * k + c];
  tot[c] = t;
  __syncthreads();
  if (c < k) {
    int run = 0;
    for (int c2 = 0; c2 < c; ++c2) run += tot[c2];
    for (int g = 0; g < nchunk; ++g) {
      const int64_t o = (bh * nchunk + g) * k + c;
      offs[o] = run;
      run += cnt[o];
    }
  }
}

// Stable scatter of one 512-token chunk: rank among equal labels within a
// warp from __match_any_sync, then an exclusive prefix over the chunk's
// warps.  grid (nchunk, BH), block 512.
__global__ void __launch_bounds__(UPD_CHUNK) sort_scatter(const int32_t* __restrict__ labels,
                                                          const int32_t* __restrict__ offs,
                                                          int64_t N, int k, int nchunk,
                                                          int32_t* __restrict__ perm) {
  constexpr int NW = UPD_CHUNK / 32;
  __shared__ int wc[NW][KMAX];
  const int64_t bh = blockIdx.y;
  const int g = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < NW * KMAX; i += UPD_CHUNK) wc[i / KMAX][i % KMAX] = 0;
  __syncthreads();
  const int64_t j = static_cast<int64_t>(g) * UPD_CHUNK + tid;
  const bool valid = j < N;
  int c = valid ? labels[bh * N + j] : -1;
  if (valid && static_cast<unsigned>(c) >= static_cast<unsigned>(k)) c = -1;  // reported by km_partial
  const unsigned same = __match_any_sync(0xffffffffu, c);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (c >= 0 && rank == 0) wc[warp][c] = __popc(same);
  __syncthreads();
  if (tid < k) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int t = wc[w][tid];
      wc[w][tid] = run;
      run += t;
    }
  }
  __syncthreads();
  if (c >= 0) perm[bh * N + offs[(bh * nchunk + g) * k + c] + wc[warp][c] + rank] = static_cast<int32_t>(j);
}

}  // namespace

size_t group_ws_layout(int64_t BH, int64_t N, int k, void* base, GroupWs* ws) {
  const int64_t nchunk = ceil_div(N, UPD_CHUNK);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return base ? static_cast<char*>(base) + o : nullptr;
  };
  GroupWs w{};
  w.cent = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * k * D * 4));
  w.part = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * nchunk * k * D * 4));
  w.cnt = reinterpret_cast<int32_t*>(take(static_cast<size_t>(BH) * nchunk * k * 4));
  w.offs = reinterpret_cast<int32_t*>(take(static_cast<size_t>(BH) * nchunk * k * 4));
  w.amb = reinterpret_cast<KmAmb*>(take(static_cast<size_t>(BH) * N * sizeof(KmAmb)));
  w.amb_count = reinterpret_cast<uint32_t*>(take(8));
  w.head_cn = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * 2 * 4));
  w.head_h = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * KMAX * 4));
  w.vnorm = reinterpret_cast<float*>(take(static_cast<size_t>(BH) * N * 4));
  if (ws) *ws = w;
  return off;
}

cudaError_t launch_group(const uint16_t* V, const RowLayout& lv, int64_t BH, int64_t N, int k, int iters,
                         const float* init, int32_t* labels, int32_t* perm, float* centroids_out,
                         const GroupWs& ws, uint32_t* err, cudaStream_t s) {
  const int nchunk = static_cast<int>(ceil_div(N, UPD_CHUNK));
  float* cent = centroids_out ? centroids_out : ws.cent;
  cudaError_t e = cudaSuccess;
  if (!init) {
    km_init<<<dim3(k, static_cast<unsigned>(BH)), D, 0, s>>>(V, lv, N, k, cent);
    e = cudaGetLastError();
  } else if (init != cent) {
    // warm start: the iterations begin from the given centroids
    e = cudaMemcpyAsync(cent, init, static_cast<size_t>(BH) * k * D * sizeof(float),
                        cudaMemcpyDeviceToDevice, s);
  }
  if (e != cudaSuccess) return e;
  // counters of the open assignments (each fix-up clears the next one)
  if ((e = cudaMemsetAsync(ws.amb_count, 0, 2 * sizeof(uint32_t), s)) != cudaSuccess) return e;
  const dim3 gchunk(nchunk, static_cast<unsigned>(BH));
  for (int it = 0; it < iters; ++it) {
    e = launch_km_assign_tc(V, lv, BH, N, k, cent, labels, ws, it, err, s);
    if (e != cudaSuccess) return e;
    km_partial<<<gchunk, 256, 0, s>>>(V, lv, labels, N, k, nchunk, ws.part, ws.cnt, err);
    km_finalize<<<dim3(k, static_cast<unsigned>(BH)), D, 0, s>>>(ws.part, ws.cnt, nchunk, k, cent);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  sort_offsets<<<static_cast<unsigned>(BH), KMAX, 0, s>>>(ws.cnt, nchunk, k, ws.offs);
  sort_scatter<<<gchunk, UPD_CHUNK, 0, s>>>(labels, ws.offs, N, k, nchunk, perm);
  return cudaGetLastError();
}

}  // namespace vc
