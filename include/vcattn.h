/*
 * vcattn.h -- C ABI of libvcattn.so: the FP8 (E4M3) smoothed attention
 * forward for GB300 (sm_103a).
 *
 * The operation, as described by the pages it comes from:
 *  - "Feat: Attention Smoothing to Improve Generation Quality" (TeleFuser
 *    PR #40), Summary and Changes: K is centred by its FP32 sequence mean
 *    before E4M3 quantisation (exact under softmax); V is centred and the
 *    mean restored.
 *  - "VC-Attention: Value Smoothing and Softmax Casting for Low-bit
 *    Attention", Key Contributions 1-3 and Methodology: V-Smooth (online
 *    k-means over value tokens, a stable sort of the labels into a
 *    permutation applied jointly to K and V, per-block mean subtraction with
 *    only the residual quantised, the means restored inside the online
 *    softmax from the per-block row sums) and ExpCast-FP8 (the probability's
 *    E4M3 byte written from the max-subtracted log2 score with one FMA and
 *    one integer rounding).
 *  - "[perf] Add opt-in SM120 sparse attention forward kernel for
 *    MiniMax-H3" (FastVideo PR #2048), Changes and Test Results: a 64x64
 *    block-sparse forward that handles partial tiles and empty selections
 *    and returns O plus the log2-LSE.
 *
 * Conventions shared by every entry point:
 *  - Tensors are contiguous.  Q, K, V, O are bf16 [B, H, N, D] with D = 128.
 *  - The caller owns and allocates every device buffer, including the
 *    workspaces sized by the *_workspace_bytes queries.  The library never
 *    allocates, never frees and never synchronises (except
 *    vcattn_last_device_error).  All pointers are device pointers unless
 *    stated otherwise; every device pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream); all work
 *    is enqueued on it in order.
 *  - Argument errors return at once and enqueue nothing.  A failed launch
 *    returns VCATTN_ERR_CUDA.  Errors found on the device (a bounded wait
 *    that ran out, a bad label) are recorded in a per-device error word and
 *    reported by the next vcattn_last_device_error().
 *  - Calls on different streams with different buffers are independent.
 */
#ifndef VCATTN_H
#define VCATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VCATTN_OK = 0,
  VCATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, small workspace */
  VCATTN_ERR_UNSUPPORTED = 2, /* D != 128, k outside [1, 64], no sm_103a device        */
  VCATTN_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed                */
  VCATTN_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out (device error word) */
  VCATTN_ERR_DEVICE = 5       /* another device-side check failed (device error word)   */
} vcattn_status;

/* Problem shape.  D must be 128; N >= 1; B, H >= 1. */
typedef struct {
  int64_t B, H, N, D;
} vcattn_shape;
/* Element strides of a [B, H, N, D] tensor whose D channels are contiguous:
 * row (b, h, n) starts at element b*b_stride + h*h_stride + n*n_stride.  The
 * *_strided entry points take them, e.g. for the (B, N, H, D) layout of
 * many models: b = N*H*D, h = D, n = H*D.  Each must be a positive multiple
 * of 8 elements (every row 16-byte aligned) below 2^38, n below 2^31; rows
 * must not overlap.  The other entry points take contiguous [B, H, N, D]
 * tensors. */
typedef struct {
  int64_t b, h, n;
} vcattn_strides;

/* Output of vcattn_prep, input of vcattn_attn.  With Npad = 128*ceil(N/128)
 * rows and nbp = Npad/64 metadata blocks per head (blocks at or past
 * ceil(N/64) are padding: scale 1, mean 0; rows at or past N are 0x00):
 *   q8      [B,H,Npad,D]  u8  E4M3 Q, original token order
 *   k8      [B,H,Npad,D]  u8  E4M3 centred K, permuted order
 *   r8t     [B,H,D,Npad]  u8  E4M3 V residual, permuted order, transposed
 *   q_scale [B,H,nbp]     f32 one scale per 64-query block
 *   k_scale [B,H,nbp]     f32 one scale per 64-key block
 *   v_scale [B,H,D]       f32 one scale per channel
 *   k_mean  [B,H,D]       f32 mu_K, the FP32 sequence mean of K
 *   v_mean  [B,H,nbp,D]   f32 mu_b, the FP32 mean of each permuted 64-block of V
 *   qmu     [B,H,N]       f32 q . mu_K (restores the true LSE)
 *   vmu_op  [B,H,nbp,D,4] f32 the block means divided by v_scale, split
 *           into tf32 parts (hi, hi, lo, 0) per channel: one 2 KiB half of
 *           the B operand of the mean-restoration MMA per 64-key block.
 * vcattn_prepped_carve() fills this struct from one buffer of
 * vcattn_prepped_bytes() bytes. */
typedef struct {
  uint8_t *q8, *k8, *r8t;
  float *q_scale, *k_scale, *v_scale, *k_mean, *v_mean, *qmu, *vmu_op;
} vcattn_prepped;

/* Padded row count 128*ceil(N/128) of the FP8 tensors. */
int64_t vcattn_npad(int64_t N);

/* ---------------------------------------------------------------- grouping */
/* V-Smooth grouping (VC-Attention, Key Contribution 1 and Methodology):
 * `iters` Lloyd iterations of k-means over the value tokens of each (b, h),
 * then a stable sort of the labels.  Init c_c = v[floor(c*N/k)]; one
 * iteration assigns every token to the cluster with the largest
 * v.c - |c|^2/2 (FP32, one fmaf chain over d ascending; ties to the lowest
 * cluster) and recomputes each centroid as the mean of its members (sums over
 * 512-token chunks in token order, chunks in order; empty clusters keep
 * their centroid).
 *   V         bf16 [B,H,N,D] (device)
 *   labels    i32  [B,H,N]   out: cluster of each token (last assignment)
 *   perm      i32  [B,H,N]   out: perm[i] = token at sorted position i,
 *                             sorted by (label, token index)
 *   centroids f32  [B,H,k,D] out, nullable: centroids after the last update
 *   ws        device scratch of at least vcattn_group_workspace_bytes(shape, k)
 * k in [1, 64], iters >= 1.  Results are bit-for-bit deterministic.
 * V must be finite: a token whose scores cannot be compared (a NaN or an
 * infinity in its row or in a centroid) gets label -1 and sets the device
 * error word (vcattn_last_device_error returns VCATTN_ERR_DEVICE); perm is
 * then not a permutation. */
size_t vcattn_group_workspace_bytes(const vcattn_shape* shape, int k);
vcattn_status vcattn_group(const vcattn_shape* shape, const void* V, int k, int iters,
                           int32_t* labels, int32_t* perm, float* centroids,
                           void* ws, size_t ws_bytes, void* stream);
/* The same grouping started from given centroids instead of the evenly
 * spaced seeds (a warm start).  The pages regroup on the first quarter of
 * the denoising steps; starting each regrouping from the previous one's
 * centroids lets it run fewer iterations.  Starting from the centroids of
 * n iterations and running m more gives exactly the result of n + m
 * iterations of vcattn_group.
 *   init_centroids  f32 [B,H,k,D] (device), required; `centroids` may be the
 *                   same buffer (updated in place), otherwise the two must
 *                   not overlap
 * Other arguments as for vcattn_group (same workspace size). */
vcattn_status vcattn_group_warm(const vcattn_shape* shape, const void* V, int k, int iters,
                                const float* init_centroids, int32_t* labels, int32_t* perm,
                                float* centroids, void* ws, size_t ws_bytes, void* stream);
/* vcattn_group (init_centroids NULL) or vcattn_group_warm (not NULL) for a
 * V with the row strides `sv` (required).  Same results as on a contiguous
 * copy of V. */
vcattn_status vcattn_group_strided(const vcattn_shape* shape, const void* V, const vcattn_strides* sv,
                                   int k, int iters, const float* init_centroids, int32_t* labels,
                                   int32_t* perm, float* centroids, void* ws, size_t ws_bytes,
                                   void* stream);

/* ----------------------------------------------------------- preprocessing */
/* Fused preprocessing (TeleFuser PR #40 Changes; VC-Attention Key
 * Contributions 1 and 3): mu_K over the original order; K gathered by perm,
 * centred and quantised per 64-key block; V gathered by perm, each 64-block
 * demeaned and only the residual quantised with one scale per channel; Q
 * quantised per 64-query block in the original order.  Quantiser: amax =
 * max|x| (amax < 2^-100 gives bytes 0 and scale 1), byte =
 * E4M3_rne_satfinite(x * fl(448/amax)), scale = fl(amax/448).  Means are
 * adjacent-pairing FP32 tree sums divided by the valid count.
 *   Q, K, V  bf16 [B,H,N,D] (device)
 *   perm     i32  [B,H,N] (device), nullable = identity; must be a
 *            permutation of [0, N) per head.  An entry outside [0, N) is
 *            never dereferenced: its row is read as zeros and the device
 *            error word reports VCATTN_ERR_DEVICE; a repeated entry is not
 *            detected.
 *   out      the prepped buffers (device pointers inside a host struct)
 *   ws       device scratch of at least vcattn_prep_workspace_bytes(shape) */
size_t vcattn_prepped_bytes(const vcattn_shape* shape);
vcattn_status vcattn_prepped_carve(const vcattn_shape* shape, void* base, size_t bytes,
                                   vcattn_prepped* out);
size_t vcattn_prep_workspace_bytes(const vcattn_shape* shape);
vcattn_status vcattn_prep(const vcattn_shape* shape, const void* Q, const void* K, const void* V,
                          const int32_t* perm, const vcattn_prepped* out,
                          void* ws, size_t ws_bytes, void* stream);
/* vcattn_prep for Q, K and V with their own row strides (all three
 * required).  The prepped tensors are the same as for contiguous copies. */
vcattn_status vcattn_prep_strided(const vcattn_shape* shape, const void* Q, const vcattn_strides* sq,
                                  const void* K, const vcattn_strides* sk, const void* V,
                                  const vcattn_strides* sv, const int32_t* perm,
                                  const vcattn_prepped* out, void* ws, size_t ws_bytes, void* stream);

/* vcattn_prep with options (`flags`, a bitwise OR of the values below; 0 =
 * vcattn_prep) and optional row strides (sq, sk, sv: NULL = contiguous).
 *
 * VCATTN_PREP_QK_HADAMARD: the QK Hadamard rotation of the fused
 * preprocessing chain (VC-Attention, Key Contribution 3 and Methodology: the
 * chain applies a Hadamard transform to Q and K after the means and the
 * gather, before the quantisers).  Each row of Q, and of K after centring,
 * is multiplied by the 128-point Sylvester-Hadamard matrix H (H[i][j] =
 * (-1)^popcount(i & j)) through a fast butterfly in a fixed FP32 order
 * (stages h = 1, 2, 4, ..., 64; each pair (x[i], x[i + h]) with i & h == 0
 * becomes (x[i] + x[i + h], x[i] - x[i + h]), rounded to FP32), then scaled
 * by 2^-4 (Q) and 2^-3 (K), so that q' . k' = q . (k - mu_K) exactly in
 * exact arithmetic (H H^T = 128 I).  The quantisers then act on the rotated
 * rows; the V side, k_mean and qmu (from the unrotated q) are unchanged, and
 * vcattn_attn consumes the result as it is.  The rotation spreads outlier
 * channels of Q and K over all 128 channels before their per-block E4M3
 * scales are set.  Rotary position embedding, the other step of the
 * pages' chain, is not included: the pages give neither its positions nor
 * its frequencies. */
#define VCATTN_PREP_QK_HADAMARD 1
vcattn_status vcattn_prep_ex(const vcattn_shape* shape, const void* Q, const vcattn_strides* sq,
                             const void* K, const vcattn_strides* sk, const void* V,
                             const vcattn_strides* sv, const int32_t* perm, int flags,
                             const vcattn_prepped* out, void* ws, size_t ws_bytes, void* stream);

/* Preprocessing without a caller-provided workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they call the preprocessing, such as a plugin
 * that receives only its input and output tensors from a host framework, or
 * a program that forbids device allocation after start-up.  It computes
 * exactly what vcattn_prep computes (same kernels, same outputs) but keeps
 * its scratch in a 16 MiB device array owned by the library, held on every
 * GPU that loads the library until the process exits.
 *   - Problems needing more than 16 MiB of scratch (256-byte-rounded
 *     B*H*(Npad/64)*512 + B*H*512 bytes; the 56-head, 32,626-token workload
 *     needs 14.7 MB) return VCATTN_ERR_UNSUPPORTED with nothing enqueued.
 *   - The first call on a device looks up the array's device address; make
 *     it before any stream capture begins.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; each call clears what must start at zero on its own stream.
 *     Calls that overlap on the GPU race on the array: order them on one
 *     stream.
 *   - It allocates and frees nothing. */
vcattn_status vcattn_prep_noalloc(const vcattn_shape* shape, const void* Q, const void* K,
                                  const void* V, const int32_t* perm, const vcattn_prepped* out,
                                  void* stream);

/* --------------------------------------------------------------- attention */
/* FP8 attention forward with ExpCast-FP8 and the rank-one mean restoration
 * (VC-Attention Key Contributions 1-2; FastVideo PR #2048 for the mask,
 * partial tiles, empty selections and the log2-LSE).  Per query i (original
 * order) over KV tiles of 128 permuted keys:
 *   x = q8_i . k8_j (FP8 tensor cores, FP32 accumulate);
 *   A = fl(fl(c0*q_scale)*k_scale), c0 = fl(8*log2(e)*sm_scale);
 *   running max m (code units) rescales when the tile max exceeds
 *   m + tau8 (tau8 = 0: exact running max);
 *   byte = ExpCast(x) = clip(rint(fmaf(x, A, C - m))), C = 56 + 8*off - 8c*,
 *   c* = (log2 1.5 - 1/2)/2, bytes below 8 flush to 0, above 126 clip;
 *   O_i = v_scale . (P8 R8 + sum_b l_ib mu_b / v_scale) / l_i  (bf16),
 *   lse2_i = m/8 - off + log2(l_i) + qmu_i * sm_scale * log2(e).
 *   in        prepped tensors from vcattn_prep
 *   sm_scale  softmax scale (> 0)
 *   tile_mask u8 [B,H,ceil(N/64),Npad/64] (device), nullable = dense:
 *             nonzero keeps (query 64-tile in original order, key 64-block
 *             in permuted order); a row with no kept key gets O = 0 and
 *             lse2 = -inf
 *   O         bf16 [B,H,N,D] (device) out
 *   lse2      f32 [B,H,N] (device) out, nullable
 * vcattn_attn uses off = 8, tau8 = 6 (the largest lazy-rescale threshold that
 * keeps every code <= 126 at off = 8: the running max, and with it O and l,
 * is rescaled only when a tile raises it by more than 6 code units = 0.75 in
 * log2 units) and writes bf16 O; vcattn_attn_ex takes off and tau8
 * (0 <= off <= 8, 0 <= tau8 <= 8*(8.75 - off); tau8 = 0 is the exact running
 * max) and, with out_f32 = 1, writes O as f32 [B,H,N,D] instead of bf16 (the
 * value before the final bf16 rounding). */
vcattn_status vcattn_attn(const vcattn_shape* shape, const vcattn_prepped* in, float sm_scale,
                          const uint8_t* tile_mask, void* O, float* lse2, void* stream);
vcattn_status vcattn_attn_ex(const vcattn_shape* shape, const vcattn_prepped* in, float sm_scale,
                             int off, float tau8, int out_f32, const uint8_t* tile_mask, void* O,
                             float* lse2, void* stream);
/* vcattn_attn_ex writing O with the row strides `so` (required; in elements
 * of O's type, bf16 or f32).  lse2 stays a contiguous [B,H,N] array. */
vcattn_status vcattn_attn_strided(const vcattn_shape* shape, const vcattn_prepped* in, float sm_scale,
                                  int off, float tau8, int out_f32, const uint8_t* tile_mask, void* O,
                                  const vcattn_strides* so, float* lse2, void* stream);

/* One call = vcattn_prep into `ws` followed by vcattn_attn.  perm is the
 * output of vcattn_group (or of an earlier step, or NULL = identity). */
size_t vcattn_fwd_workspace_bytes(const vcattn_shape* shape);
vcattn_status vcattn_fwd(const vcattn_shape* shape, const void* Q, const void* K, const void* V,
                         const int32_t* perm, float sm_scale, const uint8_t* tile_mask,
                         void* O, float* lse2, void* ws, size_t ws_bytes, void* stream);

/* -------------------------------------------------- host-resident tensors */
/* The whole path -- vcattn_group (k, iters), vcattn_prep, vcattn_attn -- for
 * Q, K, V and O in host memory, with the host<->device copies overlapped with
 * the computation.  The method never mixes heads (k-means, the permutation,
 * the quantisers and the attention are per (b, h)), so the flattened B*H
 * heads go through the device in chunks of `chunk_heads` heads (0 = 8; the
 * first two chunks have an eighth and three eighths of that, rounded up, so
 * computing starts early):
 * two device slots alternate, chunk c computes on streams[c % 2], and meanwhile
 * the next chunk's Q, K, V are copied in on streams[2] and finished chunks'
 * O (and lse2) copied out on streams[3].  streams[0] and streams[1] may be
 * the same stream (the chunks then compute in turn); distinct, one chunk's
 * k-means runs beside the other's attention.  O and lse2 equal, bit for bit,
 * those of vcattn_group followed by vcattn_fwd on the same inputs.
 *   hQ, hK, hV  bf16 [B,H,N,D] in host memory.  Page-locked buffers
 *               (cudaHostAlloc, cudaHostRegister) let the copies overlap;
 *               pageable ones give the same results, copied synchronously.
 *   k, iters    as for vcattn_group
 *   tile_mask   u8 [B,H,ceil(N/64),Npad/64] (device), nullable = dense
 *   hO          bf16 [B,H,N,D] host out; hlse2 f32 [B,H,N] host out, nullable
 *   ws          device scratch, 256-byte aligned, of at least
 *               vcattn_fwd_host_workspace_bytes(shape, k, chunk_heads) bytes
 *               (two slots of chunk_heads heads each)
 *   streams     four cudaStream_t: compute 0, compute 1 (may equal compute 0),
 *               copy in, copy out (these two distinct from all others)
 * The call's work starts after the work already enqueued on streams[0] (the
 * other three streams wait for it), and all of it is enqueued when the call
 * returns; streams[0] passes the end of the call only after the last copy
 * out, so synchronising it (or an event recorded on it afterwards) makes hO
 * and hlse2 valid, and consecutive calls may share one workspace.  The host
 * buffers must stay allocated and unchanged until then.  The call allocates
 * no device memory; it creates eleven CUDA events and releases them (each once
 * complete) before returning.  On an error return, part of the work may
 * already be enqueued. */
size_t vcattn_fwd_host_workspace_bytes(const vcattn_shape* shape, int k, int chunk_heads);
vcattn_status vcattn_fwd_host(const vcattn_shape* shape, const void* hQ, const void* hK,
                              const void* hV, int k, int iters, float sm_scale,
                              const uint8_t* tile_mask, void* hO, float* hlse2, int chunk_heads,
                              void* ws, size_t ws_bytes, void* const streams[4]);

/* ------------------------------------------------------------------ errors */
/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: VCATTN_OK, VCATTN_ERR_TIMEOUT or VCATTN_ERR_DEVICE (or
 * VCATTN_ERR_CUDA when the synchronisation itself fails). */
vcattn_status vcattn_last_device_error(void* stream);
const char* vcattn_status_string(vcattn_status s);
/* Test hook for the failure path (not part of the method): runs
 * vcattn_attn with its K/V loader switched off, so no tile ever arrives and
 * every bounded wait in the kernel (2 s each) runs out.  The kernel records
 * the timeout in the device error word and returns; O and lse2 are left
 * undefined, the context stays usable, and the next
 * vcattn_last_device_error() reports VCATTN_ERR_TIMEOUT.  Arguments as for
 * vcattn_attn (dense, no mask). */
vcattn_status vcattn_test_attn_stalled(const vcattn_shape* shape, const vcattn_prepped* in,
                                       float sm_scale, void* O, float* lse2, void* stream);
/* Test hook for the failure path while copies are in flight (not part of
 * the method): as vcattn_test_attn_stalled, but the K/V loader stops after
 * `steps` (>= 1) KV tiles, so the consumers give up part-way with loads and
 * MMAs already issued; the kernel drains what it issued before it exits and
 * records VCATTN_ERR_TIMEOUT.  tile_mask as for vcattn_attn (NULL: dense;
 * otherwise the block-sparse kernel, whose loaders walk each slot's own
 * tiles). */
vcattn_status vcattn_test_attn_stalled_after(const vcattn_shape* shape, const vcattn_prepped* in,
                                             float sm_scale, const uint8_t* tile_mask, int steps, void* O,
                                             float* lse2, void* stream);
/* Test hook for the k-means assignment's tensor-core filter (not part of the
 * method): one assign step of vcattn_group from the given centroids, with
 * the filter's inputs written out.  The tensor core computes an
 * approximation T_c of each token's FP32 score v . c_c - |c_c|^2 / 2; the
 * filter keeps the clusters within a bound E of the largest T_c and exact
 * FP32 chains decide among them, which is exact if |T_c - score_c| <= E / 2.
 *   V          bf16 [B,H,N,D] (device)
 *   centroids  f32 [B,H,k,D] (device), the centroids of the step
 *   labels     i32 [B,H,N] (device) out: the labels of this one step
 *   scores     f32 [B,H,N,65] (device) out: T_c for c < 64 (-inf for c >= k)
 *              and E at index 64, for every token
 *   ws         scratch of vcattn_group_workspace_bytes(shape, k) */
vcattn_status vcattn_test_km_scores(const vcattn_shape* shape, const void* V, int k, const float* centroids,
                                    int32_t* labels, float* scores, void* ws, size_t ws_bytes, void* stream);
/* Test hook for the byte-level check of ExpCast-FP8 (VC-Attention, Key
 * Contribution 2: the probability's E4M3 byte from one FMA and one integer
 * rounding of the max-subtracted log2 score).  Runs the attention kernel's
 * own ExpCast code on given scores: codes[i] is the byte the kernel writes
 * for score x[i] with coefficient A[i/4] and constant B[i/4] = C - m, i.e.
 * clip(rint(fmaf(x, A, B))) (rint: to nearest, ties to even) with codes
 * below 8 flushed to 0; a score of -inf marks an excluded key (byte 0).  The
 * kernel guarantees t = fmaf(x, A, B) <= C + tau8 < 126.5, so the clip at
 * 126 never binds inside that domain; outside it the bytes are not
 * specified.  x and codes hold n elements (n a multiple of 4, 16-byte
 * aligned device pointers); A and B hold n/4 (device).  Enqueued on
 * `stream`. */
vcattn_status vcattn_test_expcast(const float* x, const float* A, const float* B, uint8_t* codes, int64_t n,
                                  void* stream);
/* Text of the CUDA error behind the calling thread's most recent
 * VCATTN_ERR_CUDA (host side: a failed launch, attribute, tensor-map or
 * copy call); "no error" if there was none.  The string is static. */
const char* vcattn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* VCATTN_H */
