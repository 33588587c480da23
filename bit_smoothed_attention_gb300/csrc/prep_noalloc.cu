// vcattn_prep_noalloc: the preprocessing step for callers that cannot hand
// the library a scratch buffer.
//
// Some callers cannot allocate device memory at the point where they call
// the preprocessing: a plugin inside a framework or inference server that
// receives only its input and output tensors and has no allocator of its
// own, or a program that forbids device allocation after start-up (an
// allocation may synchronise the device, and it can fail under memory
// pressure in the middle of a run).  For them this entry point runs the same
// kernels as vcattn_prep, but its scratch (the K block sums and the V
// residual amax) lives in one file-scope device array that the library owns.
//
// Properties a user must know:
//  - The array is NOALLOC_SCRATCH_BYTES = 16 MiB.  Every GPU on which the
//    library is loaded holds it until the process exits.  A problem needs
//    256-byte-rounded B*H*(Npad/64)*128*4 + B*H*128*4 bytes; larger problems
//    are refused with VCATTN_ERR_UNSUPPORTED before any work is enqueued.
//  - The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, once per device, with that device current).
//    Make that first call before any stream capture begins.
//  - All calls on a device share the one array, and it keeps whatever the
//    last call left in it.  The part that must start at zero (the amax) is
//    cleared by every call on its stream before use.  Calls whose work
//    overlaps on the GPU (different streams, no ordering between them) race
//    on the array and give wrong results; order them on one stream.
//  - Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/vcattn.h"
#include "internal.h"

namespace vc {
vcattn_status from_cuda(cudaError_t e);             // records e for vcattn_last_cuda_error
uint32_t* device_error_word(vcattn_status* st);      // the library's device error word
}  // namespace vc

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = static_cast<size_t>(16) << 20;

// The scratch itself.  In host code this name is only a host-side stand-in:
// its device address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_prep_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEV = 64;
void* g_scratch_ptr[MAX_DEV];
std::mutex g_scratch_mu;

// Device address of g_prep_scratch on the current device (looked up once).
void* scratch_address(vcattn_status* st) {
  int dev = 0;
  const cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess || dev < 0 || dev >= MAX_DEV) {
    *st = e0 != cudaSuccess ? vc::from_cuda(e0) : VCATTN_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_prep_scratch);
    if (e != cudaSuccess || !p) {
      *st = vc::from_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" vcattn_status vcattn_prep_noalloc(const vcattn_shape* s, const void* Q, const void* K,
                                             const void* V, const int32_t* perm,
                                             const vcattn_prepped* out, void* stream) {
  if (!s) return VCATTN_ERR_INVALID_ARG;
  if (s->D != vc::D) return VCATTN_ERR_UNSUPPORTED;
  if (s->B < 1 || s->H < 1 || s->N < 1) return VCATTN_ERR_INVALID_ARG;
  if (s->N > (int64_t(1) << 30) || s->B * s->H > 65535) return VCATTN_ERR_UNSUPPORTED;
  if (!Q || !K || !V || !out || !al16(Q) || !al16(K) || !al16(V) || (perm && !al16(perm)))
    return VCATTN_ERR_INVALID_ARG;
  const void* parts[] = {out->q8, out->k8, out->r8t, out->q_scale, out->k_scale, out->v_scale,
                         out->k_mean, out->v_mean, out->qmu, out->vmu_op};
  for (const void* p : parts)
    if (!p || !al16(p)) return VCATTN_ERR_INVALID_ARG;
  const int64_t BH = s->B * s->H;
  if (vc::prep_ws_layout(BH, s->N, nullptr, nullptr) > NOALLOC_SCRATCH_BYTES)
    return VCATTN_ERR_UNSUPPORTED;  // more scratch than the built-in 16 MiB
  vcattn_status st = VCATTN_OK;
  void* base = scratch_address(&st);
  if (!base) return st;
  uint32_t* err = vc::device_error_word(&st);
  if (!err) return st;
  vc::PrepWs w{};
  vc::prep_ws_layout(BH, s->N, base, &w);
  const vc::PrepOut o{out->q8, out->k8, out->r8t, out->q_scale, out->k_scale, out->v_scale,
                      out->k_mean, out->v_mean, out->qmu, out->vmu_op};
  const vc::RowLayout lc = vc::contiguous_rows(s->H, s->N);
  const cudaError_t e = vc::launch_prep(static_cast<const uint16_t*>(Q), lc, static_cast<const uint16_t*>(K), lc,
                                        static_cast<const uint16_t*>(V), lc, perm, BH, s->N, o, w, err, 0,
                                        static_cast<cudaStream_t>(stream));
  return vc::from_cuda(e);
}
