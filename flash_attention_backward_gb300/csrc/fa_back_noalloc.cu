// fa_back_noalloc(): the backward for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: graph executors that own every device
// buffer through their own pool and expose no scratch pointer to an operator, and services
// that allocate nothing once they are set up.  This entry point serves them from one file-scope
// device array of FA_NOALLOC_SCRATCH_BYTES, resident on every GPU that loads the library until
// the process exits.  It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
// routine.  The launch sequence is fa_back()'s, given that array as its workspace.
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current context.  In host code the array's name
// is only a host-side stand-in, so the address is looked up on every call, with the caller's
// device current: a context that was reset or replaced since an earlier call may have loaded
// the module, and the array with it, at another address.
void* scratch_here(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  return *err == cudaSuccess ? p : nullptr;
}

}  // namespace

extern "C" fa_status fa_back_noalloc(const float* q, const void* k, int k_type, const void* v, int v_type,
                                     const uint16_t* mask, int mask_heads, const float* dO, float scale, int N,
                                     int M, int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK,
                                     float* dV, float* lse, float* delta, void* stream) {
  // the plan takes fewer key splits where that keeps the workspace within the scratch
  const size_t need = fab_workspace_size_capped(N, M, H, Hkv, D, Dv, kScratchBytes);
  if (need > kScratchBytes) return FA_ERR_WORKSPACE;  // larger than the static scratch
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_here(&err);
  if (!scratch) return FA_ERR_CUDA;
  return fab_back_capped(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dQ, dK,
                         dV, lse, delta, scratch, kScratchBytes, stream, kScratchBytes, nullptr, nullptr, nullptr,
                         nullptr);
}
