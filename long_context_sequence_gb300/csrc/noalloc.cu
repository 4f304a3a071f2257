// ulysses_attn_bwd_noalloc: the attention backward with its scratch held by the library.
//
// ulysses_attn_bwd needs a caller-provided workspace (an fp32 dQ accumulator, the fp32 row
// terms D_i and fp16 operand copies).  Some callers cannot hand one over: a host program
// that has given all of HBM to its own pool or caching allocator (a further cudaMalloc
// fails or fragments it), a latency-critical path that must not pay cudaMalloc's implicit
// device synchronisation, or a plain C caller that has no device allocator of its own.
// For them this entry point uses a fixed scratch array that lives in the library's own
// device memory.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes (64 MiB).  A GPU
// holds it from the moment this file's device code is loaded there until the process
// exits: with the CUDA runtime's default lazy module loading that is the first
// ulysses_plan on the device (which looks the array up, below), with eager loading the
// load of the library.  In host code the array's name only stands for it; its device
// address is looked up with cudaGetSymbolAddress in ulysses_plan, with the plan's device
// current, and kept in the plan.  The entry point itself therefore never allocates (no
// cudaMalloc, cudaFree, module load or allocating library call), its first call included.
// A plan does not survive a reset of its device (cudaDeviceReset): make a new one.
//
// All calls share the one array and it keeps the last call's contents: the backward's
// first kernels rewrite every byte they later read (the largest-magnitude slots are
// cleared, the dQ accumulator zeroed, D_i and the fp16 copies written), so nothing carries
// over from call to call.  Calls that overlap on the GPU (different streams, no ordering
// between them) race on the array: order them.
#include <cstdio>

#include "uly_internal.h"

namespace uly {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

namespace {
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// Set-up, called by ulysses_plan with the plan's device current: the array's device
// address on that device (loading this file's device code there if it is not yet loaded).
cudaError_t noalloc_setup(Plan& p) {
  void* addr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&addr, g_bwd_scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();   // not sticky: leave no error behind for the caller's next call
    p.noalloc_scratch = nullptr;
    p.noalloc_setup_error = e;
    return e;
  }
  p.noalloc_scratch = addr;
  p.noalloc_setup_error = cudaSuccess;
  return cudaSuccess;
}

}  // namespace uly

extern "C" uly_status ulysses_attn_bwd_noalloc(uly_plan plan, const void* q, const void* k,
                                               const void* v, const void* o, const void* o_lo,
                                               const float* lse, const void* d_o, void* dq,
                                               void* dk, void* dv, void* stream) {
  ULY_CALL_RANGE();
  using namespace uly;
  if (!plan) return set_error(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = attn_view(plan);
  if (p.S == 0) return set_error(ULY_OK, "");
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv)
    return set_error(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  const void* ptrs[] = {q, k, v, o, o_lo, lse, d_o, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr))
      return set_error(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const size_t need = bwd_workspace_bytes(p, nullptr, nullptr);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "this plan's backward needs %zu bytes of scratch; the built-in scratch holds "
             "%zu bytes (use ulysses_attn_bwd with a workspace)",
             need, kNoAllocScratchBytes);
    return set_error(ULY_ERR_UNSUPPORTED, msg);
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess)
    return set_error(ULY_ERR_CUDA, "cudaGetDevice failed (no usable CUDA device)");
  if (dev != p.device)
    return set_error(ULY_ERR_INVALID_ARG, "the plan's device is not the current device");
  if (!p.noalloc_scratch) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "the scratch array's address could not be looked up when the plan was made "
             "(cudaGetSymbolAddress: %s)",
             cudaGetErrorString(p.noalloc_setup_error));
    return set_error(ULY_ERR_CUDA, msg);
  }
  cudaError_t e = launch_attn_bwd(p, q, k, v, o, o_lo, lse, d_o, dq, dk, dv, p.noalloc_scratch,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc launch: %s", cudaGetErrorString(e));
    return set_error(ULY_ERR_CUDA, msg);
  }
  return set_error(ULY_OK, "");
}
