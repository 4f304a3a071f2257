// ulysses_attn_bwd_noalloc: the attention backward with its scratch held by the library.
//
// ulysses_attn_bwd needs a caller-provided workspace (an fp32 dQ accumulator and the fp32
// row terms D_i).  Some callers cannot hand one over: a host program that has given all of
// HBM to its own pool or caching allocator (a further cudaMalloc fails or fragments it), a
// latency-critical path that must not pay cudaMalloc's implicit device synchronisation,
// or a plain C caller that has no device allocator of its own.  For them this entry point
// uses a fixed scratch array that lives in the library's own device memory.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes (64 MiB): every GPU
// that loads the library holds it until the process exits.  In host code the array's name
// only stands for it; its device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made while that device is current.  Make that
// first call before any stream capture.  The entry point itself never allocates (no
// cudaMalloc, cudaFree or allocating library call).
//
// All calls share the one array and it keeps the last call's contents: the backward's
// first kernel rewrites every byte it later reads (zeroes the dQ accumulator, writes D_i),
// so nothing carries over from call to call.  Calls that overlap on the GPU (different
// streams, no ordering between them) race on the array: order them.
#include <cstdio>
#include <mutex>

#include "uly_internal.h"

namespace uly {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_bwd_scratch on `device` (which must be current).
cudaError_t scratch_address(int device, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace uly

extern "C" uly_status ulysses_attn_bwd_noalloc(uly_plan plan, const void* q, const void* k,
                                               const void* v, const void* o, const void* o_lo,
                                               const float* lse, const void* d_o, void* dq,
                                               void* dk, void* dv, void* stream) {
  using namespace uly;
  if (!plan) return set_error(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = plan->p;
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
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_error(ULY_ERR_CUDA, "no current CUDA device");
  if (dev != p.device)
    return set_error(ULY_ERR_INVALID_ARG, "the plan's device is not the current device");
  void* scratch = nullptr;
  cudaError_t e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the scratch array: %s",
             cudaGetErrorString(e));
    return set_error(ULY_ERR_CUDA, msg);
  }
  e = launch_attn_bwd(p, q, k, v, o, o_lo, lse, d_o, dq, dk, dv, scratch,
                      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc launch: %s", cudaGetErrorString(e));
    return set_error(ULY_ERR_CUDA, msg);
  }
  return set_error(ULY_OK, "");
}
