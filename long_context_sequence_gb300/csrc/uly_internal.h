// Internal declarations shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ulysses.h"

namespace uly {

// An NVTX range over one C-ABI call, named after the call: the calls show up as ranges in
// the Nsight tools, and ncu can select a call's kernels (--nvtx --nvtx-include "name/").
// Without a tool attached a range costs a few nanoseconds.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define ULY_CALL_RANGE() ::uly::CallRange uly_call_range_(__func__)

// RoPE angles are kept as a two-level table so that positions up to 2^20 and beyond
// need little memory: for s = sh * kRopeL + sl, (cos, sin)(s * w_i) is rebuilt from
// hi[sh][i] = (cos, sin)(sh * kRopeL * w_i) and lo[sl][i] = (cos, sin)(sl * w_i) by the
// angle-addition identities (fp64 on the host, fp32 in the table).
constexpr int kRopeL = 1024;

struct Plan {
  uly_config cfg;
  int device = 0;
  int rank = -1;               // >= 0: one real rank of a P-GPU group (ulysses_plan_rank)
  int64_t S = 0;
  int P = 1, hidden = 0, H = 0, G = 0, D = 0;
  float scale = 0.f;
  float2* rope_hi = nullptr;   // [ceil(S / kRopeL)][D/2]
  float2* rope_lo = nullptr;   // [kRopeL][D/2]
  int* status = nullptr;       // device status word
  uint64_t limit_ns = 0;
  std::atomic<uint64_t> bytes_moved{0};
  // Device address of the library's fixed backward scratch on this plan's device (looked up
  // when the plan is made), or null with the lookup's error.
  void* noalloc_scratch = nullptr;
  cudaError_t noalloc_setup_error = cudaSuccess;
};

// Looks up the fixed scratch array's device address for p (the plan's device current).
cudaError_t noalloc_setup(Plan& p);

// Records msg as the thread's last error (ULY_OK clears it) and returns s.
uly_status set_error(uly_status s, const char* msg);

// Launchers: each validates nothing (api.cu did) and returns the launch error.
// pos0: global position of the first token (RoPE); 0 but for one real rank's shard.
cudaError_t launch_seq_to_head(const Plan& p, const void* in, bool in_fp32, bool rope, void* q,
                               void* k, void* v, cudaStream_t st, int64_t pos0 = 0);
cudaError_t launch_permute_heads(const Plan& p, const void* in, int n_heads, void* out,
                                 bool to_head, cudaStream_t st);
cudaError_t launch_head_to_seq_qkv(const Plan& p, const void* dq, const void* dk,
                                   const void* dv, bool rope, void* out, cudaStream_t st,
                                   int64_t pos0 = 0);
cudaError_t launch_qkv_gemm(const Plan& p, const void* x, const void* w, void* out,
                            cudaStream_t st);
// y = o wo^T with o read in the head layout (bf16 [S][hidden]).
cudaError_t launch_o_proj(const Plan& p, const void* o_head, const void* wo, void* y,
                          cudaStream_t st);
// dO = dy wo written in the head layout and dwo = dy^T o (fp32 [hidden][H*D]).
cudaError_t launch_o_proj_bwd(const Plan& p, const void* o_head, const void* wo, const void* dy,
                              void* do_head, float* dwo, cudaStream_t st);
// dx = dqkv w (bf16 [S][hidden]) and dw = dqkv^T x (fp32 [C][hidden]); either may be null.
cudaError_t launch_qkv_gemm_bwd(const Plan& p, const void* x, const void* w, const void* dqkv,
                                void* dx, float* dw, cudaStream_t st);
cudaError_t launch_attn_fwd(const Plan& p, const void* q, const void* k, const void* v,
                            void* o, void* o_lo, float* lse, cudaStream_t st);
cudaError_t launch_attn_bwd(const Plan& p, const void* q, const void* k, const void* v,
                            const void* o, const void* o_lo, const float* lse,
                            const void* d_o, void* dq, void* dk, void* dv, void* workspace,
                            cudaStream_t st);

// Workspace layout of the backward pass (byte offsets, each 256-aligned): fp32 dQ
// accumulator, fp32 row terms, fp16 copies of q, dO, k, v, and 256 bytes for the call's
// largest magnitudes and power-of-two exponents.
// Ring attention: K/V ring buffers (two sets, the steps alternate), the fp32 output
// accumulator and the running max / sum of every row.
struct RingWorkspace {
  size_t k[2], v[2], acc, m, l, total;
};
RingWorkspace ring_workspace_layout(const Plan& p);
cudaError_t launch_ring_attn(const Plan& p, const void* q_seq, const void* k_seq,
                             const void* v_seq, void* o_seq, float* lse, void* workspace,
                             cudaStream_t st);

struct BwdWorkspace {
  size_t dq_acc, delta, q16, do16, k16, v16, scal, total;
};
BwdWorkspace bwd_workspace_layout(const Plan& p);
size_t bwd_workspace_bytes(const Plan& p, size_t* dq_acc_off, size_t* delta_off);

// Tensor maps (TMA descriptors), built on the host through the driver entry point.
// Returns false and sets *err on failure.
// 3-D bf16 map over [parts][rows][x] with byte strides {row, part} and a box of
// {box0, box1, 1}; 128-byte swizzle, out-of-range elements read as zero.
bool make_tmap_3d_bf16(CUtensorMap* m, const void* base, const uint64_t dims[3],
                       const uint64_t strides_bytes[2], uint32_t box0, uint32_t box1,
                       const char** err);
// 4-D bf16 map over [d3][d2][d1][d0] (d0 innermost) with byte strides s1, s2, s3 and a box
// of {box0, 1, box2, 1}; 128-byte swizzle, out-of-range elements read as zero.
bool make_tmap_4d_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], uint32_t box0, uint32_t box2,
                       const char** err);

int num_sms(int device);

#ifdef ULY_DEBUG
// Debug build: the out-of-bounds counters of the kernel files (read and cleared).
unsigned int debug_bounds_failures_permute();
unsigned int debug_bounds_failures_attn_fwd();
unsigned int debug_bounds_failures_attn_bwd();
unsigned int debug_bounds_failures_proj_gemm();
#endif

// Copies p's shared state into a view of other sizes (same device, tables, status word).
void make_view(const Plan& src, Plan& dst, int64_t S, int P, int H, int G);

}  // namespace uly

// The opaque handle of the C ABI.  For a rank plan, `heads` is the rank's head group over
// all S tokens as a one-rank plan (attention), `shard` its S/P tokens with the group's P
// ranks (projections, pack and unpack of the exchanges).
struct uly_plan_s {
  uly::Plan p;
  uly::Plan heads;
  uly::Plan shard;
};

namespace uly {
// The view an entry point works on.
inline const Plan& attn_view(const uly_plan_s* h) { return h->p.rank >= 0 ? h->heads : h->p; }
inline const Plan& rows_view(const uly_plan_s* h) { return h->p.rank >= 0 ? h->shard : h->p; }
}  // namespace uly
