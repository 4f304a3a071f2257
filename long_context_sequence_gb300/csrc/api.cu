// C-ABI layer: plan creation and validation, status handling, tensor-map encoding and
// the entry points declared in include/ulysses.h.  Every entry point validates its
// arguments on the host before anything is launched.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

thread_local char g_err[512] = "";

uly_status fail(uly_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

uly_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ULY_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(const char** err) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn && err) *err = "cuTensorMapEncodeTiled is not available from the driver";
  return fn;
}

}  // namespace

int num_sms(int device) {
  static int cached[64] = {0};
  if (device < 0 || device >= 64) return 148;
  if (!cached[device]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
      n = 148;
    cached[device] = n;
  }
  return cached[device];
}


bool make_tmap_3d_bf16(CUtensorMap* m, const void* base, const uint64_t dims_in[3],
                       const uint64_t strides_bytes[2], uint32_t box0, uint32_t box1,
                       const char** err) {
  EncodeTiledFn fn = encode_fn(err);
  if (!fn) return false;
  cuuint64_t dims[3] = {dims_in[0], dims_in[1], dims_in[2]};
  cuuint64_t strides[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled (3-D) rejected the layout";
    return false;
  }
  return true;
}

bool make_tmap_4d_bf16(CUtensorMap* m, const void* base, const uint64_t dims_in[4],
                       const uint64_t strides_bytes[3], uint32_t box0, uint32_t box2,
                       const char** err) {
  EncodeTiledFn fn = encode_fn(err);
  if (!fn) return false;
  cuuint64_t dims[4] = {dims_in[0], dims_in[1], dims_in[2], dims_in[3]};
  cuuint64_t strides[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t box[4] = {box0, 1, box2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled (4-D) rejected the layout";
    return false;
  }
  return true;
}

void make_view(const Plan& src, Plan& dst, int64_t S, int P, int H, int G) {
  dst.cfg = src.cfg;
  dst.cfg.seq_len = S;
  dst.cfg.P = P;
  dst.cfg.n_q_heads = H;
  dst.cfg.n_kv_heads = G;
  dst.device = src.device;
  dst.rank = -1;
  dst.S = S;
  dst.P = P;
  dst.hidden = src.hidden;
  dst.H = H;
  dst.G = G;
  dst.D = src.D;
  dst.scale = src.scale;
  dst.rope_hi = src.rope_hi;
  dst.rope_lo = src.rope_lo;
  dst.status = src.status;
  dst.limit_ns = src.limit_ns;
  dst.noalloc_scratch = src.noalloc_scratch;
  dst.noalloc_setup_error = src.noalloc_setup_error;
}

uly_status set_error(uly_status s, const char* msg) {
  if (s == ULY_OK) {
    g_err[0] = 0;
    return s;
  }
  return fail(s, "%s", msg);
}


}  // namespace uly

using uly::Plan;
using uly::aligned16;
using uly::fail;

namespace {

uly_status validate(const uly_config* c) {
  if (!c) return fail(ULY_ERR_INVALID_ARG, "config is NULL");
  if (c->reserved != 0) return fail(ULY_ERR_INVALID_ARG, "config.reserved must be 0");
  if (c->seq_len < 0) return fail(ULY_ERR_INVALID_ARG, "seq_len < 0");
  if (c->batch != 1) return fail(ULY_ERR_UNSUPPORTED, "batch must be 1 (got %d)", c->batch);
  if (c->causal != 1) return fail(ULY_ERR_UNSUPPORTED, "only causal attention is built");
  if (c->P < 1) return fail(ULY_ERR_INVALID_ARG, "P must be >= 1 (got %d)", c->P);
  if (c->n_q_heads < 1 || c->n_kv_heads < 1)
    return fail(ULY_ERR_INVALID_ARG, "head counts must be >= 1");
  if (c->n_q_heads % c->n_kv_heads)
    return fail(ULY_ERR_INVALID_ARG, "n_q_heads %% n_kv_heads != 0");
  if (c->n_q_heads % c->P) return fail(ULY_ERR_INVALID_ARG, "n_q_heads %% P != 0");
  if (c->n_kv_heads % c->P)
    return fail(ULY_ERR_UNSUPPORTED, "n_kv_heads %% P != 0 (KV-head replication is not built)");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(ULY_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", c->head_dim);
  if (c->hidden < 8 || c->hidden % 8)
    return fail(ULY_ERR_INVALID_ARG, "hidden must be a positive multiple of 8");
  if (c->seq_len % c->P) return fail(ULY_ERR_INVALID_ARG, "seq_len %% P != 0");
  if (c->seq_len > (int64_t(1) << 30))
    return fail(ULY_ERR_UNSUPPORTED, "seq_len above 2^30 is not supported");
  if ((int64_t)c->seq_len * (c->n_q_heads / c->P) / 128 > (int64_t(1) << 30))
    return fail(ULY_ERR_UNSUPPORTED, "grid too large");
  if (c->softmax_scale < 0 || !std::isfinite(c->softmax_scale))
    return fail(ULY_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (c->rope_theta < 0 || !std::isfinite(c->rope_theta))
    return fail(ULY_ERR_INVALID_ARG, "rope_theta must be finite and >= 0");
  if (c->wait_timeout_ms < 0) return fail(ULY_ERR_INVALID_ARG, "wait_timeout_ms < 0");
  if (c->flags & ~ULY_FLAG_INJECT_STALL) return fail(ULY_ERR_INVALID_ARG, "unknown flags");
  return ULY_OK;
}

uly_status build_rope(Plan& p) {
  const int half = p.D / 2;
  const int64_t n_hi = (p.S + uly::kRopeL - 1) / uly::kRopeL;
  std::vector<float2> hi((size_t)std::max<int64_t>(n_hi, 1) * half), lo((size_t)uly::kRopeL * half);
  const double theta = p.cfg.rope_theta;
  for (int i = 0; i < half; ++i) {
    const double w = std::pow(theta, -2.0 * i / p.D);
    for (int64_t sh = 0; sh < n_hi; ++sh) {
      const double a = (double)(sh * uly::kRopeL) * w;
      hi[(size_t)sh * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
    for (int sl = 0; sl < uly::kRopeL; ++sl) {
      const double a = (double)sl * w;
      lo[(size_t)sl * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  }
  cudaError_t e = cudaMalloc(&p.rope_hi, hi.size() * sizeof(float2));
  if (e != cudaSuccess) return fail(ULY_ERR_OOM, "RoPE table: %s", cudaGetErrorString(e));
  e = cudaMalloc(&p.rope_lo, lo.size() * sizeof(float2));
  if (e != cudaSuccess) return fail(ULY_ERR_OOM, "RoPE table: %s", cudaGetErrorString(e));
  e = cudaMemcpy(p.rope_hi, hi.data(), hi.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p.rope_lo, lo.data(), lo.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return uly::cuda_fail(e, "RoPE table upload");
  return ULY_OK;
}

void free_plan(uly_plan h) {
  if (!h) return;
  cudaFree(h->p.rope_hi);
  cudaFree(h->p.rope_lo);
  cudaFree(h->p.status);
  delete h;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

uly_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return uly::cuda_fail(e, what);
  uly::g_err[0] = 0;
  return ULY_OK;
}

uly_status reject_rank_plan(uly_plan plan, const char* what) {
  return fail(ULY_ERR_INVALID_ARG,
              "%s works on the single-GPU virtual ranks; a rank plan (rank %d) exchanges "
              "through ulysses_a2a_pack_* / ulysses_a2a_exchange / ulysses_a2a_unpack_*",
              what, plan->p.rank);
}

uly_status make_plan(const uly_config* cfg, int32_t rank, uly_plan* out) {
  if (!out) return fail(ULY_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  uly_status s = validate(cfg);
  if (s != ULY_OK) return s;
  if (rank < -1 || rank >= cfg->P)
    return fail(ULY_ERR_INVALID_ARG, "rank %d outside [0, P = %d)", rank, cfg->P);
  uly_plan h = new (std::nothrow) uly_plan_s;
  if (!h) return fail(ULY_ERR_OOM, "host allocation failed");
  Plan& p = h->p;
  p.cfg = *cfg;
  if (cudaGetDevice(&p.device) != cudaSuccess) {
    delete h;
    return fail(ULY_ERR_CUDA, "no CUDA device");
  }
  p.S = cfg->seq_len;
  p.P = cfg->P;
  p.hidden = cfg->hidden;
  p.H = cfg->n_q_heads;
  p.G = cfg->n_kv_heads;
  p.D = cfg->head_dim;
  p.scale = (float)(cfg->softmax_scale > 0 ? cfg->softmax_scale : 1.0 / std::sqrt((double)p.D));
  p.limit_ns = (uint64_t)(cfg->wait_timeout_ms > 0 ? cfg->wait_timeout_ms : 2000) * 1000000ull;
  cudaError_t e = cudaMalloc(&p.status, sizeof(int));
  if (e != cudaSuccess) {
    free_plan(h);
    return fail(ULY_ERR_OOM, "status word: %s", cudaGetErrorString(e));
  }
  e = cudaMemset(p.status, 0, sizeof(int));
  if (e != cudaSuccess) {
    free_plan(h);
    return uly::cuda_fail(e, "status word");
  }
  if (cfg->rope_theta > 0) {
    s = build_rope(p);
    if (s != ULY_OK) {
      free_plan(h);
      return s;
    }
  }
  // The allocation-free backward's scratch address, looked up here so that no call of
  // ulysses_attn_bwd_noalloc ever loads device code or allocates.  A failure only disables
  // that entry point (it reports the error); the rest of the plan works without it.
  uly::noalloc_setup(p);
  if (rank >= 0) {
    p.rank = rank;
    uly::make_view(p, h->heads, p.S, 1, p.H / p.P, p.G / p.P);
    uly::make_view(p, h->shard, p.S / p.P, p.P, p.H, p.G);
  }
  *out = h;
  uly::g_err[0] = 0;
  return ULY_OK;
}

}  // namespace

extern "C" {

uly_status ulysses_plan(const uly_config* cfg, uly_plan* out) {
  ULY_CALL_RANGE();
  return make_plan(cfg, -1, out);
}

uly_status ulysses_plan_rank(const uly_config* cfg, int32_t rank, uly_plan* out) {
  ULY_CALL_RANGE();
  if (rank < 0) return fail(ULY_ERR_INVALID_ARG, "rank must be >= 0 (got %d)", rank);
  return make_plan(cfg, rank, out);
}

uly_status ulysses_plan_destroy(uly_plan plan) {
  if (!plan) return ULY_OK;
  cudaDeviceSynchronize();
  free_plan(plan);
  return ULY_OK;
}

size_t ulysses_workspace_bytes(uly_plan plan) {
  if (!plan) return 0;
  return uly::bwd_workspace_bytes(uly::attn_view(plan), nullptr, nullptr);
}

uly_status ulysses_qkv_proj(uly_plan plan, const void* x, const void* w, void* qkv,
                            void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::rows_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!x || !w || !qkv) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(x) || !aligned16(w) || !aligned16(qkv))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if ((p.H + 2 * p.G) * p.D > (1 << 30))
    return fail(ULY_ERR_UNSUPPORTED, "projection width too large");
  return launched(uly::launch_qkv_gemm(p, x, w, qkv, as_stream(stream)), "qkv_proj launch");
}

uly_status ulysses_seq_to_head(uly_plan plan, const void* qkv_seq, int in_fp32, int apply_rope,
                               void* q, void* k, void* v, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  if (plan->p.rank >= 0) return reject_rank_plan(plan, "ulysses_seq_to_head");
  Plan& p = plan->p;
  if (p.S == 0) return ULY_OK;
  if (!qkv_seq || !q || !k || !v) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(qkv_seq) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (apply_rope && !(p.cfg.rope_theta > 0))
    return fail(ULY_ERR_INVALID_ARG, "apply_rope needs a plan with rope_theta > 0");
  const uint64_t n = (uint64_t)p.S * (p.H + 2 * p.G) * p.D;
  p.bytes_moved += n * (in_fp32 ? 4 : 2) + n * 2;
  return launched(uly::launch_seq_to_head(p, qkv_seq, in_fp32 != 0, apply_rope != 0, q, k, v,
                                          as_stream(stream)),
                  "seq_to_head launch");
}

static uly_status permute_heads(uly_plan plan, const void* in, int n_heads, void* out,
                                bool to_head, void* stream) {
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  if (plan->p.rank >= 0)
    return reject_rank_plan(plan, to_head ? "ulysses_seq_to_head_heads" : "ulysses_head_to_seq");
  Plan& p = plan->p;
  if (n_heads != p.H && n_heads != p.G)
    return fail(ULY_ERR_INVALID_ARG, "n_heads must be n_q_heads or n_kv_heads (got %d)", n_heads);
  if (p.S == 0) return ULY_OK;
  if (!in || !out) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(in) || !aligned16(out))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  p.bytes_moved += (uint64_t)p.S * n_heads * p.D * 2 * 2;
  return launched(uly::launch_permute_heads(p, in, n_heads, out, to_head, as_stream(stream)),
                  to_head ? "seq_to_head launch" : "head_to_seq launch");
}

uly_status ulysses_seq_to_head_heads(uly_plan plan, const void* x_seq, int n_heads, void* x_head,
                                     void* stream) {
  ULY_CALL_RANGE();
  return permute_heads(plan, x_seq, n_heads, x_head, true, stream);
}

uly_status ulysses_head_to_seq(uly_plan plan, const void* x_head, int n_heads, void* x_seq,
                               void* stream) {
  ULY_CALL_RANGE();
  return permute_heads(plan, x_head, n_heads, x_seq, false, stream);
}

uly_status ulysses_attn_fwd(uly_plan plan, const void* q, const void* k, const void* v, void* o,
                            void* o_lo, float* lse, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::attn_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!q || !k || !v || !o || !lse) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(o_lo))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  return launched(uly::launch_attn_fwd(p, q, k, v, o, o_lo, lse, as_stream(stream)),
                  "attn_fwd launch");
}

uly_status ulysses_attn_bwd(uly_plan plan, const void* q, const void* k, const void* v,
                            const void* o, const void* o_lo, const float* lse, const void* d_o,
                            void* dq, void* dk, void* dv, void* workspace, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::attn_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv || !workspace)
    return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  const void* ptrs[] = {q, k, v, o, o_lo, lse, d_o, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  return launched(uly::launch_attn_bwd(p, q, k, v, o, o_lo, lse, d_o, dq, dk, dv, workspace,
                                       as_stream(stream)),
                  "attn_bwd launch");
}

uly_status ulysses_head_to_seq_qkv(uly_plan plan, const void* dq, const void* dk, const void* dv,
                                   int apply_rope, void* dqkv_seq, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  if (plan->p.rank >= 0) return reject_rank_plan(plan, "ulysses_head_to_seq_qkv");
  Plan& p = plan->p;
  if (p.S == 0) return ULY_OK;
  if (!dq || !dk || !dv || !dqkv_seq) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dqkv_seq))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (apply_rope && !(p.cfg.rope_theta > 0))
    return fail(ULY_ERR_INVALID_ARG, "apply_rope needs a plan with rope_theta > 0");
  p.bytes_moved += (uint64_t)p.S * (p.H + 2 * p.G) * p.D * 4;
  return launched(uly::launch_head_to_seq_qkv(p, dq, dk, dv, apply_rope != 0, dqkv_seq,
                                              as_stream(stream)),
                  "head_to_seq_qkv launch");
}

uly_status ulysses_qkv_proj_bwd(uly_plan plan, const void* x, const void* w, const void* dqkv,
                                void* dx, float* dw, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::rows_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!x || !w || !dqkv) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(x) || !aligned16(w) || !aligned16(dqkv) || !aligned16(dx) || !aligned16(dw))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (p.S > (int64_t(1) << 31) - 1) return fail(ULY_ERR_UNSUPPORTED, "S too large");
  return launched(uly::launch_qkv_gemm_bwd(p, x, w, dqkv, dx, dw, as_stream(stream)),
                  "qkv_proj_bwd launch");
}

uly_status ulysses_o_proj(uly_plan plan, const void* o_head, const void* wo, void* y,
                          void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::rows_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!o_head || !wo || !y) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(o_head) || !aligned16(wo) || !aligned16(y))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (p.S > (int64_t(1) << 31) - 1) return fail(ULY_ERR_UNSUPPORTED, "S too large");
  return launched(uly::launch_o_proj(p, o_head, wo, y, as_stream(stream)), "o_proj launch");
}

uly_status ulysses_o_proj_bwd(uly_plan plan, const void* o_head, const void* wo, const void* dy,
                              void* do_head, float* dwo, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  const Plan& p = uly::rows_view(plan);
  if (p.S == 0) return ULY_OK;
  if (!o_head || !wo || !dy) return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(o_head) || !aligned16(wo) || !aligned16(dy) || !aligned16(do_head) ||
      !aligned16(dwo))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (p.S > (int64_t(1) << 31) - 1) return fail(ULY_ERR_UNSUPPORTED, "S too large");
  return launched(uly::launch_o_proj_bwd(p, o_head, wo, dy, do_head, dwo, as_stream(stream)),
                  "o_proj_bwd launch");
}

uly_status ulysses_sync_status(uly_plan plan, void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return uly::cuda_fail(e, "stream synchronize");
  int st = 0;
  e = cudaMemcpy(&st, plan->p.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return uly::cuda_fail(e, "status read");
  if (st != 0) {
    e = cudaMemset(plan->p.status, 0, sizeof(int));
    if (e != cudaSuccess) return uly::cuda_fail(e, "status clear");
    if (st == ULY_ERR_TIMEOUT)
      return fail(ULY_ERR_TIMEOUT, "a device-side wait ran past %llu ms",
                  (unsigned long long)(plan->p.limit_ns / 1000000ull));
    if (st == ULY_ERR_RANGE)
      return fail(ULY_ERR_RANGE, "an attention-backward input's largest magnitude is beyond "
                                 "the range its scaled fp16 copy can hold");
    return fail((uly_status)st, "device reported status %d", st);
  }
#ifdef ULY_DEBUG
  const unsigned int n_perm = uly::debug_bounds_failures_permute(),
                     n_fwd = uly::debug_bounds_failures_attn_fwd(),
                     n_bwd = uly::debug_bounds_failures_attn_bwd(),
                     n_gemm = uly::debug_bounds_failures_proj_gemm();
  if (n_perm + n_fwd + n_bwd + n_gemm)
    return fail(ULY_ERR_BOUNDS,
                "debug build: global accesses outside their buffers were skipped (permute %u, "
                "attn_fwd %u, attn_bwd %u, proj_gemm %u)",
                n_perm, n_fwd, n_bwd, n_gemm);
#endif
  uly::g_err[0] = 0;
  return ULY_OK;
}

uint64_t ulysses_bytes_moved(uly_plan plan) { return plan ? plan->p.bytes_moved.load() : 0; }

uly_status ulysses_a2a_volume(const uly_config* cfg, uint64_t* s2h, uint64_t* h2s) {
  uly_status s = validate(cfg);
  if (s != ULY_OK) return s;
  if (!s2h || !h2s) return fail(ULY_ERR_INVALID_ARG, "NULL output pointer");
  const uint64_t n = (uint64_t)(cfg->seq_len / cfg->P);
  const uint64_t D = (uint64_t)cfg->head_dim, P = (uint64_t)cfg->P;
  *s2h = n * (uint64_t)(cfg->n_q_heads + 2 * cfg->n_kv_heads) * D * 2 * (P - 1) / P;
  *h2s = n * (uint64_t)cfg->n_q_heads * D * 2 * (P - 1) / P;
  return ULY_OK;
}

size_t ulysses_ring_workspace_bytes(uly_plan plan) {
  if (!plan) return 0;
  return uly::ring_workspace_layout(plan->p).total;
}

uly_status ulysses_ring_attn_fwd(uly_plan plan, const void* q_seq, const void* k_seq,
                                 const void* v_seq, void* o_seq, float* lse, void* workspace,
                                 void* stream) {
  ULY_CALL_RANGE();
  if (!plan) return fail(ULY_ERR_INVALID_ARG, "plan is NULL");
  if (plan->p.rank >= 0) return reject_rank_plan(plan, "ulysses_ring_attn_fwd");
  Plan& p = plan->p;
  if (p.S == 0) return ULY_OK;
  if (!q_seq || !k_seq || !v_seq || !o_seq || !lse || !workspace)
    return fail(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q_seq) || !aligned16(k_seq) || !aligned16(v_seq) || !aligned16(o_seq) ||
      !aligned16(lse) || !aligned16(workspace))
    return fail(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const uint64_t shard = (uint64_t)(p.S / p.P) * p.G * p.D * 2;
  p.bytes_moved += (uint64_t)(p.P - 1) * p.P * shard * 2 * 2;   // K and V, read + write
  return launched(uly::launch_ring_attn(p, q_seq, k_seq, v_seq, o_seq, lse, workspace,
                                        as_stream(stream)),
                  "ring attention launch");
}

uly_status ulysses_ring_volume(const uly_config* cfg, uint64_t* bytes) {
  uly_status s = validate(cfg);
  if (s != ULY_OK) return s;
  if (!bytes) return fail(ULY_ERR_INVALID_ARG, "NULL output pointer");
  const uint64_t n = (uint64_t)(cfg->seq_len / cfg->P);
  *bytes = (uint64_t)(cfg->P - 1) * n * 2 * (uint64_t)cfg->n_kv_heads * (uint64_t)cfg->head_dim * 2;
  return ULY_OK;
}

const char* ulysses_last_error(void) { return uly::g_err; }

}  // extern "C"
