// The two all-to-alls of the Ulysses block as on-device permutations (virtual ranks are
// slices of one GPU's memory).
//
// "Snowflake's Ulysses trick ..." para 2: after the local QKV projection an all-to-all
// leaves every rank the full sequence for a subset of heads; another all-to-all restores
// the sequence sharding ("Ulysses Sequence Parallelism: Training with Million-Token
// Contexts", para 5).  The kernels move 16-byte vectors; for every token the source row
// is contiguous and the destination runs are (heads per rank) * D * 2 bytes long, so both
// sides stay coalesced.  The memory-bound roofline is read + write bytes / HBM bandwidth.
// The q/k/v kernels, which may apply RoPE, give each thread one 8-pair chunk of one token
// across all its heads, so the token's angles are built once, not once per head.
//
// The same kernels serve one real rank of a multi-GPU group: run over the rank's own S/P
// tokens (S := S/P) with the RoPE positions offset by the shard's first global token
// (pos0), seq->head writes the P per-peer send blocks [P][S/P][heads/P][D] of an
// all-to-all, and head->seq turns the P received blocks back into the shard's rows.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int kThreads = 256;
constexpr int kTokensPerBlock = 16;

struct RopeTab {
  const float2* hi;
  const float2* lo;
  int half;  // D / 2
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  return v;
}

// 8 consecutive elements of a row, as fp32.
template <bool kFp32>
__device__ __forceinline__ void load8(const void* row, int elem, float (&f)[8], uint4& raw) {
  if constexpr (kFp32) {
    const float* p = reinterpret_cast<const float*>(row) + elem;
    uint4 a = ld_stream(p), b = ld_stream(p + 4);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  } else {
    raw = ld_stream(reinterpret_cast<const __nv_bfloat16*>(row) + elem);
    unpack8(raw, f);
  }
}

// RoPE angles of one token for the 8 pairs (e, e + D/2), e = e0 .. e0 + 7: (cos, sin) of
// s * theta^(-2e/D), rebuilt from the two-level table by angle addition (hi: multiples of
// kRopeL positions, lo: the remainder).  The angles depend on the token and the pair only,
// so a thread computes them once and applies them to every rotated head of its token.
__device__ __forceinline__ void rope_angles8(const RopeTab& rope, int64_t s, int e0,
                                             float (&cs)[8], float (&sn)[8]) {
  const int64_t sh = s / kRopeL;
  const int sl = (int)(s - sh * kRopeL);
  const float2* th = rope.hi + sh * rope.half + e0;
  const float2* tl = rope.lo + (int64_t)sl * rope.half + e0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = __ldg(th + i), b = __ldg(tl + i);
    cs[i] = fmaf(a.x, b.x, -a.y * b.y);
    sn[i] = fmaf(a.y, b.x, a.x * b.y);
  }
}

// Thread <-> (token, chunk): a block covers kThreads / (D/16) tokens; a thread owns the
// elements [8u, 8u+8) and their RoPE partners [D/2 + 8u, D/2 + 8u + 8) of every head row of
// its token.  Per head it moves 2 x 16 bytes in and out (a warp: 4 tokens x 128-byte runs
// at D = 128).
struct TokenChunk {
  int64_t s;
  int cu;
  bool valid;
};
__device__ __forceinline__ TokenChunk token_chunk(int64_t b, int upr, int64_t S) {
  const int tpb = kThreads / upr;
  const int t = threadIdx.x / upr;
  TokenChunk r;
  r.s = b * tpb + t;
  r.cu = threadIdx.x - t * upr;
  r.valid = t < tpb && r.s < S;
  return r;
}

// seq->head with the q/k/v split, optional fp32 input and optional RoPE on q and k.
template <bool kFp32In, bool kRope>
__global__ void __launch_bounds__(kThreads) seq_to_head_kernel(
    const void* __restrict__ in, __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
    __nv_bfloat16* __restrict__ v, int64_t S, int P, int H, int G, int D, RopeTab rope,
    int64_t pos0) {
  const int C = H + 2 * G;
  const int upr = D / 16;
  const int hq = H / P, hk = G / P;
  const int64_t n_blocks = (S + kThreads / upr - 1) / (kThreads / upr);
  const size_t esz = kFp32In ? 4 : 2;
  const uint64_t ext_in = (uint64_t)S * C * D, ext_q = (uint64_t)P * S * hq * D,
                 ext_kv = (uint64_t)P * S * hk * D;   // element extents (debug checks)
  (void)ext_in; (void)ext_q; (void)ext_kv;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
    const TokenChunk tc = token_chunk(b, upr, S);
    if (!tc.valid) continue;
    const int64_t s = tc.s;
    const int e_lo = tc.cu * 8, e_hi = D / 2 + tc.cu * 8;
    float cs[8], sn[8];
    if (kRope) rope_angles8(rope, pos0 + s, e_lo, cs, sn);
    const char* row = reinterpret_cast<const char*>(in) + (size_t)s * C * D * esz;
#pragma unroll 2
    for (int c = 0; c < C; ++c) {
      const char* src = row + (size_t)c * D * esz;
      __nv_bfloat16* dst;
      size_t doff;
      uint64_t dext;
      if (c < H) {
        const int r2 = c / hq, hh = c - r2 * hq;
        doff = (((size_t)r2 * S + s) * hq + hh) * D;
        dst = q + doff;
        dext = ext_q;
      } else if (c < H + G) {
        const int g = c - H, r2 = g / hk, hh = g - r2 * hk;
        doff = (((size_t)r2 * S + s) * hk + hh) * D;
        dst = k + doff;
        dext = ext_kv;
      } else {
        const int g = c - H - G, r2 = g / hk, hh = g - r2 * hk;
        doff = (((size_t)r2 * S + s) * hk + hh) * D;
        dst = v + doff;
        dext = ext_kv;
      }
      (void)doff; (void)dext;
      const size_t soff = ((size_t)s * C + c) * D;
      (void)soff;
      if (!ULY_IN_BOUNDS(soff + e_lo, 8, ext_in) || !ULY_IN_BOUNDS(soff + e_hi, 8, ext_in) ||
          !ULY_IN_BOUNDS(doff + e_lo, 8, dext) || !ULY_IN_BOUNDS(doff + e_hi, 8, dext))
        continue;
      float lo[8], hi[8];
      uint4 raw_lo, raw_hi;
      load8<kFp32In>(src, e_lo, lo, raw_lo);
      load8<kFp32In>(src, e_hi, hi, raw_hi);
      if (kRope && c < H + G) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x0 = lo[i], x1 = hi[i];
          lo[i] = fmaf(x0, cs[i], -x1 * sn[i]);
          hi[i] = fmaf(x1, cs[i], x0 * sn[i]);
        }
        st_stream(dst + e_lo, pack8(lo));
        st_stream(dst + e_hi, pack8(hi));
      } else if (kFp32In) {
        st_stream(dst + e_lo, pack8(lo));
        st_stream(dst + e_hi, pack8(hi));
      } else {
        st_stream(dst + e_lo, raw_lo);
        st_stream(dst + e_hi, raw_hi);
      }
    }
  }
}

// Inverse of seq_to_head for the gradients: dq [P][S][H/P][D], dk, dv [P][S][G/P][D] ->
// dqkv [S][H + 2G][D], with the RoPE backward on the q and k parts (each pair turned back
// by its angle: lo' = lo cos + hi sin, hi' = hi cos - lo sin).  Same thread mapping.
template <bool kRope>
__global__ void __launch_bounds__(kThreads) head_to_seq_qkv_kernel(
    const __nv_bfloat16* __restrict__ dq, const __nv_bfloat16* __restrict__ dk,
    const __nv_bfloat16* __restrict__ dv, __nv_bfloat16* __restrict__ out, int64_t S, int P,
    int H, int G, int D, RopeTab rope, int64_t pos0) {
  const int C = H + 2 * G;
  const int upr = D / 16;
  const int hq = H / P, hk = G / P;
  const int64_t n_blocks = (S + kThreads / upr - 1) / (kThreads / upr);
  const uint64_t ext_out = (uint64_t)S * C * D, ext_q = (uint64_t)P * S * hq * D,
                 ext_kv = (uint64_t)P * S * hk * D;   // element extents (debug checks)
  (void)ext_out; (void)ext_q; (void)ext_kv;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
    const TokenChunk tc = token_chunk(b, upr, S);
    if (!tc.valid) continue;
    const int64_t s = tc.s;
    const int e_lo = tc.cu * 8, e_hi = D / 2 + tc.cu * 8;
    float cs[8], sn[8];
    if (kRope) rope_angles8(rope, pos0 + s, e_lo, cs, sn);
    __nv_bfloat16* row = out + (size_t)s * C * D;
#pragma unroll 2
    for (int c = 0; c < C; ++c) {
      const __nv_bfloat16* src;
      size_t soff;
      uint64_t sext;
      if (c < H) {
        const int r2 = c / hq, hh = c - r2 * hq;
        soff = (((size_t)r2 * S + s) * hq + hh) * D;
        src = dq + soff;
        sext = ext_q;
      } else if (c < H + G) {
        const int g = c - H, r2 = g / hk, hh = g - r2 * hk;
        soff = (((size_t)r2 * S + s) * hk + hh) * D;
        src = dk + soff;
        sext = ext_kv;
      } else {
        const int g = c - H - G, r2 = g / hk, hh = g - r2 * hk;
        soff = (((size_t)r2 * S + s) * hk + hh) * D;
        src = dv + soff;
        sext = ext_kv;
      }
      (void)soff; (void)sext;
      __nv_bfloat16* dst = row + (size_t)c * D;
      const size_t doff = ((size_t)s * C + c) * D;
      (void)doff;
      if (!ULY_IN_BOUNDS(soff + e_lo, 8, sext) || !ULY_IN_BOUNDS(soff + e_hi, 8, sext) ||
          !ULY_IN_BOUNDS(doff + e_lo, 8, ext_out) || !ULY_IN_BOUNDS(doff + e_hi, 8, ext_out))
        continue;
      const uint4 raw_lo = ld_stream(src + e_lo), raw_hi = ld_stream(src + e_hi);
      if (kRope && c < H + G) {
        float lo[8], hi[8];
        unpack8(raw_lo, lo);
        unpack8(raw_hi, hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x0 = lo[i], x1 = hi[i];
          lo[i] = fmaf(x0, cs[i], x1 * sn[i]);
          hi[i] = fmaf(x1, cs[i], -x0 * sn[i]);
        }
        st_stream(dst + e_lo, pack8(lo));
        st_stream(dst + e_hi, pack8(hi));
      } else {
        st_stream(dst + e_lo, raw_lo);
        st_stream(dst + e_hi, raw_hi);
      }
    }
  }
}

// One tensor of n heads: seq layout [S][n][D] <-> head layout [P][S][n/P][D].
// Iterates over the seq side (contiguous); the head side is written/read in runs of
// (n/P) * D elements.
template <bool kToHead>
__global__ void __launch_bounds__(kThreads) permute_heads_kernel(
    const __nv_bfloat16* __restrict__ in, __nv_bfloat16* __restrict__ out, int64_t S, int P,
    int n, int D) {
  const int upr = D / 8;
  const int U = n * upr;
  const int hl = n / P;
  const int64_t n_blocks = (S + kTokensPerBlock - 1) / kTokensPerBlock;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
    const int64_t s0 = b * kTokensPerBlock;
    const int ntok = (int)(S - s0 < kTokensPerBlock ? S - s0 : kTokensPerBlock);
    for (int w = threadIdx.x; w < ntok * U; w += kThreads) {
      const int tl = w / U;
      const int unit = w - tl * U;
      const int h = unit / upr;
      const int e = (unit - h * upr) * 8;
      const int64_t s = s0 + tl;
      const int r2 = h / hl, hh = h - r2 * hl;
      const size_t seq_off = ((size_t)s * n + h) * D + e;
      const size_t head_off = (((size_t)r2 * S + s) * hl + hh) * D + e;
      if (!ULY_IN_BOUNDS(seq_off, 8, (uint64_t)S * n * D) ||
          !ULY_IN_BOUNDS(head_off, 8, (uint64_t)S * n * D))
        continue;
      if (kToHead)
        st_stream(out + head_off, ld_stream(in + seq_off));
      else
        st_stream(out + seq_off, ld_stream(in + head_off));
    }
  }
}

int permute_grid(const Plan& p, int64_t S) {
  const int64_t blocks = (S + kTokensPerBlock - 1) / kTokensPerBlock;
  const int64_t cap = (int64_t)num_sms(p.device) * 8;
  return (int)(blocks < cap ? blocks : cap);
}

// Grid of the token-chunk kernels (kThreads / (D/16) tokens per block).
int token_chunk_grid(const Plan& p, int64_t S) {
  const int64_t tpb = kThreads / (p.D / 16);
  const int64_t blocks = (S + tpb - 1) / tpb;
  const int64_t cap = (int64_t)num_sms(p.device) * 8;
  return (int)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_seq_to_head(const Plan& p, const void* in, bool in_fp32, bool rope, void* q,
                               void* k, void* v, cudaStream_t st, int64_t pos0) {
  const int grid = token_chunk_grid(p, p.S);
  RopeTab tab{p.rope_hi, p.rope_lo, p.D / 2};
  auto* qb = static_cast<__nv_bfloat16*>(q);
  auto* kb = static_cast<__nv_bfloat16*>(k);
  auto* vb = static_cast<__nv_bfloat16*>(v);
  if (in_fp32 && rope)
    seq_to_head_kernel<true, true><<<grid, kThreads, 0, st>>>(in, qb, kb, vb, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  else if (in_fp32)
    seq_to_head_kernel<true, false><<<grid, kThreads, 0, st>>>(in, qb, kb, vb, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  else if (rope)
    seq_to_head_kernel<false, true><<<grid, kThreads, 0, st>>>(in, qb, kb, vb, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  else
    seq_to_head_kernel<false, false><<<grid, kThreads, 0, st>>>(in, qb, kb, vb, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  return cudaGetLastError();
}

cudaError_t launch_head_to_seq_qkv(const Plan& p, const void* dq, const void* dk,
                                   const void* dv, bool rope, void* out, cudaStream_t st,
                                   int64_t pos0) {
  const int grid = token_chunk_grid(p, p.S);
  RopeTab tab{p.rope_hi, p.rope_lo, p.D / 2};
  auto* a = static_cast<const __nv_bfloat16*>(dq);
  auto* b = static_cast<const __nv_bfloat16*>(dk);
  auto* c = static_cast<const __nv_bfloat16*>(dv);
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (rope)
    head_to_seq_qkv_kernel<true><<<grid, kThreads, 0, st>>>(a, b, c, o, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  else
    head_to_seq_qkv_kernel<false><<<grid, kThreads, 0, st>>>(a, b, c, o, p.S, p.P, p.H, p.G, p.D, tab, pos0);
  return cudaGetLastError();
}

cudaError_t launch_permute_heads(const Plan& p, const void* in, int n_heads, void* out,
                                 bool to_head, cudaStream_t st) {
  const int grid = permute_grid(p, p.S);
  auto* i = static_cast<const __nv_bfloat16*>(in);
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (to_head)
    permute_heads_kernel<true><<<grid, kThreads, 0, st>>>(i, o, p.S, p.P, n_heads, p.D);
  else
    permute_heads_kernel<false><<<grid, kThreads, 0, st>>>(i, o, p.S, p.P, n_heads, p.D);
  return cudaGetLastError();
}

ULY_DEBUG_COUNTER_READER(permute)

}  // namespace uly
