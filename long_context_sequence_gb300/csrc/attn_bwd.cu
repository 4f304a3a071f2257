// Backward of the per-head-group causal GQA attention (the training step of the block:
// "Ulysses Sequence Parallelism: Training with Million-Token Contexts" para 1 is about
// training; heads stay independent, "Snowflake's Ulysses trick ..." para 2).
//
// With P_ij = exp(scale q_i.k_j - lse_i) (j <= i), D_i = dO_i . o_i:
//   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
//   dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j,
// dK/dV summed over the query heads that share a KV head.
//
// Three kernels:
//   bwd_pre   D_i = rowsum(dO * O) in fp32 and zeroing of the fp32 dQ accumulator;
//   bwd_main  one CTA per (rank, KV head, 128-key block), looping over the query heads of
//             the group and the causally visible 128-row query tiles:
//               S^T  = K Q_i^T, dP^T = V dO_i^T          (tcgen05, TMEM, M = keys)
//               P^T, dS^T per key row on 4 warps -> TMEM (bf16) and dS -> smem
//               dV += P^T dO_i, dK += dS^T Q_i           (A operand from TMEM)
//               dQ_i = dS K -> TMEM -> fp32 vector reductions into the accumulator;
//   bwd_dq    fp32 dQ accumulator -> bf16.
// dS is kept as hi + lo bf16 parts for dK (hi in the smem tile that also feeds dQ, lo in
// TMEM), so the long dK sums see dS to ~16 bits.
// TMEM (512 columns): S^T [0,128) (P^T bf16 over [0,64)), dP^T [128,256) (dS^T lo part,
// bf16, over [128,192)), dV [256,256+D), dK [256+D,256+2D); dQ goes to [64,128), [192,256).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int BM = 128;  // query rows per item
constexpr int BN = 128;  // keys per CTA
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 128 * 64 * 2;

template <int D>
struct BwdLayout {
  static constexpr int kTile = (D / 64) * kBox;   // [128][D] bf16
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;             // [2] stages
  static constexpr int kDO = 4 * kTile;            // [2] stages
  static constexpr int kDS = 6 * kTile;            // [128 keys][128 q] bf16 = 2 boxes
  static constexpr int kDSBytes = 2 * kBox;
  static constexpr int kRow = kDS + kDSBytes;      // lse2[2][128], delta[2][128] fp32
  static constexpr int kBar = kRow + 4 * 128 * 4;
  static constexpr int kBytes = kBar + 256;
};

struct BwdArgs {
  const float* lse;
  const float* delta;
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int S, hl, gl, group, nkb;
  float scale, scale_log2;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {   // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(a.status, kOk, kErrUnsupported);
    return;
  }
  float* lse_s = reinterpret_cast<float*>(smem + L::kRow);   // [2][128]
  float* dlt_s = lse_s + 256;                                  // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* qd_full = bars + 1;    // [2]
  uint64_t* qd_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* dq_full = bars + 7;
  uint64_t* dq_free = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int per_rank = a.gl * a.nkb;
  const int r = blockIdx.x / per_rank;
  const int rem = blockIdx.x - r * per_rank;
  const int gg = rem / a.nkb;
  const int nb = rem - gg * a.nkb;           // key block; nb = 0 (most work) first
  const int nq = (a.S + BM - 1) / BM;
  const int n_items = a.group * (nq - nb);   // (query tile, head of the group) pairs

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtl wc{a.status, abort_flag, a.limit_ns};

  if (warp == kTmaWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_4d(smem + L::kK + b * kBox, &tm_k, kv_full, 64 * b, gg, nb * BN, r);
        tma_load_4d(smem + L::kV + b * kBox, &tm_v, kv_full, 64 * b, gg, nb * BN, r);
      }
      int issued = 0;
      for (int it = 0; it < n_items; ++it) {
        const int st = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const int i = nb + it / a.group;
        const int hh = gg * a.group + it % a.group;
        if (it >= 2 && !mbar_wait(&qd_empty[st], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&qd_full[st], 2 * L::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_4d(smem + L::kQ + st * L::kTile + b * kBox, &tm_q, &qd_full[st], 64 * b, hh,
                      i * BM, r);
          tma_load_4d(smem + L::kDO + st * L::kTile + b * kBox, &tm_do, &qd_full[st], 64 * b,
                      hh, i * BM, r);
        }
        ++issued;
      }
      mbar_drain(kv_full, 0, a.limit_ns);
      for (int it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
        mbar_drain(&qd_full[it & 1], (it >> 1) & 1, a.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BN, BM, false, false);   // M keys, N q
      constexpr uint32_t idesc_kv = idesc_bf16(BN, D, false, true);    // A tmem, B MN-major
      constexpr uint32_t idesc_q = idesc_bf16(BM, 64, true, true);     // dS, K both MN-major
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      const uint32_t sDS = smem_u32(smem + L::kDS);
      bool alive = mbar_wait(kv_full, 0, wc);
      for (int it = 0; alive && it < n_items; ++it) {
        const int st = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const uint32_t sQ = smem_u32(smem + L::kQ + st * L::kTile);
        const uint32_t sDO = smem_u32(smem + L::kDO + st * L::kTile);
        if (!mbar_wait(&qd_full[st], ph, wc)) break;
        if (it >= 1 && !mbar_wait(dq_free, (it - 1) & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBox + (kk % 4) * 32;
          mma_ss(tbase + 0, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBox + (kk % 4) * 32;
          mma_ss(tbase + 128, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (!mbar_wait(p_full, it & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ts(tbase + 256, tbase + 0 + kk * 8, sdesc_sw128(sDO + kk * 2048, kBox, 1024),
                 idesc_kv, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q with dS = hi + lo: hi from the smem tile (K-major A operand),
        // lo from TMEM, so dK sees dS to about 16 bits instead of 8.
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ss(tbase + 256 + D, sdesc_sw128(sDS + (kk / 4) * kBox + (kk % 4) * 32, 16, 1024),
                 sdesc_sw128(sQ + kk * 2048, kBox, 1024), idesc_kv,
                 (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ts(tbase + 256 + D, tbase + 128 + kk * 8, sdesc_sw128(sQ + kk * 2048, kBox, 1024),
                 idesc_kv, 1u);
#pragma unroll
        for (int half = 0; half < D / 64; ++half)
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(tbase + (half ? 192 : 64), sdesc_sw128(sDS + kk * 2048, kBox, 1024),
                   sdesc_sw128(sK + half * kBox + kk * 2048, kBox, 1024), idesc_q,
                   kk > 0 ? 1u : 0u);
        mma_commit(dq_full);
        mma_commit(&qd_empty[st]);
      }
      mma_commit(drain);
      mbar_drain(drain, 0, a.limit_ns);
    }
  } else {
    // Compute warpgroup: thread = key row (TMEM lane) for S^T/dP^T, = query row for dQ.
    const int row = warp * 32 + lane;
    const int key_g = nb * BN + row;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    uint8_t* sDS = smem + L::kDS;
    bool ok = true;
    for (int it = 0; it < n_items; ++it) {
      const int i = nb + it / a.group;
      const int hh = gg * a.group + it % a.group;
      const int q_g = i * BM + row;              // this thread's query column / dQ row
      float* lse_b = lse_s + (it & 1) * 128;
      float* dlt_b = dlt_s + (it & 1) * 128;
      const size_t rowterm = ((size_t)r * a.hl + hh) * a.S + q_g;
      lse_b[row] = q_g < a.S ? a.lse[rowterm] * 1.4426950408889634f : INFINITY;
      dlt_b[row] = q_g < a.S ? a.delta[rowterm] : 0.f;
      named_bar_sync(1, 128);
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, it & 1, wc));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tbase + lane_off + 32 * c, sv);
        tmem_ld32(tbase + lane_off + 128 + 32 * c, dp);
        uint32_t pk[16], dk[16], lo[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float pv[2], dv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ql = 32 * c + 2 * u + e;
            const int qg = i * BM + ql;
            const bool valid = key_g <= qg && qg < a.S && key_g < a.S;
            const float p = valid ? ex2_approx(fmaf(__uint_as_float(sv[2 * u + e]), sl2, -lse_b[ql]))
                                  : 0.f;
            pv[e] = p;
            dv[e] = p * (__uint_as_float(dp[2 * u + e]) - dlt_b[ql]);
          }
          pk[u] = pack_bf16x2(pv[0], pv[1]);
          dk[u] = pack_bf16x2(dv[0], dv[1]);          // dS rounded to bf16 (hi part)
          const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&dk[u]);
          const float2 hf = __bfloat1622float2(hi);
          lo[u] = pack_bf16x2(dv[0] - hf.x, dv[1] - hf.y);   // what the rounding lost
        }
        tmem_st16(tbase + lane_off + 16 * c, pk);
        tmem_st16(tbase + lane_off + 128 + 16 * c, lo);
        // dS tile in smem: [key row][q], 64-column atoms of 128-byte swizzled rows.
        uint8_t* atom = sDS + (c / 2) * kBox + row * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = (c % 2) * 4 + u;
          uint4 v = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
          *reinterpret_cast<uint4*>(atom + ((chunk ^ (row & 7)) * 16)) = v;
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, wc));
      if (!ok) break;
      tc_fence_after();
      float* dq_row = a.dq_acc + (((size_t)r * a.S + q_g) * a.hl + hh) * D;
#pragma unroll 1
      for (int half = 0; half < D / 64; ++half) {
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + (half ? 192 : 64) + 32 * c2, v);
          if (q_g < a.S) {
            float* dst = dq_row + half * 64 + c2 * 32;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v4(dst + 4 * j, __uint_as_float(v[4 * j]) * a.scale,
                         __uint_as_float(v[4 * j + 1]) * a.scale,
                         __uint_as_float(v[4 * j + 2]) * a.scale,
                         __uint_as_float(v[4 * j + 3]) * a.scale);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(dq_free);
    }
    // dK, dV of this key block (complete: the last dq_full covered every MMA).
    if (ok && n_items > 0) {
      tc_fence_after();
      const size_t out_off = (((size_t)r * a.S + key_g) * a.gl + gg) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = (which ? a.dk : a.dv) + out_off;
        const float mul = which ? a.scale : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + 256 + which * D + 32 * c, v);
          if (key_g < a.S) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * mul, __uint_as_float(v[8 * j + 1]) * mul);
              o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * mul, __uint_as_float(v[8 * j + 3]) * mul);
              o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * mul, __uint_as_float(v[8 * j + 5]) * mul);
              o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * mul, __uint_as_float(v[8 * j + 7]) * mul);
              *reinterpret_cast<uint4*>(dst + 32 * c + 8 * j) = o;
            }
          }
        }
      }
    } else if (ok && key_g < a.S) {
      // No visible query rows (cannot happen for key_g < S, kept for safety): zero grads.
      for (int d = 0; d < D; ++d) {
        a.dk[(((size_t)r * a.S + key_g) * a.gl + gg) * D + d] = __float2bfloat16_rn(0.f);
        a.dv[(((size_t)r * a.S + key_g) * a.gl + gg) * D + d] = __float2bfloat16_rn(0.f);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// D_i = sum_d dO_i[d] * O_i[d] (fp32) and zeroing of the dQ accumulator rows.
// 16 threads per row of D = 128 (8 bf16 each), 8 per row of D = 64.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ d_o,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ dq_acc, int64_t rows,
                                                      int64_t S, int hl) {
  constexpr int TPR = D / 8;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rowid = tid / TPR;       // row in [P][S][hl] order
  const int part = (int)(tid % TPR);
  float acc = 0.f;
  if (rowid < rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + rowid * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(d_o + rowid * D + part * 8);
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(ha[i]), y = __bfloat1622float2(hb[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + rowid * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (rowid < rows && part == 0) {
    const int64_t hh = rowid % hl;
    const int64_t rs = rowid / hl;     // r * S + s
    const int64_t r = rs / S, s = rs - r * S;
    delta[(r * hl + hh) * S + s] = acc;
  }
}

__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc,
                                                     __nv_bfloat16* __restrict__ dq, int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 v;
    v.x = pack_bf16x2(a.x, a.y);
    v.y = pack_bf16x2(a.z, a.w);
    v.z = pack_bf16x2(b.x, b.y);
    v.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(dq)[i] = v;
  }
}

template <int D>
cudaError_t launch_bwd_d(const Plan& p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                         void* dv, void* workspace, cudaStream_t st) {
  const int hl = p.H / p.P, gl = p.G / p.P;
  size_t acc_off = 0, delta_off = 0;
  bwd_workspace_bytes(p, &acc_off, &delta_off);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_off);
  float* delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_off);
  const int64_t rows = (int64_t)p.P * p.S * hl;
  {
    const int64_t threads = rows * (D / 8);
    const int64_t blocks = (threads + 255) / 256;
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), delta,
        dq_acc, rows, p.S, hl);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const char* err = nullptr;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t dq4[4] = {(uint64_t)D, (uint64_t)hl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)hl * D * 2, (uint64_t)p.S * hl * D * 2};
  const uint64_t dk4[4] = {(uint64_t)D, (uint64_t)gl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)gl * D * 2, (uint64_t)p.S * gl * D * 2};
  if (!make_tmap_4d_bf16(&tq, q, dq4, sq, 64, BM, &err) ||
      !make_tmap_4d_bf16(&tdo, d_o, dq4, sq, 64, BM, &err) ||
      !make_tmap_4d_bf16(&tk, k, dk4, sk, 64, BN, &err) ||
      !make_tmap_4d_bf16(&tv, v, dk4, sk, 64, BN, &err))
    return cudaErrorInvalidValue;
  BwdArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dq_acc = dq_acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.S = (int)p.S;
  a.hl = hl;
  a.gl = gl;
  a.group = p.H / p.G;
  a.nkb = (int)((p.S + BN - 1) / BN);
  a.scale = p.scale;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.status = p.status;
  a.limit_ns = p.limit_ns;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdLayout<D>::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.P * gl * a.nkb;
  attn_bwd_kernel<D><<<(unsigned)blocks, kThreads, BwdLayout<D>::kBytes, st>>>(tq, tk, tv, tdo, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * D / 8;
  const int64_t cap = (int64_t)num_sms(p.device) * 16;
  const int64_t blocks_dq = std::min<int64_t>((n8 + 255) / 256, cap);
  bwd_dq_kernel<<<(unsigned)blocks_dq, 256, 0, st>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const Plan& p, size_t* dq_acc_off, size_t* delta_off) {
  const int hl = p.H / p.P;
  const size_t acc = (size_t)p.P * p.S * hl * p.D * sizeof(float);
  const size_t acc_al = (acc + 255) & ~size_t(255);
  const size_t dl = (size_t)p.P * hl * p.S * sizeof(float);
  if (dq_acc_off) *dq_acc_off = 0;
  if (delta_off) *delta_off = acc_al;
  return acc_al + ((dl + 255) & ~size_t(255));
}

cudaError_t launch_attn_bwd(const Plan& p, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* d_o, void* dq,
                            void* dk, void* dv, void* workspace, cudaStream_t st) {
  if (p.D == 64) return launch_bwd_d<64>(p, q, k, v, o, lse, d_o, dq, dk, dv, workspace, st);
  return launch_bwd_d<128>(p, q, k, v, o, lse, d_o, dq, dk, dv, workspace, st);
}

}  // namespace uly
