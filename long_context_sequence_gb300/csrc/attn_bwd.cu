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
//   bwd_main  one CTA per (rank, KV head, 128-key block).  Work items are (64-row query
//             tile, query head of the group) pairs from the diagonal on.  Two items are in
//             flight in two TMEM regions, so one item's tensor work overlaps the other's
//             element-wise work:
//               MMA1:  S^T = K Q^T, dP^T = V dO^T      (bf16, M = 128 keys, N = 64 rows)
//               warps 0-3 / 4-7 (one group per region, thread = key row):
//                      P^T = exp2(S^T * scale*log2e - lse*log2e) -> TMEM (fp16),
//                      dS = P (dP - D) -> smem (fp16, 128-byte swizzle),
//                      Q and dO tiles converted in place to fp16;
//               MMA2:  dQ^T = K^T dS^T                  (M = 128 = d, TMEM over dP^T),
//                      dV += P^T dO, dK += dS^T Q       (fp32 accumulators in TMEM);
//               warps 8-11 (thread = d): dQ^T -> coalesced fp32 reductions into the
//                      workspace accumulator (lanes are consecutive d of one row);
//   bwd_dq    fp32 dQ accumulator -> bf16.
// The second MMA group uses fp16 operands (P in [0,1], dS, dO, Q and an fp16 copy of K,
// all clamped to the finite fp16 range): with the same tensor rate, fp16 keeps 11
// significand bits against bf16's 8, which the long dK/dQ sums need.
// TMEM (512 columns): region X in {0,1} at 128X: S^T [0,64) -> P^T [0,32); dP^T [64,128)
// -> dQ^T [64,128).  dV at [256, 256+D), dK at [256+D, 256+2D).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int BN = 128;   // keys per CTA (TMEM lanes of S^T, dP^T, dV, dK)
constexpr int BMI = 64;   // query rows per item
constexpr int NST = 3;    // Q/dO stages
constexpr int kThreads = 448;
constexpr int kDqWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;
constexpr int kBox128 = 128 * 128;   // [128 rows][128 bytes]
constexpr int kBox64 = 64 * 128;     // [64 rows][128 bytes]

template <int D>
struct BwdLayout {
  static constexpr int kKV = (D / 64) * kBox128;   // K or V tile [128][D] bf16
  static constexpr int kItem = (D / 64) * kBox64;  // Q or dO item [64][D]
  static constexpr int kK = 0;
  static constexpr int kV = kKV;
  static constexpr int kK16 = 2 * kKV;             // fp16 copy of K as two 64-column atoms
  static constexpr int kQ = kK16 + 2 * kBox128;    // [NST]
  static constexpr int kDO = kQ + NST * kItem;     // [NST]
  static constexpr int kDS = kDO + NST * kItem;    // [2] fp16 [128 keys][64 q]
  static constexpr int kRow = kDS + 2 * kBox128;   // [2 groups][2][128] fp32: lse2 | delta
  static constexpr int kBar = kRow + 2 * 2 * 128 * 4;
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

__device__ __forceinline__ void red_add(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Item -> (first query row, local query head).  Items run over the 64-row query tiles
// that see this key block (from the diagonal on) and, within a tile, the group's heads.
__device__ __forceinline__ void item_coords(int it, int nb, int gg, int group, int& q0, int& hh) {
  const int qi = it / group;
  q0 = nb * BN + qi * BMI;
  hh = gg * group + (it - qi * group);
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
  float* rowterms = reinterpret_cast<float*>(smem + L::kRow);   // [group X][u&1][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* qd_full = bars + 1;              // [NST]
  uint64_t* qd_empty = bars + 1 + NST;       // [NST]
  uint64_t* s_full = bars + 1 + 2 * NST;     // [2] per TMEM region
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* dq_full = p_full + 2;            // [2]
  uint64_t* dq_free = dq_full + 2;           // [2]
  uint64_t* k16_ready = dq_free + 2;
  uint64_t* acc_done = k16_ready + 1;
  uint64_t* drain = acc_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int per_rank = a.gl * a.nkb;
  const int r = blockIdx.x / per_rank;
  const int rem = blockIdx.x - r * per_rank;
  const int gg = rem / a.nkb;
  const int nb = rem - gg * a.nkb;                         // key block; 0 (most work) first
  const int nqi = (a.S - nb * BN + BMI - 1) / BMI;         // 64-row query tiles that see it
  const int n_items = a.group * nqi;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&dq_full[i], 1);
      mbar_init(&dq_free[i], 128);
    }
    mbar_init(k16_ready, 128);
    mbar_init(acc_done, 1);
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
      mbar_arrive_expect_tx(kv_full, 2 * L::kKV);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_4d(smem + L::kK + b * kBox128, &tm_k, kv_full, 64 * b, gg, nb * BN, r);
        tma_load_4d(smem + L::kV + b * kBox128, &tm_v, kv_full, 64 * b, gg, nb * BN, r);
      }
      int issued = 0;
      for (int it = 0; it < n_items; ++it) {
        const int st = it % NST;
        const uint32_t ph = (it / NST) & 1;
        int q0, hh;
        item_coords(it, nb, gg, a.group, q0, hh);
        if (it >= NST && !mbar_wait(&qd_empty[st], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&qd_full[st], 2 * L::kItem);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_4d(smem + L::kQ + st * L::kItem + b * kBox64, &tm_q, &qd_full[st], 64 * b,
                      hh, q0, r);
          tma_load_4d(smem + L::kDO + st * L::kItem + b * kBox64, &tm_do, &qd_full[st], 64 * b,
                      hh, q0, r);
        }
        ++issued;
      }
      mbar_drain(kv_full, 0, a.limit_ns);
      for (int it = issued > NST ? issued - NST : 0; it < issued; ++it)
        mbar_drain(&qd_full[it % NST], (it / NST) & 1, a.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // S^T, dP^T: M = keys, N = 64 query rows, K = D; bf16, both K-major.
      constexpr uint32_t id_s = idesc_bf16(BN, BMI, false, false);
      // dV += P^T dO, dK += dS^T Q: M = keys, N = D, K = 64 rows; fp16, B MN-major.
      constexpr uint32_t id_kv_t = idesc_f16(BN, D, false, true);   // A = P^T from TMEM
      constexpr uint32_t id_kv_s = idesc_f16(BN, D, false, true);   // A = dS smem, K-major
      // dQ^T = K^T dS^T: M = 128 (d, zero-padded when D = 64), N = 64 rows, K = 128 keys.
      constexpr uint32_t id_q = idesc_f16(128, BMI, true, true);
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      const uint32_t sK16 = smem_u32(smem + L::kK16);
      bool alive = mbar_wait(kv_full, 0, wc);
      auto mma1 = [&](int it) {
        const int X = it & 1, st = it % NST;
        const uint32_t sQ = smem_u32(smem + L::kQ + st * L::kItem);
        const uint32_t sDO = smem_u32(smem + L::kDO + st * L::kItem);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk / 4) * kBox128 + (kk % 4) * 32;
          const uint32_t offb = (kk / 4) * kBox64 + (kk % 4) * 32;
          mma_ss(tbase + 128 * X, sdesc_sw128(sK + offa, 16, 1024),
                 sdesc_sw128(sQ + offb, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk / 4) * kBox128 + (kk % 4) * 32;
          const uint32_t offb = (kk / 4) * kBox64 + (kk % 4) * 32;
          mma_ss(tbase + 128 * X + 64, sdesc_sw128(sV + offa, 16, 1024),
                 sdesc_sw128(sDO + offb, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[X]);
      };
      auto mma2 = [&](int it) -> bool {
        const int X = it & 1, st = it % NST;
        if (!mbar_wait(&p_full[X], (it >> 1) & 1, wc)) return false;
        if (it == 0 && !mbar_wait(k16_ready, 0, wc)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + L::kQ + st * L::kItem);     // fp16 by now
        const uint32_t sDO = smem_u32(smem + L::kDO + st * L::kItem);   // fp16 by now
        const uint32_t sDS = smem_u32(smem + L::kDS + X * kBox128);
        // dQ^T first, so its read-out overlaps the dV/dK MMAs
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tbase + 128 * X + 64, sdesc_sw128(sK16 + kk * 2048, kBox128, 1024),
                 sdesc_sw128(sDS + kk * 2048, kBox128, 1024), id_q, kk > 0 ? 1u : 0u);
        mma_commit(&dq_full[X]);
#pragma unroll
        for (int kk = 0; kk < BMI / 16; ++kk)
          mma_ts(tbase + 256, tbase + 128 * X + kk * 8, sdesc_sw128(sDO + kk * 2048, kBox64, 1024),
                 id_kv_t, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BMI / 16; ++kk)
          mma_ss(tbase + 256 + D, sdesc_sw128(sDS + kk * 32, 16, 1024),
                 sdesc_sw128(sQ + kk * 2048, kBox64, 1024), id_kv_s, (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&qd_empty[st]);
        return true;
      };
      for (int it = 0; alive && it < n_items; ++it) {
        const int X = it & 1, st = it % NST;
        if (!mbar_wait(&qd_full[st], (it / NST) & 1, wc)) { alive = false; break; }
        if (it >= 2 && !mbar_wait(&dq_free[X], ((it - 2) >> 1) & 1, wc)) { alive = false; break; }
        tc_fence_after();
        mma1(it);
        if (it >= 1 && !mma2(it - 1)) { alive = false; break; }
      }
      if (alive && n_items > 0 && mma2(n_items - 1)) mma_commit(acc_done);
      mma_commit(drain);
      mbar_drain(drain, 0, a.limit_ns);
    }
  } else if (warp >= kDqWarp0) {
    // dQ warpgroup: thread = d (TMEM lane of dQ^T).  First the fp16 copy of K.
    const int d = (warp - kDqWarp0) * 32 + lane;
    bool ok = __all_sync(0xffffffffu, mbar_wait(kv_full, 0, wc));
    if (ok) {
      uint8_t* k16 = smem + L::kK16;
      for (int c = d; c < 2 * kBox128 / 16; c += 128) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c * 16 < L::kKV)
          v = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(smem + L::kK + c * 16));
        *reinterpret_cast<uint4*>(k16 + c * 16) = v;
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(k16_ready);
    const uint32_t lane_off = (uint32_t)((warp - kDqWarp0) * 32) << 16;
    const bool active = (warp - kDqWarp0) * 32 < D;      // warp-uniform
    for (int it = 0; ok && it < n_items; ++it) {
      const int X = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&dq_full[X], (it >> 1) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      if (active) {
        int q0, hh;
        item_coords(it, nb, gg, a.group, q0, hh);
        float* base = a.dq_acc + (((size_t)r * a.S + q0) * a.hl + hh) * D + d;
        const size_t row_stride = (size_t)a.hl * D;
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + 128 * X + 64 + 32 * c2, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int qc = 32 * c2 + j;
            if (q0 + qc < a.S) red_add(base + qc * row_stride, __uint_as_float(v[j]) * a.scale);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&dq_free[X]);
    }
  } else {
    // Compute warpgroups: group X handles items X, X+2, ...; thread = key row.
    const int X = warp / 4;
    const int row = (warp % 4) * 32 + lane;
    const int t128 = threadIdx.x % 128;
    const int key_g = nb * BN + row;
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t ts = tbase + lane_off + 128 * X;   // S^T, then P^T
    const uint32_t tp = ts + 64;                       // dP^T
    const float sl2 = a.scale_log2;
    uint8_t* sDS = smem + L::kDS + X * kBox128 + row * 128;
    bool ok = true;
    for (int it = X; it < n_items; it += 2) {
      const int u = it >> 1, st = it % NST;
      int q0, hh;
      item_coords(it, nb, gg, a.group, q0, hh);
      float* terms = rowterms + (X * 2 + (u & 1)) * 128;   // [0,64) lse2, [64,128) delta
      {
        const int qc = t128 & 63;
        const int qg = q0 + qc;
        const size_t idx = ((size_t)r * a.hl + hh) * a.S + qg;
        if (t128 < 64)
          terms[t128] = qg < a.S ? a.lse[idx] * 1.4426950408889634f : INFINITY;
        else
          terms[t128] = qg < a.S ? a.delta[idx] : 0.f;
      }
      named_bar_sync(1 + X, 128);
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], u & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (q0 < nb * BN + BN) || (q0 + BMI > a.S) || (nb * BN + BN > a.S);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dp[32];
        tmem_ld32(ts + 32 * c, sv);
        tmem_ld32(tp + 32 * c, dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) {
          float pv[2], dv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int qc = 32 * c + 2 * i2 + e;
            float p = ex2_approx(fmaf(__uint_as_float(sv[2 * i2 + e]), sl2, -terms[qc]));
            if (need_mask && !(key_g <= q0 + qc && q0 + qc < a.S && key_g < a.S)) p = 0.f;
            pv[e] = p;
            dv[e] = p * (__uint_as_float(dp[2 * i2 + e]) - terms[64 + qc]);
          }
          pk[i2] = pack_f16x2_sat(pv[0], pv[1]);
          dk[i2] = pack_f16x2_sat(dv[0], dv[1]);
        }
        tmem_st16(ts + 16 * c, pk);                     // P^T (fp16) over S^T
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {                // dS row, 128-byte swizzle
          const int chunk = c * 4 + u4;
          *reinterpret_cast<uint4*>(sDS + ((chunk ^ (row & 7)) * 16)) =
              make_uint4(dk[4 * u4], dk[4 * u4 + 1], dk[4 * u4 + 2], dk[4 * u4 + 3]);
        }
      }
      // The item's Q and dO tiles are no longer needed in bf16 (S^T, dP^T are done):
      // convert them in place to fp16 for dK and dV.
      {
        uint8_t* q16 = smem + L::kQ + st * L::kItem;
        uint8_t* do16 = smem + L::kDO + st * L::kItem;
#pragma unroll 1
        for (int cidx = t128; cidx < L::kItem / 16; cidx += 128) {
          uint4* pq = reinterpret_cast<uint4*>(q16 + cidx * 16);
          uint4* pd = reinterpret_cast<uint4*>(do16 + cidx * 16);
          const uint4 vq = *pq, vd = *pd;
          *pq = bf16x8_to_f16x8(vq);
          *pd = bf16x8_to_f16x8(vd);
        }
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[X]);
    }
    // dV (group 0) and dK (group 1) of this key block, once every MMA has finished.
    if (ok && n_items > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, wc));
    if (ok && n_items > 0) {
      tc_fence_after();
      __nv_bfloat16* dst = (X ? a.dk : a.dv) + (((size_t)r * a.S + key_g) * a.gl + gg) * D;
      const float mul = X ? a.scale : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + 256 + X * D + 32 * c, v);
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
  if (!make_tmap_4d_bf16(&tq, q, dq4, sq, 64, BMI, &err) ||
      !make_tmap_4d_bf16(&tdo, d_o, dq4, sq, 64, BMI, &err) ||
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
