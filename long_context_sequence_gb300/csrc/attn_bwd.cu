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
//   bwd_pre   D_i = dO_i . (o_i + o_lo_i) in fp32 (o_lo: the forward's optional bf16 rounding
//             residual of O), zeroing of the fp32 dQ accumulator, and fp16 copies of Q,
//             dO (and, in to_f16_kernel, of K, V) for the tensor-core operands;
//   bwd_main  one CTA per (rank, KV head, 128-key block).  Work items are (64-row query
//             tile, query head of the group) pairs from the diagonal on.  Items alternate
//             between two TMEM regions so that one item's tensor work overlaps the other's
//             element-wise work.  Two threads issue the MMAs: issuer A S^T and dQ^T of both
//             regions, issuer B dP^T and every dV and dK (the accumulators both regions
//             share, so one thread orders them).  A thread issuing a tcgen05.mma stalls
//             while the tensor pipe's queue is full, and it serves its barriers in program
//             order, so one issuer would leave a region's ready MMAs behind the other
//             region's.  The pipe runs MMAs in issue order; issuer B holds dV/dK(it) until
//             A has issued dQ^T(it), which the region's next S^T waits for:
//               MMA1   S^T = K Q^T, dP^T = V dO^T            (M = 128 keys, N = 64 rows)
//               8 warps per region, thread = key row, warpgroup = 32 query columns:
//                      P^T = scale*exp(S^T scale - lse) -> TMEM (fp16, over dP^T),
//                      dS = P (dP - D) -> smem (fp16, 128-byte swizzle)
//               MMA2   dQ^T = K^T dS^T (M = d, over S^T), dV += P^T dO, dK += dS^T Q
//               the same warps, thread = d: dQ^T -> fp32 reductions into the workspace
//                      accumulator, which keeps four query rows of one (head, d) together
//                      ([P][S4/4][hl][D][4]): a thread adds its own four rows in one
//                      16-byte reduction, a warp 512 contiguous bytes;
//   bwd_dq    fp32 dQ accumulator -> bf16 [P][S][hl][D].
// Every MMA runs on fp16 operands, and P, dS keep 11 significand bits, which the long
// dK/dQ sums need.  fp16 holds full precision only in [2^-14, 65504], while the bf16 inputs
// span fp32's range (a training step's dO is often 1e-5 .. 1e-8, and q, k, v may exceed
// 65504).  So every operand is scaled by an exact power of two chosen per call from the
// tensors' largest magnitudes (bwd_amax_kernel):
//   q' = 2^eq q, k' = 2^-eq k     eq balances the two: largest |q'| and |k'| at about the
//                                 geometric mean of the two maxima (s' = q'.k' = s exactly,
//                                 so the softmax's multiplier stays a kernel constant)
//   v' = 2^ev v                   largest |v'| in [2^-1, 2^0)
//   P' = 2^kp scale P             2^kp scale in [2^7, 2^8)  (kp fixed by the plan's scale)
//   dO' = 2^edo dO                the largest edo with 2^kp scale D max|dO'| max|v'| <= 2^14
//                                 and max|dO'| < 2^15
// Then |dP' - D'| <= 2 D max|dO'| max|v'| and dS' = P' (dP' - D') stays below 2^15: no fp16
// operand can overflow, and for ordinary data none is subnormal.  The outputs take the
// inverse powers exactly (power-of-two factors in the epilogues): dV = acc / (scale
// 2^(kp+edo)), dK = 2^-(kp+edo+ev+eq) acc, dQ = 2^-(kp+edo+ev-eq) acc.  Scaling any input by
// a power of two therefore leaves every fp16 operand bit for bit as it was and scales the
// outputs exactly.  A tensor whose largest magnitude lies beyond the exponents' range
// (|e| <= 60) would saturate: the call reports ULY_ERR_RANGE through the status word.
// TMEM (512 columns): region X at [128X, 128X+128): S^T [0,64) -> dQ^T; dP^T [64,128) ->
// P^T of warpgroup w2 at [64+32 w2, 64+32 w2+16).  dV [256,256+D), dK [256+D, 256+2D).
#include <cmath>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int BN = 128;   // keys per CTA
constexpr int BMI = 64;   // query rows per item
constexpr int NST = 4;    // Q/dO stages
constexpr int kRegionThreads = 256;          // 8 warps per TMEM region
constexpr int kTmaWarp = 16, kMmaWarp = 17, kAccWarp = 18;
constexpr int kThreads = 608;
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 128 * 128;   // [128 rows][128 bytes]
constexpr int kBox64 = 64 * 128;  // [64 rows][128 bytes]

template <int D>
struct BwdLayout {
  static constexpr int kKV = (D / 64) * kBox;     // a [128][D] tile
  static constexpr int kItem = (D / 64) * kBox64; // a [64][D] tile
  static constexpr int kK = 0;                    // K: two atoms (the second zero if D = 64)
  static constexpr int kV = 2 * kBox;
  static constexpr int kQ = kV + kKV;             // [NST]
  static constexpr int kDO = kQ + NST * kItem;    // [NST]
  static constexpr int kDS = kDO + NST * kItem;   // [2] fp16 [128 keys][64 rows]
  static constexpr int kRow = kDS + 2 * kBox;     // [NST][128] fp32: lse terms | D
  static constexpr int kBar = kRow + NST * 128 * 4;
  static constexpr int kBytes = kBar + 256;
};

struct BwdArgs {
  const float* lse;
  const float* delta;
  const int* exps;        // the call's exponents eq, ek, ev, edo (bwd_amax_kernel)
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int S, hl, gl, group, nkb;
  int kp;                 // P' = 2^kp scale P
  float scale, scale_log2, log2_scale;   // log2_scale = log2(scale) + kp
  int* status;
  uint64_t limit_ns;
  uint32_t flags;
};

__device__ __forceinline__ void red_add4(float* addr, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(x), "f"(y),
               "f"(z), "f"(w)
               : "memory");
}

// Item -> (first query row, local query head): the 64-row query tiles that see this key
// block (from the diagonal on) and, within a tile, the group's heads.
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
  float* rows = reinterpret_cast<float*>(smem + L::kRow);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* qd_full = bars + 1;              // [NST]
  uint64_t* qd_empty = bars + 1 + NST;       // [NST]
  uint64_t* s_full = bars + 1 + 2 * NST;     // [2] per region
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* dq_full = s_full + 4;            // [2]
  uint64_t* dq_free = s_full + 6;            // [2]
  uint64_t* acc_done = s_full + 8;
  uint64_t* drain = s_full + 9;
  uint64_t* drain_acc = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 13);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* decision = abort_flag + 1;   // [2 regions][2]: group-wait outcomes
  volatile int* dq_issued = decision + 4;    // items whose dQ^T issuer A has issued

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int per_rank = a.gl * a.nkb;
  const int r = blockIdx.x / per_rank;
  const int rem = blockIdx.x - r * per_rank;
  const int gg = rem / a.nkb;
  const int nb = rem - gg * a.nkb;                         // key block; 0 (most work) first
  const int nqi = (a.S - nb * BN + BMI - 1) / BMI;         // 64-row query tiles that see it
  const int n_items = a.group * nqi;
  // element extents for the debug checks: row terms [P][hl][S], dQ accumulator
  // [P][S4/4][hl][D][4], dK/dV [P][S][gl][D]
  const int S4 = (a.S + 3) & ~3;
  const uint64_t n_ranks = gridDim.x / (uint64_t)per_rank;
  const uint64_t ext_rows = n_ranks * a.hl * a.S, ext_q = n_ranks * S4 * a.hl * D,
                 ext_kv = n_ranks * a.S * a.gl * D;
  (void)ext_rows; (void)ext_q; (void)ext_kv;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 2);    // S^T (issuer A) and dP^T (issuer B)
      mbar_init(&p_full[i], 1);
      mbar_init(&dq_full[i], 1);
      mbar_init(&dq_free[i], 1);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(drain_acc, 1);
    *abort_flag = 0;
    *dq_issued = 0;
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
    // TMA for K, V and every item's Q, dO (fp16 copies); the whole warp stages the item's
    // row terms (lse * log2e - log2(scale), and D) next to them.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      // K always as two 64-column atoms: for D = 64 the second box lies past the last
      // column and TMA fills it with zeros (the zero rows of K^T padded to M = 128).
      mbar_arrive_expect_tx(kv_full, 2 * kBox + L::kKV);
      for (int b = 0; b < 2; ++b)
        tma_load_4d(smem + L::kK + b * kBox, &tm_k, kv_full, 64 * b, gg, nb * BN, r);
      for (int b = 0; b < D / 64; ++b)
        tma_load_4d(smem + L::kV + b * kBox, &tm_v, kv_full, 64 * b, gg, nb * BN, r);
    }
    int issued = 0;
    for (int it = 0; it < n_items; ++it) {
      const int st = it % NST;
      const uint32_t ph = (it / NST) & 1;
      int q0, hh;
      item_coords(it, nb, gg, a.group, q0, hh);
      if (it >= NST && !__all_sync(0xffffffffu, mbar_wait(&qd_empty[st], ph ^ 1, wc))) break;
      float* rw = rows + st * 128;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int qc = lane + 32 * e;
        const int qg = q0 + qc;
        const size_t idx = ((size_t)r * a.hl + hh) * a.S + qg;
        const bool in = qg < a.S && ULY_IN_BOUNDS(idx, 1, ext_rows);
        rw[qc] = in ? a.log2_scale - a.lse[idx] * 1.4426950408889634f : -INFINITY;
        rw[64 + qc] = in ? a.delta[idx] : 0.f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&qd_full[st], 2 * L::kItem);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_4d(smem + L::kQ + st * L::kItem + b * kBox64, &tm_q, &qd_full[st], 64 * b,
                      hh, q0, r);
          tma_load_4d(smem + L::kDO + st * L::kItem + b * kBox64, &tm_do, &qd_full[st], 64 * b,
                      hh, q0, r);
        }
      }
      ++issued;
    }
    if (lane == 0) {
      mbar_drain(kv_full, 0, a.limit_ns);
      for (int it = issued > NST ? issued - NST : 0; it < issued; ++it)
        mbar_drain(&qd_full[it % NST], (it / NST) & 1, a.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    // Issuer A: S^T and dQ^T of both regions (both over a region's S^T columns).
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(BN, BMI, false, false);  // S^T (N = 64)
      constexpr uint32_t id_q = idesc_f16(128, BMI, true, true);   // dQ^T (M = d, N = 64)
      // Descriptors are built once; a K-step adds its byte offset / 16 to the address
      // field (no carry: every smem address here is below 2^18).
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + L::kK), kBox, 1024);
      // S^T of item it over region X's S^T columns, which held dQ^T(it-2) until the
      // element-wise warps read it out (dq_free).
      // ULY_FLAG_INJECT_STALL: block 0 withholds S^T(0)'s commit, so the element-wise
      // warps' bounded wait for it runs out (failure-path test; nothing faults).
      const bool stall = (a.flags & ULY_FLAG_INJECT_STALL) && blockIdx.x == 0;
      auto mma_s = [&](int it) -> bool {
        const int X = it & 1, st = it % NST;
        if (!mbar_wait(&qd_full[st], (it / NST) & 1, wc)) return false;
        if (it >= 2 && !mbar_wait(&dq_free[X], ((it - 2) >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + L::kQ + st * L::kItem), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
          const uint32_t offb = ((kk / 4) * kBox64 + (kk % 4) * 32) >> 4;
          mma_ss(tbase + 128 * X, dK_k + offa, dQ_k + offb, id_s, kk > 0 ? 1u : 0u);
        }
        if (!(stall && it == 0)) mma_commit(&s_full[X]);
        return true;
      };
      // dQ^T of item it over region X's S^T columns
      auto mma_dq = [&](int it) -> bool {
        const int X = it & 1;
        if (!mbar_wait(&p_full[X], (it >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint64_t dDS_mn = sdesc_sw128(smem_u32(smem + L::kDS + X * kBox), kBox, 1024);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tbase + 128 * X, dK_mn + ((kk * 2048) >> 4), dDS_mn + ((kk * 2048) >> 4), id_q,
                 kk > 0 ? 1u : 0u);
        mma_commit(&dq_full[X]);
        *dq_issued = it + 1;
        return true;
      };
      // Pairs, one item per region: dQ^T of both, then S^T of the next two.  (Serving
      // the regions in whatever order their barriers complete, by polling both, was
      // slower: the spinning issuer costs more than the order it saves.)
      bool alive = mbar_wait(kv_full, 0, wc);
      for (int it = 0; alive && it < 2 && it < n_items; ++it) alive = mma_s(it);
      for (int it = 0; alive && it < n_items; it += 2) {
        alive = mma_dq(it);
        if (alive && it + 1 < n_items) alive = mma_dq(it + 1);
        if (alive && it + 2 < n_items) alive = mma_s(it + 2);
        if (alive && it + 3 < n_items) alive = mma_s(it + 3);
      }
      mma_commit(drain);
      mbar_drain(drain, 0, a.limit_ns);
    }
  } else if (warp == kAccWarp) {
    // Issuer B: dP^T of both regions and every dV and dK, in item order.  dP^T(it+2) goes
    // over the columns where P^T(it) sat, after dV(it) read it (same thread, in order);
    // the dV/dK accumulators are shared by both regions, so one thread orders them.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(BN, BMI, false, false);  // dP^T (N = 64)
      constexpr uint32_t id_kv = idesc_f16(BN, D, false, true);    // dV, dK (K = 64 rows)
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + L::kV), 16, 1024);
      auto mma_dp = [&](int it) -> bool {
        const int X = it & 1, st = it % NST;
        if (!mbar_wait(&qd_full[st], (it / NST) & 1, wc)) return false;
        tc_fence_after();
        const uint64_t dDO_k = sdesc_sw128(smem_u32(smem + L::kDO + st * L::kItem), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
          const uint32_t offb = ((kk / 4) * kBox64 + (kk % 4) * 32) >> 4;
          mma_ss(tbase + 128 * X + 64, dV_k + offa, dDO_k + offb, id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[X]);
        return true;
      };
      bool alive = mbar_wait(kv_full, 0, wc);
      for (int it = 0; alive && it < 2 && it < n_items; ++it) alive = mma_dp(it);
      for (int it = 0; alive && it < n_items; ++it) {
        const int X = it & 1, st = it % NST;
        if (!mbar_wait(&p_full[X], (it >> 1) & 1, wc)) { alive = false; break; }
        // Let dQ^T(it), which a region's next S^T waits for, enter the tensor pipe ahead of
        // dV/dK(it) (the pipe runs MMAs in issue order).  Only an ordering preference: the
        // wait is bounded and gives up if the CTA aborts.
        for (uint32_t n = 0; *dq_issued <= it && n < (1u << 22) && !*wc.abort; ++n) {
        }
        tc_fence_after();
        const uint64_t dQ_mn = sdesc_sw128(smem_u32(smem + L::kQ + st * L::kItem), kBox64, 1024);
        const uint64_t dDO_mn = sdesc_sw128(smem_u32(smem + L::kDO + st * L::kItem), kBox64, 1024);
        const uint64_t dDS_k = sdesc_sw128(smem_u32(smem + L::kDS + X * kBox), 16, 1024);
        // dV += P^T dO (A = P^T from TMEM: rows 16kk.. of warpgroup kk/2, packed fp16)
#pragma unroll
        for (int kk = 0; kk < BMI / 16; ++kk)
          mma_ts(tbase + 256, tbase + 128 * X + 64 + 32 * (kk / 2) + 8 * (kk % 2),
                 dDO_mn + ((kk * 2048) >> 4), id_kv, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q (A = dS [keys][rows], K-major)
#pragma unroll
        for (int kk = 0; kk < BMI / 16; ++kk)
          mma_ss(tbase + 256 + D, dDS_k + ((kk * 32) >> 4), dQ_mn + ((kk * 2048) >> 4), id_kv,
                 (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&qd_empty[st]);
        if (it + 2 < n_items) alive = mma_dp(it + 2);
      }
      if (alive) mma_commit(acc_done);
      mma_commit(drain_acc);
      mbar_drain(drain_acc, 0, a.limit_ns);
    }
  } else {
    // 16 element-wise warps: warps [8X, 8X+8) serve TMEM region X (items X, X+2, ...);
    // within a region, warpgroup w2 owns query columns [32 w2, 32 w2 + 32) and warp % 4
    // selects the TMEM lane quarter (= key rows, and d for the dQ^T read-out).
    const int X = warp / 8;
    const int w2 = (warp / 4) % 2;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const float sl2 = a.scale_log2;     // s' = q'.k' = s: the multiplier needs no scaling
    const int key_g = nb * BN + row;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t treg = tbase + lane_off + 128 * X;
    uint8_t* ds_row = smem + L::kDS + X * kBox + row * 128;
    // The region's first warp waits on the mbarrier; the other seven sleep in a named
    // barrier (no issue slots) and read the outcome it left, so they all decide alike.
    const bool leader = (warp % 8) == 0;
    int n_waits = 0;
    auto group_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      volatile int* slot = decision + 2 * X + (n_waits & 1);
      if (leader) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
        if (lane == 0) *slot = got ? 1 : 0;
      }
      named_bar_sync(1 + X, kRegionThreads);
      ++n_waits;
      return *slot != 0;
    };
    // All threads of the region have finished (their own TMEM/smem writes fenced); one
    // thread then arrives for the whole region.
    auto group_arrive = [&](uint64_t* bar) {
      named_bar_sync(1 + X, kRegionThreads);
      if (leader && lane == 0) mbar_arrive(bar);
    };
    bool ok = true;
    for (int it = X; ok && it < n_items; it += 2) {
      const int u = it >> 1, st = it % NST;
      int q0, hh;
      item_coords(it, nb, gg, a.group, q0, hh);
      const float* rw = rows + st * 128;
      ok = group_wait(&s_full[X], u & 1);
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (q0 < nb * BN + BN) || (q0 + BMI > a.S) || (nb * BN + BN > a.S);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[16], dp[16], pk[8], dk[8];
        // row terms as packed pairs: nl = log2(scale) - lse*log2e (-inf: masked), dl = D
        uint64_t nl[8], dl[8];
        const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(rw + 32 * w2 + 16 * c);
        const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(rw + 64 + 32 * w2 + 16 * c);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const ulonglong2 x = l4[e], y = d4[e];
          nl[2 * e] = x.x; nl[2 * e + 1] = x.y;
          dl[2 * e] = y.x; dl[2 * e + 1] = y.y;
        }
        tmem_ld16x2(treg + 32 * w2 + 16 * c, treg + 64 + 32 * w2 + 16 * c, sv, dp);
        if (need_mask) {
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) {
            float n0, n1;
            f2_unpack(nl[i2], n0, n1);
            const int qg = q0 + 32 * w2 + 16 * c + 2 * i2;
            if (!(key_g <= qg && qg < a.S && key_g < a.S)) n0 = -INFINITY;          // p = 0
            if (!(key_g <= qg + 1 && qg + 1 < a.S && key_g < a.S)) n1 = -INFINITY;
            nl[i2] = f2_pack(n0, n1);
          }
        }
        const uint64_t sc2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {
          // P_s = 2^(s scale log2e + nl), dS_s = P_s (dP - D): one FFMA2, FSUB2, FMUL2 per pair
          float x0, x1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(sv[2 * i2]), __uint_as_float(sv[2 * i2 + 1])),
                          sc2, nl[i2]),
                    x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const uint64_t d2 = fsub2(f2_pack(__uint_as_float(dp[2 * i2]), __uint_as_float(dp[2 * i2 + 1])),
                                    dl[i2]);
          float ds0, ds1;
          f2_unpack(fmul2(f2_pack(p0, p1), d2), ds0, ds1);
          pk[i2] = pack_f16x2_sat(p0, p1);
          dk[i2] = pack_f16x2_sat(ds0, ds1);
        }
        // P^T over this warpgroup's own dP^T columns (read above, nobody else reads them)
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                treg + 64 + 32 * w2 + 8 * c),
            "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]),
            "r"(pk[7])
            : "memory");
#pragma unroll
        for (int u4 = 0; u4 < 2; ++u4) {
          const int chunk = w2 * 4 + c * 2 + u4;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (row & 7)) * 16)) =
              make_uint4(dk[4 * u4], dk[4 * u4 + 1], dk[4 * u4 + 2], dk[4 * u4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      group_arrive(&p_full[X]);
      // dQ^T of this item (already scaled) -> the workspace accumulator
      ok = group_wait(&dq_full[X], u & 1);
      if (!ok) break;
      tc_fence_after();
      // dQ^T to registers, hand the region's columns back at once (MMA1 of item it+2
      // writes them), then the reductions from registers.
      uint32_t v[32];
      const bool has_d = quarter * 32 < D;   // warp-uniform: lanes are d = 32*quarter + lane
      if (has_d) tmem_ld32(treg + 32 * w2, v);
      tc_fence_before();
      group_arrive(&dq_free[X]);
      if (has_d) {
        // The accumulator keeps four consecutive query rows of one (head, d) together
        // ([P][S4/4][hl][D][4]), so lane d adds its rows 4c .. 4c+3 with one 16-byte
        // reduction and a warp's 32 lanes cover 512 contiguous bytes.
        float* ptr = a.dq_acc +
                     ((((size_t)r * (S4 / 4) + (q0 + 32 * w2) / 4) * a.hl + hh) * D +
                      32 * quarter + lane) * 4;
        const size_t step = (size_t)a.hl * D * 4;   // the next four rows
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (q0 + 32 * w2 + 4 * c < a.S && ULY_IN_BOUNDS(ptr + c * step - a.dq_acc, 4, ext_q))
            red_add4(ptr + c * step, __uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                     __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
      }
    }
    // dV (warps 0-7) and dK (8-15) of this key block, once every MMA has finished.
    if (ok && n_items > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, wc));
    if (ok && n_items > 0) {
      tc_fence_after();
      const int which = warp / 8;         // 0: dV, 1: dK
      const int half = w2;                // columns [half * D/2, (half + 1) * D/2)
      __nv_bfloat16* dst = (which ? a.dk : a.dv) + (((size_t)r * a.S + key_g) * a.gl + gg) * D;
      // dV sums carry 2^(kp+edo) scale, dK sums 2^(kp+edo+ev+eq)
      const int4 ex = __ldcg(reinterpret_cast<const int4*>(a.exps));   // read here, not earlier
      const float mul = which ? 1.f : 1.f / a.scale;
      const int sh = which ? -(a.kp + ex.w + ex.z + ex.x) : -(a.kp + ex.w);
      // 2^sh as two factors of the same sign (|sh| may exceed a float exponent's range)
      const float m1 = mul * exp2i(sh / 2), m2 = exp2i(sh - sh / 2);
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + 256 + which * D + 32 * c, v);
        if (key_g < a.S &&
            ULY_IN_BOUNDS(dst + 32 * c - (which ? a.dk : a.dv), 32, ext_kv)) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            auto sc = [&](int e) { return __uint_as_float(v[8 * j + e]) * m1 * m2; };
            uint4 o;
            o.x = pack_bf16x2(sc(0), sc(1));
            o.y = pack_bf16x2(sc(2), sc(3));
            o.z = pack_bf16x2(sc(4), sc(5));
            o.w = pack_bf16x2(sc(6), sc(7));
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

// Largest magnitudes of q, k, v and dO for the call's power-of-two scaling, then (in the
// last block to finish) the exponents.
// The rule, with E(m) = floor(log2 m) and every exponent clamped to [-60, 60] (so every
// sum of two of them, and of kp, is a float exponent):
//   eq = floor((E(max|k|) - E(max|q|)) / 2), ek = -eq
//                                              -> E(max|q'|) and E(max|k'|) differ by <= 1
//   ev = -1 - E(max|v|)                        -> max|v'| in [2^-1, 2^0)
//   edo = min(14 - E(max|dO|), 13 - E(X)), X = 2^kp scale D max|dO| max|v'|
//                                              -> max|dO'| < 2^15 and X 2^edo < 2^14
// A zero (or non-finite) maximum leaves its exponent at 0.  A tensor whose scaled maximum
// would still reach 2^15 (only possible when the clamp bites) makes the call report
// kErrRange: its fp16 copy would saturate.
__device__ __forceinline__ bool finite_pos(float m) { return m > 0.f && m <= 3.4028234e38f; }
__device__ __forceinline__ int clamp_exp(int e) { return e < -60 ? -60 : (e > 60 ? 60 : e); }
// floor(log2 m) of a positive finite float, subnormals included.
__device__ __forceinline__ int floor_log2f(float m) {
  const uint32_t b = __float_as_uint(m);
  const int ex = (int)((b >> 23) & 0xFFu);
  return ex ? ex - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

__device__ void bwd_exponents(const float (&M)[4], float scale_k, int D, int (&e)[4],
                              bool& range) {
  if (finite_pos(M[0]) && finite_pos(M[1])) {
    const int d = floor_log2f(M[1]) - floor_log2f(M[0]);
    e[0] = clamp_exp(d >= 0 ? d / 2 : -((1 - d) / 2));   // floor(d / 2)
  } else {
    e[0] = 0;
  }
  e[1] = -e[0];
  e[2] = finite_pos(M[2]) ? clamp_exp(-1 - floor_log2f(M[2])) : 0;
  int edo = 0;
  if (finite_pos(M[3])) {
    edo = 14 - floor_log2f(M[3]);
    const float sd = scale_k * (float)D;
    if (finite_pos(M[2]) && finite_pos(sd)) {
      // X as a product of mantissas in [1, 2) times a power of two (nothing overflows)
      const int a = floor_log2f(sd), b = floor_log2f(M[3]), c = floor_log2f(M[2]);
      const float mm = ldexpf(sd, -a) * ldexpf(M[3], -b) * ldexpf(M[2], -c);
      const int ex = a + b + c + e[2] + floor_log2f(mm);
      edo = min(edo, 13 - ex);
    }
    edo = clamp_exp(edo);
  }
  e[3] = edo;
  range = false;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (finite_pos(M[j]) && floor_log2f(M[j]) + e[j] >= 15) range = true;
}

// Largest |x| of 8 bf16 as the bit pattern of a non-negative bf16 (whose unsigned order is
// the order of the magnitudes).
__device__ __forceinline__ uint32_t absmax8_bits(uint4 v) {
  const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                              __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// scal (zeroed before the launch): [0, 4) largest |q|, |k|, |v|, |dO| as fp32 bit patterns,
// [4] count of finished blocks, [8, 12) the exponents eq, ek, ev, edo.
__global__ void __launch_bounds__(256) bwd_amax_kernel(const uint4* __restrict__ q,
                                                       const uint4* __restrict__ k,
                                                       const uint4* __restrict__ v,
                                                       const uint4* __restrict__ d_o,
                                                       int64_t nq8, int64_t nk8,
                                                       uint32_t* scal, float scale_k, int D,
                                                       int* status) {
  uint32_t m[4] = {0u, 0u, 0u, 0u};
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = t0; i < nq8; i += stride) {
    m[0] = max(m[0], absmax8_bits(__ldcs(q + i)));
    m[3] = max(m[3], absmax8_bits(__ldcs(d_o + i)));
  }
  for (int64_t i = t0; i < nk8; i += stride) {
    m[1] = max(m[1], absmax8_bits(__ldcs(k + i)));
    m[2] = max(m[2], absmax8_bits(__ldcs(v + i)));
  }
  __shared__ uint32_t red[8][4];
  __shared__ bool last;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m[j] = max(m[j], __shfl_xor_sync(0xffffffffu, m[j], off));
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0)
    for (int j = 0; j < 4; ++j) red[warp][j] = m[j];
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int j = 0; j < 4; ++j) {
      uint32_t x = 0;
      for (int w = 0; w < (int)(blockDim.x / 32); ++w) x = max(x, red[w][j]);
      atomicMax(&scal[j], x << 16);     // bf16 bits -> fp32 bits
    }
    __threadfence();
    last = atomicAdd(&scal[4], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    float M[4];
    for (int j = 0; j < 4; ++j) M[j] = __uint_as_float(atomicOr(&scal[j], 0u));
    int e[4];
    bool range;
    bwd_exponents(M, scale_k, D, e, range);
    int* ex = reinterpret_cast<int*>(scal + 8);
    for (int j = 0; j < 4; ++j) ex[j] = e[j];
    if (range) atomicCAS(status, kOk, kErrRange);
  }
}

// D'_i = 2^(edo+ev) sum_d dO_i[d] * (O_i[d] + O_lo_i[d]) (fp32), zeroing of the dQ
// accumulator (acc8 groups of 8 floats, one per thread) and the fp16 copies q' = 2^eq q and
// dO' = 2^edo dO.  16 threads per row of D = 128 (8 elements each), 8 per row of D = 64.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ o_lo,
                                                      const __nv_bfloat16* __restrict__ d_o,
                                                      const __nv_bfloat16* __restrict__ q,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ dq_acc,
                                                      uint4* __restrict__ q16,
                                                      uint4* __restrict__ do16, int64_t rows,
                                                      int64_t S, int hl, int64_t acc8,
                                                      const int* __restrict__ exps) {
  constexpr int TPR = D / 8;
  const int4 ex = *reinterpret_cast<const int4*>(exps);
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rowid = tid / TPR;       // row in [P][S][hl] order
  const int part = (int)(tid % TPR);
  float acc = 0.f;
  if (tid < acc8 && ULY_IN_BOUNDS(tid * 8, 8, (uint64_t)acc8 * 8)) {
    float4* zq = reinterpret_cast<float4*>(dq_acc + tid * 8);
    zq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    zq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (rowid < rows && ULY_IN_BOUNDS(rowid * D + part * 8, 8, (uint64_t)rows * D)) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + rowid * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(d_o + rowid * D + part * 8);
    uint4 c = make_uint4(0, 0, 0, 0);
    if (o_lo) c = *reinterpret_cast<const uint4*>(o_lo + rowid * D + part * 8);
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
    const __nv_bfloat162* hc = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(ha[i]), y = __bfloat1622float2(hb[i]);
      const float2 z = __bfloat1622float2(hc[i]);
      acc = fmaf(x.x + z.x, y.x, acc);
      acc = fmaf(x.y + z.y, y.y, acc);
    }
    // fp16 copies of dO' and q' for the main kernel's tensor-core operands
    do16[(rowid * D + part * 8) / 8] = bf16x8_to_f16x8_scaled(b, exp2i(ex.w));
    q16[(rowid * D + part * 8) / 8] = bf16x8_to_f16x8_scaled(
        *reinterpret_cast<const uint4*>(q + rowid * D + part * 8), exp2i(ex.x));
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (rowid < rows && part == 0) {
    const int64_t hh = rowid % hl;
    const int64_t rs = rowid / hl;     // r * S + s
    const int64_t r = rs / S, s = rs - r * S;
    if (ULY_IN_BOUNDS((r * hl + hh) * S + s, 1, rows))
      delta[(r * hl + hh) * S + s] = acc * exp2i(ex.w + ex.z);
  }
}

// bf16 -> fp16 copy scaled by 2^exps[which], 8 elements per thread (k' and v' for the main
// kernel).
__global__ void __launch_bounds__(256) to_f16_kernel(const uint4* __restrict__ src,
                                                     uint4* __restrict__ dst, int64_t n8,
                                                     const int* __restrict__ exps, int which) {
  const float p2 = exp2i(exps[which]);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = bf16x8_to_f16x8_scaled(src[i], p2);
}

// fp32 dQ accumulator ([P][S4/4][hl][D][4] with S4 = S rounded up to a multiple of 4,
// holding 2^(kp+edo+ev+ek) dQ) -> bf16 dQ [P][S][hl][D].  A block reads 4 x 256 consecutive
// float4 (each four rows of one d) into shared memory, coalesced, four independent loads per
// thread; then each group of 8 threads, which holds 8 d of four rows, writes them as rows:
// thread j of the group the 4 d starting at 4 (j % 2) of row j / 2 (8 bytes).  n4 (the
// number of float4) is a multiple of 8, so a group never straddles the end.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float4* __restrict__ acc,
                                                     __nv_bfloat16* __restrict__ dq, int64_t S,
                                                     int hl, int D, int64_t n4,
                                                     const int* __restrict__ exps, int kp) {
  constexpr int U = 4;
  // per sub-tile 32 groups of 32 floats, plus one word of padding per group so that the
  // row reads below spread over the banks
  __shared__ float tile[U][32 * 33];
  const int4 ex = *reinterpret_cast<const int4*>(exps);
  const int sh = -(kp + ex.w + ex.z + ex.y);
  const float m1 = exp2i(sh / 2), m2 = exp2i(sh - sh / 2);   // 2^sh, same-sign factors
  const int64_t S4q = (S + 3) / 4;
  const int tid = threadIdx.x, grp = tid / 8, j = tid % 8;
  const int k = j / 2, h = j % 2;                             // output row, d half
  for (int64_t base = (int64_t)blockIdx.x * 256 * U; base < n4;
       base += (int64_t)gridDim.x * 256 * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = base + 256 * u + tid;
      v[u] = (g < n4 && ULY_IN_BOUNDS(g, 1, (uint64_t)n4)) ? acc[g]
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float* t = tile[u] + grp * 33 + j * 4;
      t[0] = v[u].x;
      t[1] = v[u].y;
      t[2] = v[u].z;
      t[3] = v[u].w;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g0 = base + 256 * u + 8 * grp;   // the group's first float4: d = 8 d8
      if (g0 >= n4) continue;
      const int d = (int)(g0 % D);
      int64_t t = g0 / D;
      const int hh = (int)(t % hl);
      t /= hl;
      const int64_t q4 = t % S4q, r = t / S4q;
      const int64_t qrow = 4 * q4 + k;
      if (qrow >= S) continue;
      const float* src = tile[u] + grp * 33 + (4 * h) * 4 + k;   // float4 4h + m, component k
      uint2 o;
      o.x = pack_bf16x2(src[0] * m1 * m2, src[4] * m1 * m2);
      o.y = pack_bf16x2(src[8] * m1 * m2, src[12] * m1 * m2);
      const int64_t dst = ((r * S + qrow) * hl + hh) * D + d + 4 * h;
      if (ULY_IN_BOUNDS(dst, 4, (uint64_t)(n4 / S4q) * S))
        *reinterpret_cast<uint2*>(dq + dst) = o;
    }
    __syncthreads();
  }
}

// kp of the plan's scale: 2^kp scale in [2^7, 2^8) (kp within [-30, 30]).
int p_exponent(float scale) {
  int e = 0;
  std::frexp(scale, &e);            // scale = f 2^e, f in [0.5, 1)
  int kp = 8 - e;
  return kp < -30 ? -30 : (kp > 30 ? 30 : kp);
}

template <int D>
cudaError_t launch_bwd_d(const Plan& p, const void* q, const void* k, const void* v,
                         const void* o, const void* o_lo, const float* lse, const void* d_o,
                         void* dq, void* dk, void* dv, void* workspace, cudaStream_t st) {
  const int hl = p.H / p.P, gl = p.G / p.P;
  const BwdWorkspace ws = bwd_workspace_layout(p);
  char* wsb = static_cast<char*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(wsb + ws.dq_acc);
  float* delta = reinterpret_cast<float*>(wsb + ws.delta);
  void* q16 = wsb + ws.q16;
  void* do16 = wsb + ws.do16;
  void* k16 = wsb + ws.k16;
  void* v16 = wsb + ws.v16;
  uint32_t* scal = reinterpret_cast<uint32_t*>(wsb + ws.scal);
  const int* exps = reinterpret_cast<const int*>(scal + 8);
  const int kp = p_exponent(p.scale);
  const int64_t rows = (int64_t)p.P * p.S * hl;
  const int64_t cap = (int64_t)num_sms(p.device) * 16;
  {
    cudaError_t e = cudaMemsetAsync(scal, 0, 64, st);
    if (e != cudaSuccess) return e;
    const int64_t nq8 = rows * D / 8, nk8 = (int64_t)p.P * p.S * gl * D / 8;
    const int64_t ba = std::min<int64_t>((nq8 + 255) / 256, (int64_t)num_sms(p.device) * 8);
    bwd_amax_kernel<<<(unsigned)std::max<int64_t>(ba, 1), 256, 0, st>>>(
        static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<const uint4*>(v),
        static_cast<const uint4*>(d_o), nq8, nk8, scal, std::ldexp(p.scale, kp), D, p.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the accumulator covers S rounded up to a multiple of 4 rows (S4 >= S)
    const int64_t acc8 = (int64_t)p.P * ((p.S + 3) & ~(int64_t)3) * hl * D / 8;
    const int64_t threads = std::max<int64_t>(rows * (D / 8), acc8);
    const int64_t blocks = (threads + 255) / 256;
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(o_lo),
        static_cast<const __nv_bfloat16*>(d_o), static_cast<const __nv_bfloat16*>(q), delta,
        dq_acc, static_cast<uint4*>(q16), static_cast<uint4*>(do16), rows, p.S, hl, acc8, exps);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t b8 = std::min<int64_t>((nk8 + 255) / 256, cap);
    to_f16_kernel<<<(unsigned)b8, 256, 0, st>>>(static_cast<const uint4*>(k),
                                                 static_cast<uint4*>(k16), nk8, exps, 1);
    to_f16_kernel<<<(unsigned)b8, 256, 0, st>>>(static_cast<const uint4*>(v),
                                                 static_cast<uint4*>(v16), nk8, exps, 2);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const char* err = nullptr;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t dq4[4] = {(uint64_t)D, (uint64_t)hl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)hl * D * 2, (uint64_t)p.S * hl * D * 2};
  const uint64_t dk4[4] = {(uint64_t)D, (uint64_t)gl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)gl * D * 2, (uint64_t)p.S * gl * D * 2};
  // the maps read the fp16 copies (TMA moves 16-bit elements either way)
  if (!make_tmap_4d_bf16(&tq, q16, dq4, sq, 64, BMI, &err) ||
      !make_tmap_4d_bf16(&tdo, do16, dq4, sq, 64, BMI, &err) ||
      !make_tmap_4d_bf16(&tk, k16, dk4, sk, 64, BN, &err) ||
      !make_tmap_4d_bf16(&tv, v16, dk4, sk, 64, BN, &err))
    return cudaErrorInvalidValue;
  BwdArgs a;
  a.lse = lse;
  a.delta = delta;
  a.exps = exps;
  a.kp = kp;
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
  a.log2_scale = log2f(p.scale) + (float)kp;
  a.status = p.status;
  a.limit_ns = p.limit_ns;
  a.flags = p.cfg.flags;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdLayout<D>::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.P * gl * a.nkb;
  attn_bwd_kernel<D><<<(unsigned)blocks, kThreads, BwdLayout<D>::kBytes, st>>>(tq, tk, tv, tdo, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n4 = (int64_t)p.P * ((p.S + 3) / 4) * hl * D;   // float4 of the accumulator
  const int64_t blocks_dq = std::min<int64_t>((n4 + 1023) / 1024, cap);
  bwd_dq_kernel<<<(unsigned)blocks_dq, 256, 0, st>>>(reinterpret_cast<const float4*>(dq_acc),
                                                     static_cast<__nv_bfloat16*>(dq), p.S, hl, D,
                                                     n4, exps, kp);
  return cudaGetLastError();
}

}  // namespace

BwdWorkspace bwd_workspace_layout(const Plan& p) {
  const size_t hl = p.H / p.P, gl = p.G / p.P, S = (size_t)p.S, P = p.P, D = p.D;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdWorkspace w;
  size_t off = 0;
  w.dq_acc = off; off += al(P * ((S + 3) & ~size_t(3)) * hl * D * sizeof(float));
  w.delta = off;  off += al(P * hl * S * sizeof(float));
  w.q16 = off;    off += al(P * S * hl * D * 2);
  w.do16 = off;   off += al(P * S * hl * D * 2);
  w.k16 = off;    off += al(P * S * gl * D * 2);
  w.v16 = off;    off += al(P * S * gl * D * 2);
  w.scal = off;   off += 256;
  w.total = off;
  return w;
}

size_t bwd_workspace_bytes(const Plan& p, size_t* dq_acc_off, size_t* delta_off) {
  const BwdWorkspace w = bwd_workspace_layout(p);
  if (dq_acc_off) *dq_acc_off = w.dq_acc;
  if (delta_off) *delta_off = w.delta;
  return w.total;
}

cudaError_t launch_attn_bwd(const Plan& p, const void* q, const void* k, const void* v,
                            const void* o, const void* o_lo, const float* lse, const void* d_o,
                            void* dq, void* dk, void* dv, void* workspace, cudaStream_t st) {
  if (p.D == 64) return launch_bwd_d<64>(p, q, k, v, o, o_lo, lse, d_o, dq, dk, dv, workspace, st);
  return launch_bwd_d<128>(p, q, k, v, o, o_lo, lse, d_o, dq, dk, dv, workspace, st);
}

ULY_DEBUG_COUNTER_READER(attn_bwd)

}  // namespace uly
