// Causal GQA attention forward of every virtual rank's head group, with logsumexp.
//
// "Snowflake's Ulysses trick ..." para 2: after the seq->head all-to-all each rank holds
// the full sequence for its heads and, heads not interacting, runs flash attention on
// them on its own.  "Ulysses Sequence Parallelism: Training with
// Million-Token Contexts" para 3: tiling never materialises the S x S score matrix.
//
// Design (sm_103a, tcgen05):
//   * one CTA = one (rank, query head, 256-row block) as two 128-row query tiles Q0, Q1
//     that share every K/V tile; blocks are issued heaviest (longest causal prefix) first
//     and neighbouring blocks are the query heads of one KV head, so K/V stay in L2;
//   * warp 8 (TMA): Q0/Q1 once, then K_j and V_j into a 2-deep ring (128-byte swizzle);
//   * warps 9 and 10 (MMA, one thread each, one per query tile t): S_t = Q_t K_j^T into
//     TMEM (fp32, 128 columns), then O_t += P_t V_j with P_t read from TMEM (bf16, written
//     over S_t; the same thread issues P_t V_j before the next S_t, so in order).  The two
//     threads take turns, unit by unit, in the order P_0 V_{j-1}, S_0(j), P_1 V_{j-1},
//     S_1(j), ...: so one tile's softmax runs while the tensor core works on the other
//     tile.  One thread spends ~60 cycles issuing a tcgen05.mma and ~150 on a commit,
//     against the tensor core's 64 cycles for a 128 x 128 x 16 step; with two threads the
//     barrier waits and commits of one overlap the other's issue.  They poll for P without
//     suspending, so they resume as soon as the softmax is done.  Both release K/V slots;
//   * warps 0-3 / 4-7: the online softmax of Q0 / Q1, one thread per row (= TMEM lane),
//     in the log2 domain, with lazy rescaling of O (only when the running max grows by
//     more than 2^8); they also write O / l (bf16), optionally its bf16 rounding residual
//     (so a backward pass can form dO.O to ~16 bits), and lse at the end;
//   * causal tile skipping: Q0 sees KV tiles 0..m0/128, Q1 one more.
// TMEM: S0 [0,128), S1 [128,256), O0 [256, 256+D), O1 [256+D, 256+2D) of 512 columns.
//
// The same kernel, instantiated with kRing, runs one step of ring attention (the method
// "Snowflake's Ulysses trick ..." para 3 compares against) on the virtual ranks: the sequence
// stays sharded, rank r holds its queries [S/P][H][D] and, in step t, the K/V shard
// r - t (ranks r < t hold shards after theirs, which the causal mask hides entirely, and
// do not run).  Step 0 is the causal diagonal block; later steps are full blocks.  The
// running (max, sum, fp32 accumulator) state of every row is kept in HBM between steps and
// loaded into TMEM before the first P V; rank r writes its normalised output at step r.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int BM = 128, BN = 128;
constexpr int kThreads = 352;
constexpr int kTmaWarp = 8, kMmaWarp = 9;   // MMA warps 9 (tile 0) and 10 (tile 1)
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 128 * 64 * 2;   // one [128 rows][64 elements] bf16 box

template <int D>
struct Layout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kQ = 0;
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = 4 * kTile;
  static constexpr int kBar = 6 * kTile;
  static constexpr int kBytes = kBar + 256 + 1024;
};

struct FwdArgs {
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;   // optional: bf16(O - bf16(O)), for the backward's row terms
  float* lse;
  int S, hl, gl, group, n_mb;
  float scale_log2;
  int* status;
  uint64_t limit_ns;
  uint32_t flags;
  // ring steps only: S is the shard length S/P, hl = H, gl = G
  int ring_t;
  float* acc;      // [P][S/P][H][D] fp32, unnormalised output
  float* mstate;   // [P][H][S/P] running max (log2 domain, scale applied)
  float* lstate;   // [P][H][S/P] running sum
};

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// TMEM -> registers: 32 lanes x 128 consecutive 32-bit columns in one load and one wait
// (r[c][i] = column 32 c + i), so the four 32-column parts are fetched together.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[4][32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127"
      "}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      :
        "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]), "=r"(r[0][7]),
        "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]), "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]),
        "=r"(r[0][16]), "=r"(r[0][17]), "=r"(r[0][18]), "=r"(r[0][19]), "=r"(r[0][20]), "=r"(r[0][21]), "=r"(r[0][22]), "=r"(r[0][23]),
        "=r"(r[0][24]), "=r"(r[0][25]), "=r"(r[0][26]), "=r"(r[0][27]), "=r"(r[0][28]), "=r"(r[0][29]), "=r"(r[0][30]), "=r"(r[0][31]),
        "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
        "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]), "=r"(r[1][14]), "=r"(r[1][15]),
        "=r"(r[1][16]), "=r"(r[1][17]), "=r"(r[1][18]), "=r"(r[1][19]), "=r"(r[1][20]), "=r"(r[1][21]), "=r"(r[1][22]), "=r"(r[1][23]),
        "=r"(r[1][24]), "=r"(r[1][25]), "=r"(r[1][26]), "=r"(r[1][27]), "=r"(r[1][28]), "=r"(r[1][29]), "=r"(r[1][30]), "=r"(r[1][31]),
        "=r"(r[2][0]), "=r"(r[2][1]), "=r"(r[2][2]), "=r"(r[2][3]), "=r"(r[2][4]), "=r"(r[2][5]), "=r"(r[2][6]), "=r"(r[2][7]),
        "=r"(r[2][8]), "=r"(r[2][9]), "=r"(r[2][10]), "=r"(r[2][11]), "=r"(r[2][12]), "=r"(r[2][13]), "=r"(r[2][14]), "=r"(r[2][15]),
        "=r"(r[2][16]), "=r"(r[2][17]), "=r"(r[2][18]), "=r"(r[2][19]), "=r"(r[2][20]), "=r"(r[2][21]), "=r"(r[2][22]), "=r"(r[2][23]),
        "=r"(r[2][24]), "=r"(r[2][25]), "=r"(r[2][26]), "=r"(r[2][27]), "=r"(r[2][28]), "=r"(r[2][29]), "=r"(r[2][30]), "=r"(r[2][31]),
        "=r"(r[3][0]), "=r"(r[3][1]), "=r"(r[3][2]), "=r"(r[3][3]), "=r"(r[3][4]), "=r"(r[3][5]), "=r"(r[3][6]), "=r"(r[3][7]),
        "=r"(r[3][8]), "=r"(r[3][9]), "=r"(r[3][10]), "=r"(r[3][11]), "=r"(r[3][12]), "=r"(r[3][13]), "=r"(r[3][14]), "=r"(r[3][15]),
        "=r"(r[3][16]), "=r"(r[3][17]), "=r"(r[3][18]), "=r"(r[3][19]), "=r"(r[3][20]), "=r"(r[3][21]), "=r"(r[3][22]), "=r"(r[3][23]),
        "=r"(r[3][24]), "=r"(r[3][25]), "=r"(r[3][26]), "=r"(r[3][27]), "=r"(r[3][28]), "=r"(r[3][29]), "=r"(r[3][30]), "=r"(r[3][31])
      : "r"(taddr)
      : "memory");
}

// Non-blocking test of a barrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_wait, but polls without suspending the thread, so it resumes as soon as the phase
// completes.  For the single MMA-issuing threads, whose wake-up is on the critical path.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*w.abort) return false;
    if (*reinterpret_cast<volatile int*>(w.status) != kOk) {   // another CTA gave up
      *w.abort = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > w.limit_ns) {
      atomicCAS(w.status, kOk, kErrTimeout);
      *w.abort = 1;
      __threadfence_block();
      return false;
    }
  }
}

template <int D, bool kRing>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]
  uint64_t* v_full = bars + 5;    // [2]
  uint64_t* v_empty = bars + 7;   // [2]
  uint64_t* s_full = bars + 9;    // [2] one per query tile
  uint64_t* p_full = bars + 11;   // [2]
  uint64_t* o_done = bars + 13;   // [2]
  uint64_t* drain = bars + 15;    // [2] one per MMA thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* units_done = abort_flag + 1;   // [2] issue units each MMA thread has issued

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Block -> (rank, local query head, 256-row block), heaviest blocks first.
  const int per_rank = a.hl * a.n_mb;
  const int rb = (int)blockIdx.x / per_rank;                // rank within the launch
  const int r = (kRing ? a.ring_t : 0) + rb;
  const bool full_blk = kRing && a.ring_t > 0;   // a shard before this rank's own: no mask
  const int rem = (int)blockIdx.x - rb * per_rank;
  const int mb = a.n_mb - 1 - rem / a.hl;
  const int hh = rem % a.hl;
  const int gg = hh / a.group;
  const int m0 = mb * 2 * BM;
  const int n_kv = (a.S + BN - 1) / BN;
  const int n0 = full_blk ? n_kv : min(m0 / BN + 1, n_kv);
  const int n1 = full_blk ? n_kv : min(m0 / BN + 2, n_kv);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    units_done[0] = units_done[1] = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);   // both MMA threads release a K / V slot
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 2);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);    // one arrival per softmax warp
      mbar_init(&o_done[i], 1);
      mbar_init(&drain[i], 1);
    }
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
      mbar_arrive_expect_tx(q_full, 2 * L::kTile);
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < D / 64; ++b)
          tma_load_4d(smem + L::kQ + t * L::kTile + b * kBox, &tm_q, q_full, 64 * b, hh,
                      m0 + t * BM, r);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n1; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (j >= 2 && !mbar_wait(&k_empty[st], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_4d(smem + L::kK + st * L::kTile + b * kBox, &tm_k, &k_full[st], 64 * b, gg,
                      j * BN, r);
        ++k_issued;
        if (j >= 2 && !mbar_wait(&v_empty[st], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&v_full[st], L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_4d(smem + L::kV + st * L::kTile + b * kBox, &tm_v, &v_full[st], 64 * b, gg,
                      j * BN, r);
        ++v_issued;
      }
      // Every issued copy lands before exit (immediate on the normal path).
      mbar_drain(q_full, 0, a.limit_ns);
      for (int j = k_issued > 2 ? k_issued - 2 : 0; j < k_issued; ++j)
        mbar_drain(&k_full[j & 1], (j >> 1) & 1, a.limit_ns);
      for (int j = v_issued > 2 ? v_issued - 2 : 0; j < v_issued; ++j)
        mbar_drain(&v_full[j & 1], (j >> 1) & 1, a.limit_ns);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    if (lane == 0) {
      const int t = warp - kMmaWarp;   // this thread's query tile
      const int nt = t ? n1 : n0;      // its KV steps; tile 1 may take one more than tile 0
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, false, true);
      // ULY_FLAG_INJECT_STALL: block 0 withholds S_0's first commit, so the softmax warps'
      // bounded wait for it runs out (failure-path test; nothing faults).
      const bool stall = (a.flags & ULY_FLAG_INJECT_STALL) && blockIdx.x == 0 && t == 0;
      bool alive = mbar_wait(q_full, 0, wc);
      // descriptors built once; K-steps add byte offset / 16 (smem addresses < 2^18)
      const uint64_t qa = sdesc_sw128(smem_u32(smem + L::kQ + t * L::kTile), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(smem + L::kV), kBox, 1024);
      auto issue_s = [&](int j) {
        const uint64_t kb = dk0 + (((j & 1) * L::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
          mma_ss(tbase + t * BN, qa + off, kb + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int j) {
        const uint64_t vb = dv0 + (((j & 1) * L::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tbase + 2 * BN + t * D, tbase + t * BN + kk * 8, vb + ((kk * 16 * 128) >> 4),
                 idesc_pv, (j > 0 || kk > 0 || full_blk) ? 1u : 0u);
      };
      // Waits (bounded) until the other thread has issued `need` units.
      auto wait_turn = [&](int need) -> bool {
        if (units_done[1 - t] >= need) return true;
        const uint64_t t0 = globaltimer_ns();
        while (units_done[1 - t] < need) {
          if (*wc.abort) return false;
          if (globaltimer_ns() - t0 > wc.limit_ns) {
            atomicCAS(wc.status, kOk, kErrTimeout);
            *wc.abort = 1;
            return false;
          }
        }
        return true;
      };
      // Unit u: P_t V_{u-1} (u >= 1), then S_t(u) = Q_t K_u^T over the columns P_t held
      // (u < nt).  Tile 0 takes its unit u after tile 1's unit u-1; tile 1 its unit u
      // after tile 0's unit u (or after tile 0's last unit: tile 1 may take one more step).
      // K/V slots of a step only tile 1 takes get one release; no later load waits on them.
      for (int u = 0; alive && u <= nt; ++u) {
        if (u >= 1) {
          if (!mbar_wait_spin(&p_full[t], (u - 1) & 1, wc) ||
              !mbar_wait(&v_full[(u - 1) & 1], ((u - 1) >> 1) & 1, wc)) { alive = false; break; }
        }
        if (u < nt && !mbar_wait(&k_full[u & 1], (u >> 1) & 1, wc)) { alive = false; break; }
        if (!wait_turn(t == 0 ? u : min(u + 1, n0 + 1))) { alive = false; break; }
        tc_fence_after();
        if (u >= 1) issue_pv(u - 1);
        if (u < nt) issue_s(u);
        units_done[t] = u + 1;
        if (u < nt) {
          if (!(stall && u == 0)) mma_commit(&s_full[t]);
        } else {
          mma_commit(&o_done[t]);
        }
        if (u >= 1) mma_commit(&v_empty[(u - 1) & 1]);
        if (u < nt) mma_commit(&k_empty[u & 1]);
      }
      // All issued MMAs complete before TMEM can be freed.
      mma_commit(&drain[t]);
      mbar_drain(&drain[t], 0, a.limit_ns);
    }
  } else {
    // Softmax warpgroups: t = query tile, one thread per row / TMEM lane.
    const int t = warp / 4;
    const int lane_base = (warp % 4) * 32;
    const int row = lane_base + lane;
    const int row_g = m0 + t * BM + row;
    const int nt = t ? n1 : n0;
    const uint32_t ts = tbase + ((uint32_t)lane_base << 16) + t * BN;
    const uint32_t to = tbase + ((uint32_t)lane_base << 16) + 2 * BN + t * D;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    // row offsets: output / accumulator [P][S][H][D], lse / state [P][H][S]
    auto srow = [&]() { return ((size_t)r * a.hl + hh) * a.S + row_g; };
    auto orow_off = [&]() { return (((size_t)r * a.S + row_g) * a.hl + hh) * D; };
    // element extents of o (and acc) and of lse (and the running state), for the debug checks
    // (a ring step launches the ranks ring_t .. P-1 only)
    const uint64_t n_ranks = (kRing ? a.ring_t : 0) + gridDim.x / ((uint64_t)a.hl * a.n_mb);
    const uint64_t ext_o = n_ranks * a.S * a.hl * D, ext_l = n_ranks * a.hl * a.S;
    (void)ext_o; (void)ext_l;
    if (full_blk) {
      const bool live = row_g < a.S && ULY_IN_BOUNDS(orow_off(), D, ext_o) &&
                        ULY_IN_BOUNDS(srow(), 1, ext_l);
      // the state the rank's earlier steps left: O into TMEM before the first P V
      if (live) {
        m_used = a.mstate[srow()];
        l = a.lstate[srow()];
      }
      const float4* arow = reinterpret_cast<const float4*>(a.acc + orow_off());
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 x = live ? arow[8 * c + e] : make_float4(0.f, 0.f, 0.f, 0.f);
          o[4 * e] = __float_as_uint(x.x);
          o[4 * e + 1] = __float_as_uint(x.y);
          o[4 * e + 2] = __float_as_uint(x.z);
          o[4 * e + 3] = __float_as_uint(x.w);
        }
        tmem_st32(to + 32 * c, o);
      }
    }
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[4][32];
      tmem_ld128(ts, s);
      const int kbase = j * BN;
      if ((!full_blk && kbase + BN - 1 > m0 + t * BM) || kbase + BN > a.S) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int kp = kbase + 32 * c + i;
            if ((!full_blk && kp > row_g) || kp >= a.S) s[c][i] = __float_as_uint(-INFINITY);
          }
      }
      // row max: four independent chains of 3-input max
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mq[c] = fmax3(mq[c], __uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1]));
      const float mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
      const float m_new = fmaxf(m_used, mx * sl2);
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0 && !full_blk) {
        m_used = m_new;
      } else if (m_new > m_used + 8.f) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
        rescale = true;
      }
      // p = 2^(s * scale * log2e - m) on pairs: one FFMA2, two MUFU, one FADD2 per pair
      const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_used, -m_used);
      uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])),
                          sc2, nm2),
                    x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          sum2 = fadd2(sum2, f2_pack(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(ts + 16 * c, pk);
      }
      float sum_lo, sum_hi;
      f2_unpack(sum2, sum_lo, sum_hi);
      const float sum = sum_lo + sum_hi;
      l = l * alpha + sum;
      // tcgen05.ld/st are warp-collective: the whole warp rescales when any row needs it
      // (rows that do not need it have alpha = 1).
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(to + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(to + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], 0, wc));
    if (ok && kRing && a.ring_t != r) {
      // not this rank's last step: keep the state for the next one
      tc_fence_after();
      const bool live = row_g < a.S;
      float4* arow = reinterpret_cast<float4*>(a.acc + orow_off());
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(to + 32 * c, o);
        if (live && ULY_IN_BOUNDS(orow_off() + 32 * c, 32, ext_o)) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            arow[8 * c + e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                          __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
        }
      }
      if (live && ULY_IN_BOUNDS(srow(), 1, ext_l)) {
        a.mstate[srow()] = m_used;
        a.lstate[srow()] = l;
      }
    } else if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = a.o + orow_off();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(to + 32 * c, o);
        if (row_g < a.S && ULY_IN_BOUNDS(orow_off() + 32 * c, 32, ext_o)) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * j + 0]) * inv_l, __uint_as_float(o[8 * j + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[8 * j + 2]) * inv_l, __uint_as_float(o[8 * j + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[8 * j + 4]) * inv_l, __uint_as_float(o[8 * j + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[8 * j + 6]) * inv_l, __uint_as_float(o[8 * j + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * j) = v;
            if (a.o_lo) {
              // what the bf16 rounding of O dropped, itself in bf16
              const uint32_t hw[4] = {v.x, v.y, v.z, v.w};
              uint32_t lw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[e]));
                lw[e] = pack_bf16x2(__uint_as_float(o[8 * j + 2 * e]) * inv_l - h.x,
                                    __uint_as_float(o[8 * j + 2 * e + 1]) * inv_l - h.y);
              }
              *reinterpret_cast<uint4*>(a.o_lo + orow_off() + 32 * c + 8 * j) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
      }
      if (row_g < a.S && ULY_IN_BOUNDS(srow(), 1, ext_l))
        a.lse[srow()] = (m_used + lg2_approx(l)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const Plan& p, const void* q, const void* k, const void* v, void* o,
                         void* o_lo, float* lse, cudaStream_t st) {
  const int hl = p.H / p.P, gl = p.G / p.P;
  const char* err = nullptr;
  CUtensorMap tq, tk, tv;
  const uint64_t dq[4] = {(uint64_t)D, (uint64_t)hl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)hl * D * 2, (uint64_t)p.S * hl * D * 2};
  const uint64_t dk[4] = {(uint64_t)D, (uint64_t)gl, (uint64_t)p.S, (uint64_t)p.P};
  const uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)gl * D * 2, (uint64_t)p.S * gl * D * 2};
  if (!make_tmap_4d_bf16(&tq, q, dq, sq, 64, BM, &err) ||
      !make_tmap_4d_bf16(&tk, k, dk, sk, 64, BN, &err) ||
      !make_tmap_4d_bf16(&tv, v, dk, sk, 64, BN, &err))
    return cudaErrorInvalidValue;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.o_lo = static_cast<__nv_bfloat16*>(o_lo);
  a.lse = lse;
  a.S = (int)p.S;
  a.hl = hl;
  a.gl = gl;
  a.group = p.H / p.G;
  a.n_mb = (int)((p.S + 2 * BM - 1) / (2 * BM));
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.status = p.status;
  a.limit_ns = p.limit_ns;
  a.flags = p.cfg.flags;
  a.ring_t = 0;
  a.acc = a.mstate = a.lstate = nullptr;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.P * hl * a.n_mb;
  attn_fwd_kernel<D, false><<<(unsigned)blocks, kThreads, Layout<D>::kBytes, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

// Ring exchange: every rank passes the K and V shard it holds to rank r + 1:
// dst[(r + 1) mod P] = src[r], 16-byte vectors.
__global__ void __launch_bounds__(256) ring_pass_kernel(const uint4* __restrict__ k_src,
                                                        const uint4* __restrict__ v_src,
                                                        uint4* __restrict__ k_dst,
                                                        uint4* __restrict__ v_dst, int P,
                                                        int64_t shard8) {
  const int64_t total = (int64_t)P * shard8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / shard8;
    const int64_t e = i - r * shard8;
    const int64_t d = (r + 1 == P ? 0 : r + 1) * shard8 + e;
    if (!ULY_IN_BOUNDS(d, 1, total)) continue;
    k_dst[d] = __ldcs(k_src + i);
    v_dst[d] = __ldcs(v_src + i);
  }
}

template <int D>
cudaError_t launch_ring_d(const Plan& p, const void* q_seq, const void* k_seq, const void* v_seq,
                          void* o_seq, float* lse, void* workspace, cudaStream_t st) {
  const int n = (int)(p.S / p.P);
  const RingWorkspace ws = ring_workspace_layout(p);
  char* wsb = static_cast<char*>(workspace);
  void* kbuf[2] = {wsb + ws.k[0], wsb + ws.k[1]};
  void* vbuf[2] = {wsb + ws.v[0], wsb + ws.v[1]};
  const char* err = nullptr;
  CUtensorMap tq;
  const uint64_t dq[4] = {(uint64_t)D, (uint64_t)p.H, (uint64_t)n, (uint64_t)p.P};
  const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)p.H * D * 2, (uint64_t)n * p.H * D * 2};
  const uint64_t dk[4] = {(uint64_t)D, (uint64_t)p.G, (uint64_t)n, (uint64_t)p.P};
  const uint64_t sk[3] = {(uint64_t)D * 2, (uint64_t)p.G * D * 2, (uint64_t)n * p.G * D * 2};
  if (!make_tmap_4d_bf16(&tq, q_seq, dq, sq, 64, BM, &err)) return cudaErrorInvalidValue;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o_seq);
  a.o_lo = nullptr;
  a.lse = lse;
  a.S = n;
  a.hl = p.H;
  a.gl = p.G;
  a.group = p.H / p.G;
  a.n_mb = (n + 2 * BM - 1) / (2 * BM);
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.status = p.status;
  a.limit_ns = p.limit_ns;
  a.flags = 0;
  a.acc = reinterpret_cast<float*>(wsb + ws.acc);
  a.mstate = reinterpret_cast<float*>(wsb + ws.m);
  a.lstate = reinterpret_cast<float*>(wsb + ws.l);
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t shard8 = (int64_t)n * p.G * D / 8;
  const int64_t cap = (int64_t)num_sms(p.device) * 8;
  const unsigned pass_blocks = (unsigned)std::min<int64_t>((p.P * shard8 + 255) / 256, cap);
  for (int t = 0; t < p.P; ++t) {
    const void* kc = t == 0 ? k_seq : kbuf[t % 2];
    const void* vc = t == 0 ? v_seq : vbuf[t % 2];
    CUtensorMap tk, tv;
    if (!make_tmap_4d_bf16(&tk, kc, dk, sk, 64, BN, &err) ||
        !make_tmap_4d_bf16(&tv, vc, dk, sk, 64, BN, &err))
      return cudaErrorInvalidValue;
    a.ring_t = t;
    const int64_t blocks = (int64_t)(p.P - t) * p.H * a.n_mb;
    attn_fwd_kernel<D, true><<<(unsigned)blocks, kThreads, Layout<D>::kBytes, st>>>(tq, tk, tv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (t + 1 < p.P) {
      ring_pass_kernel<<<pass_blocks, 256, 0, st>>>(
          static_cast<const uint4*>(kc), static_cast<const uint4*>(vc),
          static_cast<uint4*>(kbuf[(t + 1) % 2]), static_cast<uint4*>(vbuf[(t + 1) % 2]), p.P,
          shard8);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_fwd(const Plan& p, const void* q, const void* k, const void* v, void* o,
                            void* o_lo, float* lse, cudaStream_t st) {
  if (p.D == 64) return launch_fwd_d<64>(p, q, k, v, o, o_lo, lse, st);
  return launch_fwd_d<128>(p, q, k, v, o, o_lo, lse, st);
}

RingWorkspace ring_workspace_layout(const Plan& p) {
  const size_t S = (size_t)p.S, H = p.H, G = p.G, D = p.D;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  RingWorkspace w;
  size_t off = 0;
  for (int i = 0; i < 2; ++i) {
    w.k[i] = off; off += al(S * G * D * 2);
    w.v[i] = off; off += al(S * G * D * 2);
  }
  w.acc = off; off += al(S * H * D * 4);
  w.m = off;   off += al(S * H * 4);
  w.l = off;   off += al(S * H * 4);
  w.total = off;
  return w;
}

cudaError_t launch_ring_attn(const Plan& p, const void* q_seq, const void* k_seq,
                             const void* v_seq, void* o_seq, float* lse, void* workspace,
                             cudaStream_t st) {
  if (p.D == 64) return launch_ring_d<64>(p, q_seq, k_seq, v_seq, o_seq, lse, workspace, st);
  return launch_ring_d<128>(p, q_seq, k_seq, v_seq, o_seq, lse, workspace, st);
}

ULY_DEBUG_COUNTER_READER(attn_fwd)

}  // namespace uly
