// The block's two projections and their backward, as tcgen05 GEMMs.
//
// "Snowflake's Ulysses trick ..." para 2: each rank first computes its local QKV
// projection qkv[s][c] = sum_k x[s][k] * w[c][k].  All virtual ranks share the weight, so
// the projection of all shards is one GEMM with M = S (shard r is rows r*S/P ..).  The
// training step also needs its backward: dx = dqkv w and dw = dqkv^T x.
// After the inverse all-to-all restores the sequence sharding (same para), the block ends
// with its output projection y = o wo^T.  Its input is read straight from the attention's
// head layout o[P][S][H/P][D]: the K index c = h*D + d of token s lies in rank c / (H/P*D)
// at offset c % (H/P*D), so the GEMM's operand load performs the head->seq permutation and
// O is never written in the sequence layout.  Its backward writes dO straight into the head
// layout the attention backward reads, so the dO seq->head permutation disappears too.
//
// One tcgen05 GEMM kernel serves all six: out[m][n] = sum_k A(m, k) B(n, k) with each
// operand either K-major (k contiguous in memory) or MN-major (m or n contiguous), read
// through a 3-D tensor map {x, rows, parts}: a plain row-major operand has one part; a
// head-layout operand has P parts of H/P*D columns, and an x coordinate c is loaded from
// part c / split at column c % split (split a multiple of 64, so a 64-wide box never
// straddles two parts).
//   * 128 x 256 output tile per CTA, K in blocks of 64, a 4-deep TMA ring (128-byte
//     swizzle).  K-major tiles are [rows][64] boxes; MN-major tiles are [64 k-rows][64]
//     boxes side by side (8 KB apart) along m or n;
//   * one thread issues tcgen05.mma (M=128, N=256, K=16) into a 256-column fp32 TMEM
//     accumulator; tcgen05.commit frees ring stages;
//   * epilogue: the 4 warps read their 32 TMEM lanes (= output rows) and store bf16 (round
//     to nearest even) or fp32.
// projection:  A = x [S][hidden] (K-major), B = w [C][hidden] (K-major), out bf16 [S][C]
// dx:          A = dqkv [S][C] (K-major), B(n=h, k=c) = w[c][h] (MN-major), out bf16
// dw:          A(m=c, k=s) = dqkv[s][c] (MN-major), B(n=h, k=s) = x[s][h] (MN-major), fp32
// o_proj:      A = o (head layout, K-major), B = wo [hidden][H*D] (K-major), out bf16 [S][hidden]
// d(o):        A = dy [S][hidden] (K-major), B(n=c, k=j) = wo[j][c] (MN-major), out bf16 in
//              the head layout
// dwo^T:       A(m=c, k=s) = o (head layout, MN-major), B(n=j, k=s) = dy[s][j] (MN-major),
//              fp32 stored transposed (dwo[j][c])
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "uly_internal.h"

namespace uly {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr int kAtom = 64 * 128;   // an MN-major [64 k-rows][64] box

// Column x of a multi-part operand lives in part x / split at column x % split.
__device__ __forceinline__ int split_x(int x, int split) { return split ? x % split : x; }
__device__ __forceinline__ int split_part(int x, int split) { return split ? x / split : 0; }

template <bool A_MN, bool B_MN, bool OUT_F32>
__global__ void __launch_bounds__(128, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                void* __restrict__ out, int M, int N, int K, int a_split, int b_split,
                int out_split, int* status, uint64_t limit_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int kblocks = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtl wc{status, abort_flag, limit_ns};

  if (warp == 0 && lane == 0) {
    // TMA producer
    int issued = 0;
    for (int kb = 0; kb < kblocks; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (kb >= STAGES && !mbar_wait(&empty[s], ph ^ 1, wc)) break;
      mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
      // Every x coordinate is a multiple of 64 elements (128 bytes): m0, n0, kb * BK and
      // x % split with split a multiple of 64.  split = 0 (a one-part operand) loads x as
      // it is; past the end it reads zeros.
      if (A_MN) {
        for (int b = 0; b < BM / 64; ++b) {
          const int x = m0 + 64 * b;
          tma_load_3d(sA + s * A_BYTES + b * kAtom, &tm_a, &full[s], split_x(x, a_split), kb * BK,
                      split_part(x, a_split));
        }
      } else {
        const int x = kb * BK;
        tma_load_3d(sA + s * A_BYTES, &tm_a, &full[s], split_x(x, a_split), m0,
                    split_part(x, a_split));
      }
      if (B_MN) {
        for (int b = 0; b < BN / 64; ++b) {
          const int x = n0 + 64 * b;
          tma_load_3d(sB + s * B_BYTES + b * kAtom, &tm_b, &full[s], split_x(x, b_split), kb * BK,
                      split_part(x, b_split));
        }
      } else {
        const int x = kb * BK;
        tma_load_3d(sB + s * B_BYTES, &tm_b, &full[s], split_x(x, b_split), n0,
                    split_part(x, b_split));
      }
      ++issued;
    }
    // Every issued copy has landed before the CTA can exit (immediate on success).
    for (int kb = issued > STAGES ? issued - STAGES : 0; kb < issued; ++kb)
      mbar_drain(&full[kb % STAGES], (kb / STAGES) & 1, limit_ns);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer; descriptors built once per stage, K-steps add offset / 16
    constexpr uint32_t idesc = idesc_bf16(BM, BN, A_MN, B_MN);
    for (int kb = 0; kb < kblocks; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait(&full[s], ph, wc)) break;
      tc_fence_after();
      const uint64_t da = A_MN ? sdesc_sw128(smem_u32(sA + s * A_BYTES), kAtom, 1024)
                               : sdesc_sw128(smem_u32(sA + s * A_BYTES), 16, 1024);
      const uint64_t db = B_MN ? sdesc_sw128(smem_u32(sB + s * B_BYTES), kAtom, 1024)
                               : sdesc_sw128(smem_u32(sB + s * B_BYTES), 16, 1024);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        // K-major: 16 elements = 32 bytes along the row; MN-major: 16 k-rows = 2048 bytes
        const uint32_t oa = (A_MN ? k * 2048 : k * 32) >> 4;
        const uint32_t ob = (B_MN ? k * 2048 : k * 32) >> 4;
        mma_ss(tbase, da + oa, db + ob, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(&empty[s]);
    }
    mma_commit(acc_full);
    if (*abort_flag) mbar_drain(acc_full, 0, limit_ns);
  }
  __syncwarp();

  // Epilogue: warp w owns TMEM lanes (= tile rows) 32w .. 32w+31.
  bool ok = mbar_wait(acc_full, 0, wc);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    const int row = warp * 32 + lane;
    const int gm = m0 + row;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tbase + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      const int gn = n0 + c * 32;
      if (OUT_F32 && out_split < 0) {
        // transposed fp32 output out[n][m]: for each column the warp's 32 rows are 32
        // consecutive floats (one 128-byte store)
        if (gm < M) {
          float* ocol = static_cast<float*>(out) + gm;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (gn + j < N && ULY_IN_BOUNDS((size_t)(gn + j) * M + gm, 1, (uint64_t)M * N))
              ocol[(size_t)(gn + j) * M] = __uint_as_float(r[j]);
        }
      } else if (gm < M && gn < N &&
                 ULY_IN_BOUNDS(
                     (out_split ? ((size_t)(gn / out_split) * M + gm) * out_split + (gn % out_split)
                                : (size_t)gm * N + gn),
                     gn + 32 <= N ? 32 : N - gn, (uint64_t)M * N)) {
        // row-major [M][N], or the head layout [N/split][M][split] (32-column chunks never
        // straddle two parts since split is a multiple of 64)
        const size_t row_off = out_split ? ((size_t)(gn / out_split) * M + gm) * out_split +
                                               (gn % out_split) - gn
                                         : (size_t)gm * N;
        if (OUT_F32) {
          float* orow = static_cast<float*>(out) + row_off;
          if (gn + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(orow + gn + 4 * j) =
                  make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) orow[gn + j] = __uint_as_float(r[j]);
          }
        } else {
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + row_off;
          if (gn + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]));
              v.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
              v.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
              v.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
              *reinterpret_cast<uint4*>(orow + gn + 8 * j) = v;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) orow[gn + j] = __float2bfloat16_rn(__uint_as_float(r[j]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// One GEMM operand: a bf16 array of `parts` row-major [rows][cols] blocks stored one after
// the other (parts = 1: a plain matrix; parts = P, cols = H/P*D: a head-layout tensor whose
// logical columns are part * cols + col).
struct Operand {
  const void* base;
  uint64_t cols, rows, parts;
};

inline Operand plain(const void* base, uint64_t cols, uint64_t rows) {
  return Operand{base, cols, rows, 1};
}

// out[M][N] = sum_k A(m, k) B(n, k).  out_split = 0: out is row-major [M][N]; > 0: the head
// layout [N / out_split][M][out_split]; < 0 (fp32 only): transposed, out[n][m].
template <bool A_MN, bool B_MN, bool OUT_F32>
cudaError_t run_gemm(const Plan& p, Operand a, Operand b, void* out, int M, int N, int K,
                     int out_split, cudaStream_t st) {
  CUtensorMap ta, tb;
  const char* err = nullptr;
  // K-major operand: box {64 k, 128 or 256 rows}; MN-major: box {64 m or n, 64 k-rows}
  const uint64_t da[3] = {a.cols, a.rows, a.parts}, db[3] = {b.cols, b.rows, b.parts};
  const uint64_t sa[2] = {a.cols * 2, a.cols * a.rows * 2};
  const uint64_t sb[2] = {b.cols * 2, b.cols * b.rows * 2};
  if (!make_tmap_3d_bf16(&ta, a.base, da, sa, 64, A_MN ? 64 : BM, &err) ||
      !make_tmap_3d_bf16(&tb, b.base, db, sb, 64, B_MN ? 64 : BN, &err))
    return cudaErrorInvalidValue;
  auto kern = gemm_kernel<A_MN, B_MN, OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  const int a_split = a.parts > 1 ? (int)a.cols : 0, b_split = b.parts > 1 ? (int)b.cols : 0;
  kern<<<grid, 128, SMEM_BYTES, st>>>(ta, tb, out, M, N, K, a_split, b_split, out_split,
                                      p.status, p.limit_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qkv_gemm(const Plan& p, const void* x, const void* w, void* out,
                            cudaStream_t st) {
  const int M = (int)p.S, K = p.hidden, N = (p.H + 2 * p.G) * p.D;
  return run_gemm<false, false, false>(p, plain(x, K, M), plain(w, K, N), out, M, N, K, 0, st);
}

cudaError_t launch_qkv_gemm_bwd(const Plan& p, const void* x, const void* w, const void* dqkv,
                                void* dx, float* dw, cudaStream_t st) {
  const int S = (int)p.S, Hd = p.hidden, C = (p.H + 2 * p.G) * p.D;
  if (dx) {
    // dx[s][h] = sum_c dqkv[s][c] w[c][h]
    cudaError_t e = run_gemm<false, true, false>(p, plain(dqkv, C, S), plain(w, Hd, C), dx, S,
                                                 Hd, C, 0, st);
    if (e != cudaSuccess) return e;
  }
  if (dw) {
    // dw[c][h] = sum_s dqkv[s][c] x[s][h]
    cudaError_t e = run_gemm<true, true, true>(p, plain(dqkv, C, S), plain(x, Hd, S), dw, C, Hd,
                                               S, 0, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_o_proj(const Plan& p, const void* o_head, const void* wo, void* y,
                          cudaStream_t st) {
  const int S = (int)p.S, Hd = p.hidden, HD = p.H * p.D, part = HD / p.P;
  // y[s][j] = sum_c o(s, c) wo[j][c]
  const Operand a{o_head, (uint64_t)part, (uint64_t)S, (uint64_t)p.P};
  return run_gemm<false, false, false>(p, a, plain(wo, HD, Hd), y, S, Hd, HD, 0, st);
}

cudaError_t launch_o_proj_bwd(const Plan& p, const void* o_head, const void* wo, const void* dy,
                              void* do_head, float* dwo, cudaStream_t st) {
  const int S = (int)p.S, Hd = p.hidden, HD = p.H * p.D, part = HD / p.P;
  if (do_head) {
    // dO(s, c) = sum_j dy[s][j] wo[j][c], stored in the head layout
    cudaError_t e = run_gemm<false, true, false>(p, plain(dy, Hd, S), plain(wo, HD, Hd), do_head,
                                                 S, HD, Hd, part, st);
    if (e != cudaSuccess) return e;
  }
  if (dwo) {
    // dwo[j][c] = sum_s dy[s][j] o(s, c), computed as its transpose (m = c, n = j) so that
    // the head-layout operand is A (two boxes per stage) and dy is B; stored transposed
    const Operand a{o_head, (uint64_t)part, (uint64_t)S, (uint64_t)p.P};
    cudaError_t e = run_gemm<true, true, true>(p, a, plain(dy, Hd, S), dwo, HD, Hd, S, -1, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

ULY_DEBUG_COUNTER_READER(proj_gemm)

}  // namespace uly
