// Local QKV projection of every sequence shard and its backward.
//
// "Snowflake's Ulysses trick ..." para 2: each rank first computes its local QKV
// projection qkv[s][c] = sum_k x[s][k] * w[c][k].  All virtual ranks share the weight, so
// the projection of all shards is one GEMM with M = S (shard r is rows r*S/P ..).  The
// training step also needs its backward: dx = dqkv w and dw = dqkv^T x.
//
// One tcgen05 GEMM kernel serves all three: out[m][n] = sum_k A(m, k) B(n, k) with each
// operand either K-major (k contiguous in memory) or MN-major (m or n contiguous).
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

template <bool A_MN, bool B_MN, bool OUT_F32>
__global__ void __launch_bounds__(128, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                void* __restrict__ out, int M, int N, int K, int* status, uint64_t limit_ns) {
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
      if (A_MN) {
        for (int b = 0; b < BM / 64; ++b)
          tma_load_2d(sA + s * A_BYTES + b * kAtom, &tm_a, &full[s], m0 + 64 * b, kb * BK);
      } else {
        tma_load_2d(sA + s * A_BYTES, &tm_a, &full[s], kb * BK, m0);
      }
      if (B_MN) {
        for (int b = 0; b < BN / 64; ++b)
          tma_load_2d(sB + s * B_BYTES + b * kAtom, &tm_b, &full[s], n0 + 64 * b, kb * BK);
      } else {
        tma_load_2d(sB + s * B_BYTES, &tm_b, &full[s], kb * BK, n0);
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
      if (gm < M && gn < N) {
        if (OUT_F32) {
          float* orow = static_cast<float*>(out) + (size_t)gm * N;
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
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + (size_t)gm * N;
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

// out[M][N] = sum_k A(m, k) B(n, k); a and b are row-major [rows][cols] bf16 arrays.
template <bool A_MN, bool B_MN, bool OUT_F32>
cudaError_t run_gemm(const Plan& p, const void* a, uint64_t a_cols, uint64_t a_rows,
                     const void* b, uint64_t b_cols, uint64_t b_rows, void* out, int M, int N,
                     int K, cudaStream_t st) {
  CUtensorMap ta, tb;
  const char* err = nullptr;
  // K-major operand: box {64 k, 128 or 256 rows}; MN-major: box {64 m or n, 64 k-rows}
  if (!make_tmap_2d_bf16(&ta, a, a_cols, a_rows, a_cols * 2, 64, A_MN ? 64 : BM, &err) ||
      !make_tmap_2d_bf16(&tb, b, b_cols, b_rows, b_cols * 2, 64, B_MN ? 64 : BN, &err))
    return cudaErrorInvalidValue;
  auto kern = gemm_kernel<A_MN, B_MN, OUT_F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  kern<<<grid, 128, SMEM_BYTES, st>>>(ta, tb, out, M, N, K, p.status, p.limit_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qkv_gemm(const Plan& p, const void* x, const void* w, void* out,
                            cudaStream_t st) {
  const int M = (int)p.S, K = p.hidden, N = (p.H + 2 * p.G) * p.D;
  return run_gemm<false, false, false>(p, x, K, M, w, K, N, out, M, N, K, st);
}

cudaError_t launch_qkv_gemm_bwd(const Plan& p, const void* x, const void* w, const void* dqkv,
                                void* dx, float* dw, cudaStream_t st) {
  const int S = (int)p.S, Hd = p.hidden, C = (p.H + 2 * p.G) * p.D;
  if (dx) {
    // dx[s][h] = sum_c dqkv[s][c] w[c][h]
    cudaError_t e = run_gemm<false, true, false>(p, dqkv, C, S, w, Hd, C, dx, S, Hd, C, st);
    if (e != cudaSuccess) return e;
  }
  if (dw) {
    // dw[c][h] = sum_s dqkv[s][c] x[s][h]
    cudaError_t e = run_gemm<true, true, true>(p, dqkv, C, S, x, Hd, S, dw, C, Hd, S, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace uly
