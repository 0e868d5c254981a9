// INT8 GEMM of the INT8 route: exact int32 accumulation, per-token x per-channel scales.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science 2.A Mechanism 3 (volatile layers go
// to INT8), [ZH] 2.A weight handling (weights quantised offline).
//
// sm_103a has no tcgen05 integer MMA (ptxas rejects `.kind::i8` for this target), so the
// exact INT8 contraction runs on the warp-level IMMA path (mma.sync m16n8k32 s8.s8.s32).
// Operand tiles still arrive by TMA (128-byte swizzle) into a multi-stage mbarrier
// pipeline fed by one producer warp; eight consumer warps read fragments with ldmatrix
// (conflict-free thanks to the swizzle) and issue the MMAs.
#include "common.cuh"

namespace dit6 {
namespace i8 {

constexpr int BM = 128, BN = 128, BK = 128, STAGES = 4;
constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int TILE_BYTES = BM * BK;  // == BN * BK
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void imma(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// byte address of (row, 16-byte chunk) in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + row * 128 + (((chunk ^ (row & 7)) & 7) << 4);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_int8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const float* __restrict__ a_scale, const float* __restrict__ b_scale, int M,
                int N, int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                int32_t* __restrict__ acc_out, void* ws) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CONSUMERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();

  if (warp == CONSUMERS) {  // ------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(empty(s), ((kb / STAGES) & 1) ^ 1, ws, abort_flag)) break;
        mbar_expect_tx(full(s), STAGE_BYTES);
        tma_load_2d(sbase + s * STAGE_BYTES, &tmA, full(s), kb * BK, m0);
        tma_load_2d(sbase + s * STAGE_BYTES + TILE_BYTES, &tmB, full(s), kb * BK, n0);
        issued = kb + 1;
      }
      if (*abort_flag) {  // let copies still in flight land before the CTA exits
        volatile int no_abort = 0;
        for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
          mbar_wait(full(kb % STAGES), (kb / STAGES) & 1, ws, &no_abort);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumer warps
  const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps: 64 x 32 per warp
  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0;

  for (int kb = 0; kb < num_kb; ++kb) {
    const int s = kb % STAGES;
    if (!mbar_wait(full(s), (kb / STAGES) & 1, ws, abort_flag)) break;
    const uint32_t aB = sbase + s * STAGE_BYTES, bB = aB + TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 32; ++kk) {
      uint32_t af[4][4], bf[2][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        ldsm_x4(swz(aB, wm * 64 + mt * 16 + (lane & 15), kk * 2 + (lane >> 4)), af[mt]);
#pragma unroll
      for (int np = 0; np < 2; ++np)
        ldsm_x4(swz(bB, wn * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3),
                    kk * 2 + ((lane >> 3) & 1)),
                bf[np]);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          imma(acc[mt][nt], af[mt], bf[nt >> 1][(nt & 1) * 2], bf[nt >> 1][(nt & 1) * 2 + 1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  // ---------------------------------------------------------------- epilogue
  const int g = lane >> 2, tg = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = m0 + wm * 64 + mt * 16 + g + h * 8;
      if (row >= M) continue;
      const float sa = a_scale[row];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = n0 + wn * 32 + nt * 8 + tg * 2;
        if (col >= N) continue;
        const int c0 = acc[mt][nt][h * 2], c1 = acc[mt][nt][h * 2 + 1];
        float v0 = __fmul_rn(__fmul_rn((float)c0, sa), b_scale[col]);
        float v1 = __fmul_rn(__fmul_rn((float)c1, sa), b_scale[col + 1]);
        if (bias) {
          v0 = __fadd_rn(v0, bias[col]);
          v1 = __fadd_rn(v1, bias[col + 1]);
        }
        if (epi & EPI_GELU) {
          const float2 g = gelu_erf2(make_float2(v0, v1));
          v0 = g.x;
          v1 = g.y;
        }
        const int64_t off = (int64_t)row * N + col;
        if (epi & EPI_BF16)
          *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(y) + off) = f2_to_bf16x2(v0, v1);
        else
          *reinterpret_cast<float2*>(reinterpret_cast<float*>(y) + off) = make_float2(v0, v1);
        if (acc_out) *reinterpret_cast<int2*>(acc_out + off) = make_int2(c0, c1);
      }
    }
  }
}

}  // namespace i8
}  // namespace dit6

using namespace dit6;

namespace dit6 {
dit_status gemm_int8_tc(const void* a, const float* a_scale, const void* b, const float* b_scale, int64_t m,
                        int64_t n, int64_t k, const float* bias, void* y, int epi, int32_t* acc_out,
                        void* ws, size_t ws_bytes, cudaStream_t st);
dit_status gemm_int8_tc_requant(const void* a, const float* a_scale, const void* b, const float* b_scale, int64_t m,
                                int64_t n, int64_t k, const float* bias, bool gelu, const float* next_scale,
                                void* q_next, float* amax_out, void* ws, cudaStream_t st);
}

extern "C" dit_status dit_qgemm_int8(const void* a, const float* a_scale, const void* b,
                                     const float* b_scale, dit_dtype ab_dt, int64_t m, int64_t n,
                                     int64_t k, const float* bias, dit_act act, void* y,
                                     dit_dtype y_dt, int32_t* acc_debug, void* ws,
                                     size_t ws_bytes, dit_stream_t stream) {
  if (!a || !b || !a_scale || !b_scale || !y || !ws || ws_bytes < WS_BYTES) return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff)
    return DIT_ERR_INVALID_ARG;
  if (y_dt != DIT_F32 && y_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (ab_dt != DIT_I8 && ab_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  const int epi = (y_dt == DIT_BF16 ? EPI_BF16 : 0) | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  if (k % 16 || n % 8) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(a) || !aligned32(b) || !aligned32(y) || !aligned32(ws) ||
      (acc_debug && !aligned32(acc_debug)) || (reinterpret_cast<uintptr_t>(b_scale) & 15) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 15)))
    return DIT_ERR_ALIGNMENT;
  if (ab_dt == DIT_BF16)
    return gemm_int8_tc(a, a_scale, b, b_scale, m, n, k, bias, y, epi, acc_debug,
                        ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(a), (uint64_t)k,
                      (uint64_t)m, (uint64_t)k, i8::BK, i8::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void*>(b), (uint64_t)k,
                      (uint64_t)n, (uint64_t)k, i8::BK, i8::BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(i8::k_gemm_int8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             i8::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  dim3 grid((unsigned)((n + i8::BN - 1) / i8::BN), (unsigned)((m + i8::BM - 1) / i8::BM));
  if (grid.y > 65535) return DIT_ERR_UNSUPPORTED;
  if (launch_pdl(i8::k_gemm_int8, grid, dim3(i8::THREADS), i8::SMEM_BYTES, reinterpret_cast<cudaStream_t>(stream), 1,
                 ta, tb, a_scale, b_scale, (int)m, (int)n, (int)k, bias, y, epi, acc_debug, ws) != cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}

// INT8 GEMM with the requantising epilogue ([EN] 2.A Mechanism 3, 2.A Outlier Smoothing): the
// output quantised for the next INT8 layer with caller-supplied per-token scales, on the
// CTA-pair kernel (bf16-held codes).
extern "C" dit_status dit_qgemm_int8_requant(const void* a, const float* a_scale, const void* b,
                                             const float* b_scale, int64_t m, int64_t n, int64_t k,
                                             const float* bias, dit_act act, const float* next_scale,
                                             void* q_next, float* row_amax, void* ws, size_t ws_bytes,
                                             dit_stream_t stream) {
  if (!a || !b || !a_scale || !b_scale || !next_scale || !q_next || !row_amax || !ws || ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff)
    return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  if (k % 16 || n % 64) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(a) || !aligned32(b) || !aligned32(q_next) || !aligned32(ws) ||
      (reinterpret_cast<uintptr_t>(b_scale) & 15) || (bias && (reinterpret_cast<uintptr_t>(bias) & 15)))
    return DIT_ERR_ALIGNMENT;
  return gemm_int8_tc_requant(a, a_scale, b, b_scale, m, n, k, bias, act == DIT_ACT_GELU_ERF, next_scale, q_next,
                              row_amax, ws, reinterpret_cast<cudaStream_t>(stream));
}
