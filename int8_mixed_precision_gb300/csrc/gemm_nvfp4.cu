// NVFP4 GEMM of the NVFP4 route on the 5th-generation tensor cores.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science "1. Problem Statement" (Hardware
// Gap: Blackwell supports the NVFP4 micro-scaling format), "3. Key Contributions" 4;
// [IT] "3. Contributi Chiave" 4 (NVFP4 = E2M1).
//
// Y[m,n] = s_gA s_gB sum_k dec(A)[m,k] dec(sA)[m,k/16] dec(B)[n,k] dec(sB)[n,k/16]
//
// Design (sm_103a): tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X (E2M1 operands,
// UE4M3 scales per 16 elements, fp32 accumulator in tensor memory).  One persistent,
// warp-specialised kernel (k_gemm_nvfp4_s), instantiated on 128 x 256 tiles (one CTA per SM)
// or 128 x 128 tiles (two CTAs per SM):
//   warp 0    : TMA producer -- 2-D tiled loads (128-byte swizzle) of the packed A/B tiles and
//               1-D bulk copies of the matching 512-byte scale atoms, into a STAGES-deep ring
//               guarded by full/empty mbarriers;
//   warp 1    : allocates tensor memory; one lane issues each stage's MMAs and a
//               tcgen05.commit per stage that frees the ring slot;
//   4 warps   : scale writers -- read each stage's scale atoms from shared memory and write
//               them into the stage's tensor-memory slot with tcgen05.st (off the tensor
//               pipe), then arrive on the stage's sf_ready barrier;
//   the rest  : epilogue -- tcgen05.ld of the accumulator, global scale (+bias, GELU),
//               bf16/fp32 conversion, 256-bit stores; optionally the output's Hadamard amax.
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// DIT_ERR_TIMEOUT in the workspace, lets in-flight copies and MMAs land, frees its tensor
// memory and exits.
#include "common.cuh"

namespace dit6 {
namespace f4 {

constexpr int BM = 128;
constexpr int BK = 256;              // E2M1 elements per stage (128 bytes per row)
constexpr int KSTEP = 64;            // elements per MMA
constexpr int A_BYTES = BM * BK / 2;  // 16 KB
constexpr int SF_ATOM = 512;          // 128 rows x 4 scales

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}
// instruction descriptor: E2M1 x E2M1, UE4M3 scales, fp32 accumulate, K-major A and B
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.ld of 32 columns without the wait (the caller waits once for several loads)
__device__ __forceinline__ void tc_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}


// ---------------------------------------------------------------------------------------
// Four scale-writer warps move each stage's scale atoms from shared memory into tensor memory
// with tcgen05.st (each warp writes its own lane quarter, reproducing exactly the layout the
// 32x128b.warpx4 copy would produce), instead of tcgen05.cp on the tensor-core unit: a copy
// there costs ~110 cycles of tensor-pipe time.  The MMA thread waits on a per-stage "scales
// ready" barrier.  EPW: epilogue warps (0: one per 32 columns of the tile).
// ---------------------------------------------------------------------------------------
template <int BN, int STAGES, int CTAS, int EPW = 0>
struct SCfg {
  static constexpr int NB = BN / 128;
  static constexpr int B_BYTES = BN * BK / 2;
  static constexpr int SFA_BYTES = 4 * SF_ATOM;
  static constexpr int SFB_BYTES = NB * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 4 + 4 * NB;
  static constexpr int SF_BASE = BN;
  static constexpr int TMEM_USED = SF_BASE + STAGES * 4 * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = EPW ? EPW : BN / 32;   // 16 with BN = 256: 64 columns per warp
  static constexpr int SF_WARP0 = 2 + EPI_WARPS;
  static constexpr int THREADS = (2 + EPI_WARPS + 4) * 32;
  static_assert(TMEM_USED <= 512 / CTAS, "tensor memory");
  static_assert(SMEM_BYTES * CTAS <= 232448, "shared memory");
};

// Epilogue of 32 accumulator columns of one output row: Y = acc * (s_gA s_gB) (+ bias), then
// GELU when asked (epi_values32); stored as bf16 or fp32, with 256-bit stores when the chunk is
// whole and aligned (epi_write32).
__device__ __forceinline__ void epi_values32(const uint32_t (&r)[32], float alpha, int col0, int N,
                                             const float* __restrict__ bias, int epi, float (&v)[32]) {
  const float2 al = make_float2(alpha, alpha);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 p = mul2(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), al);
    v[2 * i] = p.x;
    v[2 * i + 1] = p.y;
  }
  if (bias) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __fadd_rn(v[i], bias[col0 + i < N ? col0 + i : N - 1]);
  }
  if (epi & EPI_GELU) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 g = gelu_erf2(make_float2(v[2 * i], v[2 * i + 1]));
      v[2 * i] = g.x;
      v[2 * i + 1] = g.y;
    }
  }
}
__device__ __forceinline__ void epi_write32(const float (&v)[32], int row, int col0, int M, int N,
                                            void* __restrict__ y, int epi) {
  if (row >= M || col0 >= N) return;
  const int64_t off = (int64_t)row * N + col0;
  if (col0 + 32 <= N && (N % 16) == 0) {
    if (epi & EPI_BF16) {
      U8x32 o0, o1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o0.w[i] = f2_to_bf16x2(v[2 * i], v[2 * i + 1]);
        o1.w[i] = f2_to_bf16x2(v[16 + 2 * i], v[16 + 2 * i + 1]);
      }
      uint16_t* yp = reinterpret_cast<uint16_t*>(y) + off;
      st256(yp, o0);
      st256(yp + 16, o1);
    } else {
      float* yp = reinterpret_cast<float*>(y) + off;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        U8x32 o;
#pragma unroll
        for (int i = 0; i < 8; ++i) o.w[i] = __float_as_uint(v[8 * b + i]);
        st256(yp + 8 * b, o);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (col0 + i >= N) continue;
      if (epi & EPI_BF16)
        reinterpret_cast<__nv_bfloat16*>(y)[off + i] = __float2bfloat16_rn(v[i]);
      else
        reinterpret_cast<float*>(y)[off + i] = v[i];
    }
  }
}
__device__ __forceinline__ void epi_store32(const uint32_t (&r)[32], float alpha, int row, int col0, int M, int N,
                                            const float* __restrict__ bias, void* __restrict__ y, int epi) {
  if (row >= M || col0 >= N) return;
  float v[32];
  epi_values32(r, alpha, col0, N, bias, epi, v);
  epi_write32(v, row, col0, M, N, y, epi);
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}


// AHB > 0 (16, 32 or 64; with EPW = 16, bf16 output): the epilogue also reduces max|H Z| over
// the output Z as stored in bf16 (block Hadamard along N in blocks of AHB, orthonormal) and the
// last CTA writes *q_sg_next = max / (6 * 448) -- the tensor scale dit_hadamard_quant_nvfp4
// derives from Z in its amax pass -- so the next NVFP4 layer's quantisation is one pass.
template <int BN, int STAGES, int CTAS, int EPW = 0, int AHB = 0>
__global__ void __launch_bounds__(SCfg<BN, STAGES, CTAS, EPW>::THREADS, CTAS)
    k_gemm_nvfp4_s(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                   const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N,
                   int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                   void* ws, int stall, float q_isb, float* __restrict__ q_sg_next) {
  pdl_launch_dependents();
  static_assert(EPW == 0 || (CTAS == 1 && EPW == BN / 16), "sixteen epilogue warps: BN = 256 only");
  static_assert(AHB == 0 || EPW != 0, "the output's Hadamard amax needs the 64-column epilogue warps");
  using C = SCfg<BN, STAGES, CTAS, EPW>;
  constexpr int S = STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  // bars: full[S], empty[S], sf_ready[S], acc_full, acc_empty, mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto sf_ready = [&](int s) { return smem_u32(bars + 2 * S + s); };
  const uint32_t afull = smem_u32(bars + 3 * S);
  const uint32_t aempty = smem_u32(bars + 3 * S + 1);
  const uint32_t mma_done = smem_u32(bars + 3 * S + 2);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfa_tile = [&](int s) { return smem + s * C::STAGE_BYTES + A_BYTES + C::B_BYTES; };
  auto sfb_tile = [&](int s) { return sfa_tile(s) + C::SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = K / KSTEP;
  const int num_kb = (ksteps + 3) / 4;
  const int k_atoms = K / KSTEP;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int n_tiles = ((M + BM - 1) / BM) * n_tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(sf_ready(s), 4);
    }
    mbar_init(afull, 1);
    mbar_init(aempty, C::EPI_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {  // -------------------------------------------------- TMA producer
    if (lane == 0 && !stall) {  // stall: a test hook that issues no loads at all
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      uint32_t kc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
        int nb_valid = (N - n0 + 127) / 128;
        if (nb_valid > C::NB) nb_valid = C::NB;
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait(empty(s), ((kc / S) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          const int nsub = min(4, ksteps - kb * 4);
          mbar_expect_tx(full(s), A_BYTES + C::B_BYTES + nsub * SF_ATOM * (1 + nb_valid));
          tma_load_2d(a_tile(s), &tmA, full(s), kb * (BK / 2), m0);
          tma_load_2d(b_tile(s), &tmB, full(s), kb * (BK / 2), n0);
          bulk_load(smem_u32(sfa_tile(s)), a_sf + ((size_t)(m0 / 128) * k_atoms + kb * 4) * SF_ATOM,
                    nsub * SF_ATOM, full(s));
          for (int nb = 0; nb < nb_valid; ++nb)
            bulk_load(smem_u32(sfb_tile(s)) + nb * 4 * SF_ATOM,
                      b_sf + ((size_t)(n0 / 128 + nb) * k_atoms + kb * 4) * SF_ATOM, nsub * SF_ATOM, full(s));
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        const uint32_t first = kc > (uint32_t)S ? kc - S : 0;
        for (uint32_t c = first; c < kc; ++c) mbar_wait(full(c % S), (c / S) & 1, ws, &no_abort);
      }
    }
  } else if (warp == 1) {  // ------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_nvf4(BM, BN);
      uint32_t kc = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
        if (!mbar_wait(aempty, (tc & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait(full(s), (kc / S) & 1, ws, abort_flag) ||
              !mbar_wait(sf_ready(s), (kc / S) & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(4, ksteps - kb * 4);
          for (int j = 0; j < nsub; ++j) {
            const uint32_t sfa_col = C::SF_BASE + (s * 4 + j) * C::SF_COLS;
            tc_mma(tmem, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc, tmem + sfa_col,
                   tmem + sfa_col + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        if (ok) tc_commit(afull);
      }
      tc_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, ws, &no_abort);
    }
    __syncwarp();
  } else if (warp >= C::SF_WARP0) {  // ------------------------------- scale writers
    const int q = warp & 3;  // the lane quarter this warp may write
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t kc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < num_kb; ++kb, ++kc) {
        const int s = kc % S;
        if (!mbar_wait(full(s), (kc / S) & 1, ws, abort_flag)) {
          ok = false;
          break;
        }
        // lane l gets the 16-byte line l of each 512-byte atom: the four scale words of
        // rows l, l+32, l+64, l+96 -- the same words the warpx4 copy puts in every quarter.
        // The stage's 4 x SF_COLS columns go out in one or two wide stores; columns of K steps
        // past the end of K, or of B atoms past N, hold stale words whose products are never
        // stored.
        uint32_t r[4 * C::SF_COLS];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int a = 0; a <= C::NB; ++a) {
            const uint8_t* src = a == 0 ? sfa_tile(s) + j * SF_ATOM : sfb_tile(s) + (a - 1) * 4 * SF_ATOM + j * SF_ATOM;
            const uint4 v = *reinterpret_cast<const uint4*>(src + lane * 16);
            r[j * C::SF_COLS + 4 * a + 0] = v.x;
            r[j * C::SF_COLS + 4 * a + 1] = v.y;
            r[j * C::SF_COLS + 4 * a + 2] = v.z;
            r[j * C::SF_COLS + 4 * a + 3] = v.w;
          }
        }
        const uint32_t col = C::SF_BASE + s * 4 * C::SF_COLS;
        tc_st32(lane_base + col, r);
        if constexpr (C::SF_COLS == 12) tc_st16(lane_base + col + 32, r + 32);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_ready(s));
      }
    }
  } else {  // ----------------------------------------------------- epilogue warps
    const int e = warp - 2;
    const int q = warp & 3;
    const int half = e >> 2;  // 128-column half of the tile (EPW = 0, BN = 256)
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    float q_amax = 0.f;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tc) {
      const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
      if (!mbar_wait(afull, tc & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
      if constexpr (EPW != 0) {
        // sixteen epilogue warps, 64 columns each: load the raw accumulator words, release the
        // accumulator, then scale, add the bias, apply the activation and store -- all of
        // the epilogue's arithmetic overlaps the next tile's MMAs
        const int part = e >> 2;  // 64-column quarter of the 256-column tile
        uint32_t r0[32], r1[32];
        tc_ld32_nowait(tq + part * 64, r0);
        tc_ld32_nowait(tq + part * 64 + 32, r1);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty);
        const int col0 = n0 + part * 64;
        if constexpr (AHB > 0) {
          if (row < M && col0 < N) {  // N % 64 == 0: the 64 columns are one transform unit
            float v0[32], v1[32];
            epi_values32(r0, alpha, col0, N, bias, epi, v0);
            epi_values32(r1, alpha, col0 + 32, N, bias, epi, v1);
            epi_write32(v0, row, col0, M, N, y, epi);
            epi_write32(v1, row, col0 + 32, M, N, y, epi);
            float2 z[32];  // the values as stored (bf16), transformed
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              z[i] = bf16x2_to_f2(f2_to_bf16x2(v0[2 * i], v0[2 * i + 1]));
              z[16 + i] = bf16x2_to_f2(f2_to_bf16x2(v1[2 * i], v1[2 * i + 1]));
            }
            fwht64<AHB>(z);
            const float2 c = make_float2(q_isb, q_isb);
#pragma unroll
            for (int p = 0; p < 32; ++p) z[p] = mul2(z[p], c);
            q_amax = fmaxf(q_amax, amax_range(z, 0, 32));
          }
        } else {
          epi_store32(r0, alpha, row, col0, M, N, bias, y, epi);
          epi_store32(r1, alpha, row, col0 + 32, M, N, bias, y, epi);
        }
        continue;  // the accumulator is already released
      }
      if constexpr (CTAS == 1) {
      if (epi & EPI_BF16) {
        // one CTA per SM: convert the thread's 128 columns to packed bf16 in registers, release
        // the accumulator, then store -- the next tile's MMAs overlap the stores
        uint32_t pk[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc_ld32(tq + half * 128 + c * 32, r);
          const int col0 = n0 + half * 128 + c * 32;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = __fmul_rn(__uint_as_float(r[i]), alpha);
            if (bias) v[i] = __fadd_rn(v[i], bias[col0 + i < N ? col0 + i : N - 1]);
          }
          if (epi & EPI_GELU) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 g = gelu_erf2(make_float2(v[2 * i], v[2 * i + 1]));
              v[2 * i] = g.x;
              v[2 * i + 1] = g.y;
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[c][i] = f2_to_bf16x2(v[2 * i], v[2 * i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col0 = n0 + half * 128 + c * 32;
          if (row >= M || col0 >= N) continue;
          const int64_t off = (int64_t)row * N + col0;
          uint16_t* yp = reinterpret_cast<uint16_t*>(y) + off;
          if (col0 + 32 <= N && (N % 16) == 0) {
            U8x32 o0, o1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              o0.w[i] = pk[c][i];
              o1.w[i] = pk[c][8 + i];
            }
            st256(yp, o0);
            st256(yp + 16, o1);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < N) yp[i] = (uint16_t)(pk[c][i >> 1] >> (16 * (i & 1)));
          }
        }
        continue;  // the accumulator is already released
      }
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // the thread's 128 columns, stored from the accumulator
        uint32_t r[32];
        tc_ld32(tq + half * 128 + c * 32, r);
        epi_store32(r, alpha, row, n0 + half * 128 + c * 32, M, N, bias, y, epi);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty);
    }
    tc_fence_before();
    if constexpr (AHB > 0) {
      const float m = warp_max_f(q_amax);
      if (lane == 0) atomicMax(ws_u32(ws, WS_AMAX), __float_as_uint(m));
    }
  }

  __syncthreads();
  if constexpr (AHB > 0) {  // the last CTA turns the whole output's max|H Z| into its tensor scale
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t t = atomicAdd(ws_u32(ws, WS_TICKET), 1u);
      if (t == gridDim.x - 1) {
        __threadfence();
        const float amax = __uint_as_float(atomicExch(ws_u32(ws, WS_AMAX), 0u));
        *q_sg_next = __fdiv_rn(amax, 2688.0f);
        *ws_u32(ws, WS_TICKET) = 0u;
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

template <int BN, int STAGES, int CTAS, int EPW = 0, int AHB = 0>
static dit_status launch_s(const uint8_t* a, const uint8_t* b, const uint8_t* a_sf, const uint8_t* b_sf,
                           const float* a_gs, const float* b_gs, int M, int N, int K, const float* bias, void* y,
                           int epi, void* ws, cudaStream_t st, float q_isb = 0.f, float* q_sg_next = nullptr) {
  using C = SCfg<BN, STAGES, CTAS, EPW>;
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(K / 2), (uint64_t)M,
                      (uint64_t)(K / 2), BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(K / 2), (uint64_t)N,
                      (uint64_t)(K / 2), BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  static bool attr_done = false;
  auto kern = k_gemm_nvfp4_s<BN, STAGES, CTAS, EPW, AHB>;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  int64_t grid = (int64_t)num_sms() * CTAS;
  if (grid > tiles) grid = tiles;
  if (launch_pdl(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, 1, ta, tb, a_sf, b_sf, a_gs, b_gs,
                 M, N, K, bias, y, epi, ws, test_stall(), q_isb, q_sg_next) != cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}

}  // namespace f4
}  // namespace dit6

using namespace dit6;

// Tile configuration per call (PFLOP/s or microseconds measured on GB300).
//  * 128 x 256 tiles, one CTA per SM, four stages, sixteen 64-column epilogue warps that
//    release their accumulator right after loading it (bias, activation and stores overlap
//    the next tile's MMAs): with the GELU epilogue it leads everywhere (CogVideoX-2B FFN-up 3.27
//    vs 2.69 on 128 x 128 tiles, 5B FFN-up 4.11 vs 3.46, 1080p FFN-up 4.26 vs 3.55); bf16
//    output without GELU when K >= 3072 (17776 tokens, 5B: QKV 224 vs 229 us, out-proj 80.5 vs
//    82.6, FFN-down 243 vs 248; 1080p FFN-up without GELU 1697 vs 1739).
//  * 128 x 256 tiles with eight 128-column epilogue warps that convert to packed bf16 before
//    the release: bf16 output without GELU when K < 3072 (2B QKV 111 vs 113 us with sixteen
//    warps); fp32 output when K >= 3072 and N is a multiple of 256.
//  * 128 x 128 tiles, two CTAs per SM (three stages each, 108 KB of shared memory): the two
//    independent MMA streams hide each other's epilogue; fp32 output otherwise, and bf16 output
//    with N off the 256 grid and K >= 4096 (2B FFN-down, N = 1920: 4.39 vs 4.32).
static dit_status nvfp4_gemm_dispatch(const uint8_t* a, const uint8_t* a_sf, const float* a_gs, const uint8_t* b,
                                      const uint8_t* b_sf, const float* b_gs, int M, int N, int K, const float* bias,
                                      void* y, int epi, void* ws, cudaStream_t st) {
  const bool wide = (epi & EPI_BF16) ? !(N % 256 != 0 && K >= 4096) : (K >= 3072 && N % 256 == 0);
  if ((epi & EPI_GELU) || (wide && (epi & EPI_BF16) && K >= 3072))
    return f4::launch_s<256, 4, 1, 16>(a, b, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y, epi, ws, st);
  if (wide) return f4::launch_s<256, 4, 1>(a, b, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y, epi, ws, st);
  return f4::launch_s<128, 3, 2>(a, b, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y, epi, ws, st);
}

extern "C" dit_status dit_qgemm_nvfp4_amax(const uint8_t* a, const uint8_t* a_sf, const float* a_gs,
                                           const uint8_t* b, const uint8_t* b_sf, const float* b_gs, int64_t m,
                                           int64_t n, int64_t k, const float* bias, dit_act act, void* y,
                                           int hblock, float* tensor_scale_out, void* ws, size_t ws_bytes,
                                           dit_stream_t stream) {
  if (!a || !a_sf || !a_gs || !b || !b_sf || !b_gs || !y || !tensor_scale_out || !ws || ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff)
    return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  if (hblock != 16 && hblock != 32 && hblock != 64) return DIT_ERR_UNSUPPORTED;
  if (k % 64 || n % 64) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(a) || !aligned32(b) || !aligned32(a_sf) || !aligned32(b_sf) || !aligned32(y) || !aligned32(ws))
    return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int epi = EPI_BF16 | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  const float isb = (float)(1.0 / sqrt((double)hblock));
#define DIT6_AM(HB_)                                                                                     \
  return f4::launch_s<256, 4, 1, 16, HB_>(a, b, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, epi, \
                                          ws, st, isb, tensor_scale_out)
  if (hblock == 16) DIT6_AM(16);
  if (hblock == 32) DIT6_AM(32);
  DIT6_AM(64);
#undef DIT6_AM
}

extern "C" dit_status dit_qgemm_nvfp4(const uint8_t* a, const uint8_t* a_sf, const float* a_gs,
                                      const uint8_t* b, const uint8_t* b_sf, const float* b_gs,
                                      int64_t m, int64_t n, int64_t k, const float* bias,
                                      dit_act act, void* y, dit_dtype y_dt, void* ws,
                                      size_t ws_bytes, dit_stream_t stream) {
  if (!a || !a_sf || !a_gs || !b || !b_sf || !b_gs || !y || !ws || ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff)
    return DIT_ERR_INVALID_ARG;
  if (y_dt != DIT_F32 && y_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  if (k % 64 || n % 8) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(a) || !aligned32(b) || !aligned32(a_sf) || !aligned32(b_sf) || !aligned32(y) ||
      !aligned32(ws))
    return DIT_ERR_ALIGNMENT;
  const int epi = (y_dt == DIT_BF16 ? EPI_BF16 : 0) | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  return nvfp4_gemm_dispatch(a, a_sf, a_gs, b, b_sf, b_gs, (int)m, (int)n, (int)k, bias, y, epi, ws,
                             reinterpret_cast<cudaStream_t>(stream));
}
