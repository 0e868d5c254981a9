// NVFP4 GEMM of the NVFP4 route on the 5th-generation tensor cores.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science "1. Problem Statement" (Hardware
// Gap: Blackwell supports the NVFP4 micro-scaling format), "3. Key Contributions" 4;
// [IT] "3. Contributi Chiave" 4 (NVFP4 = E2M1).
//
// Y[m,n] = s_gA s_gB sum_k dec(A)[m,k] dec(sA)[m,k/16] dec(B)[n,k] dec(sB)[n,k/16]
//
// Design (sm_103a): tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X (E2M1 operands,
// UE4M3 scales per 16 elements, fp32 accumulator in tensor memory).  The default kernel
// (k_gemm_nvfp4_s) is persistent and warp-specialised:
//   warp 0    : TMA producer -- 2-D tiled loads (128-byte swizzle) of the packed A/B tiles and
//               1-D bulk copies of the matching 512-byte scale atoms, into a STAGES-deep ring
//               guarded by full/empty mbarriers;
//   warp 1    : allocates tensor memory; one lane issues each stage's MMAs and a
//               tcgen05.commit per stage that frees the ring slot;
//   4 warps   : scale writers -- read each stage's scale atoms from shared memory and write
//               them into the stage's tensor-memory slot with tcgen05.st (off the tensor
//               pipe), then arrive on the stage's sf_ready barrier;
//   the rest  : epilogue -- tcgen05.ld of the accumulator, global scale (+bias, GELU),
//               bf16/fp32 conversion, 256-bit stores; optionally the output's Hadamard amax
//               or the next layer's NVFP4 encoding.
// The other tile configurations (tcgen05.cp scale copies, CTA pairs, resident scale bands)
// are kept for tests and measurements; the host picks one per call.
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

template <int BN, int STAGES>
struct Cfg {
  static constexpr int NB = BN / 128;                 // 128-row scale atoms of B per stage
  static constexpr int B_BYTES = BN * BK / 2;
  static constexpr int SFA_BYTES = 4 * SF_ATOM;       // 4 K-steps
  static constexpr int SFB_BYTES = NB * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 4 + 4 * NB;          // TMEM columns per K-step's scales
  static constexpr int TMEM_USED = BN + STAGES * 4 * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static_assert(TMEM_USED <= 512, "tensor memory");
};

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 32;  // 8 rows x 16 B core matrices, stacked along rows
  d |= (uint64_t)1 << 46;
  return d;  // no swizzle
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
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
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

template <int BN, int STAGES, bool SPLIT_N>
__global__ void __launch_bounds__(192, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                 const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N,
                 int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                 void* ws) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t tmem_full = smem_u32(bars + 2 * STAGES);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfa_tile = [&](int s) { return b_tile(s) + C::B_BYTES; };
  auto sfb_tile = [&](int s) { return sfa_tile(s) + C::SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int ksteps = K / KSTEP;
  const int num_kb = (ksteps + 3) / 4;
  const int k_atoms = K / KSTEP;  // scale atoms per 128-row block along K
  int nb_valid = (N - n0 + 127) / 128;
  if (nb_valid > C::NB) nb_valid = C::NB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(tmem_full, 1);
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

  if (warp == 0) {  // -------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(empty(s), ((kb / STAGES) & 1) ^ 1, ws, abort_flag)) break;
        const int nsub = min(4, ksteps - kb * 4);
        const uint32_t bytes = A_BYTES + C::B_BYTES + nsub * SF_ATOM * (1 + nb_valid);
        mbar_expect_tx(full(s), bytes);
        tma_load_2d(a_tile(s), &tmA, full(s), kb * (BK / 2), m0);
        tma_load_2d(b_tile(s), &tmB, full(s), kb * (BK / 2), n0);
        bulk_load(sfa_tile(s), a_sf + ((size_t)(m0 / 128) * k_atoms + kb * 4) * SF_ATOM,
                  nsub * SF_ATOM, full(s));
        for (int nb = 0; nb < nb_valid; ++nb)
          bulk_load(sfb_tile(s) + nb * 4 * SF_ATOM,
                    b_sf + ((size_t)(n0 / 128 + nb) * k_atoms + kb * 4) * SF_ATOM,
                    nsub * SF_ATOM, full(s));
        issued = kb + 1;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
          mbar_wait(full(kb % STAGES), (kb / STAGES) & 1, ws, &no_abort);
      }
    }
  } else if (warp == 1) {  // ------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr int MMA_N = SPLIT_N ? 128 : BN;
      constexpr uint32_t idesc = idesc_nvf4(BM, MMA_N);
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(full(s), (kb / STAGES) & 1, ws, abort_flag)) break;
        tc_fence_after();
        const int nsub = min(4, ksteps - kb * 4);
        for (int j = 0; j < nsub; ++j) {
          const uint32_t sfa_col = BN + (s * 4 + j) * C::SF_COLS;
          const uint32_t sfb_col = sfa_col + 4;
          tc_cp_sf(tmem + sfa_col, desc_sf(sfa_tile(s) + j * SF_ATOM));
          for (int nb = 0; nb < nb_valid; ++nb)
            tc_cp_sf(tmem + sfb_col + 4 * nb, desc_sf(sfb_tile(s) + nb * 4 * SF_ATOM + j * SF_ATOM));
          const uint64_t ad = desc_sw128(a_tile(s) + j * 32);
          const uint32_t accum = (kb | j) != 0;
          if (SPLIT_N) {
#pragma unroll
            for (int h = 0; h < C::NB; ++h)
              tc_mma(tmem + h * 128, ad, desc_sw128(b_tile(s) + h * 128 * 128 + j * 32), idesc,
                     tmem + sfa_col, tmem + sfb_col + 4 * h, accum);
          } else {
            tc_mma(tmem, ad, desc_sw128(b_tile(s) + j * 32), idesc, tmem + sfa_col,
                   tmem + sfb_col, accum);
          }
        }
        tc_commit(empty(s));
      }
      tc_commit(tmem_full);
      if (*abort_flag) {  // make sure issued MMAs have finished before TMEM is freed
        volatile int no_abort = 0;
        mbar_wait(tmem_full, 0, ws, &no_abort);
      }
    }
    __syncwarp();
  } else {  // ----------------------------------------------------- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = m0 + q * 32 + lane;
    const bool ok = mbar_wait(tmem_full, 0, ws, abort_flag);
    tc_fence_after();
    if (ok) {
      const float alpha = __fmul_rn(*a_gs, *b_gs);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
        const int col0 = n0 + c * 32;
        if (row >= M || col0 >= N) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = __fmul_rn(__uint_as_float(r[i]), alpha);
          if (bias && col0 + i < N) v[i] = __fadd_rn(v[i], bias[col0 + i]);
        }
        if (epi & EPI_GELU) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 g = gelu_erf2(make_float2(v[2 * i], v[2 * i + 1]));
            v[2 * i] = g.x;
            v[2 * i + 1] = g.y;
          }
        }
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
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------------------
// Persistent variant: one CTA per SM walks 128 x BN output tiles; the accumulator is
// ACC_BUFS-buffered in tensor memory so the epilogue of tile t overlaps the MMAs of tile
// t+1; scales get one tensor-memory slot per (stage, K step).
// ---------------------------------------------------------------------------------------
template <int BN, int STAGES, int ACC_BUFS>
struct PCfg {
  static constexpr int NB = BN / 128;
  static constexpr int B_BYTES = BN * BK / 2;
  static constexpr int SFA_BYTES = 4 * SF_ATOM;
  static constexpr int SFB_BYTES = NB * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 4 + 4 * NB;
  static constexpr int SF_BASE = ACC_BUFS * BN;
  static constexpr int TMEM_USED = SF_BASE + STAGES * 4 * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = BN / 32;          // 128 columns per epilogue thread
  static constexpr int THREADS = (2 + EPI_WARPS) * 32;
  static_assert(TMEM_USED <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <int BN, int STAGES, int ACC_BUFS>
__global__ void __launch_bounds__(PCfg<BN, STAGES, ACC_BUFS>::THREADS, 1)
    k_gemm_nvfp4_p(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                   const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N,
                   int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                   void* ws) {
  using C = PCfg<BN, STAGES, ACC_BUFS>;
  constexpr int S = STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  // bars: full[S], empty[S], acc_full[ACC_BUFS], acc_empty[ACC_BUFS], mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * ACC_BUFS + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto afull = [&](int b) { return smem_u32(bars + 2 * S + b); };
  auto aempty = [&](int b) { return smem_u32(bars + 2 * S + ACC_BUFS + b); };
  const uint32_t mma_done = smem_u32(bars + 2 * S + 2 * ACC_BUFS);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfa_tile = [&](int s) { return b_tile(s) + C::B_BYTES; };
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
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), C::EPI_WARPS);
    }
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

  if (warp == 0) {  // -------------------------------------------------- TMA producer
    if (lane == 0) {
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
          bulk_load(sfa_tile(s), a_sf + ((size_t)(m0 / 128) * k_atoms + kb * 4) * SF_ATOM, nsub * SF_ATOM,
                    full(s));
          for (int nb = 0; nb < nb_valid; ++nb)
            bulk_load(sfb_tile(s) + nb * 4 * SF_ATOM, b_sf + ((size_t)(n0 / 128 + nb) * k_atoms + kb * 4) * SF_ATOM,
                      nsub * SF_ATOM, full(s));
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
        const int n0 = (tile % n_tiles_n) * BN;
        int nb_valid = (N - n0 + 127) / 128;
        if (nb_valid > C::NB) nb_valid = C::NB;
        const int buf = tc % ACC_BUFS;
        if (!mbar_wait(aempty(buf), ((tc / ACC_BUFS) & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait(full(s), (kc / S) & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(4, ksteps - kb * 4);
          // all scale copies of the stage first, so the MMAs do not wait on them one by one
          for (int j = 0; j < nsub; ++j) {
            const uint32_t sfa_col = C::SF_BASE + (s * 4 + j) * C::SF_COLS;
            const uint32_t sfb_col = sfa_col + 4;
            tc_cp_sf(tmem + sfa_col, desc_sf(sfa_tile(s) + j * SF_ATOM));
            for (int nb = 0; nb < nb_valid; ++nb)
              tc_cp_sf(tmem + sfb_col + 4 * nb, desc_sf(sfb_tile(s) + nb * 4 * SF_ATOM + j * SF_ATOM));
          }
          for (int j = 0; j < nsub; ++j) {
            const uint32_t sfa_col = C::SF_BASE + (s * 4 + j) * C::SF_COLS;
            tc_mma(d, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc,
                   tmem + sfa_col, tmem + sfa_col + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        if (ok) tc_commit(afull(buf));
      }
      tc_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, ws, &no_abort);
    }
    __syncwarp();
  } else {  // ----------------------------------------------------- epilogue warps
    const int e = warp - 2;
    const int q = warp & 3;
    const int half = e >> 2;            // 128-column part of the tile
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tc) {
      const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
      const int buf = tc % ACC_BUFS;
      if (!mbar_wait(afull(buf), (tc / ACC_BUFS) & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + half * 128 + c * 32, r);
        const int col0 = n0 + half * 128 + c * 32;
        if (row >= M || col0 >= N) continue;
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty(buf));
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------------------
// Band-resident variant (K <= 2048): each persistent CTA walks a contiguous run of 128 x 256
// tiles in M-major order; the A-side scales of the current 128-row band (all K steps) are
// copied into tensor memory once per band, so only the B-side scales move per K step.  The
// scale copies (smem -> tensor memory) have their own limited bandwidth; this halves their
// bytes per MMA.  Single accumulator buffer.
// ---------------------------------------------------------------------------------------
struct RCfg {
  static constexpr int BN = 256, NB = 2, STAGES = 4;
  static constexpr int MAX_KSTEPS = 32;                      // K <= 2048
  static constexpr int B_BYTES = BN * BK / 2;
  static constexpr int SFB_BYTES = NB * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFB_BYTES;
  static constexpr int BAND_BYTES = MAX_KSTEPS * SF_ATOM;    // A-side scales of one band
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAND_BYTES + 1024 + 256;
  static constexpr int SFA_BASE = BN;                        // 4 columns per K step
  static constexpr int SFB_BASE = SFA_BASE + 4 * MAX_KSTEPS; // 4 K steps x 8 columns per stage
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = (2 + EPI_WARPS) * 32;
  static_assert(SFB_BASE + STAGES * 4 * 4 * NB <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__global__ void __launch_bounds__(RCfg::THREADS, 1)
    k_gemm_nvfp4_r(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                   const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N,
                   int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                   void* ws) {
  using C = RCfg;
  constexpr int S = C::STAGES, BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* band = smem + S * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(band + C::BAND_BYTES);
  // bars: full[S], empty[S], acc_full, acc_empty, band_full, band_empty, mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem), band_s = smem_u32(band);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t afull = smem_u32(bars + 2 * S), aempty = smem_u32(bars + 2 * S + 1);
  const uint32_t bfull = smem_u32(bars + 2 * S + 2), bempty = smem_u32(bars + 2 * S + 3);
  const uint32_t mma_done = smem_u32(bars + 2 * S + 4);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfb_tile = [&](int s) { return b_tile(s) + C::B_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = K / KSTEP;
  const int num_kb = (ksteps + 3) / 4;
  const int k_atoms = ksteps;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int n_tiles = ((M + BM - 1) / BM) * n_tiles_n;
  const int per = (n_tiles + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * per;
  const int t_end = min(n_tiles, t_begin + per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(afull, 1);
    mbar_init(aempty, C::EPI_WARPS);
    mbar_init(bfull, 1);
    mbar_init(bempty, 1);
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

  if (warp == 0) {  // -------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      uint32_t kc = 0, bc = 0;
      int cur_band = -1;
      bool ok = true;
      for (int tile = t_begin; tile < t_end && ok; ++tile) {
        const int mb = tile / n_tiles_n;
        const int m0 = mb * BM, n0 = (tile % n_tiles_n) * BN;
        if (mb != cur_band) {  // A-side scales of the new band, all K steps, one bulk copy
          if (!mbar_wait(bempty, (bc & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bfull, k_atoms * SF_ATOM);
          bulk_load(band_s, a_sf + (size_t)mb * k_atoms * SF_ATOM, k_atoms * SF_ATOM, bfull);
          cur_band = mb;
          ++bc;
        }
        int nb_valid = (N - n0 + 127) / 128;
        if (nb_valid > C::NB) nb_valid = C::NB;
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait(empty(s), ((kc / S) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          const int nsub = min(4, ksteps - kb * 4);
          mbar_expect_tx(full(s), A_BYTES + C::B_BYTES + nsub * SF_ATOM * nb_valid);
          tma_load_2d(a_tile(s), &tmA, full(s), kb * (BK / 2), m0);
          tma_load_2d(b_tile(s), &tmB, full(s), kb * (BK / 2), n0);
          for (int nb = 0; nb < nb_valid; ++nb)
            bulk_load(sfb_tile(s) + nb * 4 * SF_ATOM, b_sf + ((size_t)(n0 / 128 + nb) * k_atoms + kb * 4) * SF_ATOM,
                      nsub * SF_ATOM, full(s));
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        const uint32_t first = kc > (uint32_t)S ? kc - S : 0;
        for (uint32_t c = first; c < kc; ++c) mbar_wait(full(c % S), (c / S) & 1, ws, &no_abort);
        if (bc > 0) mbar_wait(bfull, (bc - 1) & 1, ws, &no_abort);
      }
    }
  } else if (warp == 1) {  // ------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_nvf4(BM, BN);
      uint32_t kc = 0, bc = 0, tc = 0;
      int cur_band = -1;
      bool ok = true;
      volatile int no_abort = 0;
      for (int tile = t_begin; tile < t_end && ok; ++tile, ++tc) {
        const int mb = tile / n_tiles_n;
        const int n0 = (tile % n_tiles_n) * BN;
        if (mb != cur_band) {
          if (cur_band >= 0) {  // every MMA reading the old band's scales has finished
            tc_commit(mma_done);
            mbar_wait(mma_done, (bc - 1) & 1, ws, &no_abort);
          }
          if (!mbar_wait(bfull, bc & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int a = 0; a < k_atoms; ++a)
            tc_cp_sf(tmem + C::SFA_BASE + 4 * a, desc_sf(band_s + a * SF_ATOM));
          tc_commit(bempty);  // the band buffer may be refilled once these copies are done
          cur_band = mb;
          ++bc;
        }
        int nb_valid = (N - n0 + 127) / 128;
        if (nb_valid > C::NB) nb_valid = C::NB;
        if (!mbar_wait(aempty, (tc & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait(full(s), (kc / S) & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(4, ksteps - kb * 4);
          for (int j = 0; j < nsub; ++j) {
            const uint32_t sfb_col = C::SFB_BASE + (s * 4 + j) * 4 * C::NB;
            for (int nb = 0; nb < nb_valid; ++nb)
              tc_cp_sf(tmem + sfb_col + 4 * nb, desc_sf(sfb_tile(s) + nb * 4 * SF_ATOM + j * SF_ATOM));
            tc_mma(tmem, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc,
                   tmem + C::SFA_BASE + 4 * (kb * 4 + j), tmem + sfb_col, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        if (ok) tc_commit(afull);
      }
      tc_commit(mma_done);
      mbar_wait(mma_done, bc > 0 ? ((bc - 1) & 1) ^ 0 : 0, ws, &no_abort);
    }
    __syncwarp();
  } else {  // ----------------------------------------------------- epilogue warps
    const int e = warp - 2;
    const int q = warp & 3;
    const int half = e >> 2;
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    uint32_t tc = 0;
    for (int tile = t_begin; tile < t_end; ++tile, ++tc) {
      const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
      if (!mbar_wait(afull, tc & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld32(tmem + ((uint32_t)(q * 32) << 16) + half * 128 + c * 32, r);
        const int col0 = n0 + half * 128 + c * 32;
        if (row >= M || col0 >= N) continue;
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty);
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

static dit_status launch_r(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf, const uint8_t* b_sf,
                           const float* a_gs, const float* b_gs, int M, int N, int K, const float* bias, void* y,
                           int epi, void* ws, cudaStream_t st) {
  using C = RCfg;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(k_gemm_nvfp4_r, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + C::BN - 1) / C::BN);
  int64_t grid = num_sms();
  if (grid > tiles) grid = tiles;
  k_gemm_nvfp4_r<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, st>>>(ta, tb, a_sf, b_sf, a_gs, b_gs, M, N, K, bias,
                                                                    y, epi, ws);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

// ---------------------------------------------------------------------------------------
// Scale-writer variant: four extra warps move each stage's scale atoms from shared memory into
// tensor memory with tcgen05.st (each warp writes its own lane quarter, reproducing exactly
// the layout the 32x128b.warpx4 copy would produce), instead of tcgen05.cp on the tensor-core
// unit.  The MMA thread waits on a per-stage "scales ready" barrier.
// ---------------------------------------------------------------------------------------
// ACC: tensor-memory accumulator buffers (2: the MMAs of tile t+1 run while the epilogue
// drains tile t)
template <int BN, int STAGES, int CTAS, int ACC = 1, int EPW = 0>
struct SCfg {
  static_assert(ACC == 1 || ACC == 2, "accumulator buffers");
  static constexpr int NB = BN / 128;
  static constexpr int B_BYTES = BN * BK / 2;
  static constexpr int SFA_BYTES = 4 * SF_ATOM;
  static constexpr int SFB_BYTES = NB * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 4 + 4 * NB;
  static constexpr int SF_BASE = BN * ACC;
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

__device__ __forceinline__ void tc_st4(uint32_t taddr, const uint4& v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
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

// QHB > 0 (16, 32 or 64): fused epilogue quantisation.  The output Z (after bias and
// activation, rounded to bf16 as it would be stored) is block-Hadamard transformed along N in
// blocks of QHB and NVFP4-encoded with the given tensor scale *q_sg into q_codes / q_sf (the
// layouts dit_hadamard_quant_nvfp4 writes, ready as the next GEMM's A operand); y (bf16) is
// written only when non-null.  max|H Z| over the whole output is reduced through the workspace
// and the last CTA writes *q_sg_next = max / (6 * 448), the tensor scale the unfused quantiser
// would derive from this Z.  Needs BN == 128 and N % 64 == 0.
// AHB > 0 (16, 32 or 64; with EPW = 16, bf16 output): the epilogue also reduces max|H Z| over
// the output Z as stored in bf16 (block Hadamard along N in blocks of AHB, orthonormal) and the
// last CTA writes *q_sg_next = max / (6 * 448) -- the tensor scale dit_hadamard_quant_nvfp4
// derives from Z in its amax pass -- so the next NVFP4 layer's quantisation is one pass.
template <int BN, int STAGES, int CTAS, int QHB = 0, int ACC = 1, int EPW = 0, int AHB = 0>
__global__ void __launch_bounds__(SCfg<BN, STAGES, CTAS, ACC, EPW>::THREADS, CTAS)
    k_gemm_nvfp4_s(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                   const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N,
                   int K, const float* __restrict__ bias, void* __restrict__ y, int epi,
                   void* ws, int stall, const float* __restrict__ q_sg, float q_isb,
                   uint8_t* __restrict__ q_codes, uint8_t* __restrict__ q_sf, float* __restrict__ q_sg_next) {
  static_assert(QHB == 0 || BN == 128, "fused quantisation works on 128-column tiles");
  static_assert(EPW == 0 || (QHB == 0 && CTAS == 1 && EPW == BN / 16), "sixteen epilogue warps: BN = 256 only");
  static_assert(AHB == 0 || EPW != 0, "the output's Hadamard amax needs the 64-column epilogue warps");
  constexpr bool TRACK_AMAX = QHB > 0 || AHB > 0;
  using C = SCfg<BN, STAGES, CTAS, ACC, EPW>;
  constexpr int S = STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  // bars: full[S], empty[S], sf_ready[S], acc_full[ACC], acc_empty[ACC], mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 2 * ACC + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto sf_ready = [&](int s) { return smem_u32(bars + 2 * S + s); };
  auto afull = [&](int b) { return smem_u32(bars + 3 * S + b); };
  auto aempty = [&](int b) { return smem_u32(bars + 3 * S + ACC + b); };
  const uint32_t mma_done = smem_u32(bars + 3 * S + 2 * ACC);
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
    for (int b = 0; b < ACC; ++b) {
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), C::EPI_WARPS);
    }
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
        const int buf = tc % ACC;
        if (!mbar_wait(aempty(buf), ((tc / ACC) & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + buf * BN;
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
            tc_mma(dacc, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc,
                   tmem + sfa_col, tmem + sfa_col + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        if (ok) tc_commit(afull(buf));
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
    const int half = e >> 2;
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    float q_s = 0.f, q_six = 0.f, q_amax = 0.f;
    const int64_t q_upr = N / 64;
    if constexpr (QHB > 0) {
      q_s = *q_sg;
      q_six = __fmul_rn(6.0f, q_s);
    }
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tc) {
      const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
      const int buf = tc % ACC;
      if (!mbar_wait(afull(buf), (tc / ACC) & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
      const uint32_t tacc = tmem + buf * BN;
      if constexpr (EPW != 0) {
        // sixteen epilogue warps, 64 columns each: load the raw accumulator words, release the
        // accumulator, then scale, add the bias, apply the activation and store -- all of the
        // epilogue's arithmetic overlaps the next tile's MMAs
        const int part = e >> 2;  // 64-column quarter of the 256-column tile
        uint32_t r0[32], r1[32];
        tc_ld32_nowait(tacc + ((uint32_t)(q * 32) << 16) + part * 64, r0);
        tc_ld32_nowait(tacc + ((uint32_t)(q * 32) << 16) + part * 64 + 32, r1);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty(buf));
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
      if constexpr (QHB == 0 && CTAS == 1) {
        if (epi & EPI_BF16) {
          // one CTA per SM: convert the thread's 128 columns to packed bf16 in registers, release
          // the accumulator, then store -- the next tile's MMAs overlap the stores
          uint32_t pk[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tc_ld32(tacc + ((uint32_t)(q * 32) << 16) + half * 128 + c * 32, r);
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
          if (lane == 0) mbar_arrive(aempty(buf));
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
      if constexpr (QHB == 0) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld32(tacc + ((uint32_t)(q * 32) << 16) + half * 128 + c * 32, r);
        const int col0 = n0 + half * 128 + c * 32;
        if (row >= M || col0 >= N) continue;
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
      } else {
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {  // two 64-column units of the 128-column tile
        const int col0 = n0 + c2 * 64;
        float2 v[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t r[32];
          tc_ld32(tacc + ((uint32_t)(q * 32) << 16) + c2 * 64 + hh * 32, r);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int cA = col0 + hh * 32 + 2 * i;
            float z0 = __fmul_rn(__uint_as_float(r[2 * i]), alpha);
            float z1 = __fmul_rn(__uint_as_float(r[2 * i + 1]), alpha);
            if (bias) {
              z0 = __fadd_rn(z0, bias[cA < N ? cA : N - 1]);
              z1 = __fadd_rn(z1, bias[cA + 1 < N ? cA + 1 : N - 1]);
            }
            // the value the output would hold in bf16 is what gets transformed
            const float2 za = epi_act2(make_float2(z0, z1), epi);
            v[hh * 16 + i] = bf16x2_to_f2(f2_to_bf16x2(za.x, za.y));
          }
        }
        if (col0 >= N) continue;
        const int ri = row & 127;
        uint32_t* sfw = reinterpret_cast<uint32_t*>(q_sf + ((int64_t)(row >> 7) * q_upr + col0 / 64) * 512 +
                                                    (ri & 31) * 16 + (ri >> 5) * 4);
        if (row >= M) {  // rows padding the scale layout to a multiple of 128: zero scales
          *sfw = 0u;
          continue;
        }
        if (y) {
          uint16_t* yp = reinterpret_cast<uint16_t*>(y) + (int64_t)row * N + col0;
#pragma unroll
          for (int b4 = 0; b4 < 4; ++b4) {
            U8x32 o;
#pragma unroll
            for (int i = 0; i < 8; ++i) o.w[i] = f2_to_bf16x2(v[b4 * 8 + i].x, v[b4 * 8 + i].y);
            st256(yp + b4 * 16, o);
          }
        }
        fwht64<QHB>(v);
        const float2 c = make_float2(q_isb, q_isb);
#pragma unroll
        for (int p = 0; p < 32; ++p) v[p] = mul2(v[p], c);
        q_amax = fmaxf(q_amax, amax_range(v, 0, 32));
        U8x32 out;
        *sfw = nvfp4_encode_unit(v, q_s, q_six, out);
        st256(q_codes + (int64_t)row * (N / 2) + col0 / 2, out);
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty(buf));
    }
    tc_fence_before();
    if constexpr (TRACK_AMAX) {
      const float m = warp_max_f(q_amax);
      if (lane == 0) atomicMax(ws_u32(ws, WS_AMAX), __float_as_uint(m));
    }
  }

  __syncthreads();
  if constexpr (TRACK_AMAX) {  // the last CTA turns the whole output's max|H Z| into its tensor scale
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

template <int BN, int STAGES, int CTAS, int QHB = 0, int ACC = 1, int EPW = 0, int AHB = 0>
static dit_status launch_s(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf, const uint8_t* b_sf,
                           const float* a_gs, const float* b_gs, int M, int N, int K, const float* bias, void* y,
                           int epi, void* ws, cudaStream_t st, const float* q_sg = nullptr, float q_isb = 0.f,
                           uint8_t* q_codes = nullptr, uint8_t* q_sf = nullptr, float* q_sg_next = nullptr) {
  using C = SCfg<BN, STAGES, CTAS, ACC, EPW>;
  static bool attr_done = false;
  auto kern = k_gemm_nvfp4_s<BN, STAGES, CTAS, QHB, ACC, EPW, AHB>;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  int64_t grid = (int64_t)num_sms() * CTAS;
  if (grid > tiles) grid = tiles;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, st>>>(ta, tb, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y,
                                                         epi, ws, test_stall(), q_sg, q_isb, q_codes, q_sf,
                                                         q_sg_next);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

template <int BN, int STAGES, int ACC_BUFS, int CTAS_PER_SM = 1>
static dit_status launch_p(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf,
                           const uint8_t* b_sf, const float* a_gs, const float* b_gs, int M, int N,
                           int K, const float* bias, void* y, int epi, void* ws, cudaStream_t st) {
  using C = PCfg<BN, STAGES, ACC_BUFS>;
  static bool attr_done = false;
  auto kern = k_gemm_nvfp4_p<BN, STAGES, ACC_BUFS>;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  int64_t grid = (int64_t)num_sms() * CTAS_PER_SM;
  if (grid > tiles) grid = tiles;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, st>>>(ta, tb, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y,
                                                         epi, ws);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

template <int BN, int STAGES, bool SPLIT_N>
static dit_status launch(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf,
                         const uint8_t* b_sf, const float* a_gs, const float* b_gs, int M, int N,
                         int K, const float* bias, void* y, int epi, void* ws,
                         cudaStream_t st) {
  using C = Cfg<BN, STAGES>;
  static bool attr_done = false;
  auto kern = k_gemm_nvfp4<BN, STAGES, SPLIT_N>;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  if (grid.y > 65535) return DIT_ERR_UNSUPPORTED;
  kern<<<grid, 192, C::SMEM_BYTES, st>>>(ta, tb, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y, epi, ws);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}


// ---------------------------------------------------------------------------------------
// CTA-pair variant: tcgen05.mma.cta_group::2 ... block_scale on 256 x 256 output tiles over
// the two SMs of a 2-CTA cluster.
//
// Each CTA stages its own 128 rows of A and its own 128-row half of the tile's B, so an SM
// moves 32 KB of operands per 256-deep K stage for the MMA work that a single-CTA 128 x 256
// tile needs 48 KB for: shared memory, which carries both the TMA writes and the MMA's operand
// reads, stops being the bound.  The even CTA (leader) issues the pair's MMAs; each CTA's
// tensor core reads A and its scales from its own memories and B from both CTAs' shared
// memory.  Scale factors reach tensor memory through WG groups of four scale-writer warps per
// CTA (tcgen05.st, off the tensor unit; the groups take alternate stages): each CTA writes the
// scales of its own A rows and those of all 256 B rows of the tile (the pair MMA reads the B
// scales of the whole N extent from each CTA's tensor memory).
// Barriers: the leader's full[s] counts both CTAs' A/B copies; each CTA's sf_full[s] its own
// scale copies; the leader's sf_ready[s] takes the eight scale-writer warps of the pair; MMA
// completion is multicast to both CTAs' empty[s] and acc_full; both epilogues release the
// accumulator on the leader's acc_empty.  One 256-column accumulator per CTA (the scale slots
// of the five stages use the other 240 columns).
// ---------------------------------------------------------------------------------------
template <int WG>
struct Pair4Cfg {
  static constexpr int STAGES = 5;
  static constexpr int B_BYTES = 128 * BK / 2;                  // this CTA's half of B
  static constexpr int SFA_BYTES = 4 * SF_ATOM;                 // own 128 rows, 4 K steps
  static constexpr int SFB_ATOMS = 2;                           // the scales of all 256 B rows
  static constexpr int SFB_BYTES = SFB_ATOMS * 4 * SF_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 4 + 4 * SFB_ATOMS;             // tensor-memory columns per K step
  static constexpr int SF_BASE = 256;
  static constexpr int TMEM_USED = SF_BASE + STAGES * 4 * SF_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int SF_WARP0 = 2 + EPI_WARPS;
  static constexpr int THREADS = (2 + EPI_WARPS + 4 * WG) * 32;
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void tc_mma_pair_f4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                               uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

template <int WG>
__global__ void __launch_bounds__(Pair4Cfg<WG>::THREADS, 1)
    k_gemm_nvfp4_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const uint8_t* __restrict__ a_sf, const uint8_t* __restrict__ b_sf,
                      const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N, int K,
                      const float* __restrict__ bias, void* __restrict__ y, int epi, void* ws, int stall) {
  using C = Pair4Cfg<WG>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  // bars: full[S], empty[S], sf_full[S], sf_ready[S], acc_full, acc_empty, mma_done (same offsets in both CTAs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * S + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto sf_full = [&](int s) { return smem_u32(bars + 2 * S + s); };
  auto sf_ready = [&](int s) { return smem_u32(bars + 3 * S + s); };
  const uint32_t acc_full = smem_u32(bars + 4 * S);
  const uint32_t acc_empty = smem_u32(bars + 4 * S + 1);
  const uint32_t mma_done = smem_u32(bars + 4 * S + 2);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfa_tile = [&](int s) { return smem + s * C::STAGE_BYTES + A_BYTES + C::B_BYTES; };
  auto sfb_tile = [&](int s) { return sfa_tile(s) + C::SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's MMAs
  const int ksteps = K / KSTEP;
  const int num_kb = (ksteps + 3) / 4;
  const int k_atoms = ksteps;             // scale atoms per 128-row block along K
  const int a_blocks = (M + 127) / 128;   // 128-row blocks present in the scale arrays
  const int b_blocks = (N + 127) / 128;
  const int n_tiles_n = (N + 255) / 256;
  const int n_items = ((M + 255) / 256) * n_tiles_n;
  const int first_item = blockIdx.x >> 1, item_step = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(sf_full(s), 1);
      mbar_init(sf_ready(s), 8);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * C::EPI_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {  // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !stall) {  // stall: a test hook that issues no loads at all
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      uint32_t kc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step) {
        const int mt = item / n_tiles_n, nt = item % n_tiles_n;
        const int m0 = mt * 256 + (int)rank * 128, n0 = nt * 256 + (int)rank * 128;
        const int ablk = mt * 2 + (int)rank;  // this CTA's row block of the A scales
        const bool a_sf_ok = ablk < a_blocks; // rows past the padded scale array: nothing to stage
        const int nb_first = nt * 2;
        int nb_cnt = b_blocks - nb_first;
        nb_cnt = nb_cnt < 0 ? 0 : (nb_cnt > C::SFB_ATOMS ? C::SFB_ATOMS : nb_cnt);
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait_cl(empty(s), ((kc / S) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(full(s), 2 * (A_BYTES + C::B_BYTES));  // both CTAs' bytes
          const uint32_t fb = mapa_rank(full(s), 0);
          tma_load_2d_pair(a_tile(s), &tmA, fb, kb * (BK / 2), m0);
          tma_load_2d_pair(b_tile(s), &tmB, fb, kb * (BK / 2), n0);
          const int nsub = min(4, ksteps - kb * 4);
          mbar_expect_tx(sf_full(s), nsub * SF_ATOM * ((a_sf_ok ? 1 : 0) + nb_cnt));
          if (a_sf_ok)
            bulk_load(smem_u32(sfa_tile(s)), a_sf + ((size_t)ablk * k_atoms + kb * 4) * SF_ATOM, nsub * SF_ATOM,
                      sf_full(s));
          for (int nb = 0; nb < nb_cnt; ++nb)
            bulk_load(smem_u32(sfb_tile(s)) + nb * 4 * SF_ATOM,
                      b_sf + ((size_t)(nb_first + nb) * k_atoms + kb * 4) * SF_ATOM, nsub * SF_ATOM, sf_full(s));
        }
      }
      if (!ok) {  // let this CTA's copies in flight land before it leaves
        volatile int no_abort = 0;
        const uint32_t first = kc > (uint32_t)S ? kc - S : 0;
        for (uint32_t c = first; c < kc; ++c) {
          mbar_wait(sf_full(c % S), (c / S) & 1, ws, &no_abort);
          if (rank == 0) mbar_wait_cl(full(c % S), (c / S) & 1, ws, &no_abort);  // counts both CTAs' A/B
        }
      }
    }
  } else if (warp == 1) {  // ----------------------------------------- MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_nvf4(256, 256);
      uint32_t kc = 0, tc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step, ++tc) {
        if (!mbar_wait_cl(acc_empty, (tc & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait_cl(full(s), (kc / S) & 1, ws, abort_flag) ||
              !mbar_wait_cl(sf_ready(s), (kc / S) & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(4, ksteps - kb * 4);
          for (int j = 0; j < nsub; ++j) {
            const uint32_t col = C::SF_BASE + (s * 4 + j) * C::SF_COLS;
            tc_mma_pair_f4(tmem, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc, tmem + col,
                           tmem + col + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(empty(s), 3);
        }
        if (ok) tc_commit_pair_mc(acc_full, 3);
      }
      tc_commit_pair(mma_done);
      volatile int no_abort = 0;
      mbar_wait_cl(mma_done, 0, ws, &no_abort);  // every issued MMA has completed
    }
    __syncwarp();
  } else if (warp >= C::SF_WARP0) {  // -------------------------- scale writers (both CTAs)
    const int q = warp & 3;                        // the lane quarter this warp may write
    const int grp = (warp - C::SF_WARP0) >> 2;     // writer group: stages kc with kc % WG == grp
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t kc = 0;
    bool ok = true;
    for (int item = first_item; item < n_items && ok; item += item_step) {
      for (int kb = 0; kb < num_kb; ++kb, ++kc) {
        if ((int)(kc % WG) != grp) continue;
        const int s = kc % S;
        if (!mbar_wait(sf_full(s), (kc / S) & 1, ws, abort_flag)) {
          ok = false;
          break;
        }
        // lane l gets the 16-byte line l of each 512-byte atom: the four scale words of rows
        // l, l+32, l+64, l+96 -- the words the 32x128b.warpx4 copy puts in every lane quarter.
        // A stage's 48 columns (per K step: A rows, B rows 0-127, B rows 128-255) go out in two
        // stores; columns of K steps past the end of K hold stale words no MMA reads.
        uint32_t r[48];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sfa_tile(s) + j * SF_ATOM + lane * 16);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sfb_tile(s) + j * SF_ATOM + lane * 16);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sfb_tile(s) + 4 * SF_ATOM + j * SF_ATOM + lane * 16);
          r[12 * j + 0] = a.x, r[12 * j + 1] = a.y, r[12 * j + 2] = a.z, r[12 * j + 3] = a.w;
          r[12 * j + 4] = b0.x, r[12 * j + 5] = b0.y, r[12 * j + 6] = b0.z, r[12 * j + 7] = b0.w;
          r[12 * j + 8] = b1.x, r[12 * j + 9] = b1.y, r[12 * j + 10] = b1.z, r[12 * j + 11] = b1.w;
        }
        const uint32_t col = C::SF_BASE + s * 4 * C::SF_COLS;
        tc_st32(lane_base + col, r);
        tc_st16(lane_base + col + 32, r + 32);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_rank(sf_ready(s), 0));
      }
    }
  } else {  // ------------------------------------------------------ epilogue warps (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;   // tensor-memory lane quarter of this warp
    const int half = e >> 2;  // which 128-column half of the 256-column tile
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    const uint32_t acc_empty_leader = mapa_rank(acc_empty, 0);
    uint32_t tc = 0;
    for (int item = first_item; item < n_items; item += item_step, ++tc) {
      const int m0 = (item / n_tiles_n) * 256 + (int)rank * 128, n0 = (item % n_tiles_n) * 256;
      if (!mbar_wait_cl(acc_full, tc & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld32(tmem + ((uint32_t)(q * 32) << 16) + half * 128 + c * 32, r);
        epi_store32(r, alpha, row, n0 + half * 128 + c * 32, M, N, bias, y, epi);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
    }
    tc_fence_before();
  }

  __syncthreads();
  cluster_sync();  // no MMA, copy or arrival of either CTA still touches the other
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

template <int WG>
static dit_status launch_pair4(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf,
                               const uint8_t* b_sf, const float* a_gs, const float* b_gs, int M, int N, int K,
                               const float* bias, void* y, int epi, void* ws, cudaStream_t st) {
  using C = Pair4Cfg<WG>;
  auto kern = k_gemm_nvfp4_pair<WG>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t items = (int64_t)((M + 255) / 256) * ((N + 255) / 256);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) return DIT_ERR_CUDA;
  int64_t pairs = clusters;
  if (pairs > items) pairs = items;
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, a_sf, b_sf, a_gs, b_gs, M, N, K, bias, y, epi, ws, test_stall()) !=
      cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}


// ---------------------------------------------------------------------------------------
// CTA-pair variant with scale copies on the tensor pipe: the same 256 x 256 tiles, but each
// CTA's scale atoms arrive by TMA with its operand tiles (one leader barrier per stage for the
// pair's A, B and scale bytes), and the leader's MMA thread moves them into both CTAs' tensor
// memory itself with tcgen05.cp.cta_group::2 (every CTA copies its own shared memory into its
// own tensor memory) right before the MMAs that read them; copies and MMAs issued by one
// thread run in order, so no scale barrier and no writer warps are needed.
// ---------------------------------------------------------------------------------------
struct PairCpCfg {
  static constexpr int STAGES = 5;
  static constexpr int B_BYTES = 128 * BK / 2;                  // this CTA's half of B
  static constexpr int SFA_BYTES = 4 * SF_ATOM;                 // own 128 rows, 4 K steps
  static constexpr int SFB_BYTES = 2 * 4 * SF_ATOM;             // all 256 B rows, 4 K steps
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int SF_COLS = 12;                            // tensor-memory columns per K step
  static constexpr int SF_BASE = 256;
  static constexpr int TMEM_USED = SF_BASE + STAGES * 4 * SF_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = (2 + EPI_WARPS) * 32;
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// EARLY: each epilogue thread first drains its 128 accumulator columns into registers and
// releases the accumulator, so the MMAs of the next tile overlap this tile's conversion and
// stores (one 256-column accumulator, no second buffer in tensor memory).
template <bool EARLY>
__global__ void __launch_bounds__(PairCpCfg::THREADS, 1)
    k_gemm_nvfp4_pair_cp(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                         const float* __restrict__ a_gs, const float* __restrict__ b_gs, int M, int N, int K,
                         const float* __restrict__ bias, void* __restrict__ y, int epi, void* ws, int stall) {
  using C = PairCpCfg;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  // bars: full[S], empty[S], acc_full, acc_empty, mma_done (same offsets in both CTAs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t acc_full = smem_u32(bars + 2 * S);
  const uint32_t acc_empty = smem_u32(bars + 2 * S + 1);
  const uint32_t mma_done = smem_u32(bars + 2 * S + 2);
  auto a_tile = [&](int s) { return sbase + s * C::STAGE_BYTES; };
  auto b_tile = [&](int s) { return a_tile(s) + A_BYTES; };
  auto sfa_tile = [&](int s) { return b_tile(s) + C::B_BYTES; };
  auto sfb_tile = [&](int s) { return sfa_tile(s) + C::SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's copies and MMAs
  const int ksteps = K / KSTEP;
  const int num_kb = (ksteps + 3) / 4;
  const int n_tiles_n = (N + 255) / 256;
  const int n_items = ((M + 255) / 256) * n_tiles_n;
  const int first_item = blockIdx.x >> 1, item_step = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * C::EPI_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {  // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !stall) {  // stall: a test hook that issues no loads at all
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmSA);
      prefetch_tmap(&tmSB);
      uint32_t kc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step) {
        const int mt = item / n_tiles_n, nt = item % n_tiles_n;
        const int m0 = mt * 256 + (int)rank * 128, n0 = nt * 256 + (int)rank * 128;
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait_cl(empty(s), ((kc / S) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(full(s), 2 * C::STAGE_BYTES);  // both CTAs' bytes
          const uint32_t fb = mapa_rank(full(s), 0);
          tma_load_2d_pair(a_tile(s), &tmA, fb, kb * (BK / 2), m0);
          tma_load_2d_pair(b_tile(s), &tmB, fb, kb * (BK / 2), n0);
          tma_load_3d_pair(sfa_tile(s), &tmSA, fb, 0, kb * 4, mt * 2 + (int)rank);
          tma_load_3d_pair(sfb_tile(s), &tmSB, fb, 0, kb * 4, nt * 2);
        }
      }
      if (!ok && rank == 0) {  // the leader's full barriers count both CTAs' copies in flight
        volatile int no_abort = 0;
        const uint32_t first = kc > (uint32_t)S ? kc - S : 0;
        for (uint32_t c = first; c < kc; ++c) mbar_wait_cl(full(c % S), (c / S) & 1, ws, &no_abort);
      }
    }
  } else if (warp == 1) {  // ----------------------------------------- MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_nvf4(256, 256);
      uint32_t kc = 0, tc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step, ++tc) {
        if (!mbar_wait_cl(acc_empty, (tc & 1) ^ 1, ws, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait_cl(full(s), (kc / S) & 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(4, ksteps - kb * 4);
          for (int j = 0; j < nsub; ++j) {
            const uint32_t col = C::SF_BASE + (s * 4 + j) * C::SF_COLS;
            tc_cp_sf_pair(tmem + col, desc_sf(sfa_tile(s) + j * SF_ATOM));
            tc_cp_sf_pair(tmem + col + 4, desc_sf(sfb_tile(s) + j * SF_ATOM));
            tc_cp_sf_pair(tmem + col + 8, desc_sf(sfb_tile(s) + 4 * SF_ATOM + j * SF_ATOM));
            tc_mma_pair_f4(tmem, desc_sw128(a_tile(s) + j * 32), desc_sw128(b_tile(s) + j * 32), idesc, tmem + col,
                           tmem + col + 4, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(empty(s), 3);
        }
        if (ok) tc_commit_pair_mc(acc_full, 3);
      }
      tc_commit_pair(mma_done);
      volatile int no_abort = 0;
      mbar_wait_cl(mma_done, 0, ws, &no_abort);  // every issued copy and MMA has completed
    }
    __syncwarp();
  } else {  // ------------------------------------------------------ epilogue warps (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;   // tensor-memory lane quarter of this warp
    const int half = e >> 2;  // which 128-column half of the 256-column tile
    const float alpha = __fmul_rn(*a_gs, *b_gs);
    const uint32_t acc_empty_leader = mapa_rank(acc_empty, 0);
    uint32_t tc = 0;
    for (int item = first_item; item < n_items; item += item_step, ++tc) {
      const int m0 = (item / n_tiles_n) * 256 + (int)rank * 128, n0 = (item % n_tiles_n) * 256;
      if (!mbar_wait_cl(acc_full, tc & 1, ws, abort_flag)) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + half * 128;
      if constexpr (EARLY) {
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc_ld32_nowait(tbase + c * 32, r[c]);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
#pragma unroll
        for (int c = 0; c < 4; ++c) epi_store32(r[c], alpha, row, n0 + half * 128 + c * 32, M, N, bias, y, epi);
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc_ld32(tbase + c * 32, r);
          epi_store32(r, alpha, row, n0 + half * 128 + c * 32, M, N, bias, y, epi);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  cluster_sync();  // no MMA, copy or arrival of either CTA still touches the other
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

template <bool EARLY>
static dit_status launch_pair_cp(const CUtensorMap& ta, const CUtensorMap& tb, const uint8_t* a_sf,
                                 const uint8_t* b_sf, const float* a_gs, const float* b_gs, int M, int N, int K,
                                 const float* bias, void* y, int epi, void* ws, cudaStream_t st) {
  using C = PairCpCfg;
  CUtensorMap tsa, tsb;
  if (!encode_tmap_sf(&tsa, a_sf, M, K, 1) || !encode_tmap_sf(&tsb, b_sf, N, K, 2)) return DIT_ERR_CUDA;
  auto kern = k_gemm_nvfp4_pair_cp<EARLY>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t items = (int64_t)((M + 255) / 256) * ((N + 255) / 256);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) return DIT_ERR_CUDA;
  int64_t pairs = clusters;
  if (pairs > items) pairs = items;
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, a_gs, b_gs, M, N, K, bias, y, epi, ws, test_stall()) !=
      cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}


}  // namespace f4
}  // namespace dit6

using namespace dit6;

// Tile configurations.  10: the persistent 128 x 128 kernel with two CTAs per SM whose scale
// atoms are written into tensor memory by four dedicated warps (tcgen05.st, one wide store per
// stage) -- scale copies on the tensor-core unit (tcgen05.cp) cost ~110 cycles of tensor time
// each -- and whose two independent MMA streams per SM hide each other's epilogue.  11: the same
// kernel on 128 x 256 tiles, one CTA per SM, four stages; with bf16 output its eight epilogue
// warps convert their 128 columns to packed bf16 registers and release the accumulator before
// storing.  23: 11 with sixteen epilogue warps of 64 columns that release the accumulator right
// after loading it, so bias, activation and stores all overlap the next tile's MMAs.  The
// CTA-pair kernels (15: scale writers, 18: tcgen05.cp with early accumulator release) are exact
// but slower on every CogVideoX shape and at 8192^3 (measured on GB300).  DIT6_NVFP4_TILE selects
// a configuration for experiments and tests.
// Without DIT6_NVFP4_TILE the call picks (PFLOP/s, GB300).  With the GELU epilogue 23 leads
// everywhere: CogVideoX-2B FFN-up 3.27 (10: 2.69, 11: 2.48), 5B FFN-up 4.11 (3.46), 1080p
// FFN-up 4.26 (3.55), 8192^3 4.84 (4.34).  Without it, for bf16 output 11 leads or ties (2B QKV
// 3.50 vs 3.08 / 3.42 for 23; 5B QKV 4.39 / 4.45; 1080p FFN-up 4.54 / 4.63) except with N off
// the 256 grid and a long K, where 10 does (2B FFN-down 4.39 vs 4.32).  fp32 output keeps the
// accumulator until stored in 10 and 11: 11 only when K >= 3072 and N is a multiple of 256.
static int nvfp4_tile_cfg(int64_t n, int64_t k, int epi) {
  const char* e = getenv("DIT6_NVFP4_TILE");
  if (e) return atoi(e);
  if (epi & EPI_GELU) return 23;
  if (epi & EPI_BF16) return (n % 256 != 0 && k >= 4096) ? 10 : 11;
  return (k >= 3072 && n % 256 == 0) ? 11 : 10;
}

extern "C" dit_status dit_qgemm_nvfp4_fused_quant(const uint8_t* a, const uint8_t* a_sf, const float* a_gs,
                                                  const uint8_t* b, const uint8_t* b_sf, const float* b_gs,
                                                  int64_t m, int64_t n, int64_t k, const float* bias,
                                                  dit_act act, void* y, int hblock, const float* q_scale_in,
                                                  uint8_t* q_codes, uint8_t* q_sf, float* q_scale_next,
                                                  void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!a || !a_sf || !a_gs || !b || !b_sf || !b_gs || !q_scale_in || !q_codes || !q_sf || !q_scale_next || !ws ||
      ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff)
    return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  if (hblock != 16 && hblock != 32 && hblock != 64) return DIT_ERR_UNSUPPORTED;
  if (k % 64 || n % 64) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(a) || !aligned32(b) || !aligned32(a_sf) || !aligned32(b_sf) || !aligned32(q_codes) ||
      !aligned32(q_sf) || !aligned32(ws) || (y && !aligned32(y)))
    return DIT_ERR_ALIGNMENT;
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(k / 2),
                      (uint64_t)m, (uint64_t)(k / 2), f4::BK / 2, f4::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(k / 2),
                      (uint64_t)n, (uint64_t)(k / 2), f4::BK / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int epi = EPI_BF16 | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  const float isb = (float)(1.0 / sqrt((double)hblock));
#define DIT6_FQ(HB_)                                                                                          \
  return f4::launch_s<128, 3, 2, HB_>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, epi, ws, \
                                      st, q_scale_in, isb, q_codes, q_sf, q_scale_next)
  if (hblock == 16) DIT6_FQ(16);
  if (hblock == 32) DIT6_FQ(32);
  DIT6_FQ(64);
#undef DIT6_FQ
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
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(k / 2),
                      (uint64_t)m, (uint64_t)(k / 2), f4::BK / 2, f4::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(k / 2),
                      (uint64_t)n, (uint64_t)(k / 2), f4::BK / 2, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int epi = EPI_BF16 | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  const float isb = (float)(1.0 / sqrt((double)hblock));
#define DIT6_AM(HB_)                                                                                             \
  return f4::launch_s<256, 4, 1, 0, 1, 16, HB_>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, \
                                                epi, ws, st, nullptr, isb, nullptr, nullptr, tensor_scale_out)
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
  const int cfg = nvfp4_tile_cfg(n, k, (y_dt == DIT_BF16 ? EPI_BF16 : 0) | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0));
  const uint32_t bn_box = (cfg == 1 || cfg == 2 || cfg == 5 || cfg == 6 || cfg == 8 || cfg == 11 || cfg == 23) ? 256 : 128;
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(k / 2),
                      (uint64_t)m, (uint64_t)(k / 2), f4::BK / 2, f4::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(k / 2),
                      (uint64_t)n, (uint64_t)(k / 2), f4::BK / 2, bn_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int yb = (y_dt == DIT_BF16 ? EPI_BF16 : 0) | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  switch (cfg) {
    case 1: return f4::launch<256, 3, true>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 2: return f4::launch<256, 3, false>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 3: return f4::launch<128, 6, false>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 4: return f4::launch_p<128, 4, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 5: return f4::launch_p<256, 3, 1>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 6: return f4::launch_p<256, 4, 1>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 7: return f4::launch_p<128, 6, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 8:
      if (k <= 64 * f4::RCfg::MAX_KSTEPS)
        return f4::launch_r(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
      return f4::launch_p<256, 4, 1>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 9: return f4::launch_p<128, 3, 1, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    default: return f4::launch_s<128, 3, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 23: return f4::launch_s<256, 4, 1, 0, 1, 16>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 11: return f4::launch_s<256, 4, 1>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 12: return f4::launch_s<128, 6, 1>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 13: return f4::launch_s<128, 6, 1, 0, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 14: return f4::launch_s<128, 4, 1, 0, 2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 0: return f4::launch<128, 3, false>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 15: return f4::launch_pair4<2>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
    case 18: return f4::launch_pair_cp<true>(ta, tb, a_sf, b_sf, a_gs, b_gs, (int)m, (int)n, (int)k, bias, y, yb, ws, st);
  }
}
