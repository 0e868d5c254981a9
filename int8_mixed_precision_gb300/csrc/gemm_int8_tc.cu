// INT8 route GEMM on the bf16 tcgen05 tensor pipe, with exact int32 accumulators.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science 2.A Mechanism 3 (volatile layers go to
// INT8).  sm_103a has no tcgen05 integer MMA and its IMMA path peaks near 151 TOPS, 13x below
// the bf16 tensor rate.  The INT8 codes (integers in [-127, 127]) are exact in bf16 and their
// products (|p| <= 16129) exact in fp32, so this kernel runs the INT8 contraction on
// tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in tensor memory) and keeps it exact by
// accumulating K in chunks of at most 1024: every partial sum of a chunk is an integer of
// magnitude <= 1024 * 16129 < 2^24, hence exactly representable in fp32 whatever the order of
// the additions.  Each finished chunk is drained from tensor memory, converted to int32
// (exact) and added to int32 running sums in the epilogue warps' registers.
//
// Persistent CTA pairs (2-CTA clusters, cta_group::2) walk 256 x 256 output tiles.  Warp 0:
// TMA producer (128-byte swizzled A/B tiles, STAGES-deep ring).  Warp 1: tensor-memory
// allocation and, in the even CTA, the MMA issuer; chunk accumulators alternate between two
// tensor-memory buffers, so the MMAs of chunk c+1 (also of the next tile) overlap the drain of
// chunk c.  Warps 2..9: epilogue.  Every wait is bounded.
#include "common.cuh"

namespace dit6 {
namespace i8tc {

constexpr int BK = 64;             // BK bf16 elements = 128 bytes per row
constexpr int KCHUNK_BLOCKS = 16;  // 16 x 64 = 1024 elements per exact chunk
constexpr int A_BYTES = 128 * BK * 2;
#ifndef I8_BAND_BYTES
#define I8_BAND_BYTES (24ll << 20)
#endif

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, K-major A and B
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
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

// ------------------------------------------------------------------------------------------
// The CTA-pair kernel: tcgen05.mma.cta_group::2, 256 x 256 tiles over two SMs.
//
// Each CTA of a 2-CTA cluster stages its own 128 rows of A and its own 128-row half of the
// tile's B (N split across the pair), so every SM moves 32 KB per 64-deep K step instead of
// the 48 KB a single-CTA 128 x 256 tile needs for the same MMA work per SM.  The even CTA (leader)
// issues the pair's MMAs; they read both CTAs' shared memory at the same offsets and write each
// CTA's 128 accumulator rows into that CTA's tensor memory.  Both producers signal the leader's
// full barrier (TMA .cta_group::2), whose expected byte count covers the pair; MMA completion
// is multicast to both CTAs' empty and chunk-full barriers; both epilogues release a drained
// chunk buffer by arriving on the leader's chunk-empty barrier.  Tensor memory is allocated and
// freed by one warp in each CTA together (cta_group::2).
// ------------------------------------------------------------------------------------------
// EPW: epilogue warps, 4 per tensor-memory lane quarter x (EPW / 4) column groups of CW.
template <int EPW>
struct PairCfgT {
  static constexpr int STAGES = 6;
  static constexpr int B_BYTES = 128 * BK * 2;                 // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // 32 KB
  static constexpr int EPI_WARPS = EPW;
  static constexpr int CW = 256 / (EPW / 4);                    // accumulator columns per thread
  static constexpr int THREADS = (2 + EPI_WARPS) * 32;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int TMEM_COLS = 512;                         // two 256-column chunk buffers
};
using PairCfg = PairCfgT<8>;
// the requantising epilogue runs sixteen warps of 64 columns (its per-thread work is heavier)
template <bool REQ>
using PairCfgFor = PairCfgT<REQ ? 16 : 8>;

__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Arguments of the requantising epilogue (REQ): the next INT8 linear's per-token scales, the
// per-row maxima it reports, and the Hadamard normalisation 1/sqrt(64).
struct ReqArgs {
  const float* scale;  // [M] s of the next layer's per-token quantisation (caller-supplied)
  float* amax;         // [M] max |H z| / 8 over the row, atomically maxed (caller zero-fills)
  float inv_sqrt_b;
};

// The requantising epilogue of one thread's CW accumulator columns of output row `row` (CW / 64
// units of 64 columns of the next layer's K): z = act((acc * s_a) * s_w (+ bias)) rounded to bf16 as
// the unfused path stores it; y = FWHT64(z) * 1/8 in the INT8 quantiser's stage order;
// q = clamp(RN(y * RN(1/s)), -127, 127) stored as bf16-held codes; the unit maxima of |y| go to
// req.amax[row].  With s = max_row |y| / 127 these are the quantiser's codes bit for bit.
template <bool GELU, int CW>
__device__ __forceinline__ void requant_row(const int (&acc)[CW], int row, int col0, int M, int N,
                                            const float* __restrict__ a_scale, const float* __restrict__ b_scale,
                                            const float* __restrict__ bias, void* __restrict__ q_out,
                                            const ReqArgs& req) {
  if (row >= M || col0 >= N) return;
  const float sa = a_scale[row];
  const float2 sa2 = make_float2(sa, sa);
  const float s = req.scale[row];
  const float inv = s == 0.f ? 0.f : __frcp_rn(s);
  const float2 iv = make_float2(inv, inv), isb = make_float2(req.inv_sqrt_b, req.inv_sqrt_b);
  float tmax = 0.f;
#pragma unroll
  for (int u = 0; u < CW / 64; ++u) {
    const int cu = col0 + 64 * u;
    if (cu >= N) break;  // N % 64 == 0: a unit is whole or absent
    float2 z[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // four columns per step, as the plain epilogue rounds them
      const int c = 64 * u + 4 * j;
      const float4 sb = reinterpret_cast<const float4*>(b_scale + col0 + c)[0];
      float2 lo = mul2(mul2(make_float2((float)acc[c], (float)acc[c + 1]), sa2), make_float2(sb.x, sb.y));
      float2 hi = mul2(mul2(make_float2((float)acc[c + 2], (float)acc[c + 3]), sa2), make_float2(sb.z, sb.w));
      if (bias) {
        const float4 bb = reinterpret_cast<const float4*>(bias + col0 + c)[0];
        lo = add2(lo, make_float2(bb.x, bb.y));
        hi = add2(hi, make_float2(bb.z, bb.w));
      }
      if (GELU) {
        lo = gelu_erf2(lo);
        hi = gelu_erf2(hi);
      }
      z[2 * j] = bf16x2_to_f2(f2_to_bf16x2(lo.x, lo.y));
      z[2 * j + 1] = bf16x2_to_f2(f2_to_bf16x2(hi.x, hi.y));
    }
    fwht64<64>(z);
#pragma unroll
    for (int p = 0; p < 32; ++p) z[p] = mul2(z[p], isb);
    tmax = fmaxf(tmax, amax_range(z, 0, 32));
    U8x32 o[4];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const float2 a = mul2(z[p], iv);
      const float q0 = fminf(fmaxf(rintf(a.x), -127.f), 127.f), q1 = fminf(fmaxf(rintf(a.y), -127.f), 127.f);
      o[p / 8].w[p % 8] = f2_to_bf16x2(q0, q1);
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(q_out) + (int64_t)row * N + cu;
#pragma unroll
    for (int c = 0; c < 4; ++c) st256(dst + 16 * c, o[c]);
  }
  atomicMax(reinterpret_cast<unsigned*>(req.amax) + row, __float_as_uint(tmax));
}

// ACCM 0: INT8 codes, exact chunks summed in int32.
// ACCM 1: INT8 codes, K spans at most two exact chunks and no raw accumulators are requested.
//         Each chunk sum is then an exact fp32 integer and one fp32 addition rounds their exact
//         total once, as the conversion of the int32 total to fp32 does, so the chunks are
//         summed in fp32 and the output is the same bit for bit without the int32 round trip.
// ACCM 2: a plain bf16 GEMM (the BF16 route of PDR): fp32 accumulation over the whole K in one
//         tensor-memory chunk, no scales.
// BANDED: the tile order in bands of N tiles (see tile_mn); a separate instantiation, so that the
// shapes that keep the plain order run exactly the code they always ran.
// REQ (ACCM 0 only): the epilogue quantises the output for the next INT8 linear (requant_row)
// instead of storing it; y then receives the bf16-held codes.
template <bool GELU, int ACCM, bool BANDED, bool REQ = false>
__global__ void __launch_bounds__(PairCfgFor<REQ>::THREADS, 1)
    k_gemm_int8_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const float* __restrict__ a_scale, const float* __restrict__ b_scale, int M, int N, int K,
                     const float* __restrict__ bias, void* __restrict__ y, int epi, int32_t* __restrict__ acc_out,
                     void* ws, int stall, int band, ReqArgs req) {
  pdl_launch_dependents();
  using P = PairCfgFor<REQ>;
  constexpr int S = P::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * P::STAGE_BYTES);
  // bars: full[S], empty[S], chunk_full[2], chunk_empty[2], mma_done (same offsets in both CTAs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + S + s); };
  auto cfull = [&](int b) { return smem_u32(bars + 2 * S + b); };
  auto cempty = [&](int b) { return smem_u32(bars + 2 * S + 2 + b); };
  const uint32_t mma_done = smem_u32(bars + 2 * S + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's MMAs
  const int n_tiles_n = (N + 255) / 256;
  const int m_tiles = (M + 255) / 256;
  const int n_items = m_tiles * n_tiles_n;
  const int first_item = blockIdx.x >> 1, item_step = gridDim.x >> 1;
  // Tile order: N fastest.  BANDED: bands of `band` N tiles, each band walked over all M tiles
  // (N fastest inside the band), so the band's slice of B stays in L2 while A streams through
  // once per band.
  auto tile_mn = [&](int item, int& m0, int& n0) {
    if constexpr (BANDED) {
      const int per_band = band * m_tiles;
      const int b = item / per_band;
      const int r = item - b * per_band;
      const int w = min(band, n_tiles_n - b * band);
      m0 = (r / w) * 256;
      n0 = (b * band + r % w) * 256;
    } else {
      m0 = (item / n_tiles_n) * 256;
      n0 = (item % n_tiles_n) * 256;
    }
  };
  const int nkb = (K + BK - 1) / BK;
  // exactness chunks of the INT8 modes; the bf16 mode accumulates all of K in one chunk
  const int kchunk = ACCM == 2 ? nkb : KCHUNK_BLOCKS;
  const int nchunks = ACCM == 2 ? 1 : (nkb + KCHUNK_BLOCKS - 1) / KCHUNK_BLOCKS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(cfull(b), 1);
      mbar_init(cempty(b), 2 * P::EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(P::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {  // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !stall) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      uint32_t kc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step) {
        int m0, n0;
        tile_mn(item, m0, n0);
        m0 += (int)rank * 128;
        n0 += (int)rank * 128;
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const int s = kc % S;
          if (!mbar_wait_cl(empty(s), ((kc / S) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(full(s), 2 * P::STAGE_BYTES);  // both CTAs' bytes
          const uint32_t fb = mapa_rank(full(s), 0);
          tma_load_2d_pair(sbase + s * P::STAGE_BYTES, &tmA, fb, kb * BK, m0);
          tma_load_2d_pair(sbase + s * P::STAGE_BYTES + A_BYTES, &tmB, fb, kb * BK, n0);
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
      constexpr uint32_t idesc = idesc_bf16(256, 256);
      uint32_t kc = 0, cc = 0;
      bool ok = true;
      for (int item = first_item; item < n_items && ok; item += item_step) {
        for (int ch = 0; ch < nchunks && ok; ++ch, ++cc) {
          const int buf = cc & 1;
          if (!mbar_wait_cl(cempty(buf), ((cc >> 1) & 1) ^ 1, ws, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * 256;
          const int kb0 = ch * kchunk;
          const int kb1 = min(nkb, kb0 + kchunk);
          for (int kb = kb0; kb < kb1; ++kb, ++kc) {
            const int s = kc % S;
            if (!mbar_wait_cl(full(s), (kc / S) & 1, ws, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_s = sbase + s * P::STAGE_BYTES, b_s = a_s + A_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)
              tc_mma_pair(d, desc_sw128(a_s + j * 32), desc_sw128(b_s + j * 32), idesc,
                          (kb > kb0 || j > 0) ? 1u : 0u);
            tc_commit_pair_mc(empty(s), 3);
          }
          if (ok) tc_commit_pair_mc(cfull(buf), 3);
        }
      }
      tc_commit_pair(mma_done);
      volatile int no_abort = 0;
      mbar_wait_cl(mma_done, 0, ws, &no_abort);  // every issued MMA has completed
    }
    __syncwarp();
  } else {  // ------------------------------------------------------ epilogue warps (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;   // tensor-memory lane quarter of this warp
    const int half = e >> 2;  // which CW-column group of the 256-column tile
    const uint32_t cempty_leader[2] = {mapa_rank(cempty(0), 0), mapa_rank(cempty(1), 0)};
    uint32_t cc = 0;
    bool ok = true;
    for (int item = first_item; item < n_items && ok; item += item_step) {
      int m0, n0;
      tile_mn(item, m0, n0);
      m0 += (int)rank * 128;
      constexpr int CW = P::CW;
      int acc[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) acc[i] = 0;
      for (int ch = 0; ch < nchunks; ++ch, ++cc) {
        const int buf = cc & 1;
        if (!mbar_wait_cl(cfull(buf), (cc >> 1) & 1, ws, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + buf * 256 + half * CW;
#pragma unroll
        for (int c = 0; c < CW / 32; ++c) {
          uint32_t r[32];
          tc_ld32(base + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if constexpr (ACCM >= 1)  // acc starts as +0.0f, and 0 + c0 = c0 exactly
              acc[c * 32 + i] = __float_as_int(__fadd_rn(__int_as_float(acc[c * 32 + i]), __uint_as_float(r[i])));
            else
              acc[c * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cempty_leader[buf]);
      }
      if (!ok) break;
      const int row = m0 + q * 32 + lane;
      const int col0 = n0 + half * CW;
      if constexpr (REQ) {
        requant_row<GELU, CW>(acc, row, col0, M, N, a_scale, b_scale, bias, y, req);
        continue;
      }
      if (row < M && col0 < N) {
        const float sa = ACCM == 2 ? 1.0f : a_scale[row];
        const int64_t off = (int64_t)row * N + col0;
#pragma unroll
        for (int c = 0; c < CW / 16; ++c) {
          const int cb = col0 + c * 16;
          if (cb >= N) break;
          float v[16];
          auto accf = [&](int i) { return ACCM >= 1 ? __int_as_float(acc[c * 16 + i]) : (float)acc[c * 16 + i]; };
          if (cb + 16 <= N) {  // packed: (acc * sa) * sb (+ bias), each product rounded as before
            const float4* sb4 = reinterpret_cast<const float4*>(b_scale + cb);
            const float4* bi4 = reinterpret_cast<const float4*>(bias + cb);
            const float2 sa2 = make_float2(sa, sa);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float2 lo = make_float2(accf(4 * j), accf(4 * j + 1));
              float2 hi = make_float2(accf(4 * j + 2), accf(4 * j + 3));
              if constexpr (ACCM != 2) {
                const float4 sb = sb4[j];
                lo = mul2(mul2(lo, sa2), make_float2(sb.x, sb.y));
                hi = mul2(mul2(hi, sa2), make_float2(sb.z, sb.w));
              }
              if (bias) {
                const float4 bb = bi4[j];
                lo = add2(lo, make_float2(bb.x, bb.y));
                hi = add2(hi, make_float2(bb.z, bb.w));
              }
              v[4 * j] = lo.x;
              v[4 * j + 1] = lo.y;
              v[4 * j + 2] = hi.x;
              v[4 * j + 3] = hi.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = cb + i < N ? cb + i : N - 1;
              v[i] = ACCM == 2 ? accf(i) : __fmul_rn(__fmul_rn(accf(i), sa), b_scale[col]);
              if (bias) v[i] = __fadd_rn(v[i], bias[col]);
            }
          }
          if (GELU) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 g = gelu_erf2(make_float2(v[2 * i], v[2 * i + 1]));
              v[2 * i] = g.x;
              v[2 * i + 1] = g.y;
            }
          }
          if (cb + 16 <= N && (N % 16) == 0) {
            if (epi & EPI_BF16) {
              U8x32 o;
#pragma unroll
              for (int i = 0; i < 8; ++i) o.w[i] = f2_to_bf16x2(v[2 * i], v[2 * i + 1]);
              st256(reinterpret_cast<uint16_t*>(y) + off + c * 16, o);
            } else {
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                U8x32 o;
#pragma unroll
                for (int i = 0; i < 8; ++i) o.w[i] = __float_as_uint(v[8 * b + i]);
                st256(reinterpret_cast<float*>(y) + off + c * 16 + 8 * b, o);
              }
            }
            if (acc_out) {
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                U8x32 o;
#pragma unroll
                for (int i = 0; i < 8; ++i) o.w[i] = (uint32_t)acc[c * 16 + 8 * b + i];
                st256(acc_out + off + c * 16 + 8 * b, o);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (cb + i >= N) continue;
              if (epi & EPI_BF16)
                reinterpret_cast<__nv_bfloat16*>(y)[off + c * 16 + i] = __float2bfloat16_rn(v[i]);
              else
                reinterpret_cast<float*>(y)[off + c * 16 + i] = v[i];
              if (acc_out) acc_out[off + c * 16 + i] = acc[c * 16 + i];
            }
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  cluster_sync();  // no MMA, copy or arrival of either CTA still touches the other
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P::TMEM_COLS)
                 : "memory");
  }
}

template <bool GELU, int ACCM, bool BANDED, bool REQ>
dit_status launch_pair_k(const CUtensorMap& ta, const CUtensorMap& tb, const float* a_scale, const float* b_scale,
                         int64_t m, int64_t n, int64_t k, const float* bias, void* y, int epi, int32_t* acc_out,
                         void* ws, cudaStream_t st, int band, const ReqArgs& req);

template <bool GELU, int ACCM, bool REQ = false>
dit_status launch_pair(const void* a, const float* a_scale, const void* b, const float* b_scale, int64_t m,
                       int64_t n, int64_t k, const float* bias, void* y, int epi, int32_t* acc_out, void* ws,
                       cudaStream_t st, const ReqArgs& req = ReqArgs{}) {
  CUtensorMap ta, tb;
  if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(a), (uint64_t)k, (uint64_t)m,
                      (uint64_t)k * 2, BK, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(b), (uint64_t)k, (uint64_t)n,
                      (uint64_t)k * 2, BK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return DIT_ERR_CUDA;
  // N tiles per band: as many as keep the band's slice of B (256 rows x K bf16 each) within
  // I8_BAND_BYTES, a share of one die's half of the L2 that leaves room for the A rows and the
  // output streaming through.  Measured on GB300 (CogVideoX-5B shapes, K = 3072): FFN-up
  // 784 -> 741 us with DRAM reads of 1.87 -> 0.42 GB per launch, QKV 530 -> 519 us with 0.74 ->
  // 0.40 GB; for K >= 7680 the plain order was ~1 % faster, so bands are used up to K = 4096.
  const int64_t n_tiles = (n + 255) / 256;
  int64_t band = I8_BAND_BYTES / (256 * 2 * k);
  if (band < 1) band = 1;
  if constexpr (ACCM != 2) {
    if (k <= 4096 && band < n_tiles)
      return launch_pair_k<GELU, ACCM, true, REQ>(ta, tb, a_scale, b_scale, m, n, k, bias, y, epi, acc_out, ws, st,
                                                  (int)band, req);
  }
  return launch_pair_k<GELU, ACCM, false, REQ>(ta, tb, a_scale, b_scale, m, n, k, bias, y, epi, acc_out, ws, st,
                                               (int)n_tiles, req);
}

template <bool GELU, int ACCM, bool BANDED, bool REQ>
dit_status launch_pair_k(const CUtensorMap& ta, const CUtensorMap& tb, const float* a_scale, const float* b_scale,
                         int64_t m, int64_t n, int64_t k, const float* bias, void* y, int epi, int32_t* acc_out,
                         void* ws, cudaStream_t st, int band, const ReqArgs& req) {
  using P = PairCfgFor<REQ>;
  auto kern = k_gemm_int8_pair<GELU, ACCM, BANDED, REQ>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES) != cudaSuccess)
      return DIT_ERR_CUDA;
    attr_done = true;
  }
  const int64_t items = ((m + 255) / 256) * ((n + 255) / 256);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(P::THREADS);
  cfg.dynamicSmemBytes = P::SMEM_BYTES;
  cfg.stream = st;
  cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) return DIT_ERR_CUDA;
  int64_t pairs = clusters;
  if (pairs > items) pairs = items;
  if (launch_pdl(kern, dim3((unsigned)(2 * pairs)), dim3(P::THREADS), P::SMEM_BYTES, st, 2, ta, tb, a_scale,
                 b_scale, (int)m, (int)n, (int)k, bias, y, epi, acc_out, ws, test_stall(), band, req) != cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}

}  // namespace i8tc

// The CTA-pair kernel (256 x 256 tiles over two SMs).  When K spans at most two exact chunks
// and no raw accumulators are requested, the chunk sums are added in fp32 (ACCM 1).
dit_status gemm_int8_tc(const void* a, const float* a_scale, const void* b, const float* b_scale, int64_t m,
                        int64_t n, int64_t k, const float* bias, void* y, int epi, int32_t* acc_out,
                        void* ws, size_t ws_bytes, cudaStream_t st) {
  (void)ws_bytes;
  const bool g = (epi & EPI_GELU) != 0;
  const bool f2 = !acc_out && (k + 1023) / 1024 <= 2;
  if (f2)
    return g ? i8tc::launch_pair<true, 1>(a, a_scale, b, b_scale, m, n, k, bias, y, epi, acc_out, ws, st)
             : i8tc::launch_pair<false, 1>(a, a_scale, b, b_scale, m, n, k, bias, y, epi, acc_out, ws, st);
  return g ? i8tc::launch_pair<true, 0>(a, a_scale, b, b_scale, m, n, k, bias, y, epi, acc_out, ws, st)
           : i8tc::launch_pair<false, 0>(a, a_scale, b, b_scale, m, n, k, bias, y, epi, acc_out, ws, st);
}

// The INT8 GEMM with the requantising epilogue (exact int32 chunk sums, ACCM 0).
dit_status gemm_int8_tc_requant(const void* a, const float* a_scale, const void* b, const float* b_scale, int64_t m,
                                int64_t n, int64_t k, const float* bias, bool gelu, const float* next_scale,
                                void* q_next, float* amax_out, void* ws, cudaStream_t st) {
  const i8tc::ReqArgs req{next_scale, amax_out, 0.125f};
  return gelu ? i8tc::launch_pair<true, 0, true>(a, a_scale, b, b_scale, m, n, k, bias, q_next, EPI_BF16 | EPI_GELU,
                                                 nullptr, ws, st, req)
              : i8tc::launch_pair<false, 0, true>(a, a_scale, b, b_scale, m, n, k, bias, q_next, EPI_BF16, nullptr,
                                                  ws, st, req);
}

}  // namespace dit6


// BF16 route of PDR ([EN] 2.C, [ZH] 2.C: full precision for a block whose input has a high
// outlier ratio): Y = act(X W^T (+ bias)) on the untransformed bf16 operands, fp32 accumulation,
// on the CTA-pair kernel in its bf16 mode.
extern "C" dit_status dit_gemm_bf16(const void* x, const void* w, int64_t m, int64_t n, int64_t k, const float* bias,
                                    dit_act act, void* y, dit_dtype y_dt, void* ws, size_t ws_bytes,
                                    dit_stream_t stream) {
  using namespace dit6;
  if (!x || !w || !y || !ws || ws_bytes < WS_BYTES) return DIT_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || m > 0x7fffffff || n > 0x7fffffff || k > 0x7fffffff) return DIT_ERR_INVALID_ARG;
  if (y_dt != DIT_F32 && y_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (act != DIT_ACT_NONE && act != DIT_ACT_GELU_ERF) return DIT_ERR_INVALID_ARG;
  if (k % 16 || n % 8) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(x) || !aligned32(w) || !aligned32(y) || !aligned32(ws) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 15)))
    return DIT_ERR_ALIGNMENT;
  const int epi = (y_dt == DIT_BF16 ? EPI_BF16 : 0) | (act == DIT_ACT_GELU_ERF ? EPI_GELU : 0);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return act == DIT_ACT_GELU_ERF
             ? dit6::i8tc::launch_pair<true, 2>(x, nullptr, w, nullptr, m, n, k, bias, y, epi, nullptr, ws, st)
             : dit6::i8tc::launch_pair<false, 2>(x, nullptr, w, nullptr, m, n, k, bias, y, epi, nullptr, ws, st);
}
