// Shared device helpers of libdit6 (sm_103a): vector memory ops, packed fp32x2 math,
// FP4/FP8 conversions, mbarrier / TMA / bounded waits, and the workspace layout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dit6.h"

namespace dit6 {

// ---------------------------------------------------------------------------------------
// Workspace layout (caller-owned, zero-filled once; the kernels keep it reusable)
// ---------------------------------------------------------------------------------------
constexpr size_t WS_STATUS = 0;      // uint32: OR of (1 << dit_status) raised on device
constexpr size_t WS_TICKET = 4;      // uint32: CTA completion counter (reset by last CTA)
constexpr size_t WS_AMAX = 8;        // uint32: float bits of a running amax (reset)
constexpr size_t WS_SG = 12;         // float : tensor scale produced by the amax pass
constexpr size_t WS_THR = 16;        // double: outlier threshold k * RMS from the first pass
constexpr size_t WS_PARTIALS = 256;  // double[MAX_RED_CTAS][4]
constexpr int MAX_RED_CTAS = 1024;   // ends at 33024
constexpr size_t WS_BYTES = 64 * 1024;

// Device-side bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t WAIT_LIMIT_NS = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t* ws_u32(void* ws, size_t off) {
  return reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws) + off);
}
__device__ __forceinline__ double* ws_partials(void* ws) {
  return reinterpret_cast<double*>(reinterpret_cast<char*>(ws) + WS_PARTIALS);
}
__device__ __forceinline__ void raise_status(void* ws, int code) {
  atomicOr(ws_u32(ws, WS_STATUS), 1u << code);
}

// ---------------------------------------------------------------------------------------
// 256-bit global memory access (sm_100+), read-only path for streamed inputs
// ---------------------------------------------------------------------------------------
struct alignas(32) U8x32 {
  uint32_t w[8];
};

__device__ __forceinline__ U8x32 ld256_nc(const void* p) {
  U8x32 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                 "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st256(void* p, const U8x32& r) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r.w[0]),
               "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]),
               "r"(r.w[7])
               : "memory");
}

// bf16 pair (element 2i in the low half) -> two floats, exact
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// two floats -> bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}


// ---------------------------------------------------------------------------------------
// packed fp32x2 arithmetic (one instruction for two lanes, no contraction)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r, x, y;
  asm("mov.b64 %0, {%1,%2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  float2 o;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t r, x, y;
  asm("mov.b64 %0, {%1,%2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  float2 o;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t r, x, y;
  asm("mov.b64 %0, {%1,%2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  float2 o;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}

// GEMM epilogue flags: bit 0 = bf16 output (else fp32), bit 1 = GELU (erf form) after bias
constexpr int EPI_BF16 = 1, EPI_GELU = 2;

// GELU(x) = x * Phi(x), Phi the standard normal CDF, from the approximation of erf in
// Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.28 (Hastings):
// for z >= 0, erfc(z) = (1 + a1 z + a2 z^2 + ... + a6 z^6)^-16 + e(z), |e(z)| <= 3e-7.
// With z = |x| / sqrt 2, Phi(x) = erfc(z) / 2 for x < 0 and 1 - erfc(z) / 2 otherwise (no
// cancellation in the negative tail).  One reciprocal and no exponential: the epilogues that
// apply it are bound by the special-function unit, which the erf forms with exp(-z^2) use
// twice per element.  Evaluated in fp32 (the 16th power amplifies the rounding of the
// reciprocal): |computed - x Phi(x)| <= 2.5e-6 |x|, far below bf16 output resolution.
__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r, x, y, z;
  asm("mov.b64 %0, {%1,%2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(z) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(z));
  float2 o;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}
__device__ __forceinline__ float2 gelu_erf2(float2 x) {
  const float2 z = mul2(make_float2(fabsf(x.x), fabsf(x.y)), make_float2(0.70710678118654752f, 0.70710678118654752f));
  float2 d = fma2(z, make_float2(0.0000430638f, 0.0000430638f), make_float2(0.0002765672f, 0.0002765672f));
  d = fma2(d, z, make_float2(0.0001520143f, 0.0001520143f));
  d = fma2(d, z, make_float2(0.0092705272f, 0.0092705272f));
  d = fma2(d, z, make_float2(0.0422820123f, 0.0422820123f));
  d = fma2(d, z, make_float2(0.0705230784f, 0.0705230784f));
  d = fma2(d, z, make_float2(1.0f, 1.0f));
  float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
  r = mul2(r, r);
  r = mul2(r, r);
  r = mul2(r, r);
  r = mul2(r, r);                                        // d^-16 = erfc(z)
  const float2 h = mul2(r, make_float2(0.5f, 0.5f));    // erfc(z) / 2
  const float2 g = sub2(make_float2(1.0f, 1.0f), h);
  return mul2(x, make_float2(x.x < 0.0f ? h.x : g.x, x.y < 0.0f ? h.y : g.y));
}
__device__ __forceinline__ float gelu_erf(float x) { return gelu_erf2(make_float2(x, 0.0f)).x; }

__device__ __forceinline__ float epi_act(float v, int epi) { return (epi & EPI_GELU) ? gelu_erf(v) : v; }
__device__ __forceinline__ float2 epi_act2(float2 v, int epi) { return (epi & EPI_GELU) ? gelu_erf2(v) : v; }

// ---------------------------------------------------------------------------------------
// In-thread fast Walsh-Hadamard transform of 64 values held as 32 pairs (2p, 2p+1).
// Stage h = 1, 2, ..., HB/2 turns every pair (i, i+h) with bit h of i clear into
// (a + b, a - b): the stage order of the Sylvester factorisation, fp32 round-to-nearest.
// ---------------------------------------------------------------------------------------
template <int HB>
__device__ __forceinline__ void fwht64(float2 (&v)[32]) {
  static_assert(HB == 16 || HB == 32 || HB == 64, "block size");
#pragma unroll
  for (int p = 0; p < 32; ++p) {  // h = 1: inside a pair
    float a = v[p].x, b = v[p].y;
    v[p].x = __fadd_rn(a, b);
    v[p].y = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < HB; h <<= 1) {
    const int hp = h >> 1;  // distance in pairs
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      if (((2 * p) & h) == 0) {
        float2 a = v[p], b = v[p + hp];
        v[p] = add2(a, b);
        v[p + hp] = sub2(a, b);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// FP4 / FP8 conversions (documented PTX cvt instructions)
// ---------------------------------------------------------------------------------------
// E2M1 of two floats: `lo` in the low nibble, `hi` in the high nibble; RN-even, saturating
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
// E4M3 code of a float (RN-even, saturating to 448)
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xffu;
}
// value of an E4M3 code (exact)
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  uint16_t c = (uint16_t)code;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// largest |v| over the pairs [p0, p0 + np)
__device__ __forceinline__ float amax_range(const float2 (&v)[32], int p0, int np) {
  float m = 0.f;
#pragma unroll
  for (int p = 0; p < 32; ++p)
    if (p >= p0 && p < p0 + np) m = fmaxf(m, fmaxf(fabsf(v[p].x), fabsf(v[p].y)));
  return m;
}

// NVFP4 encoding of one 16-element block of the transformed tensor (pairs v[0..7]) with tensor
// scale s_g (six_sg = 6 s_g): the E4M3 scale RN(amax_b / (6 s_g)), saturating; the values times
// RN(1 / (dec(scale) s_g)) rounded to E2M1.  Returns the scale code; `out` gets the 8 code bytes
// (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t nvfp4_encode_block16(const float2* v, float s_g, float six_sg, uint32_t (&out)[2]) {
  float ab = 0.f;
#pragma unroll
  for (int p = 0; p < 8; ++p) ab = fmaxf(ab, fmaxf(fabsf(v[p].x), fabsf(v[p].y)));
  uint32_t code = 0;
  float inv = 0.f;
  if (s_g > 0.f) {
    code = e4m3_code(__fdiv_rn(ab, six_sg));
    const float bs = __fmul_rn(e4m3_value(code), s_g);
    inv = bs == 0.f ? 0.f : __frcp_rn(bs);
  }
  const float2 iv = make_float2(inv, inv);
#pragma unroll
  for (int w = 0; w < 2; ++w) {  // 8 elements -> one 32-bit word of 8 codes
    uint32_t word = 0;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float2 s = mul2(v[w * 4 + pp], iv);
      word |= e2m1x2(s.x, s.y) << (8 * pp);
    }
    out[w] = inv == 0.f ? 0u : word;
  }
  return code;
}

// NVFP4 encoding of one 64-element unit of the transformed tensor (four 16-element blocks)
// with tensor scale s_g (six_sg = 6 s_g): per block the E4M3 scale RN(amax_b / (6 s_g)),
// saturating; the block's values times RN(1 / (dec(scale) s_g)) rounded to E2M1.  Returns the
// four scale codes (block g in byte g); `out` gets the 32 code bytes (element 2i low nibble).
__device__ __forceinline__ uint32_t nvfp4_encode_unit(const float2 (&v)[32], float s_g, float six_sg,
                                                      U8x32& out) {
  uint32_t sfword = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t w[2];
    sfword |= nvfp4_encode_block16(&v[g * 8], s_g, six_sg, w) << (8 * g);
    out.w[g * 2] = w[0];
    out.w[g * 2 + 1] = w[1];
  }
  return sfword;
}

// ---------------------------------------------------------------------------------------
// warp / block reductions
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------------------
// mbarrier, TMA and timing primitives
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
      "p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of `parity` to complete; give up after WAIT_LIMIT_NS (or at once when
// *abort is set by another role), raising DIT_ERR_TIMEOUT.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, void* ws,
                                          volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        raise_status(ws, DIT_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 2-D tiled TMA load into shared memory, completion counted on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// ---------------------------------------------------------------------------------------
// 2-CTA clusters (CTA pairs): rank, cross-CTA addressing, arrivals, waits, TMA and commits
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
      "p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait with cluster-scope acquire (arrivals come from the peer CTA as well)
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, void* ws, volatile int* abort) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        raise_status(ws, DIT_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
// TMA load into this CTA's shared memory whose completed bytes count on `bar_cluster`, an
// mbarrier of either CTA of the pair (shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], "
      "[%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
// 3-D tiled TMA load, completion on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], "
      "[%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace dit6

// ---------------------------------------------------------------------------------------
// host-side helpers (defined in api.cu)
// ---------------------------------------------------------------------------------------
namespace dit6 {
int num_sms();  // SM count of the current device (cached per device)
// ---------------------------------------------------------------------------------------
// Programmatic dependent launch (sm_90+).  Every kernel of the library is launched with the
// programmatic stream serialisation attribute (launch_pdl).  Its first instruction lets the
// next kernel on the stream launch once all of its own CTAs are resident
// (pdl_launch_dependents), and it waits for the previous kernel to complete, with that
// kernel's memory operations visible, before its own first global memory access (pdl_wait).
// The next kernel's CTAs thus launch and run their prologue (barrier initialisation, tensor
// memory allocation) while this one drains.  After a launch without the attribute, or after a
// stream operation other than a kernel, both are no-ops.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kern` on `st` with the programmatic stream serialisation attribute, plus a
// cluster dimension when cluster_x > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Failure-path test hook: DIT6_TEST_STALL_PRODUCER=1 makes the GEMMs' producer warp issue no
// loads, so the consumers' bounded waits run out and the kernels report DIT_ERR_TIMEOUT.
int test_stall();
bool aligned32(const void* p);
// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda needed)
// the block-scale array of an NVFP4 operand of `rows` x `k` as a TMA source (one K stage of
// box_blocks 128-row blocks per load)
bool encode_tmap_sf(CUtensorMap* map, const void* sf, int64_t rows, int64_t k, uint32_t box_blocks);
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swz);
}  // namespace dit6

#define DIT_CHECK_LAUNCH()                                  \
  do {                                                      \
    if (cudaGetLastError() != cudaSuccess) return DIT_ERR_CUDA; \
  } while (0)
