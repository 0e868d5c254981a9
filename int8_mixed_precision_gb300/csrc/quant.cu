// Online block Hadamard transform fused with NVFP4 or per-token INT8 quantisation.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science 2.A "Outlier Smoothing" (a fast
// Hadamard transform over local activation blocks, applied online), 2.A Mechanism 3 (the
// INT8 / NVFP4 routes); [IT] "3. Contributi Chiave" 4 (NVFP4 = E2M1 micro-scaled).
//
// Design: HBM-bound streaming kernels.  One thread owns one 64-element unit of a row
// (64 elements = 1, 2 or 4 Hadamard blocks), loads it with 256-bit vector loads (every
// 32-byte sector fully used), runs the butterflies in registers with packed fp32x2
// arithmetic, and writes its codes with one 256-bit store (NVFP4: 32 bytes) or two
// (INT8: 64 bytes).  No shared-memory staging and no shuffles are needed on the data path.
#include "common.cuh"

namespace dit6 {

constexpr int UNIT = 64;

template <typename T>
struct Loader;

template <>
struct Loader<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const void* base, int64_t unit, float2 (&v)[32]) {
    const char* p = reinterpret_cast<const char*>(base) + unit * (UNIT * 2);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      U8x32 r = ld256_nc(p + 32 * c);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[c * 8 + i] = bf16x2_to_f2(r.w[i]);
    }
  }
};

template <>
struct Loader<float> {
  static __device__ __forceinline__ void load(const void* base, int64_t unit, float2 (&v)[32]) {
    const char* p = reinterpret_cast<const char*>(base) + unit * (UNIT * 4);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      U8x32 r = ld256_nc(p + 32 * c);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[c * 4 + i] = make_float2(__uint_as_float(r.w[2 * i]), __uint_as_float(r.w[2 * i + 1]));
    }
  }
};

// y = fwht(x) * float(1/sqrt(b))
template <typename T, int HB>
__device__ __forceinline__ void load_transform(const void* x, int64_t unit, float2 (&v)[32],
                                               float inv_sqrt_b) {
  Loader<T>::load(x, unit, v);
  fwht64<HB>(v);
  const float2 c = make_float2(inv_sqrt_b, inv_sqrt_b);
#pragma unroll
  for (int p = 0; p < 32; ++p) v[p] = mul2(v[p], c);
}

// Raw bytes of one unit, fetched ahead of use so the next unit's loads are in flight while
// the current unit is transformed (software pipelining of the streaming loops).
template <typename T>
struct RawUnit {
  static constexpr int CHUNKS = UNIT * (int)sizeof(T) / 32;
  U8x32 r[CHUNKS];
  __device__ __forceinline__ void fetch(const void* base, int64_t unit) {
    const char* p = reinterpret_cast<const char*>(base) + unit * (UNIT * (int64_t)sizeof(T));
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) r[c] = ld256_nc(p + 32 * c);
  }
  __device__ __forceinline__ void unpack(float2 (&v)[32]) const {
    if (sizeof(T) == 2) {
#pragma unroll
      for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[c * 8 + i] = bf16x2_to_f2(r[c].w[i]);
    } else {
#pragma unroll
      for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[c * 4 + i] = make_float2(__uint_as_float(r[c].w[2 * i]), __uint_as_float(r[c].w[2 * i + 1]));
    }
  }
};

template <typename T, int HB>
__device__ __forceinline__ void transform_raw(const RawUnit<T>& raw, float2 (&v)[32], float inv_sqrt_b) {
  raw.unpack(v);
  fwht64<HB>(v);
  const float2 c = make_float2(inv_sqrt_b, inv_sqrt_b);
#pragma unroll
  for (int p = 0; p < 32; ++p) v[p] = mul2(v[p], c);
}


// ---------------------------------------------------------------------------------------
// INT8: CTA = `tr` whole rows x `upr` units per row; row amax through shared memory.
// ---------------------------------------------------------------------------------------
// OUT_BF16: the integer codes are written as bf16 values (exact for |q| <= 127), the
// operand format of the INT8 GEMM that runs on the bf16 tensor pipe.
template <typename T, int HB, bool OUT_BF16>
__global__ void __launch_bounds__(256) k_quant_int8(const void* __restrict__ x, int64_t rows,
                                                    int upr, int tr, float inv_sqrt_b,
                                                    void* __restrict__ q,
                                                    float* __restrict__ row_scale) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ unsigned row_amax[256];
  const int t = threadIdx.x;
  if (t < tr) row_amax[t] = 0u;
  __syncthreads();
  const int rl = t / upr, j = t - rl * upr;
  const int64_t row = (int64_t)blockIdx.x * tr + rl;
  const bool active = rl < tr && row < rows;
  const int64_t unit = row * upr + j;
  float2 v[32];
  if (active) {
    load_transform<T, HB>(x, unit, v, inv_sqrt_b);
    atomicMax(&row_amax[rl], __float_as_uint(amax_range(v, 0, 32)));
  }
  __syncthreads();
  if (!active) return;
  const float amax = __uint_as_float(row_amax[rl]);
  const float s = __fdiv_rn(amax, 127.0f);
  const float inv = s == 0.f ? 0.f : __frcp_rn(s);
  const float2 iv = make_float2(inv, inv);
  if (OUT_BF16) {
    U8x32 out[4];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const float2 a = mul2(v[p], iv);
      // |a| <= 127 * (1 + 3 * 2^-24): round-to-nearest-even never leaves [-127, 127]
      out[p / 8].w[p % 8] = f2_to_bf16x2(rintf(a.x), rintf(a.y));
    }
    char* dst = reinterpret_cast<char*>(q) + unit * (UNIT * 2);
#pragma unroll
    for (int c = 0; c < 4; ++c) st256(dst + 32 * c, out[c]);
  } else {
    U8x32 out[2];
#pragma unroll
    for (int p = 0; p < 32; p += 2) {
      const float2 a = mul2(v[p], iv), b = mul2(v[p + 1], iv);
      // |a|,|b| <= 127 * (1 + 3 * 2^-24): round-to-nearest-even never leaves [-127, 127]
      const int q0 = __float2int_rn(a.x), q1 = __float2int_rn(a.y);
      const int q2 = __float2int_rn(b.x), q3 = __float2int_rn(b.y);
      const uint32_t w = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) |
                         ((uint32_t)(q2 & 0xff) << 16) | ((uint32_t)(q3 & 0xff) << 24);
      out[p / 16].w[(p % 16) / 2] = w;
    }
    int8_t* dst = reinterpret_cast<int8_t*>(q) + unit * UNIT;
    st256(dst, out[0]);
    st256(dst + 32, out[1]);
  }
  if (j == 0) row_scale[row] = s;
}

// ---------------------------------------------------------------------------------------
// NVFP4 weights -> per-output-channel INT8 ([ZH] 2.A, weight handling: weights held in NVFP4
// only, converted when a layer routes INT8).  w = (dec(code) * dec(block scale)) * s_g in
// fp32 (the first product exact), then the INT8 encoding of k_quant_int8 (no transform: the
// NVFP4 weight is already in the rotated basis).  CTA = `tr` rows x `upr` 64-element units.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float e2m1_decode(uint32_t n) {
  const uint32_t e = (n >> 1) & 3u, m = n & 1u;
  const float mag = e == 0 ? (m ? 0.5f : 0.0f) : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (n & 8u) ? -mag : mag;
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(256) k_nvfp4_to_int8(const uint8_t* __restrict__ codes,
                                                       const uint8_t* __restrict__ sf,
                                                       const float* __restrict__ gs, int64_t rows, int upr,
                                                       int tr, void* __restrict__ q,
                                                       float* __restrict__ row_scale) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ unsigned row_amax[256];
  const int t = threadIdx.x;
  if (t < tr) row_amax[t] = 0u;
  __syncthreads();
  const int rl = t / upr, j = t - rl * upr;
  const int64_t row = (int64_t)blockIdx.x * tr + rl;
  const bool active = rl < tr && row < rows;
  const int64_t unit = row * upr + j;
  float2 v[32];
  if (active) {
    const float s_g = *gs;
    const U8x32 c = ld256_nc(codes + unit * 32);
    const int64_t ri = row & 127;
    const uint32_t sfw = *reinterpret_cast<const uint32_t*>(sf + ((row >> 7) * upr + j) * 512 + (ri & 31) * 16 +
                                                            (ri >> 5) * 4);
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // four 16-element blocks, one scale byte each
      const float sc = e4m3_value((sfw >> (8 * g)) & 0xffu);
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // byte p = 8g + i holds elements 2p (low nibble), 2p + 1
        const uint32_t byte = (c.w[(8 * g + i) >> 2] >> (8 * ((8 * g + i) & 3))) & 0xffu;
        v[8 * g + i] = make_float2(__fmul_rn(__fmul_rn(e2m1_decode(byte & 15u), sc), s_g),
                                   __fmul_rn(__fmul_rn(e2m1_decode(byte >> 4), sc), s_g));
      }
    }
    atomicMax(&row_amax[rl], __float_as_uint(amax_range(v, 0, 32)));
  }
  __syncthreads();
  if (!active) return;
  const float amax = __uint_as_float(row_amax[rl]);
  const float s = __fdiv_rn(amax, 127.0f);
  const float inv = s == 0.f ? 0.f : __frcp_rn(s);
  const float2 iv = make_float2(inv, inv);
  if (OUT_BF16) {
    U8x32 out[4];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const float2 a = mul2(v[p], iv);
      out[p / 8].w[p % 8] = f2_to_bf16x2(rintf(a.x), rintf(a.y));
    }
    char* dst = reinterpret_cast<char*>(q) + unit * (UNIT * 2);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) st256(dst + 32 * c4, out[c4]);
  } else {
    U8x32 out[2];
#pragma unroll
    for (int p = 0; p < 32; p += 2) {
      const float2 a = mul2(v[p], iv), b = mul2(v[p + 1], iv);
      const int q0 = __float2int_rn(a.x), q1 = __float2int_rn(a.y);
      const int q2 = __float2int_rn(b.x), q3 = __float2int_rn(b.y);
      out[p / 16].w[(p % 16) / 2] = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) |
                                    ((uint32_t)(q2 & 0xff) << 16) | ((uint32_t)(q3 & 0xff) << 24);
    }
    int8_t* dst = reinterpret_cast<int8_t*>(q) + unit * UNIT;
    st256(dst, out[0]);
    st256(dst + 32, out[1]);
  }
  if (j == 0) row_scale[row] = s;
}

// ---------------------------------------------------------------------------------------
// NVFP4 pass 1: amax of the transformed tensor -> s_g = amax / 2688 (workspace + output)
// ---------------------------------------------------------------------------------------
// raw_amax: write amax itself to tensor_scale_out (one shard of a token-sharded tensor, whose
// tensor scale follows the all-reduce-max of every shard's amax), not s_g
template <typename T, int HB>
__global__ void __launch_bounds__(256) k_nvfp4_amax(const void* __restrict__ x, int64_t units,
                                                    float inv_sqrt_b, void* ws,
                                                    float* __restrict__ tensor_scale_out, int raw_amax) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float wmax[8];
  __shared__ bool last;
  float m = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  RawUnit<T> cur;
  if (u < units) cur.fetch(x, u);
  for (; u < units; u += stride) {
    RawUnit<T> nxt;
    if (u + stride < units) nxt.fetch(x, u + stride);
    float2 v[32];
    transform_raw<T, HB>(cur, v, inv_sqrt_b);
    m = fmaxf(m, amax_range(v, 0, 32));
    cur = nxt;
  }
  m = warp_max_f(m);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b = fmaxf(b, wmax[w]);
    atomicMax(ws_u32(ws, WS_AMAX), __float_as_uint(b));
    __threadfence();
    const unsigned ticket = atomicAdd(ws_u32(ws, WS_TICKET), 1u);
    last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    const float amax = __uint_as_float(atomicExch(ws_u32(ws, WS_AMAX), 0u));
    if (raw_amax) {
      *tensor_scale_out = amax;
    } else {
      const float sg = __fdiv_rn(amax, 2688.0f);
      *reinterpret_cast<float*>(ws_u32(ws, WS_SG)) = sg;
      *tensor_scale_out = sg;
    }
    *ws_u32(ws, WS_TICKET) = 0u;
  }
}

// ---------------------------------------------------------------------------------------
// NVFP4 pass 2 (or the single pass with a given tensor scale): codes + tile-layout scales
// ---------------------------------------------------------------------------------------
template <typename T, int HB>
__global__ void __launch_bounds__(256) k_nvfp4_quant(const void* __restrict__ x, int64_t rows,
                                                     int upr, int64_t pad_units,
                                                     float inv_sqrt_b, const float* sg_ptr,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ sf,
                                                     float* __restrict__ tensor_scale_out,
                                                     int copy_scale) {
  pdl_launch_dependents();
  pdl_wait();
  const float s_g = *sg_ptr;
  if (copy_scale && blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale_out = s_g;
  const float six_sg = __fmul_rn(6.0f, s_g);
  const int64_t units = rows * upr;
  const int64_t atoms_per_row = upr;  // 4 scale columns per unit == one atom column
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  RawUnit<T> cur;
  if (u < units) cur.fetch(x, u);
  for (; u < pad_units; u += stride) {
    const int64_t row = u / upr;
    const int64_t j = u - row * upr;
    const int64_t ri = row & 127;
    uint32_t* sfw = reinterpret_cast<uint32_t*>(
        sf + ((row >> 7) * atoms_per_row + j) * 512 + (ri & 31) * 16 + (ri >> 5) * 4);
    if (u >= units) {  // rows padded up to a multiple of 128: zero scales
      *sfw = 0u;
      continue;
    }
    RawUnit<T> nxt;
    if (u + stride < units) nxt.fetch(x, u + stride);
    float2 v[32];
    transform_raw<T, HB>(cur, v, inv_sqrt_b);
    cur = nxt;
    U8x32 out;
    const uint32_t sfword = nvfp4_encode_unit(v, s_g, six_sg, out);
    st256(codes + u * 32, out);
    *sfw = sfword;
  }
}

template <typename T, bool OB>
static dit_status launch_int8(const void* x, int64_t rows, int64_t k, int hb, void* q,
                              float* rs, cudaStream_t st) {
  const int upr = (int)(k / UNIT);
  // rows per CTA: the fewest that give 64 threads (one row once K > 2048).  A CTA's barrier
  // waits for all its rows' loads, so small CTAs overlap loads and stores best (measured on
  // GB300, 17776 rows: K = 1920 29.3 us at 1-2 rows vs 33.4 at 8; K = 7680 99 vs 107 us at 2)
  const int tr = upr >= 64 ? 1 : 64 / upr;
  const int threads = tr * upr;
  const int64_t grid = (rows + tr - 1) / tr;
  if (grid > 0x7fffffff) return DIT_ERR_UNSUPPORTED;
  const float isb = (float)(1.0 / sqrt((double)hb));
  switch (hb) {
    case 16: launch_pdl(k_quant_int8<T, 16, OB>, dim3((unsigned)grid), dim3(threads), 0, st, 1, x, rows, upr, tr, isb, q, rs); break;
    case 32: launch_pdl(k_quant_int8<T, 32, OB>, dim3((unsigned)grid), dim3(threads), 0, st, 1, x, rows, upr, tr, isb, q, rs); break;
    default: launch_pdl(k_quant_int8<T, 64, OB>, dim3((unsigned)grid), dim3(threads), 0, st, 1, x, rows, upr, tr, isb, q, rs); break;
  }
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

template <typename T, int HB>
static void launch_nvfp4_t(const void* x, int64_t rows, int upr, float isb, uint8_t* codes,
                           uint8_t* sf, float* ts_out, const float* ts_in, void* ws,
                           cudaStream_t st) {
  const int64_t units = rows * upr;
  const int64_t pad_units = ((rows + 127) / 128 * 128) * upr;
  const int sms = num_sms();
  const float* sgp = ts_in;
  if (!ts_in) {
    int64_t g1 = (units + 255) / 256;
    if (g1 > 6 * sms) g1 = 6 * sms;
    if (g1 < 1) g1 = 1;
    launch_pdl(k_nvfp4_amax<T, HB>, dim3((unsigned)g1), dim3(256), 0, st, 1, x, units, isb, ws, ts_out, 0);
    sgp = reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws) + WS_SG);
  }
  int64_t g2 = (pad_units + 255) / 256;
  if (g2 > 6 * sms) g2 = 6 * sms;
  if (g2 < 1) g2 = 1;
  launch_pdl(k_nvfp4_quant<T, HB>, dim3((unsigned)g2), dim3(256), 0, st, 1, x, rows, upr, pad_units, isb, sgp, codes, sf, ts_out, ts_in ? 1 : 0);
}

}  // namespace dit6

using namespace dit6;

static dit_status check_quant_args(const void* x, dit_dtype dt, int64_t rows, int64_t k,
                                   int hblock) {
  if (!x || rows <= 0 || k <= 0) return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (k % UNIT || (hblock != 16 && hblock != 32 && hblock != 64)) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(x)) return DIT_ERR_ALIGNMENT;
  return DIT_OK;
}

extern "C" dit_status dit_hadamard_quant_int8(const void* x, dit_dtype dt, int64_t rows,
                                              int64_t k, int hblock, void* q, dit_dtype q_dt,
                                              float* row_scale, dit_stream_t stream) {
  dit_status s = check_quant_args(x, dt, rows, k, hblock);
  if (s != DIT_OK) return s;
  if (!q || !row_scale) return DIT_ERR_INVALID_ARG;
  if (q_dt != DIT_I8 && q_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (k > 256 * UNIT) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(q)) return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (q_dt == DIT_BF16)
    return dt == DIT_BF16 ? launch_int8<__nv_bfloat16, true>(x, rows, k, hblock, q, row_scale, st)
                          : launch_int8<float, true>(x, rows, k, hblock, q, row_scale, st);
  return dt == DIT_BF16 ? launch_int8<__nv_bfloat16, false>(x, rows, k, hblock, q, row_scale, st)
                        : launch_int8<float, false>(x, rows, k, hblock, q, row_scale, st);
}

extern "C" dit_status dit_hadamard_quant_nvfp4(const void* x, dit_dtype dt, int64_t rows,
                                               int64_t k, int hblock, uint8_t* codes,
                                               uint8_t* sf, float* tensor_scale_dev,
                                               const float* tensor_scale_in, void* ws,
                                               size_t ws_bytes, dit_stream_t stream) {
  dit_status s = check_quant_args(x, dt, rows, k, hblock);
  if (s != DIT_OK) return s;
  if (!codes || !sf || !tensor_scale_dev || !ws || ws_bytes < WS_BYTES) return DIT_ERR_INVALID_ARG;
  if (!aligned32(codes) || !aligned32(sf) || !aligned32(ws)) return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int upr = (int)(k / UNIT);
  const float isb = (float)(1.0 / sqrt((double)hblock));
#define DIT_NV(T, HB) \
  launch_nvfp4_t<T, HB>(x, rows, upr, isb, codes, sf, tensor_scale_dev, tensor_scale_in, ws, st)
  if (dt == DIT_BF16) {
    if (hblock == 16) DIT_NV(__nv_bfloat16, 16);
    else if (hblock == 32) DIT_NV(__nv_bfloat16, 32);
    else DIT_NV(__nv_bfloat16, 64);
  } else {
    if (hblock == 16) DIT_NV(float, 16);
    else if (hblock == 32) DIT_NV(float, 32);
    else DIT_NV(float, 64);
  }
#undef DIT_NV
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

extern "C" dit_status dit_nvfp4_to_int8(const uint8_t* codes, const uint8_t* sf, const float* tensor_scale,
                                        int64_t rows, int64_t k, void* q, dit_dtype q_dt, float* row_scale,
                                        dit_stream_t stream) {
  if (!codes || !sf || !tensor_scale || !q || !row_scale || rows <= 0 || k <= 0) return DIT_ERR_INVALID_ARG;
  if (q_dt != DIT_I8 && q_dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (k % UNIT || k > 256 * UNIT) return DIT_ERR_UNSUPPORTED;
  if (!aligned32(codes) || !aligned32(sf) || !aligned32(q)) return DIT_ERR_ALIGNMENT;
  const int upr = (int)(k / UNIT);
  const int tr = upr >= 64 ? 1 : 64 / upr;  // as in the activation quantiser
  const int64_t grid = (rows + tr - 1) / tr;
  if (grid > 0x7fffffff) return DIT_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (q_dt == DIT_BF16)
    launch_pdl(k_nvfp4_to_int8<true>, dim3((unsigned)grid), dim3(tr * upr), 0, st, 1, codes, sf, tensor_scale, rows, upr, tr, q, row_scale);
  else
    launch_pdl(k_nvfp4_to_int8<false>, dim3((unsigned)grid), dim3(tr * upr), 0, st, 1, codes, sf, tensor_scale, rows, upr, tr, q, row_scale);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

// One shard of a token-sharded tensor: max|H x| over this shard's rows (the all-reduce-max of
// every shard's value, turned into s_g = amax / (6 * 448) by dit_shard_finish, is the tensor
// scale the unsharded quantiser derives from the whole tensor).
template <typename T, int HB>
static void launch_amax_shard(const void* x, int64_t rows, int upr, float isb, float* amax_out, void* ws,
                              cudaStream_t st) {
  const int64_t units = rows * upr;
  int64_t g1 = (units + 255) / 256;
  if (g1 > 6 * num_sms()) g1 = 6 * num_sms();
  if (g1 < 1) g1 = 1;
  launch_pdl(k_nvfp4_amax<T, HB>, dim3((unsigned)g1), dim3(256), 0, st, 1, x, units, isb, ws, amax_out, 1);
}

extern "C" dit_status dit_nvfp4_amax(const void* x, dit_dtype dt, int64_t rows, int64_t k, int hblock,
                                     float* amax_dev, void* ws, size_t ws_bytes, dit_stream_t stream) {
  dit_status s = check_quant_args(x, dt, rows, k, hblock);
  if (s != DIT_OK) return s;
  if (!amax_dev || !ws || ws_bytes < WS_BYTES) return DIT_ERR_INVALID_ARG;
  if (!aligned32(ws)) return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int upr = (int)(k / UNIT);
  const float isb = (float)(1.0 / sqrt((double)hblock));
#define DIT_AS(T, HB) launch_amax_shard<T, HB>(x, rows, upr, isb, amax_dev, ws, st)
  if (dt == DIT_BF16) {
    if (hblock == 16) DIT_AS(__nv_bfloat16, 16);
    else if (hblock == 32) DIT_AS(__nv_bfloat16, 32);
    else DIT_AS(__nv_bfloat16, 64);
  } else {
    if (hblock == 16) DIT_AS(float, 16);
    else if (hblock == 32) DIT_AS(float, 32);
    else DIT_AS(float, 64);
  }
#undef DIT_AS
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}
