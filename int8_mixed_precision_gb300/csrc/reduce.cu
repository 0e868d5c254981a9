// Gamma predictor + routing and the Temporal Delta Cache device steps.
//
// 6Bit-Diffusion (arXiv 2603.18742): [EN] gist.science 2.A Mechanism 1-3 (Gamma, E_rel,
// routing); 2.B (delta cache: residual delta, similarity of the last two computed deltas,
// skip by reusing the cached delta); [IT] 2.B "Riuso" (X_out ~= X_in + Delta_{t-1}).
//
// Design: HBM-bound streaming reductions.  Grid = a fixed multiple of the SM count, each
// thread walks 32-byte vectors of every input (256-bit loads), keeps fp32 partial sums,
// the CTA folds them in fp64 and writes one partial per CTA; the last CTA to finish
// (completion ticket) sums the partials in a fixed order, so results are bit-reproducible
// for a given device and size, and resets the ticket for the next call.
#include "common.cuh"

namespace dit6 {

constexpr int RED_THREADS = 256;

struct RouteParams {
  float alpha[DIT_MAX_LAYERS], beta[DIT_MAX_LAYERS], thr[DIT_MAX_LAYERS];
  int n_layers;
};

// 16 elements per vector for bf16 (32 bytes), 8 for fp32
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 16;
  static __device__ __forceinline__ void unpack(const U8x32& r, float (&v)[16]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float2 f = bf16x2_to_f2(r.w[k]);
      v[2 * k] = f.x;
      v[2 * k + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&v)[16]) {
    unpack(ld256_nc(reinterpret_cast<const char*>(p) + i * 32), v);
  }
  static __device__ __forceinline__ float scalar(const void* p, int64_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&v)[16]) {
    U8x32 r;
#pragma unroll
    for (int k = 0; k < 8; ++k) r.w[k] = f2_to_bf16x2(v[2 * k], v[2 * k + 1]);
    st256(reinterpret_cast<char*>(p) + i * 32, r);
  }
  static __device__ __forceinline__ void store_scalar(void* p, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
  static __device__ __forceinline__ float round_store(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const U8x32& r, float (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(r.w[k]);
  }
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&v)[8]) {
    unpack(ld256_nc(reinterpret_cast<const char*>(p) + i * 32), v);
  }
  static __device__ __forceinline__ float scalar(const void* p, int64_t i) {
    return reinterpret_cast<const float*>(p)[i];
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&v)[8]) {
    U8x32 r;
#pragma unroll
    for (int k = 0; k < 8; ++k) r.w[k] = __float_as_uint(v[k]);
    st256(reinterpret_cast<char*>(p) + i * 32, r);
  }
  static __device__ __forceinline__ void store_scalar(void* p, int64_t i, float v) {
    reinterpret_cast<float*>(p)[i] = v;
  }
  static __device__ __forceinline__ float round_store(float v) { return v; }
};

// Fold NS per-thread fp32 sums into fp64 CTA partials; the last CTA reduces all partials
// in a fixed order into out[0..NS).  Returns true in the thread that holds the result.
template <int NS>
__device__ bool reduce_partials(const float (&s)[NS], void* ws, double (&out)[NS]) {
  __shared__ double sh[RED_THREADS / 32][NS];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  double d[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) d[i] = warp_sum_d((double)s[i]);
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < NS; ++i) sh[wid][i] = d[i];
  __syncthreads();
  double* part = ws_partials(ws);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      double b = 0.0;
      for (int w = 0; w < RED_THREADS / 32; ++w) b += sh[w][i];
      part[blockIdx.x * 4 + i] = b;
    }
    __threadfence();
    last = atomicAdd(ws_u32(ws, WS_TICKET), 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return false;
  __threadfence();
  // fixed-order: thread t sums partials t, t+256, ...; then a fixed tree
  double acc[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) acc[i] = 0.0;
  for (int b = threadIdx.x; b < (int)gridDim.x; b += RED_THREADS)
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] += __ldcg(part + b * 4 + i);
#pragma unroll
  for (int i = 0; i < NS; ++i) acc[i] = warp_sum_d(acc[i]);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < NS; ++i) sh[wid][i] = acc[i];
  __syncthreads();
  if (threadIdx.x != 0) return false;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    double b = 0.0;
    for (int w = 0; w < RED_THREADS / 32; ++w) b += sh[w][i];
    out[i] = b;
  }
  *ws_u32(ws, WS_TICKET) = 0u;
  return true;
}

__device__ __forceinline__ double ratio(double num, double den) {
  if (den == 0.0) return num == 0.0 ? 0.0 : __longlong_as_double(0x7ff0000000000000ll);
  return num / den;
}

template <typename T>
__global__ void __launch_bounds__(RED_THREADS) k_gamma_route(const void* __restrict__ xi,
                                                             const void* __restrict__ xo,
                                                             int64_t n, RouteParams rp,
                                                             float* gamma_out,
                                                             int32_t* routes, void* ws,
                                                             double* partials_out) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int N = Vec<T>::N;
  constexpr int U = 4;  // vectors in flight per thread
  const int64_t nv = n / N;
  float s[2] = {0.f, 0.f};
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (U - 1) * stride < nv; i += U * stride) {
    U8x32 ra[U], rb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      ra[u] = ld256_nc(reinterpret_cast<const char*>(xi) + (i + u * stride) * 32);
      rb[u] = ld256_nc(reinterpret_cast<const char*>(xo) + (i + u * stride) * 32);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float a[N], b[N];
      Vec<T>::unpack(ra[u], a);
      Vec<T>::unpack(rb[u], b);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        s[0] += fabsf(__fsub_rn(b[k], a[k]));
        s[1] += fabsf(a[k]);
      }
    }
  }
  for (; i < nv; i += stride) {
    float a[N], b[N];
    Vec<T>::load(xi, i, a);
    Vec<T>::load(xo, i, b);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      s[0] += fabsf(__fsub_rn(b[k], a[k]));
      s[1] += fabsf(a[k]);
    }
  }
  for (int64_t i = nv * N + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float a = Vec<T>::scalar(xi, i), b = Vec<T>::scalar(xo, i);
    s[0] += fabsf(__fsub_rn(b, a));
    s[1] += fabsf(a);
  }
  double r[2];
  if (!reduce_partials<2>(s, ws, r)) return;
  if (partials_out) {  // one shard of a token-sharded tensor: the sums, for an all-reduce
    partials_out[0] = r[0];
    partials_out[1] = r[1];
    return;
  }
  const double g = ratio(r[0], r[1]);
  *gamma_out = (float)g;
  for (int l = 0; l < rp.n_layers; ++l) {
    const double e = (double)rp.alpha[l] * g + (double)rp.beta[l];
    routes[l] = e > (double)rp.thr[l] ? DIT_ROUTE_INT8 : DIT_ROUTE_NVFP4;
  }
}

// PDR outlier ratio ([EN] 2.C, [ZH] 2.C; reading: the fraction of |x| > k * RMS(x) over the
// whole block input).  Pass 1: sum of squares (per-thread fp32, CTA and final sums in fp64,
// fixed order) -> threshold k * sqrt(sum / n) in fp64 in the workspace.  Pass 2: count of
// |x| > threshold (integers, exact in the fp32/fp64 partial sums) -> count and count / n.
template <typename T>
__global__ void __launch_bounds__(RED_THREADS) k_sumsq(const void* __restrict__ x, int64_t n, float k_sigma,
                                                       void* ws) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int N = Vec<T>::N;
  const int64_t nv = n / N;
  float s[1] = {0.f};
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    float a[N];
    Vec<T>::load(x, i, a);
#pragma unroll
    for (int k = 0; k < N; ++k) s[0] = fmaf(a[k], a[k], s[0]);
  }
  for (int64_t i = nv * N + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float a = Vec<T>::scalar(x, i);
    s[0] = fmaf(a, a, s[0]);
  }
  double r[1];
  if (!reduce_partials<1>(s, ws, r)) return;
  *reinterpret_cast<double*>(reinterpret_cast<char*>(ws) + WS_THR) = (double)k_sigma * sqrt(r[0] / (double)n);
}

template <typename T>
__global__ void __launch_bounds__(RED_THREADS) k_count_over(const void* __restrict__ x, int64_t n, void* ws,
                                                            float* ratio_out, int64_t* count_out) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int N = Vec<T>::N;
  const double thr = *reinterpret_cast<const double*>(reinterpret_cast<const char*>(ws) + WS_THR);
  const int64_t nv = n / N;
  uint32_t c = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    float a[N];
    Vec<T>::load(x, i, a);
#pragma unroll
    for (int k = 0; k < N; ++k) c += (double)fabsf(a[k]) > thr ? 1u : 0u;
  }
  for (int64_t i = nv * N + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    c += (double)fabsf(Vec<T>::scalar(x, i)) > thr ? 1u : 0u;
  const float s[1] = {(float)c};  // per-thread counts stay far below 2^24: exact
  double r[1];
  if (!reduce_partials<1>(s, ws, r)) return;
  const int64_t count = (int64_t)r[0];
  if (count_out) *count_out = count;
  *ratio_out = (float)((double)count / (double)n);
}

// COMMIT: delta = store(xo - xi) -> dnew; sums |xo-xi|, |xi|, |delta - d1|, |d1|
template <typename T>
__global__ void __launch_bounds__(RED_THREADS) k_tdc_commit(const void* __restrict__ xi,
                                                            const void* __restrict__ xo,
                                                            const void* __restrict__ d1,
                                                            void* __restrict__ dnew, int64_t n,
                                                            float* gamma_out, float* sim_out,
                                                            void* ws, double* partials_out) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int N = Vec<T>::N;
  const int64_t nv = n / N;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    float a[N], b[N], c[N], dl[N];
    Vec<T>::load(xi, i, a);
    Vec<T>::load(xo, i, b);
    if (d1) Vec<T>::load(d1, i, c);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const float df = __fsub_rn(b[k], a[k]);
      dl[k] = Vec<T>::round_store(df);
      s[0] += fabsf(df);
      s[1] += fabsf(a[k]);
      if (d1) {
        s[2] += fabsf(__fsub_rn(dl[k], c[k]));
        s[3] += fabsf(c[k]);
      }
    }
    Vec<T>::store(dnew, i, dl);
  }
  for (int64_t i = nv * N + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float a = Vec<T>::scalar(xi, i), b = Vec<T>::scalar(xo, i);
    const float df = __fsub_rn(b, a);
    const float dl = Vec<T>::round_store(df);
    s[0] += fabsf(df);
    s[1] += fabsf(a);
    if (d1) {
      const float c = Vec<T>::scalar(d1, i);
      s[2] += fabsf(__fsub_rn(dl, c));
      s[3] += fabsf(c);
    }
    Vec<T>::store_scalar(dnew, i, dl);
  }
  double r[4];
  if (!reduce_partials<4>(s, ws, r)) return;
  if (partials_out) {  // one shard: the four sums, for an all-reduce
#pragma unroll
    for (int i = 0; i < 4; ++i) partials_out[i] = r[i];
    return;
  }
  *gamma_out = (float)ratio(r[0], r[1]);
  *sim_out = d1 ? (float)ratio(r[2], r[3]) : __int_as_float(0x7f800000);
}

// SKIP: out = store(xi + d1)
template <typename T>
__global__ void __launch_bounds__(RED_THREADS) k_tdc_skip(const void* __restrict__ xi,
                                                          const void* __restrict__ d1,
                                                          void* __restrict__ out, int64_t n) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int N = Vec<T>::N;
  const int64_t nv = n / N;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i0 + stride < nv; i0 += 2 * stride) {  // two vectors in flight per thread
    U8x32 ra[2], rc[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      ra[u] = ld256_nc(reinterpret_cast<const char*>(xi) + (i0 + u * stride) * 32);
      rc[u] = ld256_nc(reinterpret_cast<const char*>(d1) + (i0 + u * stride) * 32);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float a[N], c[N];
      Vec<T>::unpack(ra[u], a);
      Vec<T>::unpack(rc[u], c);
#pragma unroll
      for (int k = 0; k < N; ++k) a[k] = __fadd_rn(a[k], c[k]);
      Vec<T>::store(out, i0 + u * stride, a);
    }
  }
  for (int64_t i = i0; i < nv; i += stride) {
    float a[N], c[N];
    Vec<T>::load(xi, i, a);
    Vec<T>::load(d1, i, c);
#pragma unroll
    for (int k = 0; k < N; ++k) a[k] = __fadd_rn(a[k], c[k]);
    Vec<T>::store(out, i, a);
  }
  for (int64_t i = nv * N + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    Vec<T>::store_scalar(out, i, __fadd_rn(Vec<T>::scalar(xi, i), Vec<T>::scalar(d1, i)));
}

static unsigned red_grid(int64_t n, int per_vec) {
  int64_t nv = n / per_vec;
  int64_t g = (nv + RED_THREADS - 1) / RED_THREADS;
  const int64_t cap = 4 * (int64_t)num_sms();
  if (g > cap) g = cap;
  if (g > MAX_RED_CTAS) g = MAX_RED_CTAS;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace dit6

using namespace dit6;

extern "C" dit_status dit_gamma_route(const void* x_in, const void* x_out, dit_dtype dt,
                                      int64_t n, const float* alpha, const float* beta,
                                      const float* thr, int n_layers, float* gamma_dev,
                                      int32_t* routes_dev, void* ws, size_t ws_bytes,
                                      dit_stream_t stream) {
  if (!x_in || !x_out || n <= 0 || !gamma_dev || !ws || ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (n_layers < 0 || n_layers > DIT_MAX_LAYERS) return DIT_ERR_INVALID_ARG;
  if (n_layers > 0 && (!alpha || !beta || !thr || !routes_dev)) return DIT_ERR_INVALID_ARG;
  if (!aligned32(x_in) || !aligned32(x_out) || !aligned32(ws)) return DIT_ERR_ALIGNMENT;
  RouteParams rp;
  rp.n_layers = n_layers;
  for (int l = 0; l < n_layers; ++l) {
    rp.alpha[l] = alpha[l];
    rp.beta[l] = beta[l];
    rp.thr[l] = thr[l];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dt == DIT_BF16)
    launch_pdl(k_gamma_route<__nv_bfloat16>, dim3(red_grid(n, 16)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, gamma_dev, routes_dev, ws, nullptr);
  else
    launch_pdl(k_gamma_route<float>, dim3(red_grid(n, 8)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, gamma_dev, routes_dev, ws, nullptr);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

extern "C" dit_status dit_tdc_step(int mode, const void* x_in, const void* x_out,
                                   void* x_out_skip, const void* d1, void* d_new, dit_dtype dt,
                                   int64_t n, float* gamma_dev, float* sim_dev, void* ws,
                                   size_t ws_bytes, dit_stream_t stream) {
  if (!x_in || n <= 0) return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int per = dt == DIT_BF16 ? 16 : 8;
  if (mode == DIT_TDC_SKIP) {
    if (!d1 || !x_out_skip) return DIT_ERR_INVALID_ARG;
    if (!aligned32(x_in) || !aligned32(d1) || !aligned32(x_out_skip)) return DIT_ERR_ALIGNMENT;
    int64_t g = (n / per + RED_THREADS - 1) / RED_THREADS;
    const int64_t cap = 8 * (int64_t)num_sms();
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    if (dt == DIT_BF16)
      launch_pdl(k_tdc_skip<__nv_bfloat16>, dim3((unsigned)g), dim3(RED_THREADS), 0, st, 1, x_in, d1, x_out_skip, n);
    else
      launch_pdl(k_tdc_skip<float>, dim3((unsigned)g), dim3(RED_THREADS), 0, st, 1, x_in, d1, x_out_skip, n);
    DIT_CHECK_LAUNCH();
    return DIT_OK;
  }
  if (mode != DIT_TDC_COMMIT) return DIT_ERR_INVALID_ARG;
  if (!x_out || !d_new || !gamma_dev || !sim_dev || !ws || ws_bytes < WS_BYTES)
    return DIT_ERR_INVALID_ARG;
  if (d1 == d_new) return DIT_ERR_INVALID_ARG;
  if (!aligned32(x_in) || !aligned32(x_out) || !aligned32(d_new) || (d1 && !aligned32(d1)) ||
      !aligned32(ws))
    return DIT_ERR_ALIGNMENT;
  if (dt == DIT_BF16)
    launch_pdl(k_tdc_commit<__nv_bfloat16>, dim3(red_grid(n, 16)), dim3(RED_THREADS), 0, st, 1,  x_in, x_out, d1, d_new, n, gamma_dev, sim_dev, ws, nullptr);
  else
    launch_pdl(k_tdc_commit<float>, dim3(red_grid(n, 8)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, d1, d_new, n, gamma_dev, sim_dev, ws, nullptr);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

// ---------------------------------------------------------------------------------------
// Gamma + routing without a caller-supplied workspace.
//
// Some callers cannot hand this library a device buffer: an inference-engine plugin whose
// memory is planned by the engine before execution and which may not allocate while it
// enqueues work, or a latency-critical loop that cannot pay for cudaMalloc (which may
// synchronise the whole device).  For them the per-CTA partial sums and the completion
// counter of the Gamma reduction live in the fixed device array below instead of a
// workspace.  It holds a 256-byte header (status word, completion counter) and partial
// sums for at most NOALLOC_MAX_CTAS CTAs: 20,736 bytes that every GPU which loads the
// library keeps until the process exits.  All calls share it.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace dit6 {
constexpr int NOALLOC_MAX_CTAS = 640;
constexpr size_t NOALLOC_SCRATCH_BYTES = WS_PARTIALS + (size_t)NOALLOC_MAX_CTAS * 4 * sizeof(double);
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
static void* g_noalloc_ptr[NOALLOC_MAX_DEVICES];
static std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.  The first call on a device
// looks the address up (cudaGetSymbolAddress) and zero-fills the array once, synchronously.
// The address stays cached for the life of the process, so the entry point must not be used
// across a cudaDeviceReset, after which the module may be loaded at another address.
static dit_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIT_ERR_CUDA;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return DIT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DIT_ERR_CUDA;
    if (cudaMemset(p, 0, NOALLOC_SCRATCH_BYTES) != cudaSuccess) return DIT_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DIT_OK;
}
}  // namespace dit6

extern "C" dit_status dit_gamma_route_noalloc(const void* x_in, const void* x_out, dit_dtype dt,
                                              int64_t n, const float* alpha, const float* beta,
                                              const float* thr, int n_layers, float* gamma_dev,
                                              int32_t* routes_dev, dit_stream_t stream) {
  if (!x_in || !x_out || n <= 0 || !gamma_dev) return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (n_layers < 0 || n_layers > DIT_MAX_LAYERS) return DIT_ERR_INVALID_ARG;
  if (n_layers > 0 && (!alpha || !beta || !thr || !routes_dev)) return DIT_ERR_INVALID_ARG;
  if (!aligned32(x_in) || !aligned32(x_out)) return DIT_ERR_ALIGNMENT;
  const unsigned grid = red_grid(n, dt == DIT_BF16 ? 16 : 8);
  if (grid > (unsigned)NOALLOC_MAX_CTAS) return DIT_ERR_UNSUPPORTED;  // scratch too small
  void* scratch = nullptr;
  dit_status s = noalloc_scratch(&scratch);
  if (s != DIT_OK) return s;
  RouteParams rp;
  rp.n_layers = n_layers;
  for (int l = 0; l < n_layers; ++l) {
    rp.alpha[l] = alpha[l];
    rp.beta[l] = beta[l];
    rp.thr[l] = thr[l];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the status word and completion counter must start at zero for every call
  if (cudaMemsetAsync(scratch, 0, 8, st) != cudaSuccess) return DIT_ERR_CUDA;
  if (dt == DIT_BF16)
    launch_pdl(k_gamma_route<__nv_bfloat16>, dim3(grid), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, gamma_dev, routes_dev, scratch, nullptr);
  else
    launch_pdl(k_gamma_route<float>, dim3(grid), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, gamma_dev, routes_dev, scratch, nullptr);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

extern "C" dit_status dit_outlier_ratio(const void* x, dit_dtype dt, int64_t n, float k_sigma, float* ratio_dev,
                                        int64_t* count_dev, void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!x || n <= 0 || !ratio_dev || !ws || ws_bytes < WS_BYTES || !(k_sigma >= 0.f)) return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (!aligned32(x) || !aligned32(ws)) return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dt == DIT_BF16) {
    const unsigned g = red_grid(n, 16);
    launch_pdl(k_sumsq<__nv_bfloat16>, dim3(g), dim3(RED_THREADS), 0, st, 1, x, n, k_sigma, ws);
    launch_pdl(k_count_over<__nv_bfloat16>, dim3(g), dim3(RED_THREADS), 0, st, 1, x, n, ws, ratio_dev, count_dev);
  } else {
    const unsigned g = red_grid(n, 8);
    launch_pdl(k_sumsq<float>, dim3(g), dim3(RED_THREADS), 0, st, 1, x, n, k_sigma, ws);
    launch_pdl(k_count_over<float>, dim3(g), dim3(RED_THREADS), 0, st, 1, x, n, ws, ratio_dev, count_dev);
  }
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

// ---------------------------------------------------------------------------------------
// Token-sharded form.  When one block's tokens are split across GPUs, every reduction of the
// path becomes a per-shard partial plus one all-reduce: the two (Gamma) or four (TDC commit)
// L1 sums add, and the NVFP4 tensor amax takes the maximum.  These calls produce a shard's
// partials; dit_shard_finish (device) / dit_shard_finish_host turn the reduced values into
// Gamma, the similarity, the routes and the tensor scale with the arithmetic of the
// unsharded calls.
// ---------------------------------------------------------------------------------------
namespace dit6 {
__global__ void k_shard_finish(const double* __restrict__ p, int n_partials, const float* __restrict__ amax,
                               RouteParams rp, float* gamma_out, float* sim_out, int32_t* routes,
                               float* tensor_scale_out) {
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  if (p) {
    const double g = ratio(p[0], p[1]);
    if (gamma_out) *gamma_out = (float)g;
    if (sim_out) *sim_out = n_partials == 4 ? (float)ratio(p[2], p[3]) : __int_as_float(0x7f800000);
    if (routes)
      for (int l = 0; l < rp.n_layers; ++l) {
        const double e = (double)rp.alpha[l] * g + (double)rp.beta[l];
        routes[l] = e > (double)rp.thr[l] ? DIT_ROUTE_INT8 : DIT_ROUTE_NVFP4;
      }
  }
  if (amax && tensor_scale_out) *tensor_scale_out = __fdiv_rn(*amax, 2688.0f);
}
}  // namespace dit6

extern "C" dit_status dit_l1_partials(int mode, const void* x_in, const void* x_out, const void* d1, void* d_new,
                                      dit_dtype dt, int64_t n, double* partials_dev, void* ws, size_t ws_bytes,
                                      dit_stream_t stream) {
  if (!x_in || !x_out || n <= 0 || !partials_dev || !ws || ws_bytes < WS_BYTES) return DIT_ERR_INVALID_ARG;
  if (dt != DIT_F32 && dt != DIT_BF16) return DIT_ERR_INVALID_ARG;
  if (mode != DIT_L1_GAMMA && mode != DIT_L1_TDC_COMMIT) return DIT_ERR_INVALID_ARG;
  const bool commit = mode == DIT_L1_TDC_COMMIT;
  if (commit && (!d_new || d1 == d_new)) return DIT_ERR_INVALID_ARG;
  if (!aligned32(x_in) || !aligned32(x_out) || !aligned32(ws) || (commit && !aligned32(d_new)) ||
      (commit && d1 && !aligned32(d1)) || (reinterpret_cast<uintptr_t>(partials_dev) & 7))
    return DIT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (commit) {
    if (!d1 && cudaMemsetAsync(partials_dev + 2, 0, 2 * sizeof(double), st) != cudaSuccess) return DIT_ERR_CUDA;
    if (dt == DIT_BF16)
      launch_pdl(k_tdc_commit<__nv_bfloat16>, dim3(red_grid(n, 16)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, d1, d_new, n, nullptr, nullptr, ws, partials_dev);
    else
      launch_pdl(k_tdc_commit<float>, dim3(red_grid(n, 8)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, d1, d_new, n, nullptr, nullptr, ws, partials_dev);
  } else {
    RouteParams rp;
    rp.n_layers = 0;
    if (dt == DIT_BF16)
      launch_pdl(k_gamma_route<__nv_bfloat16>, dim3(red_grid(n, 16)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, nullptr, nullptr, ws, partials_dev);
    else
      launch_pdl(k_gamma_route<float>, dim3(red_grid(n, 8)), dim3(RED_THREADS), 0, st, 1, x_in, x_out, n, rp, nullptr, nullptr, ws, partials_dev);
  }
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

static dit_status route_params(const float* alpha, const float* beta, const float* thr, int n_layers,
                               RouteParams* rp) {
  if (n_layers < 0 || n_layers > DIT_MAX_LAYERS) return DIT_ERR_INVALID_ARG;
  if (n_layers > 0 && (!alpha || !beta || !thr)) return DIT_ERR_INVALID_ARG;
  rp->n_layers = n_layers;
  for (int l = 0; l < n_layers; ++l) {
    rp->alpha[l] = alpha[l];
    rp->beta[l] = beta[l];
    rp->thr[l] = thr[l];
  }
  return DIT_OK;
}

extern "C" dit_status dit_shard_finish(const double* partials_dev, int n_partials, const float* amax_dev,
                                       const float* alpha, const float* beta, const float* thr, int n_layers,
                                       float* gamma_dev, float* sim_dev, int32_t* routes_dev,
                                       float* tensor_scale_dev, dit_stream_t stream) {
  if (partials_dev && n_partials != 2 && n_partials != 4) return DIT_ERR_INVALID_ARG;
  if (!partials_dev && (gamma_dev || sim_dev || routes_dev)) return DIT_ERR_INVALID_ARG;
  if (sim_dev && n_partials != 4) return DIT_ERR_INVALID_ARG;
  if ((amax_dev == nullptr) != (tensor_scale_dev == nullptr)) return DIT_ERR_INVALID_ARG;
  if (!partials_dev && !amax_dev) return DIT_ERR_INVALID_ARG;
  if (routes_dev && n_layers <= 0) return DIT_ERR_INVALID_ARG;
  RouteParams rp;
  dit_status s = route_params(alpha, beta, thr, routes_dev ? n_layers : 0, &rp);
  if (s != DIT_OK) return s;
  launch_pdl(k_shard_finish, dim3(1), dim3(32), 0, reinterpret_cast<cudaStream_t>(stream), 1, partials_dev, n_partials, amax_dev, rp, gamma_dev, sim_dev, routes_dev, tensor_scale_dev);
  DIT_CHECK_LAUNCH();
  return DIT_OK;
}

extern "C" dit_status dit_shard_finish_host(const double* partials, int n_partials, const float* amax,
                                            const float* alpha, const float* beta, const float* thr, int n_layers,
                                            float* gamma, float* sim, int32_t* routes, float* tensor_scale) {
  if (partials && n_partials != 2 && n_partials != 4) return DIT_ERR_INVALID_ARG;
  if (!partials && (gamma || sim || routes)) return DIT_ERR_INVALID_ARG;
  if (sim && n_partials != 4) return DIT_ERR_INVALID_ARG;
  if ((amax == nullptr) != (tensor_scale == nullptr)) return DIT_ERR_INVALID_ARG;
  if (routes && (n_layers <= 0 || n_layers > DIT_MAX_LAYERS || !alpha || !beta || !thr)) return DIT_ERR_INVALID_ARG;
  auto host_ratio = [](double num, double den) {
    if (den == 0.0) return num == 0.0 ? 0.0 : (double)INFINITY;
    return num / den;
  };
  if (partials) {
    const double g = host_ratio(partials[0], partials[1]);
    if (gamma) *gamma = (float)g;
    if (sim) *sim = (float)host_ratio(partials[2], partials[3]);
    if (routes)
      for (int l = 0; l < n_layers; ++l) {
        const double e = (double)alpha[l] * g + (double)beta[l];
        routes[l] = e > (double)thr[l] ? DIT_ROUTE_INT8 : DIT_ROUTE_NVFP4;
      }
  }
  if (amax) {
    volatile float a = *amax;  // one correctly rounded fp32 division, as on the device
    *tensor_scale = a / 2688.0f;
  }
  return DIT_OK;
}
