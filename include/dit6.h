/*
 * dit6.h -- C ABI of libdit6, the GB300 (sm_103a) hot path of the dynamically routed
 * NVFP4 / INT8 linear layer of a video diffusion transformer block, with its Temporal
 * Delta Cache.
 *
 * Method: "6Bit-Diffusion: Inference-Time Mixed-Precision Quantization for Video Diffusion
 * Models" (arXiv 2603.18742).  Passages are cited by page and section:
 *   [EN]  gist.science summary (English)   [IT] gist.science summary (Italian)
 *   [ZH]  gist.science summary (Chinese)   [ABS] the authors' abstract (chatpaper.ai)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named *_dev or passed as tensors are DEVICE pointers owned by the caller.
 *   Pointers documented as "host" are read synchronously during the call.
 * - The library never allocates, frees or synchronises.  Every call only enqueues work on
 *   `stream` and returns.  Its kernels are launched with programmatic dependent launch: one
 *   may start its prologue while the previous kernel on the stream drains, but waits for that
 *   kernel to complete before touching memory, so stream order holds as for plain launches.  The return code covers argument errors found on the host;
 *   errors found on the device (a bounded wait that ran out) are OR-ed into the status
 *   word at byte 0 of the workspace (see dit_ws_status_offset), which the caller reads
 *   after synchronising.
 * - Workspace: `ws` is a caller-owned device buffer of at least dit_workspace_bytes()
 *   bytes, zero-filled once by the caller before its first use.  The kernels keep it in a
 *   reusable state (every counter they bump is reset by the same launch).  Two calls that
 *   run concurrently on the GPU must not share one workspace.
 * - Tensors are row-major and contiguous.  Activation and delta tensors are bf16 or fp32
 *   (dit_dtype).  Device pointers must be 32-byte aligned (256-bit vector loads).
 * - All entry points are thread-compatible.  The library's only global mutable state is a
 *   cached driver entry point, per-device caches of the SM count, and the fixed scratch
 *   array of dit_gamma_route_noalloc (with its per-device address cache); calls of that entry
 *   point share the array and race when they overlap on the GPU (see its comment).
 */
#ifndef DIT6_H_
#define DIT6_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dit_stream_t; /* == cudaStream_t; NULL is the legacy stream */

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = 1, /* a null pointer, a negative or inconsistent size */
  DIT_ERR_ALIGNMENT = 2,   /* a device pointer is not 32-byte aligned */
  DIT_ERR_UNSUPPORTED = 3, /* a shape the kernels do not cover (see each call) */
  DIT_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed at launch */
  DIT_ERR_TIMEOUT = 5      /* device status bit: a bounded wait inside a kernel ran out */
} dit_status;

typedef enum { DIT_F32 = 0, DIT_BF16 = 1, DIT_I8 = 2 } dit_dtype;
typedef enum { DIT_ROUTE_NVFP4 = 0, DIT_ROUTE_INT8 = 1, DIT_ROUTE_BF16 = 2 } dit_route;
typedef enum { DIT_TDC_COMMIT = 0, DIT_TDC_SKIP = 1 } dit_tdc_mode;
/* Activation applied in the GEMM epilogue after the bias: none, or GELU in its erf form
 * x * Phi(x) (the FFN activation between the up and down projections of the CogVideoX-shaped
 * block), computed in fp32 before the output is stored, with Phi from the erf approximation
 * of Abramowitz & Stegun 7.1.28: |computed - x Phi(x)| <= 2.5e-6 |x|. */
typedef enum { DIT_ACT_NONE = 0, DIT_ACT_GELU_ERF = 1 } dit_act;

#define DIT_MAX_LAYERS 16

/* Human-readable name of a status code (static storage). */
const char* dit_status_str(dit_status s);

/* Library version, "major.minor.patch" (static storage). */
const char* dit_version(void);

/* Bytes of workspace every call below needs (a constant, 64 KiB: a status word, a completion
 * counter, a running amax, a tensor scale and the per-CTA partial sums of the reductions). */
size_t dit_workspace_bytes(void);

/* Byte offset, inside the workspace, of the uint32 device status word (bit i set means
 * status code i was raised on the device since the caller last cleared it). */
size_t dit_ws_status_offset(void);

/* ------------------------------------------------------------------------------------
 * (a1 + a2) Gamma predictor and routing.
 * [EN] 2. Methodology, A. DMPQ, Mechanism 1-3; [IT] 2.A Meccanismo / Routing Dinamico.
 *
 * Gamma = sum|x_out - x_in| / sum|x_in| over all n elements (the relative L1 distance of a
 * block's output and input at the previous step), then for each of n_layers linear layers
 * E_rel = alpha[l] * Gamma + beta[l] and route[l] = INT8 if E_rel > thr[l] else NVFP4.
 * Per-thread fp32 partial sums, fp64 across threads and CTAs in a fixed order (the result
 * is bit-reproducible run to run); E_rel and the comparison in fp64.
 *
 * x_in, x_out : device, n elements of dtype dt.
 * alpha, beta, thr : HOST arrays of n_layers floats (1 <= n_layers <= DIT_MAX_LAYERS).
 * gamma_dev   : device float, receives Gamma (sum|x_in| = 0: 0 if the numerator is 0 else
 *               +inf).
 * routes_dev  : device int32[n_layers], receives dit_route values.
 * ------------------------------------------------------------------------------------ */
dit_status dit_gamma_route(const void* x_in, const void* x_out, dit_dtype dt, int64_t n,
                           const float* alpha, const float* beta, const float* thr,
                           int n_layers, float* gamma_dev, int32_t* routes_dev, void* ws,
                           size_t ws_bytes, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * dit_gamma_route without a workspace argument.  The paper has no counterpart: this is a
 * convenience of this library for callers that cannot allocate device memory -- e.g. an
 * inference-engine plugin whose memory is planned by the engine ahead of time and which may
 * not allocate while enqueueing, or a latency-critical loop that cannot afford cudaMalloc
 * (it may synchronise the device).
 *
 * Same arguments and results as dit_gamma_route, minus ws / ws_bytes.  The reduction's
 * scratch (a status word, a completion counter and per-CTA partial sums) lives in a fixed
 * device array of 20,736 bytes inside the library, holding partials for at most 640 CTAs;
 * every GPU that loads the library keeps it until the process exits.  The launch uses
 * min(ceil(n / 4096), 4 x SM count) CTAs for bf16 (n / 2048 for fp32); a request that needs
 * more than 640 returns DIT_ERR_UNSUPPORTED.  Nothing is allocated: no cudaMalloc, cudaFree
 * or allocating library routine is called.
 *
 * The first call on a device sets the scratch up (looks up its device address with
 * cudaGetSymbolAddress and zero-fills it once, synchronously, with that device current);
 * make that first call before any stream capture.  The address is cached per device for
 * the life of the process: do not use this entry point across a cudaDeviceReset (the
 * module, and with it the array, may come back at another address).  Every call clears the
 * status word and counter asynchronously on `stream`.  All calls share the one array and it
 * keeps the last call's contents: calls whose kernels overlap on the GPU (different streams,
 * no ordering between them) race on it and give wrong results.
 * ------------------------------------------------------------------------------------ */
dit_status dit_gamma_route_noalloc(const void* x_in, const void* x_out, dit_dtype dt,
                                   int64_t n, const float* alpha, const float* beta,
                                   const float* thr, int n_layers, float* gamma_dev,
                                   int32_t* routes_dev, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a3 + a4) Online block Hadamard transform fused with NVFP4 quantisation.
 * [EN] 2.A "Outlier Smoothing" (block Hadamard on local activation blocks);
 * [IT] "3. Contributi Chiave" 4 (NVFP4 = E2M1); [ZH] 2.A (weights quantised offline).
 *
 * y = x (H_b / sqrt(b)) on every contiguous block of b elements along K (Sylvester order,
 * fp32 butterflies in stages h = 1, 2, ..., b/2, then the 1/sqrt(b) scale), then
 *   s_g = amax|y| / 2688 (whole tensor; or *tensor_scale_in when that is not NULL)
 *   s_b = E4M3_rne_sat(amax_b / (6 s_g))       per 16 elements
 *   q   = E2M1_rne_sat(y * rcp(dec(s_b) s_g))  per element
 *
 * x      : device [rows x k] of dtype dt; k % 64 == 0; hblock in {16, 32, 64}.
 * codes  : device [rows x k/2] bytes, element 2i in the low nibble, 2i+1 in the high.
 * sf     : device, dit_sf_bytes(rows, k) bytes; E4M3 scales in the tile layout of
 *          dit_sf_index (rows padded to 128 are written with zeros).
 * tensor_scale_dev : device float, receives s_g.
 * tensor_scale_in  : device float or NULL.  NULL -> two passes over x (amax, then
 *          quantise); non-NULL -> one pass with the given s_g (values beyond the range
 *          saturate).
 * ------------------------------------------------------------------------------------ */
dit_status dit_hadamard_quant_nvfp4(const void* x, dit_dtype dt, int64_t rows, int64_t k,
                                    int hblock, uint8_t* codes, uint8_t* sf,
                                    float* tensor_scale_dev, const float* tensor_scale_in,
                                    void* ws, size_t ws_bytes, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a3 + a5) Online block Hadamard transform fused with per-token INT8 quantisation.
 * [EN] 2.A Mechanism 3 (the INT8 route), "Outlier Smoothing".
 *
 * y as above; per row s = amax_row|y| / 127, q = round_half_even(y * rcp(s)) in
 * [-127, 127]; an all-zero row gives s = 0 and q = 0.  The same call quantises weights
 * per output channel (rows of W).
 *
 * x     : device [rows x k] of dtype dt; k % 64 == 0, k <= 16384; hblock in {16,32,64}.
 * q     : device [rows x k] codes in container q_dt: DIT_I8 (int8) or DIT_BF16 (the same
 *         integers stored as bf16, exact; the operand format of the INT8 GEMM on the bf16
 *         tensor pipe).
 * row_scale : device float [rows].
 * ------------------------------------------------------------------------------------ */
dit_status dit_hadamard_quant_int8(const void* x, dit_dtype dt, int64_t rows, int64_t k,
                                   int hblock, void* q, dit_dtype q_dt, float* row_scale,
                                   dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * INT8 weights from NVFP4-only weights.  [ZH] 2.A, weight handling: all weights are held
 * in NVFP4 and converted only when a layer routes INT8.
 *
 * w[r, c] = (dec(code[r, c]) * dec(sf[r, c/16])) * (*tensor_scale)  in fp32 (the first
 * product is exact), then per row s = amax_row|w| / 127, q = round_half_even(w * rcp(s)) --
 * the INT8 encoding of dit_hadamard_quant_int8, with no transform (the NVFP4 weight is
 * already in the rotated basis).
 * codes : device packed E2M1 [rows x k/2]; sf : device tile-layout scales (dit_sf_bytes);
 * tensor_scale : device float.  q : device [rows x k] in container q_dt (DIT_I8 or DIT_BF16);
 * row_scale : device float [rows].  k % 64 == 0, k <= 16384; codes, sf, q 32-byte aligned.
 * ------------------------------------------------------------------------------------ */
dit_status dit_nvfp4_to_int8(const uint8_t* codes, const uint8_t* sf, const float* tensor_scale,
                             int64_t rows, int64_t k, void* q, dit_dtype q_dt, float* row_scale,
                             dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a6) NVFP4 GEMM on the block-scaled tensor cores (tcgen05 kind::mxf4nvf4).
 * [EN] 1. Problem Statement "Hardware Gap", 3. Key Contributions 4 (NVFP4 on Blackwell).
 *
 * Y[m, n] = (*a_gs) (*b_gs) sum_k dec(A)[m,k] dec(sA)[m,k/16] dec(B)[n,k] dec(sB)[n,k/16]
 *           (+ bias[n]), then act (dit_act) elementwise
 * a, b   : device packed E2M1, [m x k/2] and [n x k/2] (both K-major, as written by
 *          dit_hadamard_quant_nvfp4); a_sf, b_sf: tile-layout scales; a_gs, b_gs: device
 *          floats (the tensor scales).  k % 64 == 0; n % 8 == 0.
 * bias   : device float [n] or NULL.     act : DIT_ACT_NONE or DIT_ACT_GELU_ERF (any other
 *          value is DIT_ERR_INVALID_ARG).     y : device [m x n] of dtype y_dt.
 * ------------------------------------------------------------------------------------ */
dit_status dit_qgemm_nvfp4(const uint8_t* a, const uint8_t* a_sf, const float* a_gs,
                           const uint8_t* b, const uint8_t* b_sf, const float* b_gs,
                           int64_t m, int64_t n, int64_t k, const float* bias, dit_act act,
                           void* y, dit_dtype y_dt, void* ws, size_t ws_bytes,
                           dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * NVFP4 GEMM whose epilogue also produces the tensor scale of its own output for the next
 * NVFP4 layer (FFN up -> down): the two-phase form of fusing the next layer's quantisation.
 * [EN] 2.A Mechanism 2-3 (online block Hadamard before NVFP4 quantisation): the dynamic
 * tensor scale of the next layer's input is max|H Z| / (6 * 448) over the whole tensor, so it
 * can only be applied once every output tile is known; this call computes it on the fly and
 * the next layer's dit_hadamard_quant_nvfp4(tensor_scale_in = *tensor_scale_out) is then one
 * pass instead of two, with the same codes and scales byte for byte.
 *
 * y = act(dit_qgemm_nvfp4 product (+ bias)) in bf16 -- the same bytes dit_qgemm_nvfp4 writes;
 * *tensor_scale_out (device float) = max over y of |block Hadamard (blocks of hblock along n,
 * orthonormal) of y as stored| / (6 * 448), exactly the tensor scale
 * dit_hadamard_quant_nvfp4(y, hblock, ...) derives.  hblock in {16, 32, 64}; n % 64 == 0;
 * k % 64 == 0; y device bf16 [m x n], 32-byte aligned.  The workspace's amax word and
 * completion ticket are used and left reset.
 * ------------------------------------------------------------------------------------ */
dit_status dit_qgemm_nvfp4_amax(const uint8_t* a, const uint8_t* a_sf, const float* a_gs,
                                const uint8_t* b, const uint8_t* b_sf, const float* b_gs,
                                int64_t m, int64_t n, int64_t k, const float* bias, dit_act act,
                                void* y, int hblock, float* tensor_scale_out, void* ws,
                                size_t ws_bytes, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * INT8 GEMM whose epilogue quantises its own output for the next INT8 layer (FFN up -> down)
 * with caller-supplied per-token scales: the INT8 form of fusing the next layer's
 * quantisation.  [EN] 2.A Mechanism 3 (per-token INT8) and 2.A Outlier Smoothing (online block
 * Hadamard before quantisation).  The method's per-token scale of the next layer's input is
 * max|H z| / 127 over the whole output row, which 30-48 output tiles hold; this call takes
 * the scales as an input (from an earlier denoising step: delayed per-token scales, a
 * variant the pages do not describe) and reports the exact row maxima of this output, so the
 * bf16 round trip of the output and the next layer's quantiser pass are skipped.
 *
 * a, b: bf16-held INT8 codes (K-major), scales as dit_qgemm_int8.  For each row m and each
 * 64-element block of n: z = act(acc * a_scale[m] * b_scale[n] (+ bias[n])) rounded to bf16
 * exactly as dit_qgemm_int8 stores it; y = H_64 z / 8 (the quantiser's butterfly order);
 * q = clamp(RN(y * RN(1 / next_scale[m])), -127, 127) (next_scale[m] = 0 gives 0), written
 * to q_next (device, bf16-held codes [m x n], 32-byte aligned); row_amax (device float [m],
 * zero-filled by the caller) receives max(row_amax[m], max over the row of |y|).  With
 * next_scale[m] = row_amax[m] / 127 of this very output, q_next equals
 * dit_hadamard_quant_int8(z, hblock = 64) bit for bit; a smaller scale saturates the entries
 * beyond 127 * next_scale[m].  n % 64 == 0, k % 16 == 0, act NONE or GELU_ERF.
 * ------------------------------------------------------------------------------------ */
dit_status dit_qgemm_int8_requant(const void* a, const float* a_scale, const void* b,
                                  const float* b_scale, int64_t m, int64_t n, int64_t k,
                                  const float* bias, dit_act act, const float* next_scale,
                                  void* q_next, float* row_amax, void* ws, size_t ws_bytes,
                                  dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * PDR outlier ratio and the BF16 route.  [EN] 2.C first bullet, [ZH] 2.C: a layer whose
 * input has a high outlier ratio runs in full precision.  The pages do not define the
 * ratio; reading: the fraction of elements with |x| > k_sigma * RMS(x) over the whole block
 * input (k_sigma = 6 in the workloads), strict >.
 *
 * dit_outlier_ratio: two passes (sum of squares, fixed-order fp64 reduction -> threshold
 * k_sigma * sqrt(sum / n); then the count of |x| > threshold).  ratio_dev: device float
 * (count / n); count_dev: device int64 or NULL.  x: device [n] of dtype dt, 32-byte aligned.
 *
 * dit_gemm_bf16: Y = act(X W^T (+ bias)) on untransformed bf16 operands (the BF16 route),
 * fp32 accumulation.  x [m x k], w [n x k] bf16 K-major; k % 16 == 0, n % 8 == 0; bias
 * device float [n] (16-byte aligned) or NULL.
 *
 * dit_route_host_pdr: dit_route_host, except that outlier_ratio > rho sends every layer to
 * DIT_ROUTE_BF16 (rho = +inf: no override).
 * ------------------------------------------------------------------------------------ */
dit_status dit_outlier_ratio(const void* x, dit_dtype dt, int64_t n, float k_sigma, float* ratio_dev,
                             int64_t* count_dev, void* ws, size_t ws_bytes, dit_stream_t stream);
dit_status dit_gemm_bf16(const void* x, const void* w, int64_t m, int64_t n, int64_t k,
                         const float* bias, dit_act act, void* y, dit_dtype y_dt, void* ws,
                         size_t ws_bytes, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a7) INT8 GEMM: exact int32 accumulation, per-row x per-column dequantisation.
 * [EN] 2.A Mechanism 3 (INT8 route); [ZH] 2.A weight handling.
 *
 * acc[m, n] = sum_k a[m, k] b[n, k] (int32, exact);
 * Y[m, n]   = act((float(acc) * a_scale[m]) * b_scale[n] (+ bias[n])), act as in a6.
 * a, b : device codes [m x k] and [n x k] in container ab_dt:
 *        DIT_I8   -> warp-level IMMA (mma.sync s8) path;
 *        DIT_BF16 -> tcgen05 bf16 path: the integer codes are exact in bf16, products exact
 *                    in fp32, and K is accumulated in chunks of <= 1024 so every partial sum
 *                    stays below 2^24 (exact), then summed in int32.  Same results, bit for
 *                    bit, as the IMMA path; ~10x its throughput on sm_103a.
 * k % 16 == 0; n % 8 == 0.
 * acc_debug : device int32 [m x n] or NULL (writes the raw accumulators as well).
 * ------------------------------------------------------------------------------------ */
dit_status dit_qgemm_int8(const void* a, const float* a_scale, const void* b,
                          const float* b_scale, dit_dtype ab_dt, int64_t m, int64_t n, int64_t k,
                          const float* bias, dit_act act, void* y, dit_dtype y_dt,
                          int32_t* acc_debug, void* ws, size_t ws_bytes, dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a8 / a10) Temporal Delta Cache device step.
 * [EN] 2.B (TDC); [IT] 2.B "Riuso" (X_out,t ~= X_in,t + Delta_{t-1}).
 *
 * mode DIT_TDC_COMMIT (a compute step just produced x_out):
 *   delta = store(x_out - x_in) -> d_new        (fp32 difference, then dtype dt)
 *   *gamma_dev = sum|x_out - x_in| / sum|x_in|  (Gamma_t, fp64 final ratio)
 *   *sim_dev   = sum|delta - d1| / sum|d1|      (relative L1 of the last two computed
 *                deltas; d1 may be NULL, then *sim_dev = +inf)
 * mode DIT_TDC_SKIP: x_out_skip = store(x_in + d1); gamma_dev / sim_dev untouched.
 * n elements; d_new must not alias d1 (the caller keeps a two-slot ring and swaps).
 * ------------------------------------------------------------------------------------ */
dit_status dit_tdc_step(int mode, const void* x_in, const void* x_out, void* x_out_skip,
                        const void* d1, void* d_new, dit_dtype dt, int64_t n,
                        float* gamma_dev, float* sim_dev, void* ws, size_t ws_bytes,
                        dit_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (a9 + a11) Host-side delta-cache decision and PDR routing (no device work).
 * [EN] 2.B "Error Control"; [EN] 2.C second bullet (INT8 after a skip); [ZH] 2.C.
 *
 * decide: n_computed < 2 -> COMMIT (compute); e_acc + d <= tau -> SKIP; else compute.
 * update after a SKIP: e_acc += d, gamma_valid = 0.
 * update after a compute: e_acc = 0, n_computed++, d = sim (if finite-or-first), gamma =
 *   the step's Gamma, gamma_valid = 1.
 * route: gamma_valid ? (alpha*gamma+beta > thr ? INT8 : NVFP4) : INT8 for every layer.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int64_t n_computed;
  double e_acc;
  double d;       /* +inf until two deltas have been computed */
  double gamma;   /* Gamma of the last step (valid iff gamma_valid) */
  int gamma_valid;
} dit_tdc_state;

void dit_tdc_state_init(dit_tdc_state* st);
int dit_tdc_decide(const dit_tdc_state* st, double tau); /* returns dit_tdc_mode */
void dit_tdc_update(dit_tdc_state* st, int mode, double gamma, double sim, int has_sim);
void dit_route_host(const dit_tdc_state* st, const float* alpha, const float* beta,
                    const float* thr, int n_layers, int32_t* routes);
void dit_route_host_pdr(const dit_tdc_state* st, const float* alpha, const float* beta,
                        const float* thr, int n_layers, double outlier_ratio, double rho,
                        int32_t* routes);

/* ------------------------------------------------------------------------------------
 * Token-sharded form (one block's tokens split across GPUs, one rank per GPU).
 * The reductions of [EN] 2.A Mechanism 1 (Gamma), 2.B (the delta similarity) and of the NVFP4
 * tensor scale ([IT] "Contributi Chiave" 4; one fp32 scale over the whole tensor) span all
 * tokens, so a rank computes its shard's partials, the ranks all-reduce them (sum for the L1
 * sums, max for the amax), and the finishing call applies the unsharded arithmetic.  Every
 * other step of the path (quantisation with the finished tensor scale, the GEMMs against
 * replicated weights, the delta-cache skip) works on a shard alone.  The library performs no
 * collective itself: the caller all-reduces with its own communicator.
 *
 * dit_l1_partials (device): mode DIT_L1_GAMMA -> partials_dev[0..1] = sum|x_out - x_in|,
 *   sum|x_in| over this shard's n elements; mode DIT_L1_TDC_COMMIT -> also writes
 *   d_new = store(x_out - x_in) as dit_tdc_step COMMIT does and partials_dev[0..3] =
 *   sum|x_out - x_in|, sum|x_in|, sum|d_new - d1|, sum|d1| (the last two 0 when d1 is NULL).
 *   Fixed-order fp64 sums (bit-reproducible for a given shard).  partials_dev: device
 *   double[2] or [4], 8-byte aligned.
 * dit_nvfp4_amax (device): *amax_dev = max|block Hadamard (x)| over this shard [rows x k]
 *   (arguments as dit_hadamard_quant_nvfp4).
 * dit_shard_finish (device) / dit_shard_finish_host (host pointers, synchronous): from the
 *   all-reduced partials, Gamma = p[0] / p[1] and sim = p[2] / p[3] (n_partials = 4) in fp64
 *   with the 0/0 -> 0, x/0 -> +inf rule, routes as dit_gamma_route; from the all-reduced
 *   amax, tensor_scale = amax / 2688 (one fp32 division, the value the unsharded quantiser
 *   derives).  Any output may be NULL; partials may be NULL when only the tensor scale is
 *   wanted, amax (with tensor_scale) when only the ratios are.
 * ------------------------------------------------------------------------------------ */
typedef enum { DIT_L1_GAMMA = 0, DIT_L1_TDC_COMMIT = 1 } dit_l1_mode;

dit_status dit_l1_partials(int mode, const void* x_in, const void* x_out, const void* d1, void* d_new,
                           dit_dtype dt, int64_t n, double* partials_dev, void* ws, size_t ws_bytes,
                           dit_stream_t stream);
dit_status dit_nvfp4_amax(const void* x, dit_dtype dt, int64_t rows, int64_t k, int hblock,
                          float* amax_dev, void* ws, size_t ws_bytes, dit_stream_t stream);
dit_status dit_shard_finish(const double* partials_dev, int n_partials, const float* amax_dev,
                            const float* alpha, const float* beta, const float* thr, int n_layers,
                            float* gamma_dev, float* sim_dev, int32_t* routes_dev,
                            float* tensor_scale_dev, dit_stream_t stream);
dit_status dit_shard_finish_host(const double* partials, int n_partials, const float* amax,
                                 const float* alpha, const float* beta, const float* thr,
                                 int n_layers, float* gamma, float* sim, int32_t* routes,
                                 float* tensor_scale);

/* ------------------------------------------------------------------------------------
 * Block-scale tile layout helpers (host).  The scales of a [rows x k] NVFP4 tensor are
 * cut into atoms of 128 rows x 4 scale columns (512 bytes), ordered with the scale-column
 * atom index fastest; inside an atom row r, column c is at (r%32)*16 + ((r%128)/32)*4 +
 * c%4.  This is the operand layout of the block-scaled tcgen05 MMA.
 * ------------------------------------------------------------------------------------ */
int64_t dit_sf_index(int64_t row, int64_t kblock, int64_t rows, int64_t k);
size_t dit_sf_bytes(int64_t rows, int64_t k);

#ifdef __cplusplus
}
#endif
#endif /* DIT6_H_ */
