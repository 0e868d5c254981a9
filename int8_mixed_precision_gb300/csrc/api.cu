// Host-side part of the libdit6 C ABI: status strings, workspace and tile-layout helpers,
// driver entry points, and the delta-cache decision logic of 6Bit-Diffusion
// ([EN] gist.science 2.B "Error Control", 2.C second bullet).
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace dit6 {

int num_sms() {
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::call_once(flags[dev], [dev]() {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  });
  return cache[dev];
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int test_stall() {
  const char* e = getenv("DIT6_TEST_STALL_PRODUCER");
  return (e && e[0] == '1') ? 1 : 0;
}

typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

static encode_tiled_fn get_encode_tiled() {
  static encode_tiled_fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<encode_tiled_fn>(p);
  });
  return fn;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swz) {
  encode_tiled_fn fn = get_encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale factors in the MMA tile layout ([row blocks of 128][K / 64 atoms][512 bytes]) as a
// 3-D tensor of 32-bit words {128 words per atom, atoms along K, row blocks}; a box of
// {128, 4, box_blocks} is one 256-deep K stage of box_blocks row blocks.  Atoms past K and
// row blocks past the padded rows read as zeros.
bool encode_tmap_sf(CUtensorMap* map, const void* sf, int64_t rows, int64_t k, uint32_t box_blocks) {
  encode_tiled_fn fn = get_encode_tiled();
  if (!fn) return false;
  const uint64_t atoms = (uint64_t)(k / 64), blocks = (uint64_t)((rows + 127) / 128);
  cuuint64_t dims[3] = {128, atoms, blocks};
  cuuint64_t strides[2] = {512, 512 * atoms};
  cuuint32_t box[3] = {128, 4, box_blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(sf), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dit6

extern "C" {

const char* dit_status_str(dit_status s) {
  switch (s) {
    case DIT_OK: return "DIT_OK";
    case DIT_ERR_INVALID_ARG: return "DIT_ERR_INVALID_ARG";
    case DIT_ERR_ALIGNMENT: return "DIT_ERR_ALIGNMENT";
    case DIT_ERR_UNSUPPORTED: return "DIT_ERR_UNSUPPORTED";
    case DIT_ERR_CUDA: return "DIT_ERR_CUDA";
    case DIT_ERR_TIMEOUT: return "DIT_ERR_TIMEOUT";
  }
  return "DIT_ERR_UNKNOWN";
}

const char* dit_version(void) { return "0.1.0"; }

size_t dit_workspace_bytes(void) { return dit6::WS_BYTES; }
size_t dit_ws_status_offset(void) { return dit6::WS_STATUS; }

int64_t dit_sf_index(int64_t row, int64_t kblock, int64_t rows, int64_t k) {
  if (row < 0 || kblock < 0 || rows <= 0 || k <= 0 || k % 16) return -1;
  const int64_t kb = k / 16;
  const int64_t cpad = (kb + 3) / 4 * 4;
  const int64_t rpad = (rows + 127) / 128 * 128;
  if (row >= rpad || kblock >= cpad) return -1;
  const int64_t atom = (row / 128) * (cpad / 4) + kblock / 4;
  const int64_t ri = row % 128;
  return atom * 512 + (ri % 32) * 16 + (ri / 32) * 4 + kblock % 4;
}

size_t dit_sf_bytes(int64_t rows, int64_t k) {
  if (rows <= 0 || k <= 0 || k % 16) return 0;
  const int64_t kb = k / 16;
  return (size_t)((rows + 127) / 128 * 128) * (size_t)((kb + 3) / 4 * 4);
}

void dit_tdc_state_init(dit_tdc_state* st) {
  if (!st) return;
  st->n_computed = 0;
  st->e_acc = 0.0;
  st->d = INFINITY;
  st->gamma = 0.0;
  st->gamma_valid = 0;
}

int dit_tdc_decide(const dit_tdc_state* st, double tau) {
  if (!st || st->n_computed < 2) return DIT_TDC_COMMIT;
  return (st->e_acc + st->d <= tau) ? DIT_TDC_SKIP : DIT_TDC_COMMIT;
}

void dit_tdc_update(dit_tdc_state* st, int mode, double gamma, double sim, int has_sim) {
  if (!st) return;
  if (mode == DIT_TDC_SKIP) {
    st->e_acc += st->d;
    st->gamma_valid = 0;
    return;
  }
  st->e_acc = 0.0;
  st->n_computed += 1;
  if (has_sim) st->d = sim;
  st->gamma = gamma;
  st->gamma_valid = 1;
}

void dit_route_host(const dit_tdc_state* st, const float* alpha, const float* beta,
                    const float* thr, int n_layers, int32_t* routes) {
  if (!routes || n_layers <= 0) return;
  for (int l = 0; l < n_layers; ++l) {
    if (!st || !st->gamma_valid) {
      routes[l] = DIT_ROUTE_INT8;
      continue;
    }
    const double e = (double)alpha[l] * st->gamma + (double)beta[l];
    routes[l] = e > (double)thr[l] ? DIT_ROUTE_INT8 : DIT_ROUTE_NVFP4;
  }
}

void dit_route_host_pdr(const dit_tdc_state* st, const float* alpha, const float* beta, const float* thr,
                        int n_layers, double outlier_ratio, double rho, int32_t* routes) {
  if (!routes || n_layers <= 0) return;
  if (outlier_ratio > rho) {
    for (int l = 0; l < n_layers; ++l) routes[l] = DIT_ROUTE_BF16;
    return;
  }
  dit_route_host(st, alpha, beta, thr, n_layers, routes);
}

}  // extern "C"
