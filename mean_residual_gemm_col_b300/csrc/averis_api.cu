// C ABI of libaveris.so: argument checks, workspace carving, tensor-map
// encoding and kernel launches.  Declarations and per-call contracts are in
// include/averis.h.
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "averis.h"
#include "gemm.cuh"
#include "quant.cuh"

namespace {

using namespace averis;

constexpr int kMaxDevices = 64;
constexpr int kStatsTargetCtas = 296;  // CTA count target of the stats pass (one wave at 2 per SM of a B300)

__device__ int g_device_error = 0;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* err_word = nullptr;
  bool attrs_set = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mutex;

// Diagnostics of the timeout path (averis_debug_starve_next_quantize): when
// non-zero, the next quantize call's statistics pass requests no input and
// waits at most this many SM cycles for it.
long long g_starve_next = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

averis_status set_attrs();

// Per-device setup: SM count, architecture check, error-word address, kernel attributes.
averis_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AVERIS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AVERIS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return AVERIS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return AVERIS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return AVERIS_ERR_CUDA;
    if (d.cc_major != 10 || d.cc_minor != 3) return AVERIS_ERR_UNSUPPORTED_ARCH;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return AVERIS_ERR_CUDA;
    d.err_word = static_cast<int*>(addr);
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return AVERIS_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  if (!d.attrs_set) {
    averis_status st = set_attrs();
    if (st != AVERIS_OK) return st;
    d.attrs_set = true;
  }
  *out = &d;
  return AVERIS_OK;
}

averis_status set_attrs() {
  if (cudaFuncSetAttribute(colstats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStatsSmem) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_nvfp4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::SMEM) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_nvfp4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::SMEM) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  return AVERIS_OK;
}

// ------------------------------------------------------------ geometry --

struct StatsGeom {
  int gx, nstrips, nrb;
  int64_t rows_per;
};

// Stats-pass grid: 64-column strips, at most kMaxStripGroups strip groups,
// and enough row blocks for about kStatsTargetCtas CTAs in all.
StatsGeom stats_geom(int64_t R, int64_t C) {
  StatsGeom g;
  g.nstrips = (int)cdiv(C, 64);
  g.gx = std::min(g.nstrips, (int)kMaxStripGroups);
  // one wave of CTAs (2 per SM), each at least 256 rows (8 per thread), row
  // blocks balanced to a multiple of 32 rows
  int64_t nrb = std::max<int64_t>(1, kStatsTargetCtas / g.gx);
  nrb = std::max<int64_t>(1, std::min<int64_t>(nrb, cdiv(R, 256)));
  int64_t rp = cdiv(R, nrb);
  rp = cdiv(rp, 32) * 32;
  g.rows_per = rp;
  g.nrb = (int)cdiv(R, rp);
  return g;
}

constexpr size_t kCtrlBytes = ((size_t)kCtrlWords * sizeof(unsigned) + 255) & ~size_t(255);
static_assert(kCtrlBytes == AVERIS_WORKSPACE_CTRL_BYTES, "control block size is part of the ABI");

size_t quant_ws_bytes(int64_t R, int64_t C) {
  const StatsGeom g = stats_geom(R, C);
  return kCtrlBytes + align256((size_t)g.nrb * (size_t)C * sizeof(ColPartial));
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes; it waits (griddepcontrol.wait)
// before touching anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

bool nvfp4_ok(const averis_nvfp4* t, int64_t rows, int64_t cols) {
  return t != nullptr && t->codes != nullptr && t->scales != nullptr && t->tensor_scale != nullptr &&
         t->rows == rows && t->cols == cols && aligned(t->codes, 16) && aligned(t->scales, 16) &&
         aligned(t->tensor_scale, 4);
}

// 2-D tiled tensor map (128-byte swizzle, zero fill out of bounds).
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------- quantize --

// Largest column count of a mean split: the NVFP4 mean is staged in the
// shared memory of the quantize pass's mean CTAs.
constexpr int64_t kMaxSplitCols = 147456;

// r_w / r_out (optional, split only): also compute the rank-one row
// r_out[N] = deq(mu_q) deq(r_w)^T for an NVFP4 r_w [N, C] blocked along C.
averis_status quantize_impl(const void* x, int64_t R, int64_t C, unsigned flags, float* mu, const averis_nvfp4* mu_q,
                            float* mu_hat, const averis_nvfp4* out_row, const averis_nvfp4* out_col, void* ws,
                            size_t ws_bytes, cudaStream_t s, const averis_nvfp4* r_w = nullptr,
                            float* r_out = nullptr) {
  if (x == nullptr || R < 1 || C < 16 || C % 16 != 0 || !aligned(x, 16)) return AVERIS_ERR_INVALID_ARG;
  if (R > (int64_t)1 << 31 || C > (int64_t)1 << 31) return AVERIS_ERR_INVALID_ARG;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  const bool had = (flags & AVERIS_HADAMARD16) != 0;
  if (out_row != nullptr && !nvfp4_ok(out_row, R, C)) return AVERIS_ERR_INVALID_ARG;
  if (out_col != nullptr && !nvfp4_ok(out_col, C, R)) return AVERIS_ERR_INVALID_ARG;
  if (split && (mu == nullptr || mu_hat == nullptr || !aligned(mu, 16) || !aligned(mu_hat, 16) ||
                !nvfp4_ok(mu_q, 1, C)))
    return AVERIS_ERR_INVALID_ARG;
  if (split && C > kMaxSplitCols) return AVERIS_ERR_INVALID_ARG;
  if ((r_w == nullptr) != (r_out == nullptr)) return AVERIS_ERR_INVALID_ARG;
  if (r_w != nullptr && (!split || r_w->rows < 1 || !nvfp4_ok(r_w, r_w->rows, C) || !aligned(r_out, 4)))
    return AVERIS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256)) return AVERIS_ERR_INVALID_ARG;
  if (ws_bytes < quant_ws_bytes(R, C)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  averis_status st = device_info(&dev);
  if (st != AVERIS_OK) return st;

  if (out_row == nullptr && out_col == nullptr && !split) return AVERIS_OK;  // nothing to compute
  uint8_t* w = static_cast<uint8_t*>(ws);
  unsigned* ctrl = reinterpret_cast<unsigned*>(w);
  ColPartial* part = reinterpret_cast<ColPartial*>(w + kCtrlBytes);
  const StatsGeom g = stats_geom(R, C);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);

  StatsParams sp{};
  sp.x = xb;
  sp.R = R;
  sp.C = C;
  sp.rows_per = g.rows_per;
  sp.nstrips = g.nstrips;
  sp.part = part;
  sp.ctrl = ctrl;
  sp.split = split ? 1 : 0;
  sp.hadamard = had ? 1 : 0;
  sp.mu = mu;
  sp.err = dev->err_word;
  sp.wait_limit = kWaitLimit;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_starve_next > 0) {
      sp.starve = 1;
      sp.wait_limit = g_starve_next;
      g_starve_next = 0;
    }
  }
  CUtensorMap tstats;  // X in boxes of 64 columns x 256 rows for the stats pass
  if (!encode_2d(&tstats, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(x), (uint64_t)C, (uint64_t)R,
                 (uint64_t)C * 2, 64u, (uint32_t)kStatsBoxRows))
    return AVERIS_ERR_CUDA;
  if (launch_pdl(colstats_kernel, dim3(g.gx, g.nrb), dim3(256), kStatsSmem, s, tstats, sp) != cudaSuccess)
    return AVERIS_ERR_CUDA;

  // The quantize pass also writes the NVFP4 mean (one of its CTAs) and resets
  // the control block, so it runs even with no residual layout requested.
  QuantParams qp{};
  qp.R = R;
  qp.C = C;
  qp.mu = split ? mu : nullptr;
  if (split) {
    qp.mu_codes = mu_q->codes;
    qp.mu_scales = mu_q->scales;
    qp.mu_ts = mu_q->tensor_scale;
    qp.mu_hat = mu_hat;
    qp.mu_kc = cdiv(C, 64);
  }
  qp.ctrl = ctrl;
  qp.err = dev->err_word;
  qp.wait_limit = kWaitLimit;
  qp.hadamard = had ? 1 : 0;
  if (out_row != nullptr) {
    qp.row_codes = out_row->codes;
    qp.row_scales = out_row->scales;
    qp.row_ts = out_row->tensor_scale;
    qp.row_ld = averis_nvfp4_ld(C);
    qp.row_kc = cdiv(C, 64);
  }
  if (out_col != nullptr) {
    qp.col_codes = out_col->codes;
    qp.col_scales = out_col->scales;
    qp.col_ts = out_col->tensor_scale;
    qp.col_ld = averis_nvfp4_ld(R);
    qp.col_kc = cdiv(R, 64);
  }
  qp.tiles_r = (int)cdiv(R, kQTile);
  qp.tiles_c = (int)cdiv(C, kQTile);
  CUtensorMap tx;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)R};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {64, kQTile};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return AVERIS_ERR_CUDA;
  }
  if (out_row == nullptr && out_col == nullptr) qp.tiles_r = 0;  // mean only
  // mean CTAs: one for the mean alone, more when they also compute the
  // rank-one row (about 128 K weights each, at most 64)
  qp.mean_ctas = 0;
  if (split) {
    qp.mean_ctas = 1;
    if (r_w != nullptr) {
      qp.w_codes = r_w->codes;
      qp.w_scales = r_w->scales;
      qp.w_ts = r_w->tensor_scale;
      qp.w_rows = r_w->rows;
      qp.w_ld = averis_nvfp4_ld(C);
      qp.w_kc = cdiv(C, 64);
      qp.r_out = r_out;
      qp.mean_ctas = (int)std::max<int64_t>(1, std::min<int64_t>(64, cdiv(r_w->rows * C, (int64_t)1 << 17)));
    }
  }
  const int ntiles = qp.tiles_r * qp.tiles_c;
  // all CTAs resident at once (2 per SM): tile CTAs fill what the mean CTAs leave
  const int tile_ctas =
      ntiles == 0 ? 0 : (int)std::max<int64_t>(1, std::min<int64_t>(ntiles, kQCtasPerSm * (int64_t)dev->sms - qp.mean_ctas));
  if (had) {
    QuantParams ap = qp;  // rotated-maximum pass: tiles only
    ap.mean_ctas = 0;
    if (launch_pdl(split_quant_kernel<true, true>, dim3(std::max(1, tile_ctas)), dim3(kQThreads), kQSmem, s, tx, ap) !=
        cudaSuccess)
      return AVERIS_ERR_CUDA;
  }
  // the rotation is a template parameter: the plain kernel carries no butterfly code
  auto* qk = had ? split_quant_kernel<false, true> : split_quant_kernel<false, false>;
  if (launch_pdl(qk, dim3(std::max(1, qp.mean_ctas + tile_ctas)), dim3(kQThreads), kQSmem, s, tx, qp) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  return AVERIS_OK;
}

// ----------------------------------------------------------------- GEMM --


// early_start: the kernel launched just before this GEMM produced none of its
// inputs (see GemmParams::early_start).
averis_status gemm_impl(const averis_nvfp4* a, const averis_nvfp4* b, const float* col_add, const float* row_vec,
                        const float* col_vec, float outer, void* out, int64_t ldo, unsigned flags, cudaStream_t s,
                        bool early_start = false) {
  if (a == nullptr || b == nullptr || out == nullptr) return AVERIS_ERR_INVALID_ARG;
  const int64_t M = a->rows, N = b->rows, K = a->cols;
  // K may be ragged (the token axis of dW): codes and scales are zero-padded to 64
  if (M < 1 || N < 1 || K < 1 || b->cols != K) return AVERIS_ERR_INVALID_ARG;
  if (M > (int64_t)1 << 30 || N > (int64_t)1 << 30 || K > (int64_t)1 << 30) return AVERIS_ERR_INVALID_ARG;
  if (!nvfp4_ok(a, M, K) || !nvfp4_ok(b, N, K)) return AVERIS_ERR_INVALID_ARG;
  const bool bf16 = (flags & AVERIS_OUT_BF16) != 0;
  const int64_t esz = bf16 ? 2 : 4;
  if (ldo < N || (ldo * esz) % 16 != 0 || !aligned(out, 16)) return AVERIS_ERR_INVALID_ARG;
  if ((row_vec == nullptr) != (col_vec == nullptr)) return AVERIS_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  averis_status st = device_info(&dev);
  if (st != AVERIS_OK) return st;

  using Cfg = GemmCfg;
  constexpr int BN = Cfg::BN;
  const int64_t ld = averis_nvfp4_ld(K);
  CUtensorMap ta, tb, td;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->codes, (uint64_t)ld, (uint64_t)M, (uint64_t)ld, Cfg::BKB,
                 Cfg::BM))
    return AVERIS_ERR_CUDA;
  if (!encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b->codes, (uint64_t)ld, (uint64_t)N, (uint64_t)ld, Cfg::BKB,
                 BN))
    return AVERIS_ERR_CUDA;
  if (!encode_2d(&td, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, (uint64_t)N,
                 (uint64_t)M, (uint64_t)(ldo * esz), bf16 ? 64u : 32u, 32u))
    return AVERIS_ERR_CUDA;

  GemmParams p{};
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.kc = (int)cdiv(K, 64);
  p.rb_b = (int)cdiv(N, 128);
  p.sfa = a->scales;
  p.sfb = b->scales;
  p.ts_a = a->tensor_scale;
  p.ts_b = b->tensor_scale;
  p.col_add = col_add;
  p.row_vec = row_vec;
  p.col_vec = col_vec;
  p.outer = outer;
  p.err = dev->err_word;
  p.early_start = early_start ? 1 : 0;
  const int64_t ntiles = cdiv(M, Cfg::BM) * cdiv(N, BN);
  const int grid = (int)std::min<int64_t>(ntiles, dev->sms);
  cudaError_t e = bf16 ? launch_pdl(gemm_nvfp4_kernel<true>, dim3(grid), dim3(kGemmThreads), Cfg::SMEM, s, ta, tb, td, p)
                       : launch_pdl(gemm_nvfp4_kernel<false>, dim3(grid), dim3(kGemmThreads), Cfg::SMEM, s, ta, tb, td, p);
  return e == cudaSuccess ? AVERIS_OK : AVERIS_ERR_CUDA;
}

averis_status rank1_impl(const averis_nvfp4* mu_q, const averis_nvfp4* w, float* out, cudaStream_t s) {
  if (w == nullptr || mu_q == nullptr || out == nullptr || !aligned(out, 4)) return AVERIS_ERR_INVALID_ARG;
  const int64_t N = w->rows, K = w->cols;
  if (N < 1 || K < 16 || K % 16 != 0) return AVERIS_ERR_INVALID_ARG;
  if (!nvfp4_ok(w, N, K) || !nvfp4_ok(mu_q, 1, K)) return AVERIS_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  averis_status st = device_info(&dev);
  if (st != AVERIS_OK) return st;
  if (launch_pdl(rank1_gemv_kernel, dim3((unsigned)cdiv(N, 8)), dim3(256), 0, s, (const uint8_t*)mu_q->codes,
                 (const uint8_t*)mu_q->scales, (const float*)mu_q->tensor_scale, (const uint8_t*)w->codes,
                 (const uint8_t*)w->scales, (const float*)w->tensor_scale, averis_nvfp4_ld(K), N, K, cdiv(K, 64),
                 out) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  return AVERIS_OK;
}

// --------------------------------------------------------------- layers --

struct Carver {
  uint8_t* p;
  size_t used = 0;
  explicit Carver(void* base) : p(static_cast<uint8_t*>(base)) {}
  void* take(size_t bytes) {
    void* r = p + used;
    used += align256(bytes);
    return r;
  }
};

size_t nvfp4_bytes(int64_t rows, int64_t cols) {
  return align256(averis_nvfp4_code_bytes(rows, cols)) + align256(averis_nvfp4_scale_bytes(rows, cols)) + 256;
}

averis_nvfp4 carve_nvfp4(Carver& c, int64_t rows, int64_t cols) {
  averis_nvfp4 t;
  t.codes = static_cast<uint8_t*>(c.take(averis_nvfp4_code_bytes(rows, cols)));
  t.scales = static_cast<uint8_t*>(c.take(averis_nvfp4_scale_bytes(rows, cols)));
  t.tensor_scale = static_cast<float*>(c.take(sizeof(float)));
  t.rows = rows;
  t.cols = cols;
  return t;
}

size_t fwd_ws(int64_t l, int64_t m, int64_t n) { return quant_ws_bytes(l, m) + align256((size_t)n * 4); }

size_t bwd_ws(int64_t l, int64_t m, int64_t n) {
  return quant_ws_bytes(l, n) + nvfp4_bytes(l, n) + nvfp4_bytes(n, l) + nvfp4_bytes(1, n) +
         2 * align256((size_t)n * 4) + align256((size_t)m * 4);
}

averis_status linear_fwd_impl(const void* x, int64_t l, int64_t m, int64_t n, const averis_nvfp4* w_m, unsigned flags,
                              void* y, const averis_fwd_state* st, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (st == nullptr || w_m == nullptr || y == nullptr) return AVERIS_ERR_INVALID_ARG;
  if (l < 1 || m < 16 || n < 16 || m % 16 || n % 16) return AVERIS_ERR_INVALID_ARG;
  if (!nvfp4_ok(w_m, n, m)) return AVERIS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256)) return AVERIS_ERR_INVALID_ARG;
  if (ws_bytes < fwd_ws(l, m, n)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  Carver c(ws);
  void* qws = c.take(quant_ws_bytes(l, m));
  float* r_x = static_cast<float*>(c.take((size_t)n * 4));
  averis_status r = quantize_impl(x, l, m, flags, st->mu, &st->mu_q, st->mu_hat, &st->x_row, &st->x_col, qws,
                                  quant_ws_bytes(l, m), s, split ? w_m : nullptr, split ? r_x : nullptr);
  if (r != AVERIS_OK) return r;
  return gemm_impl(&st->x_row, w_m, split ? r_x : nullptr, nullptr, nullptr, 0.f, y, n, flags, s);
}

averis_status linear_bwd_impl(const void* d, int64_t l, int64_t m, int64_t n, const averis_fwd_state* st,
                              const averis_nvfp4* w_n, unsigned flags, void* dx, float* dw, void* ws,
                              size_t ws_bytes, cudaStream_t s) {
  if (st == nullptr || w_n == nullptr || dx == nullptr || dw == nullptr) return AVERIS_ERR_INVALID_ARG;
  if (l < 1 || m < 16 || n < 16 || m % 16 || n % 16) return AVERIS_ERR_INVALID_ARG;
  if (!nvfp4_ok(w_n, m, n) || !nvfp4_ok(&st->x_col, m, l)) return AVERIS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256)) return AVERIS_ERR_INVALID_ARG;
  if (ws_bytes < bwd_ws(l, m, n)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  if (split && (st->mu_hat == nullptr)) return AVERIS_ERR_INVALID_ARG;
  Carver c(ws);
  void* qws = c.take(quant_ws_bytes(l, n));
  averis_nvfp4 d_row = carve_nvfp4(c, l, n);
  averis_nvfp4 d_col = carve_nvfp4(c, n, l);
  averis_nvfp4 mu_q = carve_nvfp4(c, 1, n);
  float* mu = static_cast<float*>(c.take((size_t)n * 4));
  float* mu_hat = static_cast<float*>(c.take((size_t)n * 4));
  float* r_d = static_cast<float*>(c.take((size_t)m * 4));
  averis_status r = quantize_impl(d, l, n, flags, mu, &mu_q, mu_hat, &d_row, &d_col, qws, quant_ws_bytes(l, n), s,
                                  split ? w_n : nullptr, split ? r_d : nullptr);
  if (r != AVERIS_OK) return r;
  if ((r = gemm_impl(&d_row, w_n, split ? r_d : nullptr, nullptr, nullptr, 0.f, dx, m, flags, s)) != AVERIS_OK)
    return r;
  // dW reads the forward state and D's quantized column layout, not dX: it
  // starts while the input-gradient GEMM drains
  return gemm_impl(&st->x_col, &d_col, nullptr, split ? st->mu_hat : nullptr, split ? mu_hat : nullptr, (float)l, dw,
                   n, flags & ~AVERIS_OUT_BF16, s, /*early_start=*/true);
}

// Zeroes the control block of the allocation-free call's scratch on this
// device (if that call was ever made here), ordered after `stream`.
averis_status noalloc_reset_ctrl(cudaStream_t stream);

}  // namespace

// ================================================================ C ABI ==

extern "C" {

int64_t averis_nvfp4_ld(int64_t cols) { return cdiv(cols, 64) * 32; }

size_t averis_nvfp4_code_bytes(int64_t rows, int64_t cols) {
  return (size_t)rows * (size_t)averis_nvfp4_ld(cols);
}

size_t averis_nvfp4_scale_bytes(int64_t rows, int64_t cols) {
  return (size_t)512 * (size_t)cdiv(rows, 128) * (size_t)cdiv(cols, 64);
}

size_t averis_quantize_workspace_bytes(int64_t rows, int64_t cols, unsigned flags) {
  (void)flags;
  if (rows < 1 || cols < 1) return 0;
  return quant_ws_bytes(rows, cols);
}

averis_status averis_quantize(const void* x, int64_t rows, int64_t cols, unsigned flags, float* mu,
                              const averis_nvfp4* mu_q, float* mu_hat, const averis_nvfp4* out_row,
                              const averis_nvfp4* out_col, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  return quantize_impl(x, rows, cols, flags, mu, mu_q, mu_hat, out_row, out_col, workspace, workspace_bytes, stream);
}

averis_status averis_quantize_weight(const void* w, int64_t m, int64_t n, unsigned flags, const averis_nvfp4* w_n,
                                     const averis_nvfp4* w_m, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  if (w_n == nullptr && w_m == nullptr) return AVERIS_ERR_INVALID_ARG;
  return quantize_impl(w, m, n, flags & AVERIS_HADAMARD16, nullptr, nullptr, nullptr, w_n, w_m, workspace,
                       workspace_bytes, stream);
}

averis_status averis_rank1(const averis_nvfp4* mu_q, const averis_nvfp4* w, float* out, cudaStream_t stream) {
  return rank1_impl(mu_q, w, out, stream);
}

averis_status averis_gemm(const averis_nvfp4* a, const averis_nvfp4* b, const float* col_add, const float* row_vec,
                          const float* col_vec, float outer_scale, void* out, int64_t ldo, unsigned flags,
                          cudaStream_t stream) {
  return gemm_impl(a, b, col_add, row_vec, col_vec, outer_scale, out, ldo, flags, stream);
}

size_t averis_linear_fwd_workspace_bytes(int64_t l, int64_t m, int64_t n, unsigned flags) {
  (void)flags;
  if (l < 1 || m < 1 || n < 1) return 0;
  return fwd_ws(l, m, n);
}

size_t averis_linear_bwd_workspace_bytes(int64_t l, int64_t m, int64_t n, unsigned flags) {
  (void)flags;
  if (l < 1 || m < 1 || n < 1) return 0;
  return bwd_ws(l, m, n);
}

averis_status averis_linear_fwd(const void* x, int64_t l, int64_t m, int64_t n, const averis_nvfp4* w_m,
                                unsigned flags, void* y, const averis_fwd_state* state, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  if (!(flags & AVERIS_MEAN_SPLIT)) return AVERIS_ERR_INVALID_ARG;
  return linear_fwd_impl(x, l, m, n, w_m, flags, y, state, workspace, workspace_bytes, stream);
}

averis_status averis_linear_bwd(const void* d, int64_t l, int64_t m, int64_t n, const averis_fwd_state* state,
                                const averis_nvfp4* w_n, unsigned flags, void* dx, float* dw, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  if (!(flags & AVERIS_MEAN_SPLIT)) return AVERIS_ERR_INVALID_ARG;
  return linear_bwd_impl(d, l, m, n, state, w_n, flags, dx, dw, workspace, workspace_bytes, stream);
}

averis_status nvfp4_linear_fwd(const void* x, int64_t l, int64_t m, int64_t n, const averis_nvfp4* w_m,
                               unsigned flags, void* y, const averis_fwd_state* state, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  return linear_fwd_impl(x, l, m, n, w_m, flags & ~AVERIS_MEAN_SPLIT, y, state, workspace, workspace_bytes, stream);
}

averis_status nvfp4_linear_bwd(const void* d, int64_t l, int64_t m, int64_t n, const averis_fwd_state* state,
                               const averis_nvfp4* w_n, unsigned flags, void* dx, float* dw, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  return linear_bwd_impl(d, l, m, n, state, w_n, flags & ~AVERIS_MEAN_SPLIT, dx, dw, workspace, workspace_bytes,
                         stream);
}

// ------------------------------------------------------- grouped (MoE) --

static bool offsets_ok(const int64_t* offsets, int64_t num_experts) {
  if (offsets == nullptr || num_experts < 1 || offsets[0] != 0) return false;
  for (int64_t e = 0; e < num_experts; ++e)
    if (offsets[e + 1] < offsets[e]) return false;
  return true;
}

size_t averis_grouped_linear_fwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m, int64_t n,
                                                 unsigned flags) {
  (void)flags;
  if (!offsets_ok(offsets, num_experts) || m < 1 || n < 1) return 0;
  size_t b = 0;
  for (int64_t e = 0; e < num_experts; ++e) {
    const int64_t le = offsets[e + 1] - offsets[e];
    if (le > 0) b = std::max(b, fwd_ws(le, m, n));
  }
  return std::max<size_t>(b, 256);
}

size_t averis_grouped_linear_bwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m, int64_t n,
                                                 unsigned flags) {
  (void)flags;
  if (!offsets_ok(offsets, num_experts) || m < 1 || n < 1) return 0;
  size_t b = 0;
  for (int64_t e = 0; e < num_experts; ++e) {
    const int64_t le = offsets[e + 1] - offsets[e];
    if (le > 0) b = std::max(b, bwd_ws(le, m, n));
  }
  return std::max<size_t>(b, 256);
}

averis_status averis_grouped_linear_fwd(const void* x, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_nvfp4* w_m, unsigned flags, void* y,
                                        const averis_fwd_state* states, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  if (x == nullptr || y == nullptr || w_m == nullptr || states == nullptr) return AVERIS_ERR_INVALID_ARG;
  if (!offsets_ok(offsets, num_experts)) return AVERIS_ERR_INVALID_ARG;
  const int64_t esz = (flags & AVERIS_OUT_BF16) ? 2 : 4;
  for (int64_t e = 0; e < num_experts; ++e) {
    const int64_t r0 = offsets[e], le = offsets[e + 1] - offsets[e];
    if (le == 0) continue;
    const averis_status st = linear_fwd_impl(static_cast<const uint8_t*>(x) + r0 * m * 2, le, m, n, &w_m[e], flags,
                                             static_cast<uint8_t*>(y) + r0 * n * esz, &states[e], workspace,
                                             workspace_bytes, stream);
    if (st != AVERIS_OK) return st;
  }
  return AVERIS_OK;
}

averis_status averis_grouped_linear_bwd(const void* d, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_fwd_state* states, const averis_nvfp4* w_n,
                                        unsigned flags, void* dx, float* const* dw, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  if (d == nullptr || dx == nullptr || dw == nullptr || w_n == nullptr || states == nullptr)
    return AVERIS_ERR_INVALID_ARG;
  if (!offsets_ok(offsets, num_experts)) return AVERIS_ERR_INVALID_ARG;
  const int64_t esz = (flags & AVERIS_OUT_BF16) ? 2 : 4;
  for (int64_t e = 0; e < num_experts; ++e) {
    const int64_t r0 = offsets[e], le = offsets[e + 1] - offsets[e];
    if (le == 0) continue;
    const averis_status st = linear_bwd_impl(static_cast<const uint8_t*>(d) + r0 * n * 2, le, m, n, &states[e],
                                             &w_n[e], flags, static_cast<uint8_t*>(dx) + r0 * m * esz, dw[e],
                                             workspace, workspace_bytes, stream);
    if (st != AVERIS_OK) return st;
  }
  return AVERIS_OK;
}

const char* averis_status_string(averis_status status) {
  switch (status) {
    case AVERIS_OK: return "ok";
    case AVERIS_ERR_INVALID_ARG: return "invalid argument";
    case AVERIS_ERR_UNSUPPORTED_ARCH: return "unsupported architecture (needs sm_103)";
    case AVERIS_ERR_CUDA: return "CUDA error";
    case AVERIS_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case AVERIS_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

averis_status averis_last_device_error(cudaStream_t stream, int* where) {
  DeviceInfo* dev = nullptr;
  averis_status st = device_info(&dev);
  if (st != AVERIS_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return AVERIS_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return AVERIS_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return AVERIS_ERR_CUDA;
    // the kernels leave a control block zero even when a wait gives up; the
    // library-owned one of the allocation-free call is cleared here as well,
    // since its callers have no way to do it themselves
    if (noalloc_reset_ctrl(stream) != AVERIS_OK) return AVERIS_ERR_CUDA;
  }
  if (where != nullptr) *where = v;
  return v == 0 ? AVERIS_OK : AVERIS_ERR_TIMEOUT;
}

averis_status averis_debug_starve_next_quantize(long long wait_cycles) {
  if (wait_cycles < 10000 || wait_cycles > kWaitLimit) return AVERIS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_starve_next = wait_cycles;
  return AVERIS_OK;
}

int averis_version(void) { return 100; }

}  // extern "C"

// ===================================================== allocation-free call ==

// Scratch of averis_quantize_noalloc: one array per device, alive until the
// process exits.  Host code must not pass &g_noalloc_scratch to a kernel (it
// names a host-side shadow); the device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[AVERIS_NOALLOC_SCRATCH_BYTES];

namespace {

void* g_noalloc_addr[kMaxDevices] = {};

averis_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AVERIS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AVERIS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return AVERIS_ERR_CUDA;
    g_noalloc_addr[dev] = addr;
  }
  *out = g_noalloc_addr[dev];
  return AVERIS_OK;
}

averis_status noalloc_reset_ctrl(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return AVERIS_ERR_CUDA;
  void* addr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    addr = g_noalloc_addr[dev];
  }
  if (addr == nullptr) return AVERIS_OK;
  if (cudaMemsetAsync(addr, 0, AVERIS_WORKSPACE_CTRL_BYTES, stream) != cudaSuccess) return AVERIS_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? AVERIS_OK : AVERIS_ERR_CUDA;
}

}  // namespace

extern "C" averis_status averis_quantize_noalloc(const void* x, int64_t rows, int64_t cols, unsigned flags,
                                                 float* mu, const averis_nvfp4* mu_q, float* mu_hat,
                                                 const averis_nvfp4* out_row, const averis_nvfp4* out_col,
                                                 cudaStream_t stream) {
  if (rows < 1 || cols < 1) return AVERIS_ERR_INVALID_ARG;
  if (quant_ws_bytes(rows, cols) > AVERIS_NOALLOC_SCRATCH_BYTES) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  averis_status st = noalloc_scratch(&scratch);
  if (st != AVERIS_OK) return st;
  return quantize_impl(x, rows, cols, flags, mu, mu_q, mu_hat, out_row, out_col, scratch,
                       AVERIS_NOALLOC_SCRATCH_BYTES, stream);
}
