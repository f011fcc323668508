// C ABI of libaveris.so: argument checks, workspace carving, tensor-map
// encoding and kernel launches.  Declarations and per-call contracts are in
// include/averis.h.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "averis.h"
#include "gemm.cuh"
#include "quant.cuh"

namespace {

using namespace averis;

constexpr int kMaxDevices = 64;
#ifndef AVERIS_GEMM_SFB_FULL
#define AVERIS_GEMM_SFB_FULL 1
#endif
constexpr bool kSfbFull = AVERIS_GEMM_SFB_FULL != 0;
constexpr int kStatsTargetCtas = 296;  // CTA count target of the stats pass (one wave at 2 per SM of a B300)

__device__ int g_device_error = 0;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* err_word = nullptr;
  bool attrs_set = false;
  int gemm_pairs = 0;  // clusters of two GEMM CTAs resident at once (the persistent grid's size)
  int resident_ctas = 0;  // CTAs of the single-read quantize resident at once (its cooperative grid)
  bool resident_on = false;  // AVERIS_SINGLE_READ_QUANTIZE=1 turns the single-read quantize on
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
    // a persistent grid larger than the clusters that can be resident together
    // would leave its last pairs to run after the others: size it to that count
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (d.sms / 2));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = GemmCfg<kSfbFull>::SMEM;
    int pairs = 0;
    if (cudaOccupancyMaxActiveClusters(&pairs, gemm_nvfp4_kernel<kSfbFull, 1>, &cfg) != cudaSuccess || pairs < 1)
      return AVERIS_ERR_CUDA;
    d.gemm_pairs = std::min(std::min(pairs, d.sms / 2), kMaxPairs);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_resident_kernel, kQThreads, kQSmem) !=
        cudaSuccess)
      return AVERIS_ERR_CUDA;
    d.resident_ctas = std::min(per_sm, kQCtasPerSm) * d.sms;
    const char* env = std::getenv("AVERIS_SINGLE_READ_QUANTIZE");
    d.resident_on = env != nullptr && env[0] == '1';
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
  if (cudaFuncSetAttribute(quantize_resident_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(colstats_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStatsSmem) !=
      cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_grouped_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kQSmem) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_grouped_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kQSmem) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(split_quant_grouped_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kQSmem) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_nvfp4_kernel<kSfbFull, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemmCfg<kSfbFull>::SMEM) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_nvfp4_kernel<kSfbFull, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemmCfg<kSfbFull>::SMEM) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_nvfp4_kernel<kSfbFull, kMaxGemmGroups>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemmCfg<kSfbFull>::SMEM) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  return AVERIS_OK;
}

#ifdef AVERIS_DEBUG
// The bounds predicate on fixed (offset, extent, bytes) cases -- addresses
// built from a fake base, never dereferenced -- and one recorded site.
__device__ int g_dbg_selftest[8];

__global__ void debug_self_test_kernel(int* err) {
  const char* base = reinterpret_cast<const char*>(0x10000);
  g_dbg_selftest[0] = dbg_inside(base, base, 64, 64);       // whole buffer: in
  g_dbg_selftest[1] = dbg_inside(base + 48, base, 64, 16);  // last 16 bytes: in
  g_dbg_selftest[2] = dbg_inside(base + 56, base, 64, 16);  // crosses the end: out
  g_dbg_selftest[3] = dbg_inside(base - 4, base, 64, 4);    // before the start: out
  g_dbg_selftest[4] = dbg_inside(base + 64, base, 64, 1);   // one past the end: out
  g_dbg_selftest[5] = dbg_inside(base, nullptr, 64, 4);     // no buffer: out
  g_dbg_selftest[6] = dbg_in(err, base + 64, base, 64, 4, kSiteSelfTest);  // out, recorded
  g_dbg_selftest[7] = 1;
}

// 1: predicate and recorder work; -1: they do not, an error was pending, or CUDA failed.
int debug_self_test() {
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != AVERIS_OK) return -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess || v != 0) return -1;
  debug_self_test_kernel<<<1, 1>>>(dev->err_word);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return -1;
  int got[8] = {};
  if (cudaMemcpyFromSymbol(got, g_dbg_selftest, sizeof(got)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return -1;
  const int want[8] = {1, 1, 0, 0, 0, 0, 0, 1};
  for (int i = 0; i < 8; ++i)
    if (got[i] != want[i]) return -1;
  return v == kErrBoundsBase + kSiteSelfTest ? 1 : -1;
}
#endif

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

// The single-read quantize keeps every 128 x 128 tile of X in shared memory
// (kQBufs per CTA, kQCtasPerSm CTAs per SM): tensors of at most this many
// tiles may take it (888 on a 148-SM part), and their workspace holds one
// row of column partials per tile row (at most 2 KB per tile).
constexpr int64_t kResidentMaxTiles = 1024;

bool resident_size(int64_t R, int64_t C) { return cdiv(R, kQTile) * cdiv(C, kQTile) <= kResidentMaxTiles; }

size_t quant_ws_bytes(int64_t R, int64_t C) {
  const StatsGeom g = stats_geom(R, C);
  const int64_t rows = resident_size(R, C) ? std::max<int64_t>(g.nrb, cdiv(R, kQTile)) : g.nrb;
  return kCtrlBytes + align256((size_t)rows * (size_t)C * sizeof(ColPartial));
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

// The same with a cooperative launch: every CTA of the grid is resident at
// once (the single-read quantize waits grid-wide, bounded).
template <typename... KArgs, typename... Args>
cudaError_t launch_coop_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
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
  // opt-in: a tensor whose tiles all fit the resident CTAs' buffers (and no
  // rotation, which needs the rotated maxima before any tile is quantized) in
  // one cooperative launch that reads X once.  Measured on a B300 at 8192 x
  // 1024 it takes as long as the two launches (20.1 against 20.4 us in a CUDA
  // graph): the pass is bound by its arithmetic and fixed latencies, not by the
  // second read of X (from L2), and its two grid-wide waits cost what the
  // saved launch gains

  const int64_t tile_slots = (int64_t)(dev->resident_ctas - qp.mean_ctas) * kQBufs;
  if (dev->resident_on && !had && ntiles > 0 && ntiles <= kResidentMaxTiles && ntiles <= tile_slots &&
      ws_bytes >= kCtrlBytes + (size_t)qp.tiles_r * (size_t)C * sizeof(ColPartial)) {
    ResidentParams rp{};
    rp.q = qp;
    rp.mu = split ? mu : nullptr;
    rp.part = part;
    rp.grid_wait_limit = kWaitLimit;
    if (sp.starve) {
      rp.starve = 1;
      rp.q.wait_limit = sp.wait_limit;
    }
    if (launch_coop_pdl(quantize_resident_kernel, dim3(dev->resident_ctas), dim3(kQThreads), kQSmem, s, tx, rp) !=
        cudaSuccess)
      return AVERIS_ERR_CUDA;
    return AVERIS_OK;
  }
  // with the rotation and no mean split the column statistics would give only
  // the unrotated maximum, which no layout uses (both take the rotated maxima):
  // the pass runs only when it is needed (or asked to starve)
  if ((split || !had || sp.starve) &&
      launch_pdl(colstats_kernel, dim3(g.gx, g.nrb), dim3(256), kStatsSmem, s, tstats, sp) != cudaSuccess)
    return AVERIS_ERR_CUDA;
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

// ------------------------------------------------------ grouped quantize --

// One row group (expert) of a grouped quantize: rows row0 .. row0+rows-1 of
// the grouped input, its own outputs (as in quantize_impl) and optionally its
// own rank-one row r_out = deq(mu_q) deq(r_w)^T.
struct GroupSpec {
  int64_t row0 = 0, rows = 0;
  float* mu = nullptr;
  const averis_nvfp4* mu_q = nullptr;
  float* mu_hat = nullptr;
  const averis_nvfp4* out_row = nullptr;
  const averis_nvfp4* out_col = nullptr;
  const averis_nvfp4* r_w = nullptr;
  float* r_out = nullptr;
};

// Stats geometry shared by the groups of one grouped call: the same strip
// groups, one row-block height, about four waves of CTAs over all rows.
struct GroupedGeom {
  int gx, nstrips;
  int64_t rows_per;
};
GroupedGeom grouped_geom(int64_t L, int64_t C, int ngroups) {
  GroupedGeom g;
  g.nstrips = (int)cdiv(C, 64);
  g.gx = std::min(g.nstrips, (int)kMaxStripGroups);
  const int64_t target = std::max<int64_t>(ngroups, cdiv(4 * kStatsTargetCtas, g.gx));
  g.rows_per = std::max<int64_t>(256, cdiv(cdiv(L, target), 32) * 32);
  return g;
}
// Control words of the groups of one launch (strip tickets and maxima, zero at
// rest): a fixed region at the head of every grouped workspace, the same for
// every shape, so that a workspace can serve grouped calls of any shape (every
// word of the region is zero between calls); then the groups' row-block partials.
constexpr size_t kGroupCtrlWords = kCtrlStrip + kMaxStripGroups;
static_assert(kMaxGroups * kGroupCtrlWords * sizeof(unsigned) == AVERIS_GROUPED_WORKSPACE_CTRL_BYTES,
              "grouped control region is part of the ABI");
size_t group_part_bytes(const GroupedGeom& g, int64_t rows, int64_t C) {
  return align256((size_t)cdiv(rows, g.rows_per) * (size_t)C * sizeof(ColPartial));
}
size_t grouped_quant_ws_bytes(const int64_t* rows, int ng, int64_t C) {
  int64_t L = 0;
  for (int e = 0; e < ng; ++e) L += rows[e];
  const GroupedGeom g = grouped_geom(L, C, std::min(ng, kMaxGroups));
  size_t b = AVERIS_GROUPED_WORKSPACE_CTRL_BYTES;
  for (int e = 0; e < ng; ++e)
    if (rows[e] > 0) b += group_part_bytes(g, rows[e], C);
  return b;
}

// The quantize pass of up to kMaxGroups groups of one grouped input x
// [L, C]: one stats launch and one quantize launch (two with the rotation)
// for all of them.  Groups with no rows are skipped.  ctrl: the control
// region (zero at rest); ws: the groups' partials, in group order.
averis_status grouped_quantize_chunk(const void* x, int64_t L, int64_t C, unsigned flags, const GroupSpec* gs, int ng,
                                     const GroupedGeom& geo, unsigned* ctrl_region, uint8_t* ws, DeviceInfo* dev,
                                     cudaStream_t s) {
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  const bool had = (flags & AVERIS_HADAMARD16) != 0;
  GroupedStatsParams sp{};
  GroupedQuantParams qp{};
  GroupedQuantParams ap{};  // rotated-maximum pass: tiles only
  int n = 0, rbs = 0, ctas = 0, mctas = 0, actas = 0;
  int64_t tiles_all = 0;
  for (int e = 0; e < ng; ++e)
    if (gs[e].rows > 0) tiles_all += cdiv(gs[e].rows, kQTile) * cdiv(C, kQTile);
  const int64_t budget = kQCtasPerSm * (int64_t)dev->sms;  // tile CTAs of one wave, shared out by tiles
  // rank-one work of all groups: the mean CTAs of a launch (launched ahead of
  // every tile CTA) take at most one wave, shared out by the groups' weight
  // rows (one each at least, about 128 K weights each at most), so that the
  // mean phase is short and the tile CTAs start together when it ends
  int64_t w_rows_all = 0;
  for (int e = 0; e < ng; ++e)
    if (gs[e].rows > 0 && gs[e].r_w != nullptr) w_rows_all += gs[e].r_w->rows;
  long long starve = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    std::swap(starve, g_starve_next);
  }
  for (int e = 0; e < ng; ++e) {
    const GroupSpec& G = gs[e];
    if (G.rows <= 0) continue;
    unsigned* ctrl = ctrl_region + (size_t)n * kGroupCtrlWords;
    ColPartial* part = reinterpret_cast<ColPartial*>(ws);
    ws += group_part_bytes(geo, G.rows, C);
    const int nrb = (int)cdiv(G.rows, geo.rows_per);
    StatsParams& st = sp.g[n];
    st.x = static_cast<const __nv_bfloat16*>(x);
    st.R = G.rows;
    st.C = C;
    st.rows_per = cdiv(cdiv(G.rows, nrb), 32) * 32;
    st.nstrips = geo.nstrips;
    st.part = part;
    st.ctrl = ctrl;
    st.err = dev->err_word;
    st.split = split ? 1 : 0;
    st.hadamard = had ? 1 : 0;
    st.mu = G.mu;
    st.wait_limit = starve > 0 ? starve : kWaitLimit;
    st.starve = starve > 0 ? 1 : 0;
    st.row_base = G.row0;
    sp.rb0[n] = rbs;
    rbs += (int)cdiv(G.rows, st.rows_per);

    QuantParams& q = qp.g[n];
    q.R = G.rows;
    q.C = C;
    q.mu = split ? G.mu : nullptr;
    if (split) {
      q.mu_codes = G.mu_q->codes;
      q.mu_scales = G.mu_q->scales;
      q.mu_ts = G.mu_q->tensor_scale;
      q.mu_hat = G.mu_hat;
      q.mu_kc = cdiv(C, 64);
    }
    q.ctrl = ctrl;
    q.err = dev->err_word;
    q.wait_limit = kWaitLimit;
    q.hadamard = had ? 1 : 0;
    if (G.out_row != nullptr) {
      q.row_codes = G.out_row->codes;
      q.row_scales = G.out_row->scales;
      q.row_ts = G.out_row->tensor_scale;
      q.row_ld = averis_nvfp4_ld(C);
      q.row_kc = cdiv(C, 64);
    }
    if (G.out_col != nullptr) {
      q.col_codes = G.out_col->codes;
      q.col_scales = G.out_col->scales;
      q.col_ts = G.out_col->tensor_scale;
      q.col_ld = averis_nvfp4_ld(G.rows);
      q.col_kc = cdiv(G.rows, 64);
    }
    q.tiles_r = (int)cdiv(G.rows, kQTile);
    q.tiles_c = (int)cdiv(C, kQTile);
    if (G.out_row == nullptr && G.out_col == nullptr) q.tiles_r = 0;
    q.row_base = G.row0;
    q.mean_ctas = 0;
    if (split) {
      q.mean_ctas = 1;
      if (G.r_w != nullptr) {
        q.w_codes = G.r_w->codes;
        q.w_scales = G.r_w->scales;
        q.w_ts = G.r_w->tensor_scale;
        q.w_rows = G.r_w->rows;
        q.w_ld = averis_nvfp4_ld(C);
        q.w_kc = cdiv(C, 64);
        q.r_out = G.r_out;
        q.mean_ctas = (int)std::max<int64_t>(
            1, std::min<int64_t>(std::min<int64_t>(16, cdiv(G.r_w->rows * C, (int64_t)1 << 17)),
                                 budget * G.r_w->rows / std::max<int64_t>(1, w_rows_all)));
      }
    }
    const int64_t tiles = (int64_t)q.tiles_r * q.tiles_c;
    const int tile_ctas =
        tiles == 0 ? 0 : (int)std::max<int64_t>(1, std::min<int64_t>(tiles, budget * tiles / std::max<int64_t>(1, tiles_all)));
    qp.cta0[n] = ctas;     // tile CTAs (at least one CTA per group: its last one resets its words)
    qp.mcta0[n] = mctas;   // mean CTAs
    ctas += q.mean_ctas + tile_ctas > 0 ? tile_ctas : 1;
    mctas += q.mean_ctas;
    ap.g[n] = q;
    ap.g[n].mean_ctas = 0;
    ap.cta0[n] = actas;
    actas += std::max(1, tile_ctas);
    ++n;
  }
  if (n == 0) return AVERIS_OK;
  sp.rb0[n] = rbs;
  sp.ngroups = n;
  qp.cta0[n] = ctas;
  qp.mcta0[n] = mctas;
  qp.ngroups = n;
  ap.cta0[n] = actas;
  ap.ngroups = n;

  CUtensorMap tstats, tx;
  if (!encode_2d(&tstats, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(x), (uint64_t)C, (uint64_t)L,
                 (uint64_t)C * 2, 64u, (uint32_t)kStatsBoxRows))
    return AVERIS_ERR_CUDA;
  if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(x), (uint64_t)C, (uint64_t)L,
                 (uint64_t)C * 2, 64u, (uint32_t)kQTile))
    return AVERIS_ERR_CUDA;
  // the statistics are unused with the rotation and no mean split (see quantize_impl)
  if ((split || !had || starve > 0) &&
      launch_pdl(colstats_grouped_kernel, dim3(geo.gx, rbs), dim3(256), kStatsSmem, s, tstats, sp) != cudaSuccess)
    return AVERIS_ERR_CUDA;
  if (had && launch_pdl(split_quant_grouped_kernel<true, true>, dim3(actas), dim3(kQThreads), kQSmem, s, tx, ap) !=
                 cudaSuccess)
    return AVERIS_ERR_CUDA;
  auto* qk = had ? split_quant_grouped_kernel<false, true> : split_quant_grouped_kernel<false, false>;
  if (launch_pdl(qk, dim3(mctas + ctas), dim3(kQThreads), kQSmem, s, tx, qp) != cudaSuccess) return AVERIS_ERR_CUDA;
  return AVERIS_OK;
}

// All groups of a grouped input, kMaxGroups at a time.  Checks every group's
// outputs; rows of the groups must tile [0, L) in order.
averis_status grouped_quantize_impl(const void* x, int64_t L, int64_t C, unsigned flags, const GroupSpec* gs, int ng,
                                    void* ws, size_t ws_bytes, cudaStream_t s) {
  if (x == nullptr || gs == nullptr || ng < 1 || L < 1 || C < 16 || C % 16 != 0 || !aligned(x, 16))
    return AVERIS_ERR_INVALID_ARG;
  if (L > (int64_t)1 << 31 || C > (int64_t)1 << 31) return AVERIS_ERR_INVALID_ARG;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  if (split && C > kMaxSplitCols) return AVERIS_ERR_INVALID_ARG;
  std::vector<int64_t> rows(ng);
  int64_t next = 0;
  for (int e = 0; e < ng; ++e) {
    const GroupSpec& G = gs[e];
    if (G.rows < 0 || G.row0 != next) return AVERIS_ERR_INVALID_ARG;
    next += G.rows;
    rows[e] = G.rows;
    if (G.rows == 0) continue;
    if (G.out_row != nullptr && !nvfp4_ok(G.out_row, G.rows, C)) return AVERIS_ERR_INVALID_ARG;
    if (G.out_col != nullptr && !nvfp4_ok(G.out_col, C, G.rows)) return AVERIS_ERR_INVALID_ARG;
    if (split && (G.mu == nullptr || G.mu_hat == nullptr || !aligned(G.mu, 16) || !aligned(G.mu_hat, 16) ||
                  !nvfp4_ok(G.mu_q, 1, C)))
      return AVERIS_ERR_INVALID_ARG;
    if ((G.r_w == nullptr) != (G.r_out == nullptr)) return AVERIS_ERR_INVALID_ARG;
    if (G.r_w != nullptr && (!split || G.r_w->rows < 1 || !nvfp4_ok(G.r_w, G.r_w->rows, C) || !aligned(G.r_out, 4)))
      return AVERIS_ERR_INVALID_ARG;
  }
  if (next != L) return AVERIS_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256)) return AVERIS_ERR_INVALID_ARG;
  if (ws_bytes < grouped_quant_ws_bytes(rows.data(), ng, C)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  averis_status st = device_info(&dev);
  if (st != AVERIS_OK) return st;
  const GroupedGeom geo = grouped_geom(L, C, std::min(ng, kMaxGroups));
  unsigned* ctrl = static_cast<unsigned*>(ws);  // reused by every chunk: each leaves it zero
  uint8_t* w = static_cast<uint8_t*>(ws) + AVERIS_GROUPED_WORKSPACE_CTRL_BYTES;
  for (int e0 = 0; e0 < ng; e0 += kMaxGroups) {
    const int cnt = std::min(kMaxGroups, ng - e0);
    if ((st = grouped_quantize_chunk(x, L, C, flags, gs + e0, cnt, geo, ctrl, w, dev, s)) != AVERIS_OK) return st;
    for (int e = e0; e < e0 + cnt; ++e)
      if (rows[e] > 0) w += group_part_bytes(geo, rows[e], C);
  }
  return AVERIS_OK;
}

// ----------------------------------------------------------------- GEMM --


// One GEMM of a launch: the operands and epilogue terms of averis_gemm.
struct GemmSpec {
  const averis_nvfp4* a = nullptr;
  const averis_nvfp4* b = nullptr;
  const float* col_add = nullptr;
  const float* row_vec = nullptr;
  const float* col_vec = nullptr;
  float outer = 0.f;
  void* out = nullptr;
  int64_t ldo = 0;
  bool bf16 = false;  // output in bf16 (else binary32)
};

// Argument checks of one GEMM (before anything touches the device).
averis_status gemm_check(const GemmSpec& g) {
  const bool bf16 = g.bf16;
  const averis_nvfp4* a = g.a;
  const averis_nvfp4* b = g.b;
  if (a == nullptr || b == nullptr || g.out == nullptr) return AVERIS_ERR_INVALID_ARG;
  const int64_t M = a->rows, N = b->rows, K = a->cols;
  // K may be ragged (the token axis of dW): codes and scales are zero-padded to 64
  if (M < 1 || N < 1 || K < 1 || b->cols != K) return AVERIS_ERR_INVALID_ARG;
  if (M > (int64_t)1 << 30 || N > (int64_t)1 << 30 || K > (int64_t)1 << 30) return AVERIS_ERR_INVALID_ARG;
  if (!nvfp4_ok(a, M, K) || !nvfp4_ok(b, N, K)) return AVERIS_ERR_INVALID_ARG;
  const int64_t esz = bf16 ? 2 : 4;
  if (g.ldo < N || (g.ldo * esz) % 16 != 0 || !aligned(g.out, 16)) return AVERIS_ERR_INVALID_ARG;
  if ((g.row_vec == nullptr) != (g.col_vec == nullptr)) return AVERIS_ERR_INVALID_ARG;
  return AVERIS_OK;
}

// Fills one checked GEMM's tensor maps and scalars.
averis_status gemm_fill(const GemmSpec& g, CUtensorMap* ta, CUtensorMap* tb, CUtensorMap* td, GemmGroup* gg) {
  const bool bf16 = g.bf16;
  const averis_nvfp4* a = g.a;
  const averis_nvfp4* b = g.b;
  const int64_t M = a->rows, N = b->rows, K = a->cols;
  const int64_t esz = bf16 ? 2 : 4;
  using Cfg = GemmCfg<kSfbFull>;
  const int64_t ld = averis_nvfp4_ld(K);
  if (!encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->codes, (uint64_t)ld, (uint64_t)M, (uint64_t)ld, Cfg::BKB,
                 Cfg::BM))
    return AVERIS_ERR_CUDA;
  if (!encode_2d(tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b->codes, (uint64_t)ld, (uint64_t)N, (uint64_t)ld, Cfg::BKB,
                 Cfg::BNH))
    return AVERIS_ERR_CUDA;
  if (!encode_2d(td, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.out, (uint64_t)N,
                 (uint64_t)M, (uint64_t)(g.ldo * esz), bf16 ? 64u : 32u, 32u))
    return AVERIS_ERR_CUDA;
  gg->sfa = a->scales;
  gg->sfb = b->scales;
  gg->ts_a = a->tensor_scale;
  gg->ts_b = b->tensor_scale;
  gg->col_add = g.col_add;
  gg->row_vec = g.row_vec;
  gg->col_vec = g.col_vec;
  gg->outer = g.outer;
  gg->M = (int)M;
  gg->N = (int)N;
  gg->kc = (int)cdiv(K, 64);
  gg->rb_a = (int)cdiv(M, 128);
  gg->rb_b = (int)cdiv(N, 128);
  gg->num_m = (int)cdiv(M, Cfg::PM);
  gg->bf16 = bf16 ? 1 : 0;
  return AVERIS_OK;
}

// Up to G GEMMs in one persistent launch of CTA pairs.  Each pair runs a
// contiguous range of work units (GEMM after GEMM, tile after tile); the ranges
// are cut so that every pair gets about the same cost, a unit costing its K
// tiles plus an allowance for its epilogue, so that a launch mixing long-K
// and short-K GEMMs (dW and dX of one layer, or the experts of a grouped
// layer) keeps every pair busy.
template <int G>
averis_status gemm_launch(const GemmSpec* specs, int n, cudaStream_t s) {
  if (n < 1 || n > G) return AVERIS_ERR_INVALID_ARG;
  averis_status st = AVERIS_OK;
  for (int e = 0; e < n; ++e)
    if ((st = gemm_check(specs[e])) != AVERIS_OK) return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != AVERIS_OK) return st;
  using Cfg = GemmCfg<kSfbFull>;
  static thread_local GemmArgs<G> args;  // about 31 KB for G = 64: kept off the stack
  std::memset(&args, 0, sizeof(args));
  int64_t units = 0;
  double total = 0.0;
  auto unit_cost = [](const GemmGroup& g) { return (double)(cdiv(g.kc, 4) + (g.bf16 ? 2 : 4)); };
  for (int e = 0; e < n; ++e) {
    if ((st = gemm_fill(specs[e], &args.tmA[e], &args.tmB[e], &args.tmD[e], &args.g[e])) != AVERIS_OK) return st;
    args.g[e].unit0 = (int)units;
    const int64_t t = (int64_t)args.g[e].num_m * cdiv(args.g[e].N, Cfg::BN);
    units += t;
    total += (double)t * unit_cost(args.g[e]);
    if (units > (int64_t)1 << 30) return AVERIS_ERR_INVALID_ARG;
  }
  args.ngroups = n;
  args.nunits = (int)units;
  args.err = dev->err_word;
  args.wait_limit = kWaitLimit;
  args.early_start = 0;
  const int pairs = (int)std::min<int64_t>(units, dev->gemm_pairs);
  // contiguous cost-balanced ranges: pair p ends at the first unit whose cost
  // prefix reaches (p + 1) / pairs of the total
  int p = 0, e = 0;
  double acc = 0.0;
  args.range0[0] = 0;
  for (int64_t u = 0; u < units && p < pairs - 1; ++u) {
    while (e + 1 < n && args.g[e + 1].unit0 <= u) ++e;
    acc += unit_cost(args.g[e]);
    if (acc >= total * (double)(p + 1) / (double)pairs) args.range0[++p] = (int)(u + 1);
  }
  while (p < pairs) args.range0[++p] = (int)units;
  const cudaError_t err =
      launch_pdl(gemm_nvfp4_kernel<kSfbFull, G>, dim3(2 * pairs), dim3(kGemmThreads), Cfg::SMEM, s, args);
  return err == cudaSuccess ? AVERIS_OK : AVERIS_ERR_CUDA;
}

averis_status gemm_impl(const averis_nvfp4* a, const averis_nvfp4* b, const float* col_add, const float* row_vec,
                        const float* col_vec, float outer, void* out, int64_t ldo, unsigned flags, cudaStream_t s) {
  GemmSpec g;
  g.a = a;
  g.b = b;
  g.col_add = col_add;
  g.row_vec = row_vec;
  g.col_vec = col_vec;
  g.outer = outer;
  g.out = out;
  g.ldo = ldo;
  g.bf16 = (flags & AVERIS_OUT_BF16) != 0;
  return gemm_launch<1>(&g, 1, s);
}

// Many GEMMs, kMaxGemmGroups per launch.
averis_status grouped_gemm_impl(const GemmSpec* specs, int n, cudaStream_t s) {
  for (int e0 = 0; e0 < n; e0 += kMaxGemmGroups) {
    const averis_status st = gemm_launch<kMaxGemmGroups>(specs + e0, std::min(kMaxGemmGroups, n - e0), s);
    if (st != AVERIS_OK) return st;
  }
  return AVERIS_OK;
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
                 out, dev->err_word) != cudaSuccess)
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
  // dW (long K: the tokens) and dX in one launch, the pairs' ranges balanced by cost
  GemmSpec g[2];
  g[0].a = &st->x_col;
  g[0].b = &d_col;
  g[0].row_vec = split ? st->mu_hat : nullptr;
  g[0].col_vec = split ? mu_hat : nullptr;
  g[0].outer = (float)l;
  g[0].out = dw;
  g[0].ldo = n;
  g[1].a = &d_row;
  g[1].b = w_n;
  g[1].col_add = split ? r_d : nullptr;
  g[1].out = dx;
  g[1].ldo = m;
  g[1].bf16 = (flags & AVERIS_OUT_BF16) != 0;
  return gemm_launch<2>(g, 2, s);
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

size_t averis_quantize_weight_grouped_workspace_bytes(int64_t num_experts, int64_t m, int64_t n) {
  if (num_experts < 1 || m < 1 || n < 1) return 0;
  const std::vector<int64_t> rows((size_t)num_experts, m);
  return grouped_quant_ws_bytes(rows.data(), (int)num_experts, n);
}

averis_status averis_quantize_weight_grouped(const void* w, int64_t num_experts, int64_t m, int64_t n,
                                             unsigned flags, const averis_nvfp4* w_n, const averis_nvfp4* w_m,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (num_experts < 1 || num_experts > (int64_t)1 << 20 || m < 1 || (w_n == nullptr && w_m == nullptr))
    return AVERIS_ERR_INVALID_ARG;
  if (m > ((int64_t)1 << 31) / num_experts) return AVERIS_ERR_INVALID_ARG;
  // the experts are the row groups of one [num_experts * m, n] input
  std::vector<GroupSpec> gs((size_t)num_experts);
  for (int64_t e = 0; e < num_experts; ++e) {
    GroupSpec& G = gs[(size_t)e];
    G.row0 = e * m;
    G.rows = m;
    G.out_row = w_n != nullptr ? &w_n[e] : nullptr;
    G.out_col = w_m != nullptr ? &w_m[e] : nullptr;
  }
  return grouped_quantize_impl(w, num_experts * m, n, flags & AVERIS_HADAMARD16, gs.data(), (int)num_experts,
                               workspace, workspace_bytes, stream);
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
  if (offsets == nullptr || num_experts < 1 || num_experts > (1 << 20) || offsets[0] != 0) return false;
  for (int64_t e = 0; e < num_experts; ++e)
    if (offsets[e + 1] < offsets[e]) return false;
  return true;
}

static std::vector<int64_t> group_rows(const int64_t* offsets, int64_t num_experts) {
  std::vector<int64_t> r((size_t)num_experts);
  for (int64_t e = 0; e < num_experts; ++e) r[(size_t)e] = offsets[e + 1] - offsets[e];
  return r;
}

// Forward workspace: the grouped quantize's control words and partials, then
// one rank-one row [n] per expert.
static size_t grouped_fwd_ws(const int64_t* offsets, int64_t E, int64_t m, int64_t n) {
  const std::vector<int64_t> rows = group_rows(offsets, E);
  return align256(grouped_quant_ws_bytes(rows.data(), (int)E, m)) + (size_t)E * align256((size_t)n * 4);
}

// Backward workspace: the grouped quantize's, then per expert with rows its
// quantized D (both layouts), mean, NVFP4 mean, dequantized mean and rank-one row [m].
static size_t grouped_bwd_ws(const int64_t* offsets, int64_t E, int64_t m, int64_t n) {
  const std::vector<int64_t> rows = group_rows(offsets, E);
  size_t b = align256(grouped_quant_ws_bytes(rows.data(), (int)E, n));
  for (int64_t e = 0; e < E; ++e) {
    const int64_t le = rows[(size_t)e];
    if (le > 0)
      b += nvfp4_bytes(le, n) + nvfp4_bytes(n, le) + nvfp4_bytes(1, n) + 2 * align256((size_t)n * 4) +
           align256((size_t)m * 4);
  }
  return b;
}

size_t averis_grouped_linear_fwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m, int64_t n,
                                                 unsigned flags) {
  (void)flags;
  if (!offsets_ok(offsets, num_experts) || m < 1 || n < 1) return 0;
  return grouped_fwd_ws(offsets, num_experts, m, n);
}

size_t averis_grouped_linear_bwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m, int64_t n,
                                                 unsigned flags) {
  (void)flags;
  if (!offsets_ok(offsets, num_experts) || m < 1 || n < 1) return 0;
  return grouped_bwd_ws(offsets, num_experts, m, n);
}

averis_status averis_grouped_linear_fwd(const void* x, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_nvfp4* w_m, unsigned flags, void* y,
                                        const averis_fwd_state* states, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  if (x == nullptr || y == nullptr || w_m == nullptr || states == nullptr) return AVERIS_ERR_INVALID_ARG;
  if (!offsets_ok(offsets, num_experts)) return AVERIS_ERR_INVALID_ARG;
  if (m < 16 || n < 16 || m % 16 || n % 16) return AVERIS_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return AVERIS_ERR_INVALID_ARG;
  if (workspace_bytes < grouped_fwd_ws(offsets, num_experts, m, n)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  const int64_t E = num_experts, L = offsets[E];
  if (L < 1) return AVERIS_OK;
  for (int64_t e = 0; e < E; ++e)
    if (offsets[e + 1] > offsets[e] && !nvfp4_ok(&w_m[e], n, m)) return AVERIS_ERR_INVALID_ARG;
  const std::vector<int64_t> rows = group_rows(offsets, E);
  Carver c(workspace);
  void* qws = c.take(grouped_quant_ws_bytes(rows.data(), (int)E, m));
  std::vector<GroupSpec> gs((size_t)E);
  std::vector<float*> r_x((size_t)E);
  for (int64_t e = 0; e < E; ++e) {
    r_x[(size_t)e] = static_cast<float*>(c.take((size_t)n * 4));
    GroupSpec& G = gs[(size_t)e];
    G.row0 = offsets[e];
    G.rows = rows[(size_t)e];
    if (G.rows == 0) continue;
    const averis_fwd_state& st = states[e];
    G.mu = st.mu;
    G.mu_q = &st.mu_q;
    G.mu_hat = st.mu_hat;
    G.out_row = &st.x_row;
    G.out_col = &st.x_col;
    if (split) {
      G.r_w = &w_m[e];
      G.r_out = r_x[(size_t)e];
    }
  }
  averis_status r = grouped_quantize_impl(x, L, m, flags, gs.data(), (int)E, qws,
                                          grouped_quant_ws_bytes(rows.data(), (int)E, m), stream);
  if (r != AVERIS_OK) return r;
  const int64_t esz = (flags & AVERIS_OUT_BF16) ? 2 : 4;
  std::vector<GemmSpec> gm;
  for (int64_t e = 0; e < E; ++e) {
    if (rows[(size_t)e] == 0) continue;
    GemmSpec g;
    g.a = &states[e].x_row;
    g.b = &w_m[e];
    g.col_add = split ? r_x[(size_t)e] : nullptr;
    g.out = static_cast<uint8_t*>(y) + offsets[e] * n * esz;
    g.ldo = n;
    g.bf16 = esz == 2;
    gm.push_back(g);
  }
  return grouped_gemm_impl(gm.data(), (int)gm.size(), stream);
}

averis_status averis_grouped_linear_bwd(const void* d, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_fwd_state* states, const averis_nvfp4* w_n,
                                        unsigned flags, void* dx, float* const* dw, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  if (d == nullptr || dx == nullptr || dw == nullptr || w_n == nullptr || states == nullptr)
    return AVERIS_ERR_INVALID_ARG;
  if (!offsets_ok(offsets, num_experts)) return AVERIS_ERR_INVALID_ARG;
  if (m < 16 || n < 16 || m % 16 || n % 16) return AVERIS_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return AVERIS_ERR_INVALID_ARG;
  if (workspace_bytes < grouped_bwd_ws(offsets, num_experts, m, n)) return AVERIS_ERR_WORKSPACE_TOO_SMALL;
  const bool split = (flags & AVERIS_MEAN_SPLIT) != 0;
  const int64_t E = num_experts, L = offsets[E];
  if (L < 1) return AVERIS_OK;
  for (int64_t e = 0; e < E; ++e) {
    const int64_t le = offsets[e + 1] - offsets[e];
    if (le == 0) continue;
    if (!nvfp4_ok(&w_n[e], m, n) || !nvfp4_ok(&states[e].x_col, m, le) || dw[e] == nullptr)
      return AVERIS_ERR_INVALID_ARG;
    if (split && states[e].mu_hat == nullptr) return AVERIS_ERR_INVALID_ARG;
  }
  const std::vector<int64_t> rows = group_rows(offsets, E);
  Carver c(workspace);
  void* qws = c.take(grouped_quant_ws_bytes(rows.data(), (int)E, n));
  struct DState {
    averis_nvfp4 row, col, mu_q;
    float *mu, *mu_hat, *r_d;
  };
  std::vector<DState> ds((size_t)E);
  std::vector<GroupSpec> gs((size_t)E);
  for (int64_t e = 0; e < E; ++e) {
    const int64_t le = rows[(size_t)e];
    GroupSpec& G = gs[(size_t)e];
    G.row0 = offsets[e];
    G.rows = le;
    if (le == 0) continue;
    DState& D = ds[(size_t)e];
    D.row = carve_nvfp4(c, le, n);
    D.col = carve_nvfp4(c, n, le);
    D.mu_q = carve_nvfp4(c, 1, n);
    D.mu = static_cast<float*>(c.take((size_t)n * 4));
    D.mu_hat = static_cast<float*>(c.take((size_t)n * 4));
    D.r_d = static_cast<float*>(c.take((size_t)m * 4));
    G.mu = D.mu;
    G.mu_q = &D.mu_q;
    G.mu_hat = D.mu_hat;
    G.out_row = &D.row;
    G.out_col = &D.col;
    if (split) {
      G.r_w = &w_n[e];
      G.r_out = D.r_d;
    }
  }
  averis_status r = grouped_quantize_impl(d, L, n, flags, gs.data(), (int)E, qws,
                                          grouped_quant_ws_bytes(rows.data(), (int)E, n), stream);
  if (r != AVERIS_OK) return r;
  const int64_t esz = (flags & AVERIS_OUT_BF16) ? 2 : 4;
  std::vector<GemmSpec> gx, gw;
  for (int64_t e = 0; e < E; ++e) {
    const int64_t le = rows[(size_t)e];
    if (le == 0) continue;
    const DState& D = ds[(size_t)e];
    GemmSpec a;
    a.a = &D.row;
    a.b = &w_n[e];
    a.col_add = split ? D.r_d : nullptr;
    a.out = static_cast<uint8_t*>(dx) + offsets[e] * m * esz;
    a.ldo = m;
    a.bf16 = esz == 2;
    gx.push_back(a);
    GemmSpec w;
    w.a = &states[e].x_col;
    w.b = &D.col;
    w.row_vec = split ? states[e].mu_hat : nullptr;
    w.col_vec = split ? D.mu_hat : nullptr;
    w.outer = (float)le;
    w.out = dw[e];
    w.ldo = n;
    gw.push_back(w);
  }
  // the weight gradients first (the longest units), then the input gradients
  if ((r = grouped_gemm_impl(gw.data(), (int)gw.size(), stream)) != AVERIS_OK) return r;
  return grouped_gemm_impl(gx.data(), (int)gx.size(), stream);
}

const char* averis_status_string(averis_status status) {
  switch (status) {
    case AVERIS_OK: return "ok";
    case AVERIS_ERR_INVALID_ARG: return "invalid argument";
    case AVERIS_ERR_UNSUPPORTED_ARCH: return "unsupported architecture (needs sm_103)";
    case AVERIS_ERR_CUDA: return "CUDA error";
    case AVERIS_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case AVERIS_ERR_TIMEOUT: return "device-side wait timed out";
    case AVERIS_ERR_OUT_OF_BOUNDS: return "out-of-range access caught by a debug-build check";
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
  return v == 0 ? AVERIS_OK : v >= kErrBoundsBase ? AVERIS_ERR_OUT_OF_BOUNDS : AVERIS_ERR_TIMEOUT;
}

averis_status averis_debug_starve_next_quantize(long long wait_cycles) {
  if (wait_cycles < 10000 || wait_cycles > kWaitLimit) return AVERIS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_starve_next = wait_cycles;
  return AVERIS_OK;
}

int averis_version(void) { return 20000; }

int averis_debug_checks(void) {
#ifndef AVERIS_DEBUG
  return 0;
#else
  return debug_self_test();
#endif
}

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
