// Bounds checks of the debug build (compiled with -DAVERIS_DEBUG).
//
// A memory checker is not available on every machine this library runs its
// tests on, so the debug build checks every global-memory address that a
// kernel computes itself (the plain loads and stores, not the TMA copies,
// which clip to their tensor maps) against the extent of the buffer it must
// fall in, and the inner coordinate of every TMA copy against the 16-byte
// rule.  A failed check skips the access and records kErrBoundsBase + site
// in the device error word (the first failure wins; averis_last_device_error
// reads it back).  Kernels write the checks as AVERIS_DBG_IN(...) and
// AVERIS_DBG_TMA_X(...), which the release build replaces by the literal true,
// arguments and all, so its code is what it would be without them.
#pragma once

#include <cstdint>

namespace averis {

constexpr int kErrBoundsBase = 100;  // error word = kErrBoundsBase + site

// Where a check sits (the site is part of the recorded code).
enum : int {
  kSiteSelfTest = 0,       // averis_debug_checks' own test of the recorder
  kSiteStatsPartial = 1,   // stats pass: row-block partial store
  kSiteStatsCombine = 2,   // stats pass: partial loads of the last CTA of a strip group
  kSiteStatsMean = 3,      // stats pass: mean store
  kSiteMeanLoad = 4,       // quantize pass, mean CTAs: mean loads
  kSiteMeanCodes = 5,      // quantize pass: NVFP4 mean codes / block scales
  kSiteMeanHat = 6,        // quantize pass: dequantized mean
  kSiteRank1Weight = 7,    // rank-one row: weight codes / block scales
  kSiteRank1Out = 8,       // rank-one row: output
  kSiteRowCodes = 9,       // quantize pass: row-layout codes
  kSiteColCodes = 10,      // quantize pass: column-layout codes
  kSiteScaleAtoms = 11,    // quantize pass: block-scale atoms
  kSiteResidentPart = 12,  // single-read quantize: per-tile column partials
  kSiteGemmVectors = 13,   // GEMM epilogue: broadcast row / outer-product vectors
  kSiteTmaInner = 14,      // any kernel: a TMA copy's inner coordinate off the 16-byte rule
  kSiteGemvOut = 15        // standalone rank-one GEMV: output
};

#ifdef AVERIS_DEBUG
constexpr bool kDebugChecks = true;

// True when the `bytes` at p lie inside [base, base + extent); the test alone,
// with no access and no recording (the self-test of averis_debug_checks uses it).
__host__ __device__ __forceinline__ bool dbg_inside(const void* p, const void* base, int64_t extent, int bytes) {
  const int64_t off = reinterpret_cast<const char*>(p) - reinterpret_cast<const char*>(base);
  return base != nullptr && off >= 0 && off <= extent - bytes;
}

__device__ __forceinline__ void dbg_record(int* err, int site) { atomicCAS(err, 0, kErrBoundsBase + site); }

__device__ __forceinline__ bool dbg_in(int* err, const void* p, const void* base, int64_t extent, int bytes,
                                       int site) {
  if (dbg_inside(p, base, extent, bytes)) return true;
  dbg_record(err, site);
  return false;
}

// inner TMA coordinate x of elements of `elem_bytes`: x * elem_bytes must be a multiple of 16
__device__ __forceinline__ bool dbg_tma_x(int* err, int64_t x, int elem_bytes) {
  if ((x * elem_bytes) % 16 == 0) return true;
  dbg_record(err, kSiteTmaInner);
  return false;
}
#define AVERIS_DBG_IN(...) ::averis::dbg_in(__VA_ARGS__)
#define AVERIS_DBG_TMA_X(...) ::averis::dbg_tma_x(__VA_ARGS__)
#else
constexpr bool kDebugChecks = false;
// the release build: the checks and their arguments vanish before compilation
#define AVERIS_DBG_IN(...) true
#define AVERIS_DBG_TMA_X(...) true
#endif

}  // namespace averis
