// Mean-split NVFP4 quantize pass and the rank-one GEMV.
//
// Pass 1  colstats         : per column compensated sum, max and min of the
//                            bf16 input in one coalesced read; the last CTAs
//                            to finish combine them into the mean mu
//                            (binary32), the residual's exact maximum
//                            magnitude, the tensor scales, and the NVFP4
//                            quantization of mu itself.
// Pass 2  split_quant      : r = fl32(x - mu) (optionally rotated by H16/4),
//                            NVFP4 along the columns AND along the rows, both
//                            layouts written in one read of the tile.
// rank1_gemv               : r = deq(mu_q) deq(W)^T.
//
// Method: "均值偏置的诅咒与祝福：FP4量化大语言模型训练" (paper.rainbus.top summary),
// section 方法步骤详情: mu = (1/l) 1^T X, X_R = X - 1 mu, mu and X_R quantized
// independently; background 块量化 for the blockwise quantizer; background
// Hadamard变换 for the 16x16 rotation.  The quantizer's binary32 steps:
//   s_g = fl32(A / 2688), den = fl32(6 s_g), e = E4M3(fl32(a_b / den)),
//   sb = fl32(e4m3(e) s_g), inv = min(fl32(1/sb), FLT_MAX) (0 if sb == 0),
//   code = E2M1(fl32(r * inv)); all round-to-nearest-even, saturating.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "debug.cuh"
#include "ptx.cuh"

namespace averis {

// Control block at the head of every workspace.  Every word is zero at rest:
// the stats pass accumulates maxima with atomicMax and resets its strip
// tickets itself; the last CTA of the quantize pass (ticket) resets the
// maxima after every reader is done.  A workspace that starts zeroed stays
// usable for any later call without a memset.
enum : int {
  kCtrlAmaxRes = 1,      // residual max magnitude (float bits), both layouts
  kCtrlAmaxRowH = 5,     // rotated residual max, layout blocked along columns (Hadamard)
  kCtrlAmaxColH = 6,     // rotated residual max, layout blocked along rows (Hadamard)
  kCtrlQuantTicket = 7,  // quantize pass: CTAs finished
  kCtrlGridBar = 9,      // single-read quantize: arrivals at its grid-wide waits
  kCtrlStrip = 64,       // per-strip-group tickets of the stats pass
  kMaxStripGroups = 1024,
  kCtrlWords = kCtrlStrip + kMaxStripGroups
};

struct ColPartial {
  float s_hi, s_lo, mx, mn;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Offset of (row r, 16-block k) in the tiled scale layout of a tensor with
// `kc` 64-column chunks per row: see averis_nvfp4 in averis.h.
__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t k, int64_t kc) {
  return ((r >> 7) * kc + (k >> 2)) * 512 + 16 * (r & 31) + 4 * ((r & 127) >> 5) + (k & 3);
}


__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
// Two binary32 subtractions / multiplications, each rounded to nearest even (packed issue).
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// fl32(bf16 - binary32) for both halves of a packed bf16 word (mixed-precision subtract; the
// bf16 operand converts exactly, so this is the binary32 subtraction of the widened value).
__device__ __forceinline__ uint64_t bf2_sub_f2(uint32_t w, uint64_t m) {
  float d0, d1;
  asm("{\n .reg .b16 l, h;\n .reg .f32 m0, m1;\n mov.b32 {l, h}, %2;\n mov.b64 {m0, m1}, %3;\n"
      " sub.rn.f32.bf16 %0, l, m0;\n sub.rn.f32.bf16 %1, h, m1;\n}"
      : "=f"(d0), "=f"(d1)
      : "r"(w), "l"(m));
  return f2pack(d0, d1);
}
// fl32(bf16 - m) of one half (hi: the upper one) of each of two words.
__device__ __forceinline__ uint64_t bf_pair_sub(uint32_t wa, uint32_t wb, bool hi, float m) {
  float d0, d1;
  if (hi)
    asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %2;\n mov.b32 {l1, h1}, %3;\n"
        " sub.rn.f32.bf16 %0, h0, %4;\n sub.rn.f32.bf16 %1, h1, %4;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(wa), "r"(wb), "f"(m));
  else
    asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %2;\n mov.b32 {l1, h1}, %3;\n"
        " sub.rn.f32.bf16 %0, l0, %4;\n sub.rn.f32.bf16 %1, l1, %4;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(wa), "r"(wb), "f"(m));
  return f2pack(d0, d1);
}
// (fl32(bf16 a - ma), fl32(bf16 b - mb)) of one half (hi: the upper one) of each of two words.
__device__ __forceinline__ uint64_t bf_pair_sub2(uint32_t wa, uint32_t wb, bool hi, float ma, float mb) {
  float d0, d1;
  if (hi)
    asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %2;\n mov.b32 {l1, h1}, %3;\n"
        " sub.rn.f32.bf16 %0, h0, %4;\n sub.rn.f32.bf16 %1, h1, %5;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(wa), "r"(wb), "f"(ma), "f"(mb));
  else
    asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %2;\n mov.b32 {l1, h1}, %3;\n"
        " sub.rn.f32.bf16 %0, l0, %4;\n sub.rn.f32.bf16 %1, l1, %5;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(wa), "r"(wb), "f"(ma), "f"(mb));
  return f2pack(d0, d1);
}
// The two bf16 values of a packed word as a binary32 pair (exact).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return f2pack(bf16lo(w), bf16hi(w)); }
// Element-wise max / min of two packed bf16 pairs (exact).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Unevaluated sum hi + lo of two binary32 values (|lo| <= ulp(hi) / 2): the
// column sums are combined in this form, exactly enough for the mean and
// without float64 arithmetic (slow on this part).
struct F2 {
  float hi, lo;
};
__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ F2 fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ F2 df_add(F2 a, F2 b) {
  const F2 s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
// binary32 of (hi + lo) / n for an integer count n < 2^24 (exact in binary32).
__device__ __forceinline__ float df_div_count(F2 a, float n) {
  const float q = __fdiv_rn(a.hi, n);
  const float r = __fadd_rn(__fmaf_rn(-q, n, a.hi), a.lo);  // a - q n, the product residual is exact
  return __fadd_rn(q, __fdiv_rn(r, n));
}

// Block-wide max of non-negative floats (blockDim 256).
__device__ __forceinline__ float block_max256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}

// In-register 16-point Walsh-Hadamard butterfly, strides 1, 2, 4, 8, then * 1/4.
__device__ __forceinline__ void fwht16(float (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (!(j & h)) {
        const float a = v[j], b = v[j + h];
        v[j] = __fadd_rn(a, b);
        v[j + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// The same butterfly on packed pairs, for the tile quantizer: on entry
// p[k] = (v[k], v[k+8]), k < 8.  Strides 1, 2 and 4 pair whole registers
// (packed adds and subtractions), stride 8 pairs the two halves of each
// register; on exit p[m] = (v[2m], v[2m+1]) * 1/4.  Every element sees the
// same binary32 operations in the same order as fwht16.
__device__ __forceinline__ void fwht16_x2(uint64_t (&p)[8]) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (!(k & h)) {
        const uint64_t a = p[k], b = p[k + h];
        p[k] = add2(a, b);
        p[k + h] = sub2(a, b);
      }
    }
  }
  float o[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a = f2lo(p[k]), b = f2hi(p[k]);
    o[k] = __fadd_rn(a, b);
    o[k + 8] = __fsub_rn(a, b);
  }
  const uint64_t quarter = f2pack(0.25f, 0.25f);
#pragma unroll
  for (int m = 0; m < 8; ++m) p[m] = mul2(f2pack(o[2 * m], o[2 * m + 1]), quarter);
}

struct BlockQ {
  uint32_t scale;   // E4M3 code
  uint32_t lo, hi;  // 16 E2M1 codes, element 0 in the low nibble of lo
  float amax;
};

__device__ __forceinline__ float tensor_scale_of(float amax) { return __fdiv_rn(amax, 2688.0f); }

// NVFP4 of one 16-element block, given the tensor scale s_g (binary32 steps
// as in the file header).
__device__ __forceinline__ BlockQ quant_block16(const float (&r)[16], float s_g) {
  BlockQ q;
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(r[e]));
  q.amax = a;
  uint32_t code = 0;
  if (s_g > 0.f) code = ptx::cvt_e4m3(__fdiv_rn(a, __fmul_rn(6.0f, s_g)));
  const float sb = __fmul_rn(e4m3_value(code), s_g);
  const float inv = sb > 0.f ? fminf(__frcp_rn(sb), FLT_MAX) : 0.f;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t b = ptx::cvt_e2m1x2(__fmul_rn(r[2 * e], inv), __fmul_rn(r[2 * e + 1], inv));
    w[e >> 2] |= b << (8 * (e & 3));
  }
  q.scale = code;
  q.lo = w[0];
  q.hi = w[1];
  return q;
}

__device__ __forceinline__ float e2m1_mag(uint32_t c3) {
  // 0, .5, 1, 1.5, 2, 3, 4, 6
  const uint32_t e = (c3 >> 1) & 3u, m = c3 & 1u;
  return e == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
}
__device__ __forceinline__ float e2m1_val(uint32_t c4) {
  const float v = e2m1_mag(c4 & 7u);
  return (c4 & 8u) ? -v : v;
}

// ------------------------------------------------------------ pass 1 ----

struct StatsParams {
  const __nv_bfloat16* x;
  int64_t R, C;
  int64_t rows_per;   // rows per CTA row block (multiple of 32)
  int nstrips;        // ceil(C / 64) column strips of 64
  ColPartial* part;   // [gridDim.y][C] per-row-block partials
  unsigned* ctrl;
  int* err;           // device error word (a box that never arrived)
  int split;          // mean split on
  int hadamard;       // rotation on (the rotated residual's maximum comes from the amax pass)
  float* mu;          // [C] out (split)
  long long wait_limit;  // bound of every wait, in SM clock cycles
  // diagnostics only: issue no input loads, so that every wait for a box runs
  // out (exercises the timeout path with no copy in flight)
  int starve;
  int64_t row_base;   // first row of these R rows in the tensor map (a group of a grouped input)
};

// Column statistics in one pass over X, with the combine fused in.
//
// grid (strip groups, row blocks), 256 threads.  CTA (g, b) reads rows
// [b*rows_per, (b+1)*rows_per) of the 64-column strips g, g+gridDim.x, ...:
// thread t owns 8 adjacent columns (16-byte loads) of rows t/8, t/8+32, ...,
// keeps a Kahan-compensated binary32 sum plus max and min per column (packed
// bf16 max / min, pairs of columns summed with packed binary32 adds), and the
// 32 row lanes are combined as hi + lo binary32 pairs in a fixed order.  The
// last CTA of a strip group to finish (ticket) combines the row-block
// partials of its strips in row-block order -- the result does not depend on
// which CTA is last -- giving mu_j = fl32(S_j / R) and the residual's exact
// maximum magnitude max(|fl32(max_j - mu_j)|, |fl32(min_j - mu_j)|) (binary32
// subtraction is monotone), folded into the control block with atomicMax.
constexpr int kStatsBoxRows = 256;                           // rows per TMA box (8 per thread)
constexpr int kStatsBufs = 3;                                 // boxes in flight per CTA
constexpr int kStatsBox = kStatsBoxRows * 128;                // 64 bf16 columns x 256 rows (32 KB)
constexpr int kStatsSmem = kStatsBufs * kStatsBox + 1024;     // + alignment slack for the 128-byte swizzle

// The pass of one CTA: strip group bx of nbx, row block by of nby.
__device__ __forceinline__ void colstats_body(const CUtensorMap& tmX, const StatsParams& p, int bx, int nbx, int by,
                                              int nby) {
  extern __shared__ uint8_t stats_raw[];
  uint8_t* ring = stats_raw + ((1024u - (ptx::smem_u32(stats_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  __shared__ F2 s_sum[8][64];
  __shared__ float s_mx[8][64], s_mn[8][64];
  __shared__ float red[8];
  __shared__ int s_last;
  __shared__ uint64_t s_full[kStatsBufs];
  __shared__ int s_done[kStatsBufs];  // warps done with the buffer's current box
  __shared__ int s_failed;
  __shared__ int s_issued;  // boxes of the current strip requested so far
  if (threadIdx.x == 0) {
    for (int b = 0; b < kStatsBufs; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      s_done[b] = 0;
    }
    s_failed = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmX);
  }
  __syncthreads();
  ptx::pdl_wait_and_release();
  // the quantize pass reads X again right after: keep its lines in L2
  const uint64_t keep = ptx::l2_policy_evict_last();
  uint32_t it = 0;  // boxes consumed by this CTA (buffer it % kStatsBufs, phase it / kStatsBufs)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = tid & 7;     // 8-column group inside the strip
  const int rl = tid >> 3;    // row lane 0..31
  const int64_t rb0 = (int64_t)by * p.rows_per;
  const int64_t rb1 = min(p.R, rb0 + p.rows_per);

  bool failed = false;  // a box never arrived (uniform over the CTA)
  for (int strip = bx; strip < p.nstrips && !failed; strip += nbx) {
    // column pairs (2w, 2w+1): Kahan-compensated binary32 sums, packed bf16 max / min
    uint64_t s2[4], c2[4];
    uint32_t mx2[4], mn2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      s2[w] = 0ull;
      c2[w] = 0ull;
      mx2[w] = 0xFF80FF80u;  // -inf, -inf
      mn2[w] = 0x7F807F80u;  // +inf, +inf
    }
    auto kahan = [&](int w, uint64_t t) {
      const uint64_t y = sub2(t, c2[w]);
      const uint64_t tt = add2(s2[w], y);
      c2[w] = sub2(sub2(tt, s2[w]), y);
      s2[w] = tt;
    };
    // 8 rows (stride 32) at a time: pairwise sums, then one compensated add.
    // nv < 8: only the first nv rows count (the others repeat a counted row,
    // harmless for max / min, and are left out of the sum)
    auto group = [&](const uint4 (&v)[8], int nv) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = w == 0 ? v[j].x : w == 1 ? v[j].y : w == 2 ? v[j].z : v[j].w;
        mx2[w] = bmax2(mx2[w], bmax2(bmax2(bmax2(x[0], x[1]), bmax2(x[2], x[3])), bmax2(bmax2(x[4], x[5]), bmax2(x[6], x[7]))));
        mn2[w] = bmin2(mn2[w], bmin2(bmin2(bmin2(x[0], x[1]), bmin2(x[2], x[3])), bmin2(bmin2(x[4], x[5]), bmin2(x[6], x[7]))));
#pragma unroll
        for (int j = 1; j < 8; ++j)
          if (j >= nv) x[j] = 0u;  // +0 + +0: adds nothing
        const uint64_t t = add2(add2(add2(bf2_to_f2(x[0]), bf2_to_f2(x[1])), add2(bf2_to_f2(x[2]), bf2_to_f2(x[3]))),
                                add2(add2(bf2_to_f2(x[4]), bf2_to_f2(x[5])), add2(bf2_to_f2(x[6]), bf2_to_f2(x[7]))));
        kahan(w, t);
      }
    };
    // the strip's rows arrive by TMA in boxes of 256 rows x 64 columns (128-byte
    // swizzle: 16-byte chunk j of box row r at chunk j ^ (r % 8)); thread rows
    // rl, rl + 32, ... of a box are one 8-row group.  Rows past this CTA's block
    // are left out (max / min see a repeat of a counted row, the sum zeros).
    const int64_t nbox = (rb1 - rb0 + kStatsBoxRows - 1) / kStatsBoxRows;
    if (threadIdx.x == 0) {
      s_issued = 0;
      if (!p.starve)
        for (int64_t k = 0; k < kStatsBufs && k < nbox; ++k) {
          const uint32_t b = (it + (uint32_t)k) % kStatsBufs;
          ptx::mbar_arrive_expect_tx(&s_full[b], (uint32_t)kStatsBox);
          if (AVERIS_DBG_TMA_X(p.err, (int64_t)strip * 64, 2))
            ptx::tma_load_2d_hint(ring + b * kStatsBox, &tmX, strip * 64,
                                  (int32_t)(p.row_base + rb0 + k * kStatsBoxRows), &s_full[b], keep);
          s_issued = (int)k + 1;
        }
    }
    __syncthreads();
    // every warp walks the boxes on its own; the last warp done with a box
    // refills its buffer (no CTA-wide barrier per box)
    uint32_t it0 = it;  // first box of this strip
    for (int64_t k = 0; k < nbox; ++k, ++it) {
      const uint32_t b = it % kStatsBufs;
      int ok = 1;
      if (lane == 0) ok = ptx::mbar_wait(&s_full[b], (it / kStatsBufs) & 1u, p.wait_limit) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        // this warp gives up; the others give up on their own waits.  The
        // results of this call are invalid; the CTA still takes its ticket
        // below so that the control block returns to zero
        if (lane == 0) {
          atomicExch(p.err, kErrQuantLoad);
          s_failed = 1;
        }
        break;
      }
      const int64_t row0 = rb0 + k * kStatsBoxRows + rl;  // this thread's first row of the box
      const int64_t left = row0 < rb1 ? (rb1 - row0 + 31) / 32 : 0;  // this thread's rows left in the block
      const int nv = left < 8 ? (int)left : 8;
      if (nv > 0) {
        const uint8_t* box = ring + b * kStatsBox;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = rl + 32 * j;
          v[j] = *reinterpret_cast<const uint4*>(box + r * 128 + ((g8 ^ (r & 7)) << 4));
        }
#pragma unroll
        for (int j = 1; j < 8; ++j)
          if (j >= nv) v[j] = v[0];  // a counted row: harmless for max / min; group() drops it from the sum
        if (nv == 8)
          group(v, 8);
        else
          group(v, nv);
      }
      // count this warp done with the box; the last of the 8 warps refills the buffer
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&s_done[b], 1) == 7) {
          s_done[b] = 0;
          if (k + kStatsBufs < nbox) {
            ptx::mbar_arrive_expect_tx(&s_full[b], (uint32_t)kStatsBox);
            if (AVERIS_DBG_TMA_X(p.err, (int64_t)strip * 64, 2))
              ptx::tma_load_2d_hint(ring + b * kStatsBox, &tmX, strip * 64,
                                    (int32_t)(p.row_base + rb0 + (k + kStatsBufs) * kStatsBoxRows), &s_full[b], keep);
            s_issued = (int)(k + kStatsBufs) + 1;
          }
        }
      }
    }
    __syncthreads();  // every warp is done with this strip's boxes (or gave up)
    if (s_failed) {
      if (threadIdx.x == 0) {
        // let the boxes still in flight land (bounded) before the buffers are
        // given up: only the last kStatsBufs requested can be (a box is
        // requested only after the box kStatsBufs before it was consumed)
        for (int k = max(0, s_issued - kStatsBufs); k < s_issued; ++k)
          ptx::mbar_wait(&s_full[(it0 + (uint32_t)k) % kStatsBufs], ((it0 + (uint32_t)k) / kStatsBufs) & 1u,
                         p.wait_limit);
      }
      failed = true;
      break;
    }
    it = it0 + (uint32_t)nbox;
    // combine the 4 row lanes of this warp that share the columns (lanes differ by 8, 16)
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = 2 * w + h;
        const float sv = h ? f2hi(s2[w]) : f2lo(s2[w]), cv = h ? f2hi(c2[w]) : f2lo(c2[w]);
        F2 d = fast_two_sum(sv, -cv);
        F2 o{__shfl_xor_sync(0xffffffffu, d.hi, 8), __shfl_xor_sync(0xffffffffu, d.lo, 8)};
        d = (lane & 8) ? df_add(o, d) : df_add(d, o);
        o = F2{__shfl_xor_sync(0xffffffffu, d.hi, 16), __shfl_xor_sync(0xffffffffu, d.lo, 16)};
        d = (lane & 16) ? df_add(o, d) : df_add(d, o);
        const float mxv = h ? bf16hi(mx2[w]) : bf16lo(mx2[w]), mnv = h ? bf16hi(mn2[w]) : bf16lo(mn2[w]);
        float m1 = fmaxf(mxv, __shfl_xor_sync(0xffffffffu, mxv, 8));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 16));
        float m2 = fminf(mnv, __shfl_xor_sync(0xffffffffu, mnv, 8));
        m2 = fminf(m2, __shfl_xor_sync(0xffffffffu, m2, 16));
        if (lane < 8) {
          s_sum[warp][8 * lane + e] = d;
          s_mx[warp][8 * lane + e] = m1;
          s_mn[warp][8 * lane + e] = m2;
        }
      }
    }
    __syncthreads();
    if (tid < 64) {
      const int64_t col = (int64_t)strip * 64 + tid;
      F2 acc = s_sum[0][tid];
      float m1 = s_mx[0][tid], m2 = s_mn[0][tid];
#pragma unroll
      for (int w = 1; w < 8; ++w) {
        acc = df_add(acc, s_sum[w][tid]);
        m1 = fmaxf(m1, s_mx[w][tid]);
        m2 = fminf(m2, s_mn[w][tid]);
      }
      if (col < p.C && AVERIS_DBG_IN(p.err, p.part + (int64_t)by * p.C + col, p.part, (int64_t)nby * p.C * 16, 16,
                                     kSiteStatsPartial))
        *reinterpret_cast<float4*>(p.part + (int64_t)by * p.C + col) = make_float4(acc.hi, acc.lo, m1, m2);
    }
    __syncthreads();
  }

  // ---- last row block of this strip group combines the partials
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(&p.ctrl[kCtrlStrip + bx], 1u);
    s_last = (t == (unsigned)nby - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  float a_res = 0.f;
  const int nrb = nby;
  const float Rf = (float)p.R;
  for (int strip = bx; strip < p.nstrips; strip += nbx) {
    const int cl = tid & 63, part = tid >> 6;
    const int64_t col = (int64_t)strip * 64 + cl;
    F2 acc{0.f, 0.f};
    float m1 = -FLT_MAX, m2 = FLT_MAX;
    if (col < p.C) {
      // row blocks part, part + 4, ... in order; up to 32 row blocks in one round of loads
      for (int rb = part; rb < nrb; rb += 32) {
        float4 q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          q[j] = rb + 4 * j < nrb && AVERIS_DBG_IN(p.err, p.part + (int64_t)(rb + 4 * j) * p.C + col, p.part,
                                                   (int64_t)nrb * p.C * 16, 16, kSiteStatsCombine)
                     ? __ldcg(reinterpret_cast<const float4*>(p.part + (int64_t)(rb + 4 * j) * p.C + col))
                     : make_float4(0.f, 0.f, -FLT_MAX, FLT_MAX);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc = df_add(acc, F2{q[j].x, q[j].y});
          m1 = fmaxf(m1, q[j].z);
          m2 = fminf(m2, q[j].w);
        }
      }
    }
    s_sum[part][cl] = acc;
    s_mx[part][cl] = m1;
    s_mn[part][cl] = m2;
    __syncthreads();
    if (tid < 64 && col < p.C) {
      const F2 S = df_add(df_add(df_add(s_sum[0][cl], s_sum[1][cl]), s_sum[2][cl]), s_sum[3][cl]);
      const float M1 = fmaxf(fmaxf(s_mx[0][cl], s_mx[1][cl]), fmaxf(s_mx[2][cl], s_mx[3][cl]));
      const float M2 = fminf(fminf(s_mn[0][cl], s_mn[1][cl]), fminf(s_mn[2][cl], s_mn[3][cl]));
      if (p.split) {
        const float mu = df_div_count(S, Rf);
        if (AVERIS_DBG_IN(p.err, p.mu + col, p.mu, p.C * 4, 4, kSiteStatsMean)) p.mu[col] = mu;
        a_res = fmaxf(a_res, fmaxf(fabsf(__fsub_rn(M1, mu)), fabsf(__fsub_rn(M2, mu))));
      } else {
        a_res = fmaxf(a_res, fmaxf(fabsf(M1), fabsf(M2)));
      }
    }
    __syncthreads();
  }
  if (tid == 0) p.ctrl[kCtrlStrip + bx] = 0u;  // every row block has arrived: reset for the next call
  a_res = block_max256(a_res, red);
  if (tid == 0) atomicMax(&p.ctrl[kCtrlAmaxRes], __float_as_uint(a_res));
}

__global__ void __launch_bounds__(256, 2) colstats_kernel(const __grid_constant__ CUtensorMap tmX,
                                                          const __grid_constant__ StatsParams p) {
  colstats_body(tmX, p, blockIdx.x, gridDim.x, blockIdx.y, gridDim.y);
}

// Groups (experts) of a grouped input, one launch: at most kMaxGroups per launch.
constexpr int kMaxGroups = 64;

// The stats pass over the row groups of a grouped input: group e owns row
// blocks rb0[e] .. rb0[e+1]-1 of the grid's y dimension; g[e] holds its rows,
// partials, control words and mean.
struct GroupedStatsParams {
  StatsParams g[kMaxGroups];
  int rb0[kMaxGroups + 1];
  int ngroups;
};

__global__ void __launch_bounds__(256, 2) colstats_grouped_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                  const __grid_constant__ GroupedStatsParams gp) {
  int e = 0;
  while (e + 1 < gp.ngroups && gp.rb0[e + 1] <= (int)blockIdx.y) ++e;
  colstats_body(tmX, gp.g[e], blockIdx.x, gridDim.x, (int)blockIdx.y - gp.rb0[e], gp.rb0[e + 1] - gp.rb0[e]);
}

// NVFP4 of the mean as one [1, C] row, into SMEM (codes: C/2 bytes, one E4M3
// byte per block) and, when `p.mu_codes` is to be written by this CTA, into
// the caller's tensor (codes, tiled scales, tensor scale) and mu_hat.  Under
// the Hadamard variant the mean is rotated block-wise first, and mu_hat is
// the dequantized mean rotated back (H16/4 is its own inverse).  The tensor
// scale comes from the maximum magnitude of the (rotated) mean.  All 256
// threads of the CTA take part; returns the tensor scale.
template <typename P>
__device__ float quantize_mean(const P& p, bool write_global, uint8_t* s_codes, uint8_t* s_scales, float* red) {
  const int64_t nb = p.C / 16;
  const bool had = p.hadamard != 0;
  float a = 0.f;
  for (int64_t b = threadIdx.x; b < nb; b += 256) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      v[e] = AVERIS_DBG_IN(p.err, p.mu + 16 * b + e, p.mu, p.C * 4, 4, kSiteMeanLoad) ? __ldcg(p.mu + 16 * b + e) : 0.f;
    if (had) fwht16(v);
#pragma unroll
    for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(v[e]));
  }
  const float s_g = tensor_scale_of(block_max256(a, red));
  if (write_global && threadIdx.x == 0) *p.mu_ts = s_g;
  for (int64_t b = threadIdx.x; b < nb; b += 256) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
      const float4 m4 = AVERIS_DBG_IN(p.err, p.mu + 16 * b + e, p.mu, p.C * 4, 16, kSiteMeanLoad)
                            ? __ldcg(reinterpret_cast<const float4*>(p.mu + 16 * b + e))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      v[e] = m4.x;
      v[e + 1] = m4.y;
      v[e + 2] = m4.z;
      v[e + 3] = m4.w;
    }
    if (had) fwht16(v);
    const BlockQ q = quant_block16(v, s_g);
    *reinterpret_cast<uint2*>(s_codes + 8 * b) = make_uint2(q.lo, q.hi);
    s_scales[b] = (uint8_t)q.scale;
    if (!write_global) continue;
    if (AVERIS_DBG_IN(p.err, p.mu_codes + 8 * b, p.mu_codes, (p.C + 63) / 64 * 32, 8, kSiteMeanCodes))
      *reinterpret_cast<uint2*>(p.mu_codes + 8 * b) = make_uint2(q.lo, q.hi);
    if (AVERIS_DBG_IN(p.err, p.mu_scales + scale_offset(0, b, p.mu_kc), p.mu_scales, 512 * p.mu_kc, 1, kSiteMeanCodes))
      p.mu_scales[scale_offset(0, b, p.mu_kc)] = (uint8_t)q.scale;
    const float sc = e4m3_value(q.scale);
    float d[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c4 = ((e < 8 ? q.lo : q.hi) >> (4 * (e & 7))) & 15u;
      d[e] = __fmul_rn(__fmul_rn(e2m1_val(c4), sc), s_g);
    }
    if (had) fwht16(d);
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      if (AVERIS_DBG_IN(p.err, p.mu_hat + 16 * b + e, p.mu_hat, p.C * 4, 16, kSiteMeanHat))
        *reinterpret_cast<float4*>(p.mu_hat + 16 * b + e) = make_float4(d[e], d[e + 1], d[e + 2], d[e + 3]);
  }
  __syncthreads();
  return s_g;
}

// The four bytes of a code word (eight E2M1 codes) as four f16 pairs.  E2M1
// values are exact in f16, and a dot product does not depend on the order
// of the pair halves, so the two operands just have to be unpacked alike.
__device__ __forceinline__ void e2m1x8_to_h2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Dot product of one 16-element block of codes (two words, already unpacked
// into f16 pairs for the mean) with the same block of another code row.
// Each product of E2M1 values is a multiple of 1/4 of magnitude <= 36, and
// each f16 half accumulates 8 of them (<= 288, 1152 quarter units < 2^11):
// every step is exact in f16, and the final binary32 sum is exact too.
__device__ __forceinline__ float dot16_h2(const uint32_t (&mh)[8], uint32_t w0, uint32_t w1) {
  uint32_t wh[4];
  __half2 acc = __float2half2_rn(0.f);
  e2m1x8_to_h2(w0, wh);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    acc = __hfma2(*reinterpret_cast<const __half2*>(&mh[k]), *reinterpret_cast<__half2*>(&wh[k]), acc);
  e2m1x8_to_h2(w1, wh);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    acc = __hfma2(*reinterpret_cast<const __half2*>(&mh[4 + k]), *reinterpret_cast<__half2*>(&wh[k]), acc);
  const float2 f = __half22float2(acc);
  return f.x + f.y;
}

// Rank-one row r[n] = s_mu s_w sum_k deq(mu)_k deq(W)_{n,k} for rows
// [n0, n1) of W, with the NVFP4 mean in SMEM.  A warp handles 4 rows at a
// time (all their loads in flight together), lanes over 32-element chunks;
// block products in f16 (exact), scaled per 16-block in binary32.
template <typename P>
__device__ void rank1_rows(const P& p, int64_t n0, int64_t n1, const uint8_t* s_codes, const uint8_t* s_scales,
                           float s_mu) {
  constexpr int RW = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float s = __fmul_rn(s_mu, __ldg(p.w_ts));
  const int64_t nb = p.C / 16;
  const int64_t nch = (nb + 1) / 2;  // 32-element chunks (the last may hold one block)
  for (int64_t nr = n0 + RW * warp; nr < n1; nr += RW * 8) {
    float acc[RW];
#pragma unroll
    for (int i = 0; i < RW; ++i) acc[i] = 0.f;
    for (int64_t j = lane; j < nch; j += 32) {
      const bool two = 2 * j + 1 < nb;
      uint4 wc[RW];
      uint32_t wsc[RW];
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        const int64_t n = min(nr + i, n1 - 1);
        const uint8_t* wrow = p.w_codes + n * p.w_ld + 16 * j;
        wc[i] = !AVERIS_DBG_IN(p.err, wrow, p.w_codes, p.w_rows * p.w_ld, two ? 16 : 8, kSiteRank1Weight)
                    ? make_uint4(0u, 0u, 0u, 0u)
                : two ? __ldg(reinterpret_cast<const uint4*>(wrow))
                      : make_uint4(__ldg(reinterpret_cast<const uint32_t*>(wrow)),
                                   __ldg(reinterpret_cast<const uint32_t*>(wrow + 4)), 0u, 0u);
        // blocks 2j, 2j+1 of a row sit in adjacent bytes of one scale atom
        const uint8_t* sp = p.w_scales + scale_offset(n, 2 * j, p.w_kc);
        wsc[i] = !AVERIS_DBG_IN(p.err, sp, p.w_scales, 512 * ((p.w_rows + 127) / 128) * p.w_kc, two ? 2 : 1,
                                kSiteRank1Weight)
                     ? 0u
                 : two ? __ldg(reinterpret_cast<const uint16_t*>(sp)) : __ldg(sp);
      }
      const uint4 mc = two ? *reinterpret_cast<const uint4*>(s_codes + 16 * j)
                           : make_uint4(*reinterpret_cast<const uint32_t*>(s_codes + 16 * j),
                                        *reinterpret_cast<const uint32_t*>(s_codes + 16 * j + 4), 0u, 0u);
      uint32_t m0[8], m1[8];
      e2m1x8_to_h2(mc.x, *reinterpret_cast<uint32_t(*)[4]>(&m0[0]));
      e2m1x8_to_h2(mc.y, *reinterpret_cast<uint32_t(*)[4]>(&m0[4]));
      e2m1x8_to_h2(mc.z, *reinterpret_cast<uint32_t(*)[4]>(&m1[0]));
      e2m1x8_to_h2(mc.w, *reinterpret_cast<uint32_t(*)[4]>(&m1[4]));
      const float ms0 = e4m3_value(s_scales[2 * j]);
      const float ms1 = two ? e4m3_value(s_scales[2 * j + 1]) : 0.f;
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        acc[i] = fmaf(dot16_h2(m0, wc[i].x, wc[i].y), __fmul_rn(e4m3_value(wsc[i] & 0xFFu), ms0), acc[i]);
        if (two) acc[i] = fmaf(dot16_h2(m1, wc[i].z, wc[i].w), __fmul_rn(e4m3_value(wsc[i] >> 8), ms1), acc[i]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int i = 0; i < RW; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
    }
    if (lane < RW && nr + lane < n1) {
      float v = acc[0];
#pragma unroll
      for (int i = 1; i < RW; ++i)
        if (lane == i) v = acc[i];
      if (AVERIS_DBG_IN(p.err, p.r_out + nr + lane, p.r_out, p.w_rows * 4, 4, kSiteRank1Out)) p.r_out[nr + lane] = v * s;
    }
  }
}

// ------------------------------------------------------------ pass 2 ----

struct QuantParams {
  int64_t R, C;
  const float* mu;  // null: no split (r = x)
  // quantized mean (split): [1, C]
  uint8_t* mu_codes;
  uint8_t* mu_scales;
  float* mu_ts;
  float* mu_hat;    // [C] dequantized, unrotated
  int64_t mu_kc;    // ceil(C / 64)
  unsigned* ctrl;
  int* err;
  int hadamard;
  // blocked along C: [R, C]
  uint8_t* row_codes;
  uint8_t* row_scales;
  float* row_ts;
  int64_t row_ld, row_kc;
  // blocked along R: [C, R]
  uint8_t* col_codes;
  uint8_t* col_scales;
  float* col_ts;
  int64_t col_ld, col_kc;
  int tiles_r, tiles_c;
  // CTAs [0, mean_ctas) quantize the mean and compute the rank-one row; the
  // rest quantize tiles
  int mean_ctas;
  long long wait_limit;  // bound of every wait, in SM clock cycles
  int64_t row_base;      // first row of these R rows in the tensor map (a group of a grouped input)
  // optional rank-one row (split only): r[N] = deq(mu_q) deq(W)^T, with W an
  // NVFP4 [N, C] tensor blocked along C (the blocking of the mean)
  const uint8_t* w_codes;
  const uint8_t* w_scales;
  const float* w_ts;
  int64_t w_rows, w_ld, w_kc;
  float* r_out;
};

constexpr int kQTile = 128;
constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr int kQBufs = 3;                         // tile buffers per CTA
constexpr int kQCtasPerSm = 2;                    // resident CTAs per SM (registers, SMEM)
constexpr int kQHalf = kQTile * 64 * 2;          // one 128-row x 64-column bf16 box (16 KB)
constexpr int kQTileBytes = 2 * kQHalf;           // 32 KB
// SMEM: tile buffers | mu [kQBufs][128] | inverse-scale tables [2][128] |
// scale-atom staging [kQBufs][row atoms 1 KB | column atoms 1 KB] | barriers, counters
constexpr int kQOffMu = kQBufs * kQTileBytes;
constexpr int kQOffInv = kQOffMu + kQBufs * 128 * 4;
constexpr int kQOffStage = kQOffInv + 2 * 128 * 4;
constexpr int kQStageBytes = 2048;
constexpr int kQOffBar = kQOffStage + kQBufs * kQStageBytes;
constexpr int kQSmem = kQOffBar + 64 + 1024;      // + alignment slack

// inv(e) = min(fl32(1 / fl32(e4m3(e) s_g)), FLT_MAX), or 0 when the decode scale is 0.
__device__ __forceinline__ float inv_scale_of(uint32_t e, float s_g) {
  const float sb = __fmul_rn(e4m3_value(e), s_g);
  return sb > 0.f ? fminf(__frcp_rn(sb), FLT_MAX) : 0.f;
}

__device__ __forceinline__ float absmax16(const float (&r)[16]) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    a0 = fmaxf(a0, fabsf(r[e]));
    a1 = fmaxf(a1, fabsf(r[e + 1]));
  }
  return fmaxf(a0, a1);
}

// Eight binary32 values (four packed pairs, element 0 in the low half of q[0])
// -> eight E2M1 codes in one word, element 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8(uint64_t q0, uint64_t q1, uint64_t q2, uint64_t q3) {
  uint32_t out;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n .reg .f32 l0, h0, l1, h1, l2, h2, l3, h3;\n"
      " mov.b64 {l0, h0}, %1;\n mov.b64 {l1, h1}, %2;\n mov.b64 {l2, h2}, %3;\n mov.b64 {l3, h3}, %4;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(out)
      : "l"(q0), "l"(q1), "l"(q2), "l"(q3));
  return out;
}

// NVFP4 of one 16-element block with a per-tensor table of reciprocal decode
// scales (same binary32 steps as quant_block16).  Returns the E4M3 code.
__device__ __forceinline__ uint32_t quant16_tab(const float (&r)[16], float den, bool s_pos, const float* inv_tab,
                                                uint32_t& lo, uint32_t& hi) {
  const float a = absmax16(r);
  const uint32_t code = s_pos ? ptx::cvt_e4m3(__fdiv_rn(a, den)) : 0u;
  const float inv = inv_tab[code];
  const uint64_t inv2 = f2pack(inv, inv);
  uint64_t q[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) q[e] = mul2(f2pack(r[2 * e], r[2 * e + 1]), inv2);
  lo = e2m1x8(q[0], q[1], q[2], q[3]);
  hi = e2m1x8(q[4], q[5], q[6], q[7]);
  return code;
}

// One 128 x 128 tile, both layouts, by one warp: warp w owns tile rows
// 32(w/2) .. +31 of the 64-column half w%2 (exactly one TMA box).  The box
// sits in SMEM as 128 rows x 128 bytes, 16-byte chunk j of row r at chunk
// j ^ (r % 8) (the TMA 128-byte swizzle).
//
// Blocks along C (row layout): lane = (block kb = lane % 4, row rs = lane / 4);
// rows rs, rs + 8, rs + 16, rs + 24 of the warp's 32.  A quarter-warp reads
// 2 rows x 4 blocks: 8 distinct chunk positions, no bank conflict.
// Blocks along R (column layout): lane = (column quad cq = lane % 16, row
// block rb = lane / 16); 4 columns x 16 rows.  Each half-warp reads one full
// 128-byte row per load: no bank conflict.
// Codes go to global memory directly; block scales to the SMEM staging of
// this buffer (the tile fills exactly two 512-byte atoms of each layout).
// EDGE: the tile crosses row R or column C (masked, zero-filled blocks).
template <bool AMAX_ONLY, bool HAD, bool EDGE>
__device__ __forceinline__ void quant_tile_warp(const QuantParams& p, const uint8_t* buf, const float* mub,
                                                uint8_t* stage, int64_t r0, int64_t c0, float den_row, float den_col,
                                                bool pos_row, bool pos_col, const float* inv_s, bool rows_on,
                                                bool cols_on, float& amax_row, float& amax_col) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = w & 1, rq = w >> 1;
  const uint8_t* hb = buf + half * kQHalf;
  const float* mh = mub + 64 * half;
  const int64_t ch = c0 + 64 * half;  // first column of the half
  if (rows_on) {
    const int kb = lane & 3, rs = lane >> 2;
    uint64_t m2[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 m4 = *reinterpret_cast<const float4*>(mh + 16 * kb + 4 * k);
      m2[2 * k] = f2pack(m4.x, m4.y);
      m2[2 * k + 1] = f2pack(m4.z, m4.w);
    }
    const bool cvalid = !EDGE || ch + 16 * kb < p.C;
#pragma unroll 2
    for (int i = 0; i < 4; ++i) {
      const int row = 32 * rq + rs + 8 * i;
      const int64_t gr = r0 + row;
      const uint4 v0 = *reinterpret_cast<const uint4*>(hb + row * 128 + (((2 * kb) ^ (row & 7)) << 4));
      const uint4 v1 = *reinterpret_cast<const uint4*>(hb + row * 128 + (((2 * kb + 1) ^ (row & 7)) << 4));
      const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      const bool valid = !EDGE || (cvalid && gr < p.R);
      float rx[16];
      if constexpr (HAD) {
        // residual pairs (k, k + 8), then the packed butterfly
        uint64_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = k >> 1;
          const bool h = (k & 1) != 0;
          pk[k] = bf_pair_sub2(wv[e], wv[e + 4], h, h ? f2hi(m2[e]) : f2lo(m2[e]),
                               h ? f2hi(m2[e + 4]) : f2lo(m2[e + 4]));
          if (EDGE && !valid) pk[k] = 0ull;
        }
        fwht16_x2(pk);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          rx[2 * e] = f2lo(pk[e]);
          rx[2 * e + 1] = f2hi(pk[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint64_t d = bf2_sub_f2(wv[e], m2[e]);
          rx[2 * e] = f2lo(d);
          rx[2 * e + 1] = f2hi(d);
        }
        if (EDGE && !valid) {
#pragma unroll
          for (int e = 0; e < 16; ++e) rx[e] = 0.f;
        }
      }
      if (AMAX_ONLY) {
        amax_row = fmaxf(amax_row, absmax16(rx));
      } else {
        uint32_t lo, hi;
        const uint32_t sc = quant16_tab(rx, den_row, pos_row, inv_s, lo, hi);
        if (valid && AVERIS_DBG_IN(p.err, p.row_codes + gr * p.row_ld + ch / 2 + 8 * kb, p.row_codes, p.R * p.row_ld, 8,
                                   kSiteRowCodes))
          *reinterpret_cast<uint2*>(p.row_codes + gr * p.row_ld + ch / 2 + 8 * kb) = make_uint2(lo, hi);
        stage[half * 512 + 16 * (row & 31) + 4 * (row >> 5) + kb] = (uint8_t)sc;
      }
    }
  }
  if (cols_on) {
    const int cq = lane & 15, rb = lane >> 4;
    const int row0 = 32 * rq + 16 * rb;  // first tile row of this lane's blocks
    const float4 m4 = *reinterpret_cast<const float4*>(mh + 4 * cq);
    const float mc[4] = {m4.x, m4.y, m4.z, m4.w};
    uint2 x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int row = row0 + e;
      x[e] = *reinterpret_cast<const uint2*>(hb + row * 128 + (((cq >> 1) ^ (row & 7)) << 4) + 8 * (cq & 1));
    }
    const int64_t off = (r0 + row0) / 2;  // code byte offset of the block within a column
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int cc = 64 * half + 4 * cq + j;  // tile column
      const bool cvalid = !EDGE || c0 + cc < p.C;
      float rx[16];
      if constexpr (HAD) {
        // residual pairs (rows k, k + 8), then the packed butterfly
        uint64_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t wa = (j >> 1) ? x[k].y : x[k].x;
          const uint32_t wb = (j >> 1) ? x[k + 8].y : x[k + 8].x;
          pk[k] = bf_pair_sub(wa, wb, (j & 1) != 0, mc[j]);
          if (EDGE) {
            const float lo = !cvalid || r0 + row0 + k >= p.R ? 0.f : f2lo(pk[k]);
            const float hi = !cvalid || r0 + row0 + k + 8 >= p.R ? 0.f : f2hi(pk[k]);
            pk[k] = f2pack(lo, hi);
          }
        }
        fwht16_x2(pk);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          rx[2 * e] = f2lo(pk[e]);
          rx[2 * e + 1] = f2hi(pk[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const uint32_t wa = (j >> 1) ? x[e].y : x[e].x;
          const uint32_t wb = (j >> 1) ? x[e + 1].y : x[e + 1].x;
          const uint64_t d = bf_pair_sub(wa, wb, (j & 1) != 0, mc[j]);
          rx[e] = f2lo(d);
          rx[e + 1] = f2hi(d);
        }
        if (EDGE) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (!cvalid || r0 + row0 + e >= p.R) rx[e] = 0.f;
        }
      }
      if (AMAX_ONLY) {
        amax_col = fmaxf(amax_col, absmax16(rx));
      } else {
        uint32_t lo, hi;
        const uint32_t sc = quant16_tab(rx, den_col, pos_col, inv_s + 128, lo, hi);
        if (cvalid && (!EDGE || off < p.col_ld) &&
            AVERIS_DBG_IN(p.err, p.col_codes + (c0 + cc) * p.col_ld + off, p.col_codes, p.C * p.col_ld, 8, kSiteColCodes))
          *reinterpret_cast<uint2*>(p.col_codes + (c0 + cc) * p.col_ld + off) = make_uint2(lo, hi);
        stage[1024 + (rq >> 1) * 512 + 16 * (cc & 31) + 4 * (cc >> 5) + 2 * (rq & 1) + rb] = (uint8_t)sc;
      }
    }
  }
}

// Split + quantize, both layouts from one read of each 128 x 128 tile.
// Persistent CTAs with kQBufs tile buffers, each filled by TMA together with
// the tile's 128 mean values (bulk copy) on one mbarrier.  Every warp does
// the same share of every tile (both layouts of a 32 x 64 sub-tile) and
// counts itself done in the buffer's counter; the warp that completes the
// count writes the tile's four staged scale atoms and refills the buffer.
// Dedicated CTAs quantize the mean and compute the rank-one row; the last
// CTA to finish resets the control block's maxima.  AMAX_ONLY: compute the
// rotated residual's per-layout maximum magnitude (Hadamard variant)
// instead of quantizing.
// The pass of CTA `cta` of the `ncta` CTAs given to one tensor (or group).
template <bool AMAX_ONLY, bool HAD>
__device__ __forceinline__ void split_quant_body(const CUtensorMap& tmX, const QuantParams& p, int cta, int ncta) {
  extern __shared__ uint8_t qraw[];
  uint8_t* sm = qraw + ((1024u - (ptx::smem_u32(qraw) & 1023u)) & 1023u);  // stays a shared-space pointer
  float* mu_s = reinterpret_cast<float*>(sm + kQOffMu);
  float* inv_s = reinterpret_cast<float*>(sm + kQOffInv);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kQOffBar);
  int* done = reinterpret_cast<int*>(sm + kQOffBar + 8 * kQBufs);
  __shared__ float red[8];

  const int tid = threadIdx.x, lane = tid & 31;
  const int ntiles = p.tiles_r * p.tiles_c;
  const bool split = p.mu != nullptr;
  const bool mean_cta = cta < p.mean_ctas;
  const int tcta = cta - p.mean_ctas, ntcta = ncta - p.mean_ctas;  // tile CTA index, count
  const bool rows_on = AMAX_ONLY || p.row_codes != nullptr;
  const bool cols_on = AMAX_ONLY || p.col_codes != nullptr;

  auto mu_bytes = [&](int tile) {
    const int64_t left = p.C - (int64_t)(tile % p.tiles_c) * kQTile;
    return (uint32_t)(left < kQTile ? left : kQTile) * 4u;
  };
  auto issue_x = [&](int tile, int b) {
    const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
    ptx::mbar_arrive_expect_tx(&full[b], (uint32_t)kQTileBytes + (split ? mu_bytes(tile) : 0u));
    const int32_t y = (int32_t)(p.row_base + (int64_t)tr * kQTile);
    // the last read of X in this call (the stats pass kept it in L2)
    const uint64_t last_use = ptx::l2_policy_evict_first();
    if (!AVERIS_DBG_TMA_X(p.err, (int64_t)tc * kQTile, 2)) return;
    ptx::tma_load_2d_hint(sm + b * kQTileBytes, &tmX, tc * kQTile, y, &full[b], last_use);
    ptx::tma_load_2d_hint(sm + b * kQTileBytes + kQHalf, &tmX, tc * kQTile + 64, y, &full[b], last_use);
  };
  auto issue_mu = [&](int tile, int b) {
    if (split) ptx::bulk_load(mu_s + 128 * b, p.mu + (int64_t)(tile % p.tiles_c) * kQTile, mu_bytes(tile), &full[b]);
  };
  if (tid < kQBufs) done[tid] = 0;
  if (!split)
    for (int k = tid; k < kQBufs * 128; k += kQThreads) mu_s[k] = 0.f;  // x - 0 = x exactly
  if (tid == 0) {
    for (int b = 0; b < kQBufs; ++b) ptx::mbar_init(&full[b], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmX);
    // the input was written before the previous kernel started: fetch while it finishes
    if (!mean_cta)
      for (int b = 0; b < kQBufs; ++b)
        if (tcta + b * ntcta < ntiles) issue_x(tcta + b * ntcta, b);
  }
  ptx::pdl_wait_and_release();
  if (tid == 0 && !mean_cta)
    for (int b = 0; b < kQBufs; ++b)
      if (tcta + b * ntcta < ntiles) issue_mu(tcta + b * ntcta, b);  // the mean comes from the stats pass

  float s_row = 0.f, s_col = 0.f;
  if (!AMAX_ONLY) {
    // tensor scales from the maxima of the stats pass (or of the rotated-maximum pass)
    s_row = tensor_scale_of(__uint_as_float(__ldcg(&p.ctrl[p.hadamard ? kCtrlAmaxRowH : kCtrlAmaxRes])));
    s_col = tensor_scale_of(__uint_as_float(__ldcg(&p.ctrl[p.hadamard ? kCtrlAmaxColH : kCtrlAmaxRes])));
    if (tid < 128) {
      inv_s[tid] = tid < 127 ? inv_scale_of(tid, s_row) : 0.f;
      inv_s[128 + tid] = tid < 127 ? inv_scale_of(tid, s_col) : 0.f;
    }
    if (cta == 0 && tid == 0) {
      if (p.row_ts) *p.row_ts = s_row;
      if (p.col_ts) *p.col_ts = s_col;
    }
  }
  __syncthreads();  // tables, counters, barrier init
  const float den_row = __fmul_rn(6.0f, s_row), den_col = __fmul_rn(6.0f, s_col);
  float amax_row = 0.f, amax_col = 0.f;
  if (!AMAX_ONLY && split && mean_cta) {
    // the mean as NVFP4 (CTA 0 writes it out) and this CTA's share of the rank-one row
    uint8_t* s_codes = sm;                        // tile buffers are unused in a mean CTA
    uint8_t* s_scales = sm + kQOffMu - kQBufs * kQTileBytes / 4;
    const float s_mu = quantize_mean(p, cta == 0, s_codes, s_scales, red);
    if (p.r_out != nullptr) {
      const int64_t per = (p.w_rows + p.mean_ctas - 1) / p.mean_ctas;
      const int64_t n0 = (int64_t)cta * per;
      rank1_rows(p, n0, min(p.w_rows, n0 + per), s_codes, s_scales, s_mu);
    }
  }

  int i = 0;
  bool failed = false;
  for (int tile = mean_cta ? ntiles : tcta; tile < ntiles; tile += ntcta, ++i) {
    const int b = i % kQBufs;
    const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
    const int64_t r0 = (int64_t)tr * kQTile, c0 = (int64_t)tc * kQTile;
    if (!ptx::mbar_wait(&full[b], (uint32_t)((i / kQBufs) & 1), p.wait_limit)) {
      if (lane == 0) atomicExch(p.err, kErrQuantLoad);
      failed = true;
      break;
    }
    const uint8_t* buf = sm + b * kQTileBytes;
    uint8_t* stage = sm + kQOffStage + b * kQStageBytes;
    const float* mub = mu_s + 128 * b;
    if (r0 + kQTile > p.R || c0 + kQTile > p.C)
      quant_tile_warp<AMAX_ONLY, HAD, true>(p, buf, mub, stage, r0, c0, den_row, den_col, s_row > 0.f, s_col > 0.f, inv_s,
                                       rows_on, cols_on, amax_row, amax_col);
    else
      quant_tile_warp<AMAX_ONLY, HAD, false>(p, buf, mub, stage, r0, c0, den_row, den_col, s_row > 0.f, s_col > 0.f,
                                        inv_s, rows_on, cols_on, amax_row, amax_col);
    // count this warp done with the buffer; the last of the kQWarps writes the
    // staged scale atoms, then refills the buffer (its own reads are done too)
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(&done[b], 1) == kQWarps - 1;
      if (last) {
        done[b] = 0;
        __threadfence_block();
      }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __syncwarp();
      if (!AMAX_ONLY) {
        // 4 atoms x 512 B: row layout (row chunk tr, column chunks 2tc, 2tc+1),
        // column layout (row chunk tc, column chunks 2tr, 2tr+1)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const bool is_col = a >= 2;
          const int64_t kc = (is_col ? 2 * (int64_t)tr : 2 * (int64_t)tc) + (a & 1);
          const bool on = is_col ? (p.col_codes != nullptr && kc < p.col_kc) : (p.row_codes != nullptr && kc < p.row_kc);
          if (on) {
            uint8_t* dst = is_col ? p.col_scales + ((int64_t)tc * p.col_kc + kc) * 512
                                  : p.row_scales + ((int64_t)tr * p.row_kc + kc) * 512;
            if (AVERIS_DBG_IN(p.err, dst + 16 * lane, is_col ? p.col_scales : p.row_scales,
                              is_col ? 512 * ((p.C + 127) / 128) * p.col_kc : 512 * ((p.R + 127) / 128) * p.row_kc, 16,
                              kSiteScaleAtoms))
              *reinterpret_cast<uint4*>(dst + 16 * lane) = *reinterpret_cast<const uint4*>(stage + 512 * a + 16 * lane);
          }
        }
        __syncwarp();
      }
      if (lane == 0 && tile + kQBufs * ntcta < ntiles) {
        issue_x(tile + kQBufs * ntcta, b);
        issue_mu(tile + kQBufs * ntcta, b);
      }
    }
  }
  if (failed && tid == 0) {
    // this call's results are invalid; let the tiles already requested for this
    // CTA's buffers land (bounded) before its shared memory is given up
    for (int j = i; j < i + kQBufs; ++j)
      if (tcta + j * ntcta < ntiles) ptx::mbar_wait(&full[j % kQBufs], (uint32_t)((j / kQBufs) & 1), p.wait_limit);
  }
  if (AMAX_ONLY) {
    // rotated maxima, read by the quantize pass that follows
    amax_row = block_max256(amax_row, red);
    amax_col = block_max256(amax_col, red);
    if (tid == 0) {
      atomicMax(&p.ctrl[kCtrlAmaxRowH], __float_as_uint(amax_row));
      atomicMax(&p.ctrl[kCtrlAmaxColH], __float_as_uint(amax_col));
    }
  } else {
    // every CTA has read the maxima: the last one to finish resets them
    __shared__ int s_last;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned t = atomicAdd(&p.ctrl[kCtrlQuantTicket], 1u);
      s_last = (t == (unsigned)ncta - 1);
      if (s_last) {
        p.ctrl[kCtrlAmaxRes] = 0u;
        p.ctrl[kCtrlAmaxRowH] = 0u;
        p.ctrl[kCtrlAmaxColH] = 0u;
        p.ctrl[kCtrlQuantTicket] = 0u;
      }
    }
  }
}

template <bool AMAX_ONLY, bool HAD>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    split_quant_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ QuantParams p) {
  split_quant_body<AMAX_ONLY, HAD>(tmX, p, blockIdx.x, gridDim.x);
}

// The quantize pass over the row groups of a grouped input: g[e] holds group
// e's rows, outputs and control words, and its CTAs are its mean CTAs and its
// tile CTAs (below).
struct GroupedQuantParams {
  QuantParams g[kMaxGroups];
  // the launch's CTAs: first the mean CTAs of every group (group e: mcta0[e] ..
  // mcta0[e+1]-1), then the tile CTAs (group e: mcta0[ngroups] + cta0[e] ..
  // mcta0[ngroups] + cta0[e+1]-1); in a group the mean CTAs come first too
  int cta0[kMaxGroups + 1];
  int mcta0[kMaxGroups + 1];
  int ngroups;
};

// kernel parameters are limited to 32764 bytes (with the tensor map)
static_assert(sizeof(GroupedQuantParams) + sizeof(CUtensorMap) <= 32000, "grouped quantize parameters too large");
static_assert(sizeof(GroupedStatsParams) + sizeof(CUtensorMap) <= 32000, "grouped stats parameters too large");

template <bool AMAX_ONLY, bool HAD>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    split_quant_grouped_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ GroupedQuantParams gp) {
  // all groups' mean CTAs run in the first wave and then make room for tile CTAs,
  // which thus mostly start together instead of the last groups' starting late
  const int nmean = gp.mcta0[gp.ngroups];
  const int b = (int)blockIdx.x;
  int e = 0;
  if (b < nmean) {
    while (e + 1 < gp.ngroups && gp.mcta0[e + 1] <= b) ++e;
  } else {
    while (e + 1 < gp.ngroups && gp.cta0[e + 1] <= b - nmean) ++e;
  }
  const int means = gp.mcta0[e + 1] - gp.mcta0[e];
  const int cta = b < nmean ? b - gp.mcta0[e] : means + (b - nmean - gp.cta0[e]);
  split_quant_body<AMAX_ONLY, HAD>(tmX, gp.g[e], cta, means + gp.cta0[e + 1] - gp.cta0[e]);
}

// ------------------------------------------------ single-read quantize ----
//
// For inputs whose 128 x 128 tiles all fit the tile buffers of one wave of
// CTAs (2 per SM x kQBufs each: about 29 MB of bf16 on a B300), one
// cooperative launch reads every tile of X from HBM once and keeps it in
// shared memory: (1) column partials of each resident tile (compensated sum,
// max, min) into the workspace; a grid-wide wait; (2) each CTA combines a
// share of the columns (the same binary32 hi + lo arithmetic as the stats
// pass) into mu and the residual's maximum magnitude; a grid-wide wait; (3)
// the quantize pass of the two-launch path, tile by tile, from the resident
// tiles, with the mean CTAs quantizing the mean and computing the rank-one
// row.  Grid-wide waits count arrivals in the control block, bounded; the
// last CTA resets the words.  No rotation (the Hadamard variant needs the
// rotated maxima first and keeps the two-launch path).

struct ResidentParams {
  QuantParams q;     // the quantize pass's parameters (outputs, mean, rank-one row, control block)
  float* mu;         // [C] out (split; q.mu is the same pointer), null without the split
  ColPartial* part;  // [tiles_r][C] column partials of each tile
  long long grid_wait_limit;  // bound of each grid-wide wait, in SM clock cycles
  int starve;        // diagnostics only: request no tiles, so that every wait for one runs out
};

// the column partials of one tile ([4 row quarters][128 columns] float4) reuse
// the mean / table / staging area, which the quantize phase fills only later
static_assert(kQOffMu + 4 * 128 * 16 <= kQOffBar, "tile partials do not fit the staging area");

// Column partials of one resident tile (all 256 threads): thread t sums the
// column pair 2(t % 64), 2(t % 64) + 1 over rows 32(t / 64) .. +31 (groups of 8
// rows added pairwise, then compensated, as in the stats pass); the four row
// quarters are combined as hi + lo pairs in a fixed order.  Rows at or past R
// count neither in the sum nor in the extremes.
__device__ __forceinline__ void resident_tile_stats(const uint8_t* buf, float4* scratch, int64_t r0, int64_t c0,
                                                    int64_t R, int64_t C, ColPartial* part_row,
                                                    [[maybe_unused]] const ColPartial* part,
                                                    [[maybe_unused]] int64_t part_extent, [[maybe_unused]] int* err) {
  const int tid = threadIdx.x;
  const int cp = tid & 63, rq = tid >> 6;
  const uint8_t* hb = buf + (cp >> 5) * kQHalf;
  const int w = cp & 31;  // word of the column pair in the 128-byte box row
  const int64_t rows_left = R - r0;
  uint64_t s2 = 0ull, c2 = 0ull;
  uint32_t mx2 = 0xFF80FF80u, mn2 = 0x7F807F80u;  // -inf, +inf
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t xs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int row = 32 * rq + 8 * g + j;
      const uint32_t v = *reinterpret_cast<const uint32_t*>(hb + row * 128 + ((((w >> 2) ^ (row & 7))) << 4) + 4 * (w & 3));
      const bool valid = row < rows_left;
      mx2 = bmax2(mx2, valid ? v : 0xFF80FF80u);
      mn2 = bmin2(mn2, valid ? v : 0x7F807F80u);
      xs[j] = valid ? v : 0u;  // +0 + +0: adds nothing
    }
    const uint64_t t = add2(add2(add2(bf2_to_f2(xs[0]), bf2_to_f2(xs[1])), add2(bf2_to_f2(xs[2]), bf2_to_f2(xs[3]))),
                            add2(add2(bf2_to_f2(xs[4]), bf2_to_f2(xs[5])), add2(bf2_to_f2(xs[6]), bf2_to_f2(xs[7]))));
    const uint64_t y = sub2(t, c2);
    const uint64_t tt = add2(s2, y);
    c2 = sub2(sub2(tt, s2), y);
    s2 = tt;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float sv = h ? f2hi(s2) : f2lo(s2), cv = h ? f2hi(c2) : f2lo(c2);
    const F2 d = fast_two_sum(sv, -cv);
    scratch[rq * 128 + 2 * cp + h] =
        make_float4(d.hi, d.lo, h ? bf16hi(mx2) : bf16lo(mx2), h ? bf16hi(mn2) : bf16lo(mn2));
  }
  __syncthreads();
  if (tid < 128 && c0 + tid < C) {
    float4 q = scratch[tid];
    F2 acc{q.x, q.y};
    float m1 = q.z, m2 = q.w;
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      q = scratch[k * 128 + tid];
      acc = df_add(acc, F2{q.x, q.y});
      m1 = fmaxf(m1, q.z);
      m2 = fminf(m2, q.w);
    }
    if (AVERIS_DBG_IN(err, part_row + c0 + tid, part, part_extent, 16, kSiteResidentPart))
      *reinterpret_cast<float4*>(part_row + c0 + tid) = make_float4(acc.hi, acc.lo, m1, m2);
  }
  __syncthreads();  // scratch is free for the next tile
}

// Columns [c_begin, c_end) of the tiles' partials -> mu (split) and this
// CTA's share of the residual's maximum magnitude.  One warp per column:
// lanes add the tile rows lane, lane + 32, ... in order, then a fixed
// butterfly over the lanes.  All 256 threads call it; returns the maximum
// (valid in every thread).
__device__ __forceinline__ float resident_combine(const QuantParams& p, const ColPartial* part, float* mu_out,
                                                  int64_t c_begin, int64_t c_end, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tiles_r = p.tiles_r;
  const float Rf = (float)p.R;
  float a_res = 0.f;
  for (int64_t c = c_begin + warp; c < c_end; c += 8) {
    F2 acc{0.f, 0.f};
    float m1 = -FLT_MAX, m2 = FLT_MAX;
    for (int j = lane; j < tiles_r; j += 32) {
      const float4 q = AVERIS_DBG_IN(p.err, part + (int64_t)j * p.C + c, part, (int64_t)tiles_r * p.C * 16, 16,
                                     kSiteResidentPart)
                           ? __ldcg(reinterpret_cast<const float4*>(part + (int64_t)j * p.C + c))
                           : make_float4(0.f, 0.f, -FLT_MAX, FLT_MAX);
      acc = df_add(acc, F2{q.x, q.y});
      m1 = fmaxf(m1, q.z);
      m2 = fminf(m2, q.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const F2 other{__shfl_xor_sync(0xffffffffu, acc.hi, o), __shfl_xor_sync(0xffffffffu, acc.lo, o)};
      acc = (lane & o) ? df_add(other, acc) : df_add(acc, other);
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      m2 = fminf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
    }
    if (mu_out != nullptr) {
      const float mu = df_div_count(acc, Rf);
      if (lane == 0 && AVERIS_DBG_IN(p.err, mu_out + c, mu_out, p.C * 4, 4, kSiteStatsMean)) mu_out[c] = mu;
      a_res = fmaxf(a_res, fmaxf(fabsf(__fsub_rn(m1, mu)), fabsf(__fsub_rn(m2, mu))));
    } else {
      a_res = fmaxf(a_res, fmaxf(fabsf(m1), fabsf(m2)));
    }
  }
  return block_max256(a_res, red);
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* a) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// Grid-wide wait of the single-read quantize: every CTA adds one to the
// control word, then (when `wait`) waits until `target` arrivals are counted.
// A CTA that has already given up still arrives, so that the others are not
// held until their own limit.  Returns false (uniform over the CTA) when the
// wait ran out.
__device__ __forceinline__ bool resident_grid_wait(unsigned* ctrl, unsigned target, bool wait, long long limit,
                                                   int* s_ok) {
  __syncthreads();  // this CTA's writes are issued
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&ctrl[kCtrlGridBar], 1u);
    int ok = 1;
    if (wait) {
      const long long t0 = clock64();
      while (ld_acquire_gpu(&ctrl[kCtrlGridBar]) < target) {
        if (clock64() - t0 > limit) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
      __threadfence();
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    quantize_resident_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ ResidentParams rp) {
  const QuantParams& p = rp.q;
  extern __shared__ uint8_t qraw[];
  uint8_t* sm = qraw + ((1024u - (ptx::smem_u32(qraw) & 1023u)) & 1023u);  // stays a shared-space pointer
  float* mu_s = reinterpret_cast<float*>(sm + kQOffMu);
  float* inv_s = reinterpret_cast<float*>(sm + kQOffInv);
  float4* scratch = reinterpret_cast<float4*>(sm + kQOffMu);  // column partials of a tile, before mu_s is used
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kQOffBar);
  __shared__ float red[8];
  __shared__ int s_ok, s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int ntiles = p.tiles_r * p.tiles_c;
  const bool split = rp.mu != nullptr;
  const bool mean_cta = cta < p.mean_ctas;
  const int tcta = cta - p.mean_ctas, ntcta = ncta - p.mean_ctas;  // tile CTA index, count
  int nmine = 0;  // this CTA's tiles: tcta, tcta + ntcta, ... (buffer k holds the k-th)
  if (!mean_cta)
    while (nmine < kQBufs && tcta + nmine * ntcta < ntiles) ++nmine;

  if (tid == 0) {
    for (int b = 0; b < kQBufs; ++b) ptx::mbar_init(&full[b], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmX);
  }
  __syncthreads();
  // X may come from the kernel just before this one: load it after the wait
  ptx::pdl_wait_and_release();
  if (tid == 0 && !rp.starve) {
    const uint64_t once = ptx::l2_policy_evict_first();  // the only read of X
    for (int k = 0; k < nmine; ++k) {
      const int tile = tcta + k * ntcta;
      const int32_t x0 = (tile % p.tiles_c) * kQTile, y = (tile / p.tiles_c) * kQTile;
      ptx::mbar_arrive_expect_tx(&full[k], (uint32_t)kQTileBytes);
      ptx::tma_load_2d_hint(sm + k * kQTileBytes, &tmX, x0, y, &full[k], once);
      ptx::tma_load_2d_hint(sm + k * kQTileBytes + kQHalf, &tmX, x0 + 64, y, &full[k], once);
    }
  }

  // (1) column partials of each resident tile
  bool failed = false;
  int landed = 0;  // tiles known to have arrived
  for (; landed < nmine; ++landed) {
    if (!__syncthreads_and(ptx::mbar_wait(&full[landed], 0u, p.wait_limit) ? 1 : 0)) {
      if (tid == 0) atomicExch(p.err, kErrQuantLoad);
      failed = true;
      break;
    }
    const int tile = tcta + landed * ntcta;
    const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
    resident_tile_stats(sm + landed * kQTileBytes, scratch, (int64_t)tr * kQTile, (int64_t)tc * kQTile, p.R, p.C,
                        rp.part + (int64_t)tr * p.C, rp.part, (int64_t)p.tiles_r * p.C * 16, p.err);
  }
  if (!resident_grid_wait(p.ctrl, (unsigned)ncta, !failed, rp.grid_wait_limit, &s_ok) && !failed) {
    if (tid == 0) atomicCAS(p.err, 0, kErrQuantGrid);  // keep the cause if another CTA reported one
    failed = true;
  }

  // (2) mu and the residual's maximum over this CTA's share of the columns
  if (!failed) {
    const int64_t per = (p.C + ncta - 1) / ncta;
    const int64_t c_begin = min(p.C, (int64_t)cta * per), c_end = min(p.C, c_begin + per);
    const float a_res = resident_combine(p, rp.part, rp.mu, c_begin, c_end, red);
    if (tid == 0) atomicMax(&p.ctrl[kCtrlAmaxRes], __float_as_uint(a_res));
  }
  if (!resident_grid_wait(p.ctrl, 2u * (unsigned)ncta, !failed, rp.grid_wait_limit, &s_ok) && !failed) {
    if (tid == 0) atomicCAS(p.err, 0, kErrQuantGrid);
    failed = true;
  }

  // (3) the quantize pass over the resident tiles, the mean and the rank-one row
  if (!failed) {
    const float amax = __uint_as_float(__ldcg(&p.ctrl[kCtrlAmaxRes]));
    const float s_g = tensor_scale_of(amax);  // one tensor scale for both layouts (no rotation)
    if (tid < 128) {
      const float inv = tid < 127 ? inv_scale_of(tid, s_g) : 0.f;
      inv_s[tid] = inv;
      inv_s[128 + tid] = inv;
    }
    if (cta == 0 && tid == 0) {
      if (p.row_ts) *p.row_ts = s_g;
      if (p.col_ts) *p.col_ts = s_g;
    }
    for (int k = 0; k < nmine; ++k) {
      const int64_t c0 = (int64_t)((tcta + k * ntcta) % p.tiles_c) * kQTile;
      if (tid < 128) mu_s[128 * k + tid] = split && c0 + tid < p.C ? __ldcg(rp.mu + c0 + tid) : 0.f;  // x - 0 = x
    }
    __syncthreads();
    if (split && mean_cta) {
      uint8_t* s_codes = sm;  // a mean CTA holds no tiles
      uint8_t* s_scales = sm + kQOffMu - kQBufs * kQTileBytes / 4;
      const float s_mu = quantize_mean(p, cta == 0, s_codes, s_scales, red);
      if (p.r_out != nullptr) {
        const int64_t per = (p.w_rows + p.mean_ctas - 1) / p.mean_ctas;
        const int64_t n0 = (int64_t)cta * per;
        rank1_rows(p, n0, min(p.w_rows, n0 + per), s_codes, s_scales, s_mu);
      }
    }
    const float den = __fmul_rn(6.0f, s_g);
    const bool rows_on = p.row_codes != nullptr, cols_on = p.col_codes != nullptr;
    float unused_r = 0.f, unused_c = 0.f;
    for (int k = 0; k < nmine; ++k) {
      const int tile = tcta + k * ntcta;
      const int64_t r0 = (int64_t)(tile / p.tiles_c) * kQTile, c0 = (int64_t)(tile % p.tiles_c) * kQTile;
      const uint8_t* buf = sm + k * kQTileBytes;
      uint8_t* stage = sm + kQOffStage + k * kQStageBytes;
      if (r0 + kQTile > p.R || c0 + kQTile > p.C)
        quant_tile_warp<false, false, true>(p, buf, mu_s + 128 * k, stage, r0, c0, den, den, s_g > 0.f, s_g > 0.f,
                                            inv_s, rows_on, cols_on, unused_r, unused_c);
      else
        quant_tile_warp<false, false, false>(p, buf, mu_s + 128 * k, stage, r0, c0, den, den, s_g > 0.f, s_g > 0.f,
                                             inv_s, rows_on, cols_on, unused_r, unused_c);
    }
    __syncthreads();  // every warp's scale atoms are staged
    // 4 atoms x 512 B per tile: row layout (row chunk tr, column chunks 2tc,
    // 2tc+1), column layout (row chunk tc, column chunks 2tr, 2tr+1)
    for (int a = warp; a < 4 * nmine; a += kQWarps) {
      const int k = a >> 2, tile = tcta + k * ntcta;
      const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
      const bool is_col = (a & 2) != 0;
      const int64_t kc = (is_col ? 2 * (int64_t)tr : 2 * (int64_t)tc) + (a & 1);
      const bool on = is_col ? (cols_on && kc < p.col_kc) : (rows_on && kc < p.row_kc);
      if (on) {
        uint8_t* dst = is_col ? p.col_scales + ((int64_t)tc * p.col_kc + kc) * 512
                              : p.row_scales + ((int64_t)tr * p.row_kc + kc) * 512;
        if (AVERIS_DBG_IN(p.err, dst + 16 * lane, is_col ? p.col_scales : p.row_scales,
                          is_col ? 512 * ((p.C + 127) / 128) * p.col_kc : 512 * ((p.R + 127) / 128) * p.row_kc, 16,
                          kSiteScaleAtoms))
          *reinterpret_cast<uint4*>(dst + 16 * lane) =
              *reinterpret_cast<const uint4*>(sm + kQOffStage + k * kQStageBytes + 512 * (a & 3) + 16 * lane);
      }
    }
  }

  // (4) a CTA that gave up lets the tiles it requested land (bounded) before
  // its shared memory is given up; the last CTA resets the control words
  if (failed && tid == 0 && !rp.starve)
    for (int k = landed; k < nmine; ++k) ptx::mbar_wait(&full[k], 0u, p.wait_limit);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned t = atomicAdd(&p.ctrl[kCtrlQuantTicket], 1u);
    s_last = (t == (unsigned)ncta - 1);
    if (s_last) {
      p.ctrl[kCtrlAmaxRes] = 0u;
      p.ctrl[kCtrlGridBar] = 0u;
      p.ctrl[kCtrlQuantTicket] = 0u;
    }
  }
}

// --------------------------------------------------------- rank-one GEMV --

// out[r] = s_mu s_w sum_k e2m1(mu_k) e4m3(mu scale) e2m1(w_rk) e4m3(w scale);
// one warp per output row, fixed reduction order.
__global__ void __launch_bounds__(256) rank1_gemv_kernel(const uint8_t* __restrict__ mu_codes,
                                                         const uint8_t* __restrict__ mu_scales,
                                                         const float* __restrict__ mu_ts,
                                                         const uint8_t* __restrict__ w_codes,
                                                         const uint8_t* __restrict__ w_scales,
                                                         const float* __restrict__ w_ts, int64_t w_ld, int64_t N,
                                                         int64_t K, int64_t kc, float* __restrict__ out,
                                                         [[maybe_unused]] int* err) {
  __shared__ float lut[16];
  ptx::pdl_wait_and_release();
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_val(threadIdx.x);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= N) return;
  const int64_t nb = K / 16;
  float acc = 0.f;
  for (int64_t b = lane; b < nb; b += 32) {
    const uint2 wc = *reinterpret_cast<const uint2*>(w_codes + r * w_ld + 8 * b);
    const uint2 mc = *reinterpret_cast<const uint2*>(mu_codes + 8 * b);
    const float sc = e4m3_value(w_scales[scale_offset(r, b, kc)]) * e4m3_value(mu_scales[scale_offset(0, b, kc)]);
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      part += lut[(wc.x >> (4 * e)) & 15u] * lut[(mc.x >> (4 * e)) & 15u];
      part += lut[(wc.y >> (4 * e)) & 15u] * lut[(mc.y >> (4 * e)) & 15u];
    }
    acc += part * sc;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && AVERIS_DBG_IN(err, out + r, out, N * 4, 4, kSiteGemvOut)) out[r] = (acc * __ldg(mu_ts)) * __ldg(w_ts);
}

}  // namespace averis
