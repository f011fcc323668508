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

#include "ptx.cuh"

namespace averis {

// Control block at the head of every quantize workspace.  Every word below
// kCtrlScaleRow is zero at rest: the kernel that counts on a ticket or
// accumulates a maximum resets it before it finishes, so a workspace that
// starts zeroed stays usable for any later call without a memset.
enum : int {
  kCtrlTicket = 0,       // stats pass: strips finished
  kCtrlAmaxRow = 1,      // residual max magnitude, layout blocked along columns (float bits)
  kCtrlAmaxCol = 2,      // same, layout blocked along rows
  kCtrlAmaxMu = 3,       // max |mu|
  kCtrlAmaxTicket = 4,   // rotated-amax pass: CTAs finished
  kCtrlScaleRow = 8,     // tensor scales handed to the quantize pass (written every call)
  kCtrlScaleCol = 9,
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
  int64_t rows_per;   // rows per CTA row block (multiple of 128)
  int nstrips;        // ceil(C / 64) column strips of 64
  ColPartial* part;   // [gridDim.y][C] per-row-block partials
  unsigned* ctrl;
  int split;          // mean split on
  int hadamard;       // rotation on (the rotated residual's maximum comes from the amax pass)
  float* mu;          // [C] out (split)
  // quantized mean (split): [1, C]
  uint8_t* mu_codes;
  uint8_t* mu_scales;
  float* mu_ts;
  float* mu_hat;      // [C] dequantized, unrotated
  int64_t kc;         // ceil(C / 64)
};

// Column statistics in one pass over X, with the combine fused in.
//
// grid (strip groups, row blocks), 256 threads.  CTA (g, b) reads rows
// [b*rows_per, (b+1)*rows_per) of the 64-column strips g, g+gridDim.x, ...:
// thread t owns 8 adjacent columns (16-byte loads) of rows t/8, t/8+32, ...,
// keeps a Kahan-compensated binary32 sum plus max and min per column, and the
// 32 row lanes are combined in float64 in a fixed order.  The last CTA of a
// strip group to finish (ticket) combines the row-block partials of its
// strips in row-block order -- the result does not depend on which CTA is
// last -- giving mu_j = fl32(S_j / R) and the residual's exact maximum
// magnitude max(|fl32(max_j - mu_j)|, |fl32(min_j - mu_j)|) (binary32
// subtraction is monotone).  The last strip group overall turns the maxima
// into the two tensor scales and quantizes mu as a [1, C] NVFP4 row.
__global__ void __launch_bounds__(256) colstats_kernel(StatsParams p) {
  __shared__ double s_sum[8][64];
  __shared__ float s_mx[8][64], s_mn[8][64];
  __shared__ float red[8];
  __shared__ int s_last;
  ptx::pdl_wait_and_release();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = tid & 7;     // 8-column group inside the strip
  const int rl = tid >> 3;    // row lane 0..31
  const int64_t rb0 = (int64_t)blockIdx.y * p.rows_per;
  const int64_t rb1 = min(p.R, rb0 + p.rows_per);

  for (int strip = blockIdx.x; strip < p.nstrips; strip += gridDim.x) {
    const int64_t c0 = (int64_t)strip * 64 + 8 * g8;
    float s[8], c[8], mx[8], mn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s[e] = 0.f;
      c[e] = 0.f;
      mx[e] = -FLT_MAX;
      mn[e] = FLT_MAX;
    }
    if (c0 < p.C) {
      const __nv_bfloat16* base = p.x + c0;
      for (int64_t r = rb0 + rl; r < rb1; r += 128) {
        uint4 v[4];
        bool ok[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t rr = r + 32 * j;
          ok[j] = rr < rb1;
          v[j] = ok[j] ? __ldg(reinterpret_cast<const uint4*>(base + rr * p.C)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float a[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w = (e >> 1) == 0 ? v[j].x : (e >> 1) == 1 ? v[j].y : (e >> 1) == 2 ? v[j].z : v[j].w;
            a[j] = (e & 1) ? bf16hi(w) : bf16lo(w);
            if (ok[j]) {
              mx[e] = fmaxf(mx[e], a[j]);
              mn[e] = fminf(mn[e], a[j]);
            }
          }
          // rows that are out of range contribute an exact 0 to the sum
          const float t = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
          const float y = __fsub_rn(t, c[e]);
          const float tt = __fadd_rn(s[e], y);
          c[e] = __fsub_rn(__fsub_rn(tt, s[e]), y);
          s[e] = tt;
        }
      }
    }
    // combine the 4 row lanes of this warp that share the columns (lanes differ by 8, 16)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      double d = (double)s[e] - (double)c[e];
      d += __shfl_xor_sync(0xffffffffu, d, 8);
      d += __shfl_xor_sync(0xffffffffu, d, 16);
      float m1 = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 16));
      float m2 = fminf(mn[e], __shfl_xor_sync(0xffffffffu, mn[e], 8));
      m2 = fminf(m2, __shfl_xor_sync(0xffffffffu, m2, 16));
      if (lane < 8) {
        s_sum[warp][8 * lane + e] = d;
        s_mx[warp][8 * lane + e] = m1;
        s_mn[warp][8 * lane + e] = m2;
      }
    }
    __syncthreads();
    if (tid < 64) {
      const int64_t col = (int64_t)strip * 64 + tid;
      double acc = 0.0;
      float m1 = -FLT_MAX, m2 = FLT_MAX;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        acc += s_sum[w][tid];
        m1 = fmaxf(m1, s_mx[w][tid]);
        m2 = fminf(m2, s_mn[w][tid]);
      }
      if (col < p.C) {
        ColPartial q;
        q.s_hi = (float)acc;
        q.s_lo = (float)(acc - (double)q.s_hi);
        q.mx = m1;
        q.mn = m2;
        *reinterpret_cast<float4*>(p.part + (int64_t)blockIdx.y * p.C + col) = make_float4(q.s_hi, q.s_lo, q.mx, q.mn);
      }
    }
    __syncthreads();
  }

  // ---- last row block of this strip group combines the partials
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(&p.ctrl[kCtrlStrip + blockIdx.x], 1u);
    s_last = (t == gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  float a_res = 0.f, a_mu = 0.f;
  const int nrb = (int)gridDim.y;
  for (int strip = blockIdx.x; strip < p.nstrips; strip += gridDim.x) {
    const int cl = tid & 63, part = tid >> 6;
    const int64_t col = (int64_t)strip * 64 + cl;
    double acc = 0.0;
    float m1 = -FLT_MAX, m2 = FLT_MAX;
    if (col < p.C) {
      for (int rb = part; rb < nrb; rb += 4) {
        const float4 q = __ldcg(reinterpret_cast<const float4*>(p.part + (int64_t)rb * p.C + col));
        acc += (double)q.x + (double)q.y;
        m1 = fmaxf(m1, q.z);
        m2 = fminf(m2, q.w);
      }
    }
    s_sum[part][cl] = acc;
    s_mx[part][cl] = m1;
    s_mn[part][cl] = m2;
    __syncthreads();
    if (tid < 64 && col < p.C) {
      const double S = ((s_sum[0][cl] + s_sum[1][cl]) + s_sum[2][cl]) + s_sum[3][cl];
      const float M1 = fmaxf(fmaxf(s_mx[0][cl], s_mx[1][cl]), fmaxf(s_mx[2][cl], s_mx[3][cl]));
      const float M2 = fminf(fminf(s_mn[0][cl], s_mn[1][cl]), fminf(s_mn[2][cl], s_mn[3][cl]));
      if (p.split) {
        const float mu = (float)(S / (double)p.R);
        p.mu[col] = mu;
        a_res = fmaxf(a_res, fmaxf(fabsf(__fsub_rn(M1, mu)), fabsf(__fsub_rn(M2, mu))));
        a_mu = fmaxf(a_mu, fabsf(mu));
      } else {
        a_res = fmaxf(a_res, fmaxf(fabsf(M1), fabsf(M2)));
      }
    }
    __syncthreads();
  }
  if (tid == 0) p.ctrl[kCtrlStrip + blockIdx.x] = 0u;  // every row block has arrived: reset for the next call
  a_res = block_max256(a_res, red);
  a_mu = block_max256(a_mu, red);
  __threadfence();  // publish mu before taking the overall ticket
  if (tid == 0) {
    if (!p.hadamard) {
      atomicMax(&p.ctrl[kCtrlAmaxRow], __float_as_uint(a_res));
      atomicMax(&p.ctrl[kCtrlAmaxCol], __float_as_uint(a_res));
    }
    atomicMax(&p.ctrl[kCtrlAmaxMu], __float_as_uint(a_mu));
    __threadfence();
    const unsigned t = atomicAdd(&p.ctrl[kCtrlTicket], 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last strip group overall: tensor scales, reset, quantize mu
  __shared__ float s_amax_mu;
  if (tid == 0) {
    if (!p.hadamard) {
      const float ar = __uint_as_float(atomicExch(&p.ctrl[kCtrlAmaxRow], 0u));
      const float ac = __uint_as_float(atomicExch(&p.ctrl[kCtrlAmaxCol], 0u));
      p.ctrl[kCtrlScaleRow] = __float_as_uint(tensor_scale_of(ar));
      p.ctrl[kCtrlScaleCol] = __float_as_uint(tensor_scale_of(ac));
    }
    s_amax_mu = __uint_as_float(atomicExch(&p.ctrl[kCtrlAmaxMu], 0u));
    p.ctrl[kCtrlTicket] = 0u;
    __threadfence();
  }
  __syncthreads();
  if (!p.split) return;

  // Quantize mu along C as one row ([1, C]).  Under the Hadamard variant mu
  // is rotated block-wise first, and mu_hat is the dequantized mean rotated
  // back (H16/4 is its own inverse).
  const int64_t nb = p.C / 16;
  float amax_mu = s_amax_mu;
  if (p.hadamard) {
    float a = 0.f;
    for (int64_t b = tid; b < nb; b += 256) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __ldcg(p.mu + 16 * b + e);
      fwht16(v);
#pragma unroll
      for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(v[e]));
    }
    amax_mu = block_max256(a, red);
  }
  const float s_g = tensor_scale_of(amax_mu);
  if (tid == 0) *p.mu_ts = s_g;
  for (int64_t b = tid; b < nb; b += 256) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __ldcg(p.mu + 16 * b + e);
    if (p.hadamard) fwht16(v);
    const BlockQ q = quant_block16(v, s_g);
    *reinterpret_cast<uint2*>(p.mu_codes + 8 * b) = make_uint2(q.lo, q.hi);
    p.mu_scales[scale_offset(0, b, p.kc)] = (uint8_t)q.scale;
    const float sc = e4m3_value(q.scale);
    float d[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c4 = ((e < 8 ? q.lo : q.hi) >> (4 * (e & 7))) & 15u;
      d[e] = __fmul_rn(__fmul_rn(e2m1_val(c4), sc), s_g);
    }
    if (p.hadamard) fwht16(d);
#pragma unroll
    for (int e = 0; e < 16; ++e) p.mu_hat[16 * b + e] = d[e];
  }
}

// ------------------------------------------------------------ pass 2 ----

struct QuantParams {
  const __nv_bfloat16* x;
  int64_t R, C;
  const float* mu;  // null: no split (r = x)
  unsigned* ctrl;
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
};

constexpr int kQTile = 128;
constexpr int kQThreads = 256;
// smem: 2 x bf16 tile (64 KB) + column-layout code staging (8 KB) + scale staging (2 KB)
constexpr int kQSmemTile = kQTile * kQTile * 2;
constexpr int kQSmem = 2 * kQSmemTile + kQTile * 64 + 2048 + 64;

// 16-byte chunk k (0..15) of a 256-byte tile row lives at chunk k ^ ((k >> 3) & 1):
// row-wise 32-byte reads and column-wise reads are then conflict-free.
__device__ __forceinline__ int qswz(int k) { return k ^ ((k >> 3) & 1); }

__device__ __forceinline__ void quant_issue_tile(const QuantParams& p, uint8_t* buf, int tile) {
  const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
  const int64_t r0 = (int64_t)tr * kQTile, c0 = (int64_t)tc * kQTile;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int q = threadIdx.x + kQThreads * i;
    const int row = q >> 4, k = q & 15;
    const int64_t gr = r0 + row, gc = c0 + 8 * k;
    const bool ok = gr < p.R && gc < p.C;
    const __nv_bfloat16* src = ok ? p.x + gr * p.C + gc : p.x;
    ptx::cp_async16(buf + row * 256 + qswz(k) * 16, src, ok ? 16u : 0u);
  }
}

// AMAX_ONLY: compute the rotated residual's per-layout maximum magnitude
// (Hadamard variant) instead of quantizing.
template <bool AMAX_ONLY>
__global__ void __launch_bounds__(kQThreads, 2) split_quant_kernel(QuantParams p) {
  extern __shared__ __align__(128) uint8_t qsm[];
  uint8_t* cstage = qsm + 2 * kQSmemTile;                 // [128 rows][64 B], 8-byte granules swizzled
  uint8_t* sstage_row = cstage + kQTile * 64;             // 1 KB: 2 scale chunks of the row layout
  uint8_t* sstage_col = sstage_row + 1024;                // 1 KB: 2 scale chunks of the column layout
  __shared__ float red[8];

  __shared__ int s_last;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntiles = p.tiles_r * p.tiles_c;
  const bool split = p.mu != nullptr;

  // the input was written before the previous kernel started: fetch the
  // first tile while that kernel finishes
  int buf = 0;
  if ((int)blockIdx.x < ntiles) quant_issue_tile(p, qsm, blockIdx.x);
  ptx::cp_async_commit();
  ptx::pdl_wait_and_release();

  const float s_row = AMAX_ONLY ? 0.f : __uint_as_float(__ldcg(&p.ctrl[kCtrlScaleRow]));
  const float s_col = AMAX_ONLY ? 0.f : __uint_as_float(__ldcg(&p.ctrl[kCtrlScaleCol]));
  if (!AMAX_ONLY && blockIdx.x == 0 && threadIdx.x == 0) {
    if (p.row_ts) *p.row_ts = s_row;
    if (p.col_ts) *p.col_ts = s_col;
  }
  float amax_row = 0.f, amax_col = 0.f;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int next = tile + gridDim.x;
    if (next < ntiles) quant_issue_tile(p, qsm + (buf ^ 1) * kQSmemTile, next);
    ptx::cp_async_commit();
    ptx::cp_async_wait<1>();
    __syncthreads();

    const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
    const int64_t r0 = (int64_t)tr * kQTile, c0 = (int64_t)tc * kQTile;
    const uint8_t* t = qsm + buf * kQSmemTile;

    // ---- blocks along C (row layout): thread = (row, 16-column block), 4 per thread
    if (p.row_codes != nullptr || AMAX_ONLY) {
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int row = warp * 4 + (lane >> 3) + 32 * i;
        const int kb = lane & 7;
        const int64_t gr = r0 + row, gc = c0 + 16 * kb;
        const bool valid = gr < p.R && gc < p.C;
        const uint4 v0 = *reinterpret_cast<const uint4*>(t + row * 256 + qswz(2 * kb) * 16);
        const uint4 v1 = *reinterpret_cast<const uint4*>(t + row * 256 + qswz(2 * kb + 1) * 16);
        const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float r[16];
        if (valid) {
          if (split) {
            const float4* mp = reinterpret_cast<const float4*>(p.mu + gc);
            float mu[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float4 m4 = __ldg(mp + q4);
              mu[4 * q4] = m4.x;
              mu[4 * q4 + 1] = m4.y;
              mu[4 * q4 + 2] = m4.z;
              mu[4 * q4 + 3] = m4.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              r[2 * e] = __fsub_rn(bf16lo(wv[e]), mu[2 * e]);
              r[2 * e + 1] = __fsub_rn(bf16hi(wv[e]), mu[2 * e + 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              r[2 * e] = bf16lo(wv[e]);
              r[2 * e + 1] = bf16hi(wv[e]);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0.f;
        }
        if (p.hadamard) fwht16(r);
        if (AMAX_ONLY) {
#pragma unroll
          for (int e = 0; e < 16; ++e) amax_row = fmaxf(amax_row, fabsf(r[e]));
        } else {
          const BlockQ q = quant_block16(r, s_row);
          if (valid) *reinterpret_cast<uint2*>(p.row_codes + gr * p.row_ld + c0 / 2 + 8 * kb) = make_uint2(q.lo, q.hi);
          sstage_row[(kb >> 2) * 512 + 16 * (row & 31) + 4 * (row >> 5) + (kb & 3)] = (uint8_t)q.scale;
        }
      }
    }

    // ---- blocks along R (column layout): thread = (2 columns, 16-row block), 2 per thread
    if (p.col_codes != nullptr || AMAX_ONLY) {
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int cp = lane + 32 * (warp & 1);         // column pair 0..63
        const int rb = (warp >> 1) + 4 * i;            // 16-row block 0..7
        const int col = 2 * cp;
        const int64_t gc = c0 + col;
        const bool cvalid = gc < p.C;
        float mu0 = 0.f, mu1 = 0.f;
        if (split && cvalid) {
          const float2 m2 = __ldg(reinterpret_cast<const float2*>(p.mu + gc));
          mu0 = m2.x;
          mu1 = m2.y;
        }
        float ra[16], rbv[16];
        const int choff = qswz(col >> 3) * 16 + (col & 7) * 2;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = 16 * rb + e;
          const uint32_t w = *reinterpret_cast<const uint32_t*>(t + row * 256 + choff);
          const bool valid = cvalid && (r0 + row < p.R);
          if (valid) {
            ra[e] = split ? __fsub_rn(bf16lo(w), mu0) : bf16lo(w);
            rbv[e] = split ? __fsub_rn(bf16hi(w), mu1) : bf16hi(w);
          } else {
            ra[e] = 0.f;
            rbv[e] = 0.f;
          }
        }
        if (p.hadamard) {
          fwht16(ra);
          fwht16(rbv);
        }
        if (AMAX_ONLY) {
#pragma unroll
          for (int e = 0; e < 16; ++e) amax_col = fmaxf(amax_col, fmaxf(fabsf(ra[e]), fabsf(rbv[e])));
        } else {
          const BlockQ qa = quant_block16(ra, s_col);
          const BlockQ qb = quant_block16(rbv, s_col);
          *reinterpret_cast<uint2*>(cstage + col * 64 + 8 * (rb ^ (col & 7))) = make_uint2(qa.lo, qa.hi);
          *reinterpret_cast<uint2*>(cstage + (col + 1) * 64 + 8 * (rb ^ ((col + 1) & 7))) = make_uint2(qb.lo, qb.hi);
          sstage_col[(rb >> 2) * 512 + 16 * (col & 31) + 4 * (col >> 5) + (rb & 3)] = (uint8_t)qa.scale;
          sstage_col[(rb >> 2) * 512 + 16 * ((col + 1) & 31) + 4 * ((col + 1) >> 5) + (rb & 3)] = (uint8_t)qb.scale;
        }
      }
    }
    __syncthreads();

    if (!AMAX_ONLY) {
      // column-layout codes: row (c0 + c) bytes r0/2 .. r0/2+63, four 8-byte granules per thread
      if (p.col_codes != nullptr) {
        const int c = threadIdx.x >> 1, half = threadIdx.x & 1;
        const int64_t grow = c0 + c;
        if (grow < p.C) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t boff = r0 / 2 + 32 * half + 16 * h;
            if (boff < p.col_ld) {
              const int g0 = 4 * half + 2 * h;
              const uint2 a = *reinterpret_cast<const uint2*>(cstage + c * 64 + 8 * (g0 ^ (c & 7)));
              const uint2 b = *reinterpret_cast<const uint2*>(cstage + c * 64 + 8 * ((g0 + 1) ^ (c & 7)));
              *reinterpret_cast<uint4*>(p.col_codes + grow * p.col_ld + boff) = make_uint4(a.x, a.y, b.x, b.y);
            }
          }
        }
        // scale chunks of the column layout: row chunk tc, chunks 2*tr, 2*tr+1
        if (threadIdx.x < 64) {
          const int ch = threadIdx.x >> 5;
          const int64_t kc = 2 * (int64_t)tr + ch;
          if (kc < p.col_kc)
            *reinterpret_cast<uint4*>(p.col_scales + ((int64_t)tc * p.col_kc + kc) * 512 + 16 * (threadIdx.x & 31)) =
                *reinterpret_cast<const uint4*>(sstage_col + 16 * threadIdx.x);
        }
      }
      if (p.row_codes != nullptr && threadIdx.x >= 64 && threadIdx.x < 128) {
        const int tt = threadIdx.x - 64, ch = tt >> 5;
        const int64_t kc = 2 * (int64_t)tc + ch;
        if (kc < p.row_kc)
          *reinterpret_cast<uint4*>(p.row_scales + ((int64_t)tr * p.row_kc + kc) * 512 + 16 * (tt & 31)) =
              *reinterpret_cast<const uint4*>(sstage_row + 16 * tt);
      }
      __syncthreads();
    }
    buf ^= 1;
  }
  ptx::cp_async_wait<0>();
  if (AMAX_ONLY) {
    // rotated maxima -> tensor scales; the last CTA converts and resets
    amax_row = block_max256(amax_row, red);
    amax_col = block_max256(amax_col, red);
    if (threadIdx.x == 0) {
      atomicMax(&p.ctrl[kCtrlAmaxRow], __float_as_uint(amax_row));
      atomicMax(&p.ctrl[kCtrlAmaxCol], __float_as_uint(amax_col));
      __threadfence();
      const unsigned t = atomicAdd(&p.ctrl[kCtrlAmaxTicket], 1u);
      s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
      __threadfence();
      const float ar = __uint_as_float(atomicExch(&p.ctrl[kCtrlAmaxRow], 0u));
      const float ac = __uint_as_float(atomicExch(&p.ctrl[kCtrlAmaxCol], 0u));
      p.ctrl[kCtrlScaleRow] = __float_as_uint(tensor_scale_of(ar));
      p.ctrl[kCtrlScaleCol] = __float_as_uint(tensor_scale_of(ac));
      p.ctrl[kCtrlAmaxTicket] = 0u;
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
                                                         int64_t K, int64_t kc, float* __restrict__ out) {
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
  if (lane == 0) out[r] = (acc * __ldg(mu_ts)) * __ldg(w_ts);
}

}  // namespace averis
