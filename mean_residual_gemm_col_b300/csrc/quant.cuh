// Mean-split NVFP4 quantize pass and the rank-one GEMV.
//
// Pass 1  colstats_partial : per (row block, column) compensated sum, max, min
//                            of the bf16 input (one coalesced read).
// Pass 1b colstats_finalize: column mean mu (binary32), the residual's exact
//                            maximum magnitude, and -- in the last block to
//                            finish -- the NVFP4 quantization of mu itself.
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

// control words at the head of a quantize workspace
enum : int { kCtrlTicket = 0, kCtrlAmaxRow = 1, kCtrlAmaxCol = 2, kCtrlAmaxMu = 3, kCtrlWords = 64 };

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

// ------------------------------------------------------------ pass 1 ----

// grid (strips of 256 columns, row blocks); 256 threads.  Thread: 8 columns,
// rows warp, warp+8, ... of its row block, four rows per step.  The four rows
// are summed pairwise and the step sum is added with Kahan compensation.
__global__ void __launch_bounds__(256) colstats_partial_kernel(const __nv_bfloat16* __restrict__ x, int64_t R,
                                                               int64_t C, int64_t rows_per,
                                                               ColPartial* __restrict__ part,
                                                               unsigned* __restrict__ ctrl) {
  __shared__ double s_sum[8][256];
  __shared__ float s_mx[8][256], s_mn[8][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kCtrlWords) ctrl[threadIdx.x] = 0u;

  const int64_t c0 = (int64_t)blockIdx.x * 256 + lane * 8;
  const bool col_ok = c0 < C;
  const int64_t rb0 = (int64_t)blockIdx.y * rows_per;
  const int64_t rb1 = min(R, rb0 + rows_per);

  float s[8], c[8], mx[8], mn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    s[e] = 0.f;
    c[e] = 0.f;
    mx[e] = -FLT_MAX;
    mn[e] = FLT_MAX;
  }
  if (col_ok) {
    for (int64_t r = rb0 + warp; r < rb1; r += 32) {
      uint4 v[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t rr = r + 8 * j;
        ok[j] = rr < rb1;
        v[j] = ok[j] ? __ldg(reinterpret_cast<const uint4*>(x + rr * C + c0)) : make_uint4(0, 0, 0, 0);
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
        const float t = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
        const float y = __fsub_rn(t, c[e]);
        const float tt = __fadd_rn(s[e], y);
        c[e] = __fsub_rn(__fsub_rn(tt, s[e]), y);
        s[e] = tt;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    s_sum[warp][lane * 8 + e] = (double)s[e] - (double)c[e];
    s_mx[warp][lane * 8 + e] = mx[e];
    s_mn[warp][lane * 8 + e] = mn[e];
  }
  __syncthreads();
  const int64_t col = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (col < C) {
    double acc = 0.0;
    float m1 = -FLT_MAX, m2 = FLT_MAX;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      acc += s_sum[w][threadIdx.x];
      m1 = fmaxf(m1, s_mx[w][threadIdx.x]);
      m2 = fminf(m2, s_mn[w][threadIdx.x]);
    }
    ColPartial p;
    p.s_hi = (float)acc;
    p.s_lo = (float)(acc - (double)p.s_hi);
    p.mx = m1;
    p.mn = m2;
    part[(int64_t)blockIdx.y * C + col] = p;
  }
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

struct FinalizeParams {
  const ColPartial* part;
  int nrb;
  int64_t R, C;
  int split;     // mean split on
  int hadamard;  // rotation on (amax of the residual comes from the amax pass)
  float* mu;     // [C] out (split)
  unsigned* ctrl;
  // quantized mean (split): [1, C]
  uint8_t* mu_codes;
  uint8_t* mu_scales;
  float* mu_ts;
  float* mu_hat;  // [C] dequantized, unrotated
  int64_t kc;     // ceil(C/64)
};

// grid ceil(C/256) x 256 threads; thread = column.
__global__ void __launch_bounds__(256) colstats_finalize_kernel(FinalizeParams p) {
  __shared__ float red[8];
  __shared__ int s_last;
  const int64_t j = (int64_t)blockIdx.x * 256 + threadIdx.x;
  float a_col = 0.f, a_mu = 0.f;
  if (j < p.C) {
    double s = 0.0;
    float mx = -FLT_MAX, mn = FLT_MAX;
    for (int rb = 0; rb < p.nrb; ++rb) {
      const ColPartial q = p.part[(int64_t)rb * p.C + j];
      s += (double)q.s_hi + (double)q.s_lo;
      mx = fmaxf(mx, q.mx);
      mn = fminf(mn, q.mn);
    }
    if (p.split) {
      const float mu = (float)(s / (double)p.R);
      p.mu[j] = mu;
      a_col = fmaxf(fabsf(__fsub_rn(mx, mu)), fabsf(__fsub_rn(mn, mu)));
      a_mu = fabsf(mu);
    } else {
      a_col = fmaxf(fabsf(mx), fabsf(mn));
    }
  }
  __threadfence();  // publish mu before this block takes its ticket
  a_col = block_max256(a_col, red);
  a_mu = block_max256(a_mu, red);
  if (threadIdx.x == 0) {
    if (!p.hadamard) {
      atomicMax(&p.ctrl[kCtrlAmaxRow], __float_as_uint(a_col));
      atomicMax(&p.ctrl[kCtrlAmaxCol], __float_as_uint(a_col));
    }
    atomicMax(&p.ctrl[kCtrlAmaxMu], __float_as_uint(a_mu));
    __threadfence();
    const unsigned t = atomicAdd(&p.ctrl[kCtrlTicket], 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last || !p.split) return;
  __threadfence();

  // Last block: quantize mu along C as one row ([1, C]).  Under the
  // Hadamard variant mu is rotated block-wise first, and mu_hat is the
  // dequantized mean rotated back (H16/4 is its own inverse).
  const int64_t nb = p.C / 16;
  float amax_mu;
  if (!p.hadamard) {
    amax_mu = __uint_as_float(atomicAdd(&p.ctrl[kCtrlAmaxMu], 0u));
  } else {
    float a = 0.f;
    for (int64_t b = threadIdx.x; b < nb; b += 256) {
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
  if (threadIdx.x == 0) *p.mu_ts = s_g;
  for (int64_t b = threadIdx.x; b < nb; b += 256) {
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

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntiles = p.tiles_r * p.tiles_c;
  const bool split = p.mu != nullptr;
  const float s_row = AMAX_ONLY ? 0.f : tensor_scale_of(__uint_as_float(p.ctrl[kCtrlAmaxRow]));
  const float s_col = AMAX_ONLY ? 0.f : tensor_scale_of(__uint_as_float(p.ctrl[kCtrlAmaxCol]));
  if (!AMAX_ONLY && blockIdx.x == 0 && threadIdx.x == 0) {
    if (p.row_ts) *p.row_ts = s_row;
    if (p.col_ts) *p.col_ts = s_col;
  }
  float amax_row = 0.f, amax_col = 0.f;

  int buf = 0;
  if ((int)blockIdx.x < ntiles) quant_issue_tile(p, qsm, blockIdx.x);
  ptx::cp_async_commit();
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
    amax_row = block_max256(amax_row, red);
    amax_col = block_max256(amax_col, red);
    if (threadIdx.x == 0) {
      atomicMax(&p.ctrl[kCtrlAmaxRow], __float_as_uint(amax_row));
      atomicMax(&p.ctrl[kCtrlAmaxCol], __float_as_uint(amax_col));
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
