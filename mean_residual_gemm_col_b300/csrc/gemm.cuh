// Block-scaled NVFP4 GEMM on the 5th-generation tensor cores (tcgen05) with
// the Averis epilogue.
//
//   out[i][j] = s_a s_b * sum_k A[i][k] B[j][k] + col_add[j] + outer * u[i] v[j]
//
// A [M, K] and B [N, K] are NVFP4 (E2M1 codes, E4M3 scale per 16 along K);
// the broadcast term col_add is the 1 (mu_bar W_bar) / 1 (mu_bar_D W_bar^T)
// row of the forward and input-gradient equations, and outer * u v^T is the
// l mu_bar_X^T mu_bar_D term of the weight gradient (paper.rainbus.top
// summary "均值偏置的诅咒与祝福：FP4量化大语言模型训练", section 方法步骤详情;
// the mean term is broadcast, never materialised: paperlayer.ai summary,
// section 3 Method).
//
// Design: persistent CTAs (one per SM), 128 x 256 output tiles (M fastest,
// so CTAs running together share B tiles in L2), K tiles of 256 elements
// (128 bytes of codes per row), a 3-deep shared-memory ring.  Warp roles:
//   warp 0     TMA producer: codes by 2-D tensor TMA (128-byte swizzle),
//              block scales by 1-D bulk copies.
//   warp 1     TMEM owner and MMA issuer: tcgen05.mma kind::mxf4nvf4
//              128x256x64 accumulating in TMEM; tcgen05.commit frees the
//              stage and, after the last K tile, hands the accumulator to
//              the epilogue.
//   warps 2-9  epilogue, two per TMEM lane quarter (warp % 4), each
//              draining half of the accumulator columns: tcgen05.ld 32
//              columns at a time, alpha scaling and the rank-one terms in
//              binary32 (vector entries staged once per tile in SMEM and read
//              as broadcasts), SMEM staging (128-byte swizzle), TMA tensor
//              stores (which clip ragged edges).
//   warps 10-13 scale feed: each writes a whole stage's block scales into
//              its TMEM lane quarter with two tcgen05.st (registers -> TMEM),
//              the same words a 32x128b.warpx4 copy of each SMEM scale atom
//              would place there (lane 32 w + i, columns base_g .. +3 = atom
//              row i).  This keeps the tensor pipe free of the 12 SMEM->TMEM
//              copies per stage that would otherwise issue between the MMAs
//              (each costs about as much tensor-pipe time as an MMA).
// One 256-column accumulator leaves TMEM room for the scale stages.  With a
// bf16 output the epilogue moves the accumulator into registers (packed
// bf16) and releases TMEM before storing, so the next tile's MMAs
// overlap the stores.  Every wait is bounded; on timeout the kernel sets the
// error word, drains its own tensor-core work and frees its TMEM.  Launched
// with programmatic dependent launch: set-up runs before the wait for the
// previous kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace averis {

struct GemmParams {
  int M, N, K;
  int kc;        // ceil(K / 64): 64-element scale chunks per row chunk (same for A and B)
  int rb_b;      // ceil(N / 128): row chunks of B's scales
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ts_a;
  const float* ts_b;
  const float* col_add;  // [N] or null
  const float* row_vec;  // [M] or null
  const float* col_vec;  // [N] or null
  float outer;
  int* err;
  // 1: none of this GEMM's inputs comes from the kernel launched just before
  // it (the library issues it right after an independent GEMM): start at
  // once, and wait for that kernel only before exiting, so that this
  // kernel's completion still implies the previous one's.
  int early_start;
};


struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 256;
  static constexpr int BKB = 128;  // bytes of codes per row per K tile (256 elements)
  static constexpr int STAGES = 3;
  static constexpr int A_BYTES = BM * BKB;
  static constexpr int B_BYTES = BN * BKB;
  static constexpr int SFA_BYTES = 4 * 512;
  static constexpr int SFB_BYTES = (BN / 128) * 4 * 512;
  static constexpr int EPI_WARPS = 8;             // 2 per TMEM lane quarter, each half of the columns
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // accumulator columns per epilogue warp
  static constexpr int EPI_NBUF = EPI_WARPS == 4 ? 2 : 1;  // staging boxes per epilogue warp
  static constexpr int EPI_BUF = 32 * 128;        // one warp's 32 rows x 128 bytes
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_NBUF * EPI_BUF;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int OFF_VEC = OFF_EPI + EPI_BYTES;  // [2 tile parities][col_add, col_vec][BN] floats
  static constexpr int OFF_BAR = OFF_VEC + 2 * 2 * BN * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + alignment slack
  // TMEM columns: the accumulator, then per stage 16 SFA columns + BN/8 SFB columns
  static constexpr int SF_BASE = BN;
  static constexpr int SFB_COLS_PER_STEP = BN / 32;
  static constexpr int SF_STAGE_COLS = 16 + 4 * SFB_COLS_PER_STEP;
  static constexpr int TMEM_COLS = 512;
  static_assert(OFF_EPI % 1024 == 0, "epilogue staging must be 1024-byte aligned");
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM overflow");
  static_assert(SMEM <= 227 * 1024, "shared memory overflow");
  // instruction descriptor: E2M1 x E2M1 (format 1), K-major A and B, UE4M3 scales,
  // N >> 3 at bit 17, M >> 4 at bit 24
  static constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

// Epilogue value of one accumulator column chunk: alpha * acc + col_add + rterm * col_vec.
// `cadd`/`cvec` point at the chunk's 32 vector entries in SMEM (broadcast reads).
__device__ __forceinline__ void epi_math(float (&f)[32], const float (&acc)[32], bool has_add, const float* cadd,
                                         bool has_outer, float rterm, const float* cvec) {
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 a4 = has_add ? *reinterpret_cast<const float4*>(cadd + 4 * j4) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 v4 = has_outer ? *reinterpret_cast<const float4*>(cvec + 4 * j4) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x = acc[4 * j4 + k];
      if (has_add) x += a[k];
      if (has_outer) x = fmaf(rterm, v[k], x);
      f[4 * j4 + k] = x;
    }
  }
}

// Named barrier of the four epilogue warps (ids 1 and up are free for this).
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * GemmCfg::EPI_WARPS) : "memory");
}

// warps: producer, MMA issuer, GemmCfg::EPI_WARPS epilogue warps, 4 scale-feed warps
constexpr int kGemmThreads = 32 * (2 + GemmCfg::EPI_WARPS + 4);

template <bool BF16_OUT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using Cfg = GemmCfg;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* smem = gsm_raw + ((1024u - (ptx::smem_u32(gsm_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* sf_full = drain + 1;            // [STAGES]: the stage's scales are in TMEM
  uint64_t* sf_loaded = sf_full + STAGES;  // [STAGES]: the stage's scale atoms are in SMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_loaded + STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&sf_full[s], 4);
      ptx::mbar_init(&sf_loaded[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(tempty, Cfg::EPI_WARPS);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // operands, scales and epilogue vectors may come from the previous kernel
  if (p.early_start)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  else
    ptx::pdl_wait_and_release();

  const int num_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int num_n = (p.N + BN - 1) / BN;
  const int ntiles = num_m * num_n;
  const int nkt = (p.kc + 3) / 4;
  // output tile `tile` -> (mt, nt), M fastest; every tile runs over all K tiles
  auto decode = [&](int tile, int& mt, int& nt, int& kt0, int& kt1) {
    mt = tile % num_m;
    nt = tile / num_m;
    kt0 = 0;
    kt1 = nkt;
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        int mt, nt, kt0, kt1;
        decode(tile, mt, nt, kt0, kt1);
        int nsfb = 0;
#pragma unroll
        for (int h = 0; h < BN / 128; ++h) nsfb += (nt * (BN / 128) + h) < p.rb_b ? 1 : 0;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, kWaitLimit)) {
            atomicExch(p.err, kErrProducer);
            goto done;
          }
          const int ns = min(4, p.kc - 4 * kt);
          // the small scale atoms first, on their own barrier: the scale warps
          // move them into TMEM while the operand tiles are still arriving
          ptx::mbar_arrive_expect_tx(&sf_loaded[stage], (uint32_t)ns * 512u * (1u + (uint32_t)nsfb));
          ptx::bulk_load(smem + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES, p.sfa + ((int64_t)mt * p.kc + 4 * kt) * 512,
                         ns * 512u, &sf_loaded[stage]);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            const int rb = nt * (BN / 128) + h;
            if (rb < p.rb_b)
              ptx::bulk_load(smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES + h * 2048,
                             p.sfb + ((int64_t)rb * p.kc + 4 * kt) * 512, ns * 512u, &sf_loaded[stage]);
          }
          ptx::mbar_arrive_expect_tx(&full[stage], (uint32_t)(Cfg::A_BYTES + Cfg::B_BYTES));
          ptx::tma_load_2d(smem + Cfg::OFF_A + stage * Cfg::A_BYTES, &tmA, kt * Cfg::BKB, mt * Cfg::BM, &full[stage]);
          ptx::tma_load_2d(smem + Cfg::OFF_B + stage * Cfg::B_BYTES, &tmB, kt * Cfg::BKB, nt * BN, &full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool issued = false;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        int mt, nt, kt0, kt1;
        decode(tile, mt, nt, kt0, kt1);
        if (!ptx::mbar_wait(tempty, (it & 1) ^ 1u, kWaitLimit)) {
          atomicExch(p.err, kErrMma);
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kt = kt0; kt < kt1; ++kt) {
          // operand tiles in SMEM, scales in TMEM
          if (!ptx::mbar_wait(&full[stage], phase, kWaitLimit) || !ptx::mbar_wait(&sf_full[stage], phase, kWaitLimit)) {
            atomicExch(p.err, kErrMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int ns = min(4, p.kc - 4 * kt);
          const uint32_t sfa_t = tmem + (uint32_t)(Cfg::SF_BASE + stage * Cfg::SF_STAGE_COLS);
          const uint32_t sfb_t = sfa_t + 16u;
          const uint32_t a_s = ptx::smem_u32(smem + Cfg::OFF_A + stage * Cfg::A_BYTES);
          const uint32_t b_s = ptx::smem_u32(smem + Cfg::OFF_B + stage * Cfg::B_BYTES);
          for (int g = 0; g < ns; ++g) {
            const uint64_t adesc = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
            const uint64_t bdesc = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
            ptx::tc_mma_nvf4(tmem, adesc, bdesc, Cfg::IDESC, sfa_t + 4u * g,
                             sfb_t + (uint32_t)(Cfg::SFB_COLS_PER_STEP * g), (kt != kt0 || g != 0) ? 1u : 0u);
          }
          issued = true;
          ptx::tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit(tfull);
      }
      if (issued) {
        // drain: every MMA and copy this thread issued has completed
        ptx::tc_commit(drain);
        if (!ptx::mbar_wait(drain, 0, kWaitLimit)) atomicExch(p.err, kErrDrain);
      }
    }
  } else if (warp >= 2 + Cfg::EPI_WARPS) {
    // scale feed: every lane quarter q = warp % 4 gets the same words: lane
    // 32 q + i, columns 4 g .. 4 g + 3 (A chunk g) and 16 + 8 g + 4 h .. +3
    // (B half h, chunk g) = row i of that 512-byte SMEM atom, whose word j
    // holds the 4 block scales of row i + 32 j.
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      int mt, nt, kt0, kt1;
      decode(tile, mt, nt, kt0, kt1);
      for (int kt = kt0; kt < kt1; ++kt) {
        if (!ptx::mbar_wait(&sf_loaded[stage], phase, kWaitLimit)) {
          if (lane == 0) atomicExch(p.err, kErrScaleFeed);
          goto done;
        }
        const uint8_t* sa = smem + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES + 16 * lane;
        const uint8_t* sb = smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES + 16 * lane;
        uint32_t ra[16], rb[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(sa + 512 * g);
          ra[4 * g] = v.x;
          ra[4 * g + 1] = v.y;
          ra[4 * g + 2] = v.z;
          ra[4 * g + 3] = v.w;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 v = *reinterpret_cast<const uint4*>(sb + 2048 * h + 512 * g);
            rb[8 * g + 4 * h] = v.x;
            rb[8 * g + 4 * h + 1] = v.y;
            rb[8 * g + 4 * h + 2] = v.z;
            rb[8 * g + 4 * h + 3] = v.w;
          }
        const uint32_t t = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(Cfg::SF_BASE + stage * Cfg::SF_STAGE_COLS);
        ptx::tmem_st16(t, ra);
        ptx::tmem_st32(t + 16u, rb);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sf_full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // epilogue warps: TMEM lane quarter (warp % 4) holds tile rows 32*(warp%4) .. +31;
    // warp 2 + 4 k + .. drains accumulator columns EPI_COLS * k .. +EPI_COLS - 1
    const int q = warp & 3;
    const int cb = Cfg::EPI_COLS * ((warp - 2) >> 2);  // this warp's first column
    const int et = threadIdx.x - 64;  // 0 .. 32 EPI_WARPS - 1 over the epilogue warps
    const float alpha = __ldg(p.ts_a) * __ldg(p.ts_b);
    const bool has_add = p.col_add != nullptr;
    const bool has_outer = p.row_vec != nullptr;
    uint8_t* stage_base = smem + Cfg::OFF_EPI + (warp - 2) * Cfg::EPI_NBUF * Cfg::EPI_BUF;
    float* vec_base = reinterpret_cast<float*>(smem + Cfg::OFF_VEC);
    __shared__ int s_ok[2];
    int sbuf = 0;
    int it = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
      int mt, nt, kt0, kt1;
      decode(tile, mt, nt, kt0, kt1);
      const int row = mt * Cfg::BM + q * 32 + lane;
      const int row0 = mt * Cfg::BM + q * 32;
      const float rterm = (has_outer && row < p.M) ? p.outer * __ldg(p.row_vec + row) : 0.f;
      // this tile's vector entries -> SMEM (double-buffered by tile parity: a warp
      // reaches the next tile's writes only after every warp passed this barrier)
      float* cadd_s = vec_base + (it & 1) * 2 * BN;
      float* cvec_s = cadd_s + BN;
      for (int c = et; c < BN; c += 32 * Cfg::EPI_WARPS) {
        const int col = nt * BN + c;
        cadd_s[c] = (has_add && col < p.N) ? __ldg(p.col_add + col) : 0.f;
        cvec_s[c] = (has_outer && col < p.N) ? __ldg(p.col_vec + col) : 0.f;
      }
      // one thread waits for the accumulator; the barrier hands its verdict (and
      // the staged vectors) to all epilogue warps, so they leave the loop together
      if (et == 0) s_ok[it & 1] = ptx::mbar_wait(tfull, it & 1, kWaitLimit) ? 1 : 0;
      epi_bar();
      if (!s_ok[it & 1]) {
        if (et == 0) atomicExch(p.err, kErrEpilogue);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);

      // stage one 32-row x 128-byte box in swizzled SMEM and store it with TMA
      auto store_box = [&](const uint4 (&w)[8], int col0) {
        uint8_t* sb = stage_base + sbuf * Cfg::EPI_BUF;
        if (lane == 0) ptx::bulk_wait_read<Cfg::EPI_NBUF - 1>();
        __syncwarp();
        uint8_t* srow = sb + lane * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(srow + ((k ^ (lane & 7)) * 16)) = w[k];
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmD, sb, col0, row0);
          ptx::bulk_commit();
        }
        sbuf = (sbuf + 1) % Cfg::EPI_NBUF;
      };
      auto store_f32 = [&](const float (&f)[32], int c) {
        uint4 w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w[k] = make_uint4(__float_as_uint(f[4 * k]), __float_as_uint(f[4 * k + 1]), __float_as_uint(f[4 * k + 2]),
                            __float_as_uint(f[4 * k + 3]));
        store_box(w, nt * BN + c);
      };

      if (BF16_OUT) {
        // this warp's accumulator columns -> packed bf16 registers, release TMEM, then store
        uint32_t packed[Cfg::EPI_COLS / 2];
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + (uint32_t)(cb + c), v);
          ptx::tmem_ld_wait();
          float acc[32], f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = alpha * __uint_as_float(v[j]);
          epi_math(f, acc, has_add, cadd_s + cb + c, has_outer, rterm, cvec_s + cb + c);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
            packed[c / 2 + j] = *reinterpret_cast<uint32_t*>(&b2);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty);
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 64) {
          uint4 w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = make_uint4(packed[c / 2 + 4 * k], packed[c / 2 + 4 * k + 1], packed[c / 2 + 4 * k + 2],
                              packed[c / 2 + 4 * k + 3]);
          store_box(w, nt * BN + cb + c);
        }
      } else {
#pragma unroll 1
        for (int c = cb; c < cb + Cfg::EPI_COLS; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + (uint32_t)c, v);
          ptx::tmem_ld_wait();
          if (c + 32 == cb + Cfg::EPI_COLS) {
            // last chunk is in registers: the accumulator may be overwritten
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty);
          }
          float acc[32], f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = alpha * __uint_as_float(v[j]);
          epi_math(f, acc, has_add, cadd_s + c, has_outer, rterm, cvec_s + c);
          store_f32(f, c);
        }
      }
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }
done:
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
  if (p.early_start) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace averis
