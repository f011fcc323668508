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
// Design: pairs of CTAs (clusters of two on one TPC), persistent, one pair
// per two SMs.  A pair computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 64 per instruction): each
// CTA loads its own 128 rows of A and its own 128 rows of B (half of the
// tile's N), so every SM streams 32 KB of operands per 256-element K tile
// instead of the 48 KB a one-CTA 128 x 256 tile needs, and the shared-memory
// ring is deeper for the same capacity (5 stages).  A launch runs up to G GEMMs (the
// dW and dX of a layer, or the experts of a grouped layer), each with its own
// output type; every pair runs a contiguous range of work units (GEMM after
// GEMM, tiles M fastest), the ranges cut by the host so that the pairs' K
// tiles balance.  Warp roles, in each CTA:
//   warp 0     TMA producer: this CTA's A and B halves by 2-D tensor TMA
//              (128-byte swizzle), completing on the leader CTA's stage
//              barrier; block scales by 1-D bulk copies into its own SMEM.
//   warp 1     TMEM owner (both CTAs allocate together); in the leader CTA
//              also the MMA issuer.  tcgen05.commit multicast to both CTAs
//              frees a stage and hands the accumulator to both epilogues.
//   warps 2-9  epilogue, two per TMEM lane quarter, each draining half of the
//              256 accumulator columns of this CTA's 128 rows: tcgen05.ld,
//              alpha scaling and the rank-one terms in binary32 (vector
//              entries staged once per tile in SMEM), SMEM staging (128-byte
//              swizzle), TMA tensor stores (which clip ragged edges).
//   warps 10-13 scale feed: write each stage's block scales from SMEM into
//              this CTA's TMEM with tcgen05.st (the words a 32x128b.warpx4
//              copy of each scale atom would place), then arrive on the
//              leader's stage barrier, the one the operands complete on, so
//              the MMA thread waits once per stage and issues only MMAs.
// Every wait is bounded; on timeout the kernel sets the error word, lets its
// copies in flight land, drains its tensor-core work, and both CTAs meet at a
// cluster barrier before freeing TMEM.  Launched with programmatic dependent
// launch: set-up runs before the wait for the previous kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "debug.cuh"
#include "ptx.cuh"

namespace averis {

// One GEMM of a launch (a launch runs one, or one per expert of a grouped layer).
struct GemmGroup {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ts_a;
  const float* ts_b;
  const float* col_add;  // [N] or null
  const float* row_vec;  // [M] or null
  const float* col_vec;  // [N] or null
  float outer;
  int M, N;
  int kc;      // ceil(K / 64): 64-element scale chunks per row chunk (same for A and B)
  int rb_a;    // ceil(M / 128): row chunks of A's scales
  int rb_b;    // ceil(N / 128): row chunks of B's scales
  int num_m;   // ceil(M / 256): pair tiles along M
  int unit0;   // first work unit of this GEMM in the launch
  int bf16;    // output in bf16 (else binary32)
};

constexpr int kMaxPairs = 128;  // CTA pairs of one launch at most (74 on a B300)

// Kernel arguments for up to G GEMMs: their tensor maps (A, B codes and the
// output, kept in parameter space, where TMA reads them) and scalars.
template <int G>
struct GemmArgs {
  CUtensorMap tmA[G], tmB[G], tmD[G];
  GemmGroup g[G];
  int ngroups;
  int nunits;          // work units of all GEMMs
  int* err;
  long long wait_limit;  // bound of every wait, in SM clock cycles
  // 1: none of these GEMMs' inputs comes from the kernel launched just before
  // (the library never sets it today): start at once, and wait for that kernel
  // only before exiting, so that this kernel's completion still implies the
  // previous one's.
  int early_start;
  // G > 1: pair p runs the contiguous units range0[p] .. range0[p+1]-1, cut
  // by the host so that every pair gets about the same number of K tiles
  // (units of different GEMMs of a launch can differ widely in K).  G = 1:
  // every unit costs the same, and pair p runs units p, p + P, p + 2P, ... of
  // the P pairs, which then work on neighbouring tiles at any one time
  // (8192^3: 174 us against 189 us with contiguous ranges)
  int range0[kMaxPairs + 1];
};
// kernel parameters are limited to 32764 bytes
constexpr int kMaxGemmGroups = 64;
static_assert(sizeof(GemmArgs<kMaxGemmGroups>) <= 32000, "grouped GEMM arguments too large");

// SFB_FULL: each CTA holds the block scales of all 256 B rows of the tile in
// its TMEM (8 columns per MMA); otherwise only those of its own 128 rows.
template <bool SFB_FULL>
struct GemmCfg {
  static constexpr int BM = 128;       // rows of A and of the output per CTA
  static constexpr int PM = 2 * BM;    // rows per pair tile
  static constexpr int BN = 256;       // output columns per tile (the MMA's N)
  static constexpr int BNH = BN / 2;   // rows of B per CTA
  static constexpr int BKB = 128;      // bytes of codes per row per K tile (256 elements)
  // 5 stages x (32 KB of operands + 6 KB of scales) per CTA: 160 KB of operands in
  // flight per SM; the epilogue gets one staging box per warp and one buffer of
  // vector entries to make room (4 stages left the MMAs waiting for operands)
  static constexpr int STAGES = 5;
  static constexpr int A_BYTES = BM * BKB;
  static constexpr int B_BYTES = BNH * BKB;
  static constexpr int SFA_BYTES = 4 * 512;
  static constexpr int SFB_HALVES = SFB_FULL ? 2 : 1;
  static constexpr int SFB_BYTES = SFB_HALVES * 4 * 512;
  static constexpr int EPI_WARPS = 8;                  // 2 per TMEM lane quarter, each half of the columns
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // accumulator columns per epilogue warp
  static constexpr int EPI_BUF = 32 * 128;             // one warp's 32 rows x 128 bytes
  static constexpr int EPI_NBUF = 1;                   // staging boxes per epilogue warp
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_NBUF * EPI_BUF;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int OFF_VEC = OFF_EPI + EPI_BYTES;  // [col_add, col_vec][BN] floats of the current tile
  static constexpr int OFF_BAR = OFF_VEC + 2 * BN * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;    // + alignment slack
  // TMEM columns: the accumulator, then per stage 16 SFA columns + the SFB columns
  static constexpr int SF_BASE = BN;
  static constexpr int SFB_STEP = 4 * SFB_HALVES;      // SFB columns per MMA (64 elements of K)
  static constexpr int SF_STAGE_COLS = 16 + 4 * SFB_STEP;
  static constexpr int TMEM_COLS = 512;
  static_assert(OFF_EPI % 1024 == 0, "epilogue staging must be 1024-byte aligned");
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM overflow");
  static_assert(SMEM <= 227 * 1024, "shared memory overflow");
  // instruction descriptor: E2M1 x E2M1 (format 1), K-major A and B, UE4M3 scales,
  // N >> 3 at bit 17, M >> 4 at bit 24 (M = 256: the pair's rows)
  static constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
};

// Named barrier of the epilogue warps (ids 1 and up are free for this).
template <int EPI_WARPS>
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b2);
}

// warps: producer, TMEM owner / MMA issuer, 8 epilogue warps, 4 scale-feed warps
constexpr int kGemmThreads = 32 * (2 + 8 + 4);

template <bool SFB_FULL, int G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ GemmArgs<G> p) {
  using Cfg = GemmCfg<SFB_FULL>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  constexpr int EPI_WARPS = Cfg::EPI_WARPS;
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* smem = gsm_raw + ((1024u - (ptx::smem_u32(gsm_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  // [STAGES] leader: both CTAs' operands landed and both CTAs' scales are in TMEM
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + STAGES;       // [STAGES] both: the stage's MMAs completed
  uint64_t* sf_loaded = empty + STAGES;  // [STAGES] both: this CTA's scale atoms are in SMEM
  uint64_t* tfull = sf_loaded + STAGES;  // both: the accumulator holds a finished tile
  uint64_t* tempty = tfull + 1;          // leader: both CTAs' epilogues drained the accumulator
  uint64_t* drain = tempty + 1;          // leader: every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = ptx::cluster_ctarank();  // 0: leader (issues the MMAs), 1: follower
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1 + 2 * 4);  // the leader's producer (with the bytes), the scale warps of both CTAs
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&sf_loaded[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(tempty, 2 * EPI_WARPS);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (G == 1 && warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.tmA[0]);
    ptx::prefetch_tmap(&p.tmB[0]);
    ptx::prefetch_tmap(&p.tmD[0]);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers are initialised and their TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // operands, scales and epilogue vectors may come from the previous kernel
  if (p.early_start)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  else
    ptx::pdl_wait_and_release();

  const int pair = blockIdx.x >> 1;
  constexpr bool kStrided = G == 1;
  const int u_begin = kStrided ? pair : p.range0[pair];
  const int u_end = kStrided ? p.nunits : p.range0[pair + 1];
  const int u_step = kStrided ? (int)(gridDim.x >> 1) : 1;
  // work unit -> its GEMM (the last one whose first unit is not after it),
  // output tile (mt, nt), M fastest, and K-tile range (all of K)
  struct Unit {
    int e, tile, mt, nt, kt0, kt1;
  };
  auto decode = [&](int unit) {
    Unit u;
    u.e = 0;
    if (G > 1) {
      int lo = 0, hi = p.ngroups - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.g[mid].unit0 <= unit) lo = mid;
        else hi = mid - 1;
      }
      u.e = lo;
    }
    const GemmGroup& gg = p.g[u.e];
    u.tile = unit - gg.unit0;
    u.mt = u.tile % gg.num_m;
    u.nt = u.tile / gg.num_m;
    u.kt0 = 0;
    u.kt1 = (gg.kc + 3) / 4;
    return u;
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // stages this thread has filled at least once (bit mask)
      bool failed = false;
      int cur_e = -1;
      for (int unit = u_begin; unit < u_end && !failed; unit += u_step) {
        const Unit u = decode(unit);
        const GemmGroup& gg = p.g[u.e];
        const CUtensorMap* tmA = &p.tmA[u.e];
        const CUtensorMap* tmB = &p.tmB[u.e];
        if (G > 1 && u.e != cur_e) {
          ptx::prefetch_tmap(tmA);
          ptx::prefetch_tmap(tmB);
          cur_e = u.e;
        }
        const int mt = u.mt, nt = u.nt;
        const int rba = mt * 2 + (int)cta;  // 128-row scale chunk of this CTA's A rows
        int nsfb = 0;
#pragma unroll
        for (int h = 0; h < Cfg::SFB_HALVES; ++h) nsfb += (nt * 2 + (SFB_FULL ? h : (int)cta)) < gg.rb_b ? 1 : 0;
        const uint32_t nsf = (rba < gg.rb_a ? 1u : 0u) + (uint32_t)nsfb;
        for (int kt = u.kt0; kt < u.kt1; ++kt) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit)) {
            atomicExch(p.err, kErrProducer);
            failed = true;
            break;
          }
          const int ns = min(4, gg.kc - 4 * kt);
          // the small scale atoms first, on their own barrier: the scale warps
          // move them into TMEM while the operand tiles are still arriving
          ptx::mbar_arrive_expect_tx(&sf_loaded[stage], (uint32_t)ns * 512u * nsf);
          if (rba < gg.rb_a)
            ptx::bulk_load(smem + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES,
                           gg.sfa + ((int64_t)rba * gg.kc + 4 * kt) * 512, ns * 512u, &sf_loaded[stage]);
          if constexpr (SFB_FULL) {
            // both CTAs need the scales of all 256 B rows: each loads the half of
            // its own B rows once, multicast to both (the partner's stage slot is
            // free: the commit that freed this stage here freed it there too, after
            // both CTAs' scale warps had read it)
            const int rb = nt * 2 + (int)cta;
            if (rb < gg.rb_b)
              ptx::bulk_load_mc(smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES + (int)cta * 2048,
                                gg.sfb + ((int64_t)rb * gg.kc + 4 * kt) * 512, ns * 512u, &sf_loaded[stage], 0x3);
          } else {
            const int rb = nt * 2 + (int)cta;
            if (rb < gg.rb_b)
              ptx::bulk_load(smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES, gg.sfb + ((int64_t)rb * gg.kc + 4 * kt) * 512,
                             ns * 512u, &sf_loaded[stage]);
          }
          // both CTAs' operand halves complete on the leader's stage barrier
          const uint32_t full_leader = ptx::mapa(ptx::smem_u32(&full[stage]), 0);
          if (cta == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2u * (uint32_t)(Cfg::A_BYTES + Cfg::B_BYTES));
          if (AVERIS_DBG_TMA_X(p.err, (int64_t)kt * Cfg::BKB, 1)) {
            ptx::tma_load_2d_pair(smem + Cfg::OFF_A + stage * Cfg::A_BYTES, tmA, kt * Cfg::BKB,
                                  mt * Cfg::PM + (int)cta * Cfg::BM, full_leader);
            ptx::tma_load_2d_pair(smem + Cfg::OFF_B + stage * Cfg::B_BYTES, tmB, kt * Cfg::BKB,
                                  nt * BN + (int)cta * Cfg::BNH, full_leader);
          }
          issued |= 1u << stage;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        // let this CTA's copies in flight land before its shared memory can be
        // given up: the scale atoms on its own barriers, and (leader) both
        // CTAs' operands on the stage barriers; give up again after the bound
        for (int s = 0; s < STAGES; ++s) {
          if (!(issued & (1u << s))) continue;
          const uint32_t par = s < stage ? phase : phase ^ 1u;  // parity of the stage's last fill
          ptx::mbar_wait(&sf_loaded[s], par, p.wait_limit);
          if (cta == 0) ptx::mbar_wait(&full[s], par, p.wait_limit);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && cta == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool issued = false;
      for (int unit = u_begin; unit < u_end; unit += u_step, ++it) {
        const Unit u = decode(unit);
        const int kc = p.g[u.e].kc, kt0 = u.kt0, kt1 = u.kt1;
        if (!ptx::mbar_wait(tempty, (it & 1) ^ 1u, p.wait_limit)) {
          atomicExch(p.err, kErrMma);
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kt = kt0; kt < kt1; ++kt) {
          // both CTAs' operand tiles in SMEM, both CTAs' scales in TMEM (one barrier)
          if (!ptx::mbar_wait(&full[stage], phase, p.wait_limit)) {
            atomicExch(p.err, kErrMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int ns = min(4, kc - 4 * kt);
          const uint32_t sfa_t = tmem + (uint32_t)(Cfg::SF_BASE + stage * Cfg::SF_STAGE_COLS);
          const uint32_t sfb_t = sfa_t + 16u;
          const uint32_t a_s = ptx::smem_u32(smem + Cfg::OFF_A + stage * Cfg::A_BYTES);
          const uint32_t b_s = ptx::smem_u32(smem + Cfg::OFF_B + stage * Cfg::B_BYTES);
          const uint64_t adesc0 = ptx::smem_desc(a_s, 16u, 1024u, ptx::kSwizzle128B);
          const uint64_t bdesc0 = ptx::smem_desc(b_s, 16u, 1024u, ptx::kSwizzle128B);
          const uint32_t acc0 = kt != kt0 ? 1u : 0u;
          if (ns == 4) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              ptx::tc_mma_nvf4_pair(tmem, adesc0 + 2u * g, bdesc0 + 2u * g, Cfg::IDESC, sfa_t + 4u * g,
                                    sfb_t + (uint32_t)(Cfg::SFB_STEP * g), g != 0 ? 1u : acc0);
          } else {
            for (int g = 0; g < ns; ++g)
              ptx::tc_mma_nvf4_pair(tmem, adesc0 + 2u * g, bdesc0 + 2u * g, Cfg::IDESC, sfa_t + 4u * g,
                                    sfb_t + (uint32_t)(Cfg::SFB_STEP * g), g != 0 ? 1u : acc0);
          }
          issued = true;
          ptx::tc_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit_pair(tfull, 0x3);
      }
      if (issued) {
        // drain: every MMA this thread issued has completed
        ptx::tc_commit_pair(drain, 0x1);
        if (!ptx::mbar_wait(drain, 0, p.wait_limit)) atomicExch(p.err, kErrDrain);
      }
    }
  } else if (warp >= 2 + EPI_WARPS) {
    // scale feed: every lane quarter q = warp % 4 gets the same words: lane
    // 32 q + i, columns 4 g .. 4 g + 3 (A chunk g) and 16 + SFB_STEP g + 4 h
    // .. +3 (B half h, chunk g) = row i of that 512-byte SMEM atom, whose word
    // j holds the 4 block scales of row i + 32 j.
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool failed = false;
    for (int unit = u_begin; unit < u_end && !failed; unit += u_step) {
      const Unit u = decode(unit);
      for (int kt = u.kt0; kt < u.kt1; ++kt) {
        if (!ptx::mbar_wait(&sf_loaded[stage], phase, p.wait_limit)) {
          if (lane == 0) atomicExch(p.err, kErrScaleFeed);
          failed = true;
          break;
        }
        const uint8_t* sa = smem + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES + 16 * lane;
        const uint8_t* sb = smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES + 16 * lane;
        uint32_t ra[16], rb[16 * Cfg::SFB_HALVES];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(sa + 512 * g);
          ra[4 * g] = v.x;
          ra[4 * g + 1] = v.y;
          ra[4 * g + 2] = v.z;
          ra[4 * g + 3] = v.w;
        }
#pragma unroll
        for (int h = 0; h < Cfg::SFB_HALVES; ++h)
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 v = *reinterpret_cast<const uint4*>(sb + 2048 * h + 512 * g);
            const int o = Cfg::SFB_STEP * g + 4 * h;
            rb[o] = v.x;
            rb[o + 1] = v.y;
            rb[o + 2] = v.z;
            rb[o + 3] = v.w;
          }
        const uint32_t t = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(Cfg::SF_BASE + stage * Cfg::SF_STAGE_COLS);
        ptx::tmem_st16(t, ra);
        if constexpr (SFB_FULL) {
          ptx::tmem_st32(t + 16u, rb);
        } else {
          ptx::tmem_st16(t + 16u, rb);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&full[stage]), 0));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // epilogue warps: TMEM lane quarter (warp % 4) holds this CTA's tile rows
    // 32*(warp%4) .. +31; warp 2 + 4 k + .. drains accumulator columns
    // EPI_COLS * k .. +EPI_COLS - 1
    const int q = warp & 3;
    const int cb = Cfg::EPI_COLS * ((warp - 2) >> 2);  // this warp's first column
    const int et = threadIdx.x - 64;  // 0 .. 32 EPI_WARPS - 1 over the epilogue warps
    uint8_t* stage_base = smem + Cfg::OFF_EPI + (warp - 2) * Cfg::EPI_NBUF * Cfg::EPI_BUF;
    int sbuf = 0;
    float* vec_base = reinterpret_cast<float*>(smem + Cfg::OFF_VEC);
    const uint32_t tempty_leader = ptx::mapa(ptx::smem_u32(tempty), 0);
    __shared__ int s_ok[2];    // per tile parity: the accumulator arrived
    int it = 0;
    int cur_e = -1;
    for (int unit = u_begin; unit < u_end; unit += u_step, ++it) {
      const Unit u = decode(unit);
      const GemmGroup& gg = p.g[u.e];
      const CUtensorMap* tmD = &p.tmD[u.e];
      if (G > 1 && u.e != cur_e && lane == 0) ptx::prefetch_tmap(tmD);
      cur_e = u.e;
      const int mt = u.mt, nt = u.nt;
      const float alpha = __ldg(gg.ts_a) * __ldg(gg.ts_b);
      const bool has_add = gg.col_add != nullptr;
      const bool has_outer = gg.row_vec != nullptr;
      const int row0 = mt * Cfg::PM + (int)cta * Cfg::BM + q * 32;
      const int row = row0 + lane;
      const float rterm = (has_outer && row < gg.M &&
                           AVERIS_DBG_IN(p.err, gg.row_vec + row, gg.row_vec, (int64_t)gg.M * 4, 4, kSiteGemmVectors))
                              ? gg.outer * __ldg(gg.row_vec + row)
                              : 0.f;
      // this tile's vector entries -> SMEM (one buffer: the barrier at the end of
      // the previous tile kept every warp from writing while another still read)
      float* cadd_s = vec_base;
      float* cvec_s = cadd_s + BN;
      for (int c = et; c < BN; c += 32 * EPI_WARPS) {
        const int col = nt * BN + c;
        cadd_s[c] = (has_add && col < gg.N &&
                     AVERIS_DBG_IN(p.err, gg.col_add + col, gg.col_add, (int64_t)gg.N * 4, 4, kSiteGemmVectors))
                        ? __ldg(gg.col_add + col)
                        : 0.f;
        cvec_s[c] = (has_outer && col < gg.N &&
                     AVERIS_DBG_IN(p.err, gg.col_vec + col, gg.col_vec, (int64_t)gg.N * 4, 4, kSiteGemmVectors))
                        ? __ldg(gg.col_vec + col)
                        : 0.f;
      }
      // one thread waits for the accumulator; the barrier hands its verdict (and
      // the staged vectors) to all epilogue warps, so they leave the loop together
      if (et == 0) s_ok[it & 1] = ptx::mbar_wait(tfull, it & 1, p.wait_limit) ? 1 : 0;
      epi_bar<EPI_WARPS>();
      if (!s_ok[it & 1]) {
        if (et == 0) atomicExch(p.err, kErrEpilogue);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
      const bool rows_live = row0 < gg.M;  // a box wholly below the last row stores nothing

      // stage one 32-row x 128-byte box in swizzled SMEM and store it with TMA
      auto store_box = [&](const uint4 (&w)[8], int col0) {
        uint8_t* stage_buf = stage_base + sbuf * Cfg::EPI_BUF;
        sbuf = (sbuf + 1) % Cfg::EPI_NBUF;
        if (lane == 0) ptx::bulk_wait_read<Cfg::EPI_NBUF - 1>();  // this box's previous store has read it
        __syncwarp();
        uint8_t* srow = stage_buf + lane * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(srow + ((k ^ (lane & 7)) * 16)) = w[k];
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (AVERIS_DBG_TMA_X(p.err, col0, gg.bf16 ? 2 : 4)) ptx::tma_store_2d(tmD, stage_buf, col0, row0);
          ptx::bulk_commit();
        }
      };
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(tempty_leader);
      };

      if (gg.bf16) {
        // this warp's accumulator columns -> packed bf16 registers, release TMEM, then store
        uint32_t packed[Cfg::EPI_COLS / 2];
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + (uint32_t)(cb + c), v);
          ptx::tmem_ld_wait();
          const float* ca = cadd_s + cb + c;
          const float* cv = cvec_s + cb + c;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(ca + j);
            const float4 v4 = *reinterpret_cast<const float4*>(cv + j);
            float x0 = __fmaf_rn(alpha, __uint_as_float(v[j]), a4.x);
            float x1 = __fmaf_rn(alpha, __uint_as_float(v[j + 1]), a4.y);
            float x2 = __fmaf_rn(alpha, __uint_as_float(v[j + 2]), a4.z);
            float x3 = __fmaf_rn(alpha, __uint_as_float(v[j + 3]), a4.w);
            if (has_outer) {
              x0 = __fmaf_rn(rterm, v4.x, x0);
              x1 = __fmaf_rn(rterm, v4.y, x1);
              x2 = __fmaf_rn(rterm, v4.z, x2);
              x3 = __fmaf_rn(rterm, v4.w, x3);
            }
            packed[(c + j) / 2] = pack_bf16x2(x0, x1);
            packed[(c + j) / 2 + 1] = pack_bf16x2(x2, x3);
          }
        }
        release();
        if (rows_live) {
#pragma unroll
          for (int c = 0; c < Cfg::EPI_COLS; c += 64) {
            uint4 w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = make_uint4(packed[c / 2 + 4 * k], packed[c / 2 + 4 * k + 1], packed[c / 2 + 4 * k + 2],
                                packed[c / 2 + 4 * k + 3]);
            store_box(w, nt * BN + cb + c);
          }
        }
      } else {
#pragma unroll 1
        for (int c = cb; c < cb + Cfg::EPI_COLS; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + (uint32_t)c, v);
          ptx::tmem_ld_wait();
          if (c + 32 == cb + Cfg::EPI_COLS) release();  // last chunk is in registers
          if (!rows_live) continue;
          const float* ca = cadd_s + c;
          const float* cv = cvec_s + c;
          uint4 w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 a4 = *reinterpret_cast<const float4*>(ca + 4 * k);
            const float4 v4 = *reinterpret_cast<const float4*>(cv + 4 * k);
            // fl32(alpha acc + broadcast row), then the outer product (the bf16
            // path computes the same binary32 values before rounding them)
            float x0 = __fmaf_rn(alpha, __uint_as_float(v[4 * k]), a4.x);
            float x1 = __fmaf_rn(alpha, __uint_as_float(v[4 * k + 1]), a4.y);
            float x2 = __fmaf_rn(alpha, __uint_as_float(v[4 * k + 2]), a4.z);
            float x3 = __fmaf_rn(alpha, __uint_as_float(v[4 * k + 3]), a4.w);
            if (has_outer) {
              x0 = __fmaf_rn(rterm, v4.x, x0);
              x1 = __fmaf_rn(rterm, v4.y, x1);
              x2 = __fmaf_rn(rterm, v4.z, x2);
              x3 = __fmaf_rn(rterm, v4.w, x3);
            }
            w[k] = make_uint4(__float_as_uint(x0), __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
          }
          store_box(w, nt * BN + c);
        }
      }
      epi_bar<EPI_WARPS>();  // every warp has read this tile's vector entries (one buffer)
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }
  __syncthreads();
  // neither CTA frees TMEM or leaves while the pair's MMAs may still use its
  // shared memory or TMEM: the leader has drained them above
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
  }
  if (p.early_start) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace averis
