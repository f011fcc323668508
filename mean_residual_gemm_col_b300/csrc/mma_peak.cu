// Tensor-core instruction throughput on this GPU: how many SM cycles one
// tcgen05.mma takes when MMAs are issued back to back with their operands
// already in shared memory (no loads, one commit at the end), and the
// resulting rate with one CTA per SM on every SM.
//
// Measured forms (the ones the library's GEMM uses, and bf16 for reference):
//   nvf4  kind::mxf4nvf4.block_scale.scale_vec::4X, M = 128, N = 256 / 128, K = 64
//   pair  the same with cta_group::2 (M = 256 over two CTAs), N = 256 / 128
//   bf16  kind::f16 (bf16 inputs, binary32 accumulate), M = 128, N = 256 / 128, K = 16
//   stage nvf4 N = 256 with the GEMM's per-stage bookkeeping between every four
//         MMAs: a commit (mode 1), plus two waits on completed barriers and a
//         tcgen05 fence (mode 2)
//   st    pair MMAs reading their scales from four rotating 48-column TMEM
//         stages, while four more warps per CTA write one stage of scales
//         (tcgen05.st, 16 + 32 columns per lane quarter) per four MMAs, as the
//         GEMM's scale-feed warps do
//   pipe  the pair GEMM's dependency loop: a stage's 32 KB per CTA is reloaded
//         (bulk copies from a 64 MB L2-resident source) only after the MMAs
//         that read it completed (commit multicast to both CTAs), and its
//         four MMAs are issued only after both CTAs' copies landed; 4 and 6
//         stages
//   tma   the same loop fed the way the GEMM feeds it: 2-D tiled TMA loads
//         (128 rows x 128 bytes, 128-byte swizzle) of two 32 MB operand
//         matrices, each CTA's loads completing on the leader's stage barrier
//   scales the tma loop with each stage's block scales (2 KB of A scales, 4 KB
//         of B scales per CTA): (st) loaded by bulk copies and written into
//         TMEM by four scale warps per CTA that then arrive on the leader's
//         barrier; (cp) loaded by TMA with the operands and moved into TMEM by
//         tcgen05.cp from the MMA thread
//   copy  a second warp of every CTA streams 32 KB bulk copies (an L2-resident
//         8 MB source) into a 4-slot shared-memory ring, one copy per four MMAs
//         (the pair GEMM's operand bytes per stage), alone and beside the pair
//         MMAs: does the tensor pipe slow down while the same shared memory is
//         being written?
// Every wait is bounded; the operands are fixed bit patterns.
//
// Build and run: python -m mean_residual_gemm_col_b300.mma_peak
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

using namespace averis;

namespace {

constexpr int kSmem = 16384 + 32768 + 1024;  // A 128 x 128 B, B 256 x 128 B, alignment slack
constexpr long long kLimit = 1ll << 31;

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 1, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
                   d),
               "l"(a), "l"(b), "r"(idesc)
               : "memory");
}

// Shared set-up: operand bytes, TMEM (512 columns), E4M3 scale 1.0 in columns 256..511.
template <bool PAIR>
__device__ uint32_t setup(uint8_t* sm, uint32_t* slot, uint64_t* bars, int nbars) {
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x35733573u * (uint32_t)(i + 7);
  if (threadIdx.x == 0) {
    for (int b = 0; b < nbars; ++b) ptx::mbar_init(&bars[b], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    if (PAIR) {
      ptx::tmem_alloc_pair(slot, 512);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(slot, 512);
      ptx::tmem_relinquish();
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *slot;
  uint32_t r[32];
  for (int j = 0; j < 32; ++j) r[j] = 0x38383838u;
  if (warp < 4)
    for (int c = 256; c < 512; c += 32) ptx::tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + c, r);
  ptx::tmem_st_wait();
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  return tmem;
}

template <bool PAIR>
__device__ void teardown(uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  if ((threadIdx.x >> 5) == 0) {
    if (PAIR) ptx::tmem_dealloc_pair(tmem, 512);
    else ptx::tmem_dealloc(tmem, 512);
  }
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return raw + ((1024u - (ptx::smem_u32(raw) & 1023u)) & 1023u);
}

// KIND 0: nvf4; 1: bf16.  MODE (nvf4 only): 0 plain, 1 commit per 4 MMAs, 2 commit + waits + fence.
template <int KIND, int N, int MODE>
__global__ void __launch_bounds__(128, 1) bench_one(long long* cycles, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  __shared__ uint64_t bars[3];  // end, per-stage commits, always-complete
  __shared__ uint32_t slot;
  const uint32_t tmem = setup<false>(sm, &slot, bars, 3);
  if (threadIdx.x == 0) {
    ptx::mbar_arrive(&bars[2]);  // phase 0 of bars[2] completes: its waits return at once
    const uint32_t a_s = ptx::smem_u32(sm), b_s = ptx::smem_u32(sm + 16384);
    const uint32_t idesc = KIND == 0 ? (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (8u << 24)
                                     : (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (8u << 24);
    const long long t0 = clock64();
    for (int i = 0; i < iters; i += 4) {
      if (MODE == 2) {
        ptx::mbar_wait(&bars[2], 0, kLimit);
        ptx::mbar_wait(&bars[2], 0, kLimit);
        ptx::tc_fence_after();
      }
      for (int g = 0; g < 4; ++g) {
        const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        if (KIND == 0)
          ptx::tc_mma_nvf4(tmem, ad, bd, idesc, tmem + 256 + 4 * g, tmem + 272 + 8 * g, 1u);
        else
          mma_bf16(tmem, ad, bd, idesc);
      }
      if (MODE >= 1) ptx::tc_commit(&bars[1]);
    }
    ptx::tc_commit(&bars[0]);
    const bool ok = ptx::mbar_wait(&bars[0], 0, kLimit);
    cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
  }
  teardown<false>(tmem);
}

template <int N>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) bench_pair(long long* cycles, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  __shared__ uint64_t bars[1];
  __shared__ uint32_t slot;
  const uint32_t tmem = setup<true>(sm, &slot, bars, 1);
  if (ptx::cluster_ctarank() == 0 && threadIdx.x == 0) {
    const uint32_t a_s = ptx::smem_u32(sm), b_s = ptx::smem_u32(sm + 16384);
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (16u << 24);
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int g = i & 3;
      const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, tmem + 256 + 4 * g, tmem + 272 + 8 * g, 1u);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    const bool ok = ptx::mbar_wait(&bars[0], 0, kLimit);
    cycles[blockIdx.x >> 1] = ok ? clock64() - t0 : -1;
  }
  teardown<true>(tmem);
}

// Pair MMAs with scales in four rotating TMEM stages (columns 256 + 48 s:
// 16 for A, 32 for B); FEED: warps 4..7 of every CTA rewrite one stage per
// four MMAs (paced by the clock, one stage at a time).
template <bool FEED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1) bench_pair_st(long long* cycles, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  __shared__ uint64_t bars[1];
  __shared__ uint32_t slot;
  const uint32_t tmem = setup<true>(sm, &slot, bars, 1);
  const int warp = threadIdx.x >> 5;
  if (ptx::cluster_ctarank() == 0 && threadIdx.x == 0) {
    const uint32_t a_s = ptx::smem_u32(sm), b_s = ptx::smem_u32(sm + 16384);
    const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (16u << 24);
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int g = i & 3;
      const uint32_t st = 256u + 48u * (uint32_t)((i >> 2) & 3);
      const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, tmem + st + 4 * g, tmem + st + 16 + 8 * g, 1u);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    const bool ok = ptx::mbar_wait(&bars[0], 0, kLimit);
    cycles[blockIdx.x >> 1] = ok ? clock64() - t0 : -1;
  }
  if (FEED && warp >= 4) {
    const uint32_t q = (uint32_t)(warp & 3);
    uint32_t ra[16], rb[32];
    for (int j = 0; j < 16; ++j) ra[j] = 0x38383838u;
    for (int j = 0; j < 32; ++j) rb[j] = 0x38383838u;
    const long long t0 = clock64();
    for (int k = 0; k < iters / 4; ++k) {
      // one stage per 512 cycles (four MMAs at 128 cycles); the wait is bounded by its own count
      for (int spin = 0; spin < 100000 && clock64() - t0 < 512ll * k; ++spin) {
      }
      const uint32_t t = tmem + ((q * 32u) << 16) + 256u + 48u * (uint32_t)((k + 2) & 3);
      ptx::tmem_st16(t, ra);
      ptx::tmem_st32(t + 16u, rb);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
    }
  }
  teardown<true>(tmem);
}

void run_st(bool feed, int sms, int iters) {
  const int ctas = 2 * (sms / 2), pairs = ctas / 2;
  long long* d = nullptr;
  if (cudaMalloc(&d, pairs * sizeof(long long)) != cudaSuccess) return;
  auto k = feed ? bench_pair_st<true> : bench_pair_st<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  k<<<ctas, 256, kSmem>>>(d, 64);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<ctas, 256, kSmem>>>(d, iters);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  long long h[256];
  cudaMemcpy(h, d, pairs * sizeof(long long), cudaMemcpyDeviceToHost);
  double mc = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) {
    if (h[i] < 0) ++bad;
    else mc += (double)h[i];
  }
  mc /= pairs;
  printf("%-12s N=256  %6.1f cycles/MMA  %8.1f TFLOP/s  (%.3f ms, %s%s)\n", feed ? "pair+st" : "pair stages", mc / iters,
         2.0 * 2 * 128 * 64 * 256 * (double)iters * pairs / (ms * 1e-3) / 1e12, ms, cudaGetErrorString(err),
         bad ? ", a wait gave up" : "");
  cudaFree(d);
}

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    bench_pair_pipe(long long* cycles, const uint8_t* src, int chunks, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  // done | full[S] (leader, both CTAs' forwarders arrive) | empty[S] | own[S] (this CTA's copies)
  __shared__ uint64_t bars[1 + 3 * STAGES];
  __shared__ uint32_t slot;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + STAGES;
  uint64_t* own = empty + STAGES;
  const uint32_t cta = ptx::cluster_ctarank();
  if (threadIdx.x == 0)
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 2);
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&own[s], 1);
    }
  const uint32_t tmem = setup<true>(sm, &slot, bars, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = iters / 4;
  if (warp == 1 && lane == 0) {
    // producer: refill stage s once the MMAs that read it completed
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&empty[s], (uint32_t)(((k / STAGES) & 1) ^ 1), kLimit)) break;
      ptx::mbar_arrive_expect_tx(&own[s], 32768u);
      const size_t c = (size_t)(((blockIdx.x >> 1) * 131 + k * 2 + (int)cta) % chunks) * 32768;
      ptx::bulk_load(sm + s * 32768, src + c, 16384u, &own[s]);
      ptx::bulk_load(sm + s * 32768 + 16384, src + c + 16384, 16384u, &own[s]);
    }
  } else if (warp == 2 && lane == 0) {
    // forwarder: this CTA's copies of stage s landed -> the leader's full[s]
    // (also lets every copy this CTA requested land before it exits)
    const uint32_t full_leader = ptx::mapa(ptx::smem_u32(&full[0]), 0);
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&own[s], (uint32_t)((k / STAGES) & 1), kLimit)) break;
      ptx::mbar_arrive_cluster(full_leader + 8u * (uint32_t)s);
    }
  } else if (warp == 0 && lane == 0 && cta == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (16u << 24);
    const long long t0 = clock64();
    bool ok = true;
    for (int k = 0; k < nk && ok; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&full[s], (uint32_t)((k / STAGES) & 1), kLimit)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a_s = ptx::smem_u32(sm + s * 32768), b_s = a_s + 16384u;
      for (int g = 0; g < 4; ++g) {
        const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, tmem + 256 + 4 * g, tmem + 272 + 8 * g, 1u);
      }
      ptx::tc_commit_pair(&empty[s], 0x3);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    if (!ptx::mbar_wait(&bars[0], 0, kLimit)) ok = false;
    cycles[blockIdx.x >> 1] = ok ? clock64() - t0 : -1;
  }
  teardown<true>(tmem);
}

template <int STAGES>
void run_pipe(int sms, int iters) {
  const int ctas = 2 * (sms / 2), pairs = ctas / 2, chunks = 2048;
  const int smem = STAGES * 32768 + 1024;
  long long* d = nullptr;
  uint8_t* src = nullptr;
  if (cudaMalloc(&d, pairs * sizeof(long long)) != cudaSuccess ||
      cudaMalloc(&src, (size_t)chunks * 32768) != cudaSuccess)
    return;
  cudaMemset(src, 0x35, (size_t)chunks * 32768);
  cudaFuncSetAttribute(bench_pair_pipe<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  bench_pair_pipe<STAGES><<<ctas, 128, smem>>>(d, src, chunks, 64);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  bench_pair_pipe<STAGES><<<ctas, 128, smem>>>(d, src, chunks, iters);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  long long h[256];
  cudaMemcpy(h, d, pairs * sizeof(long long), cudaMemcpyDeviceToHost);
  double mc = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) {
    if (h[i] < 0) ++bad;
    else mc += (double)h[i];
  }
  mc /= pairs;
  printf("pipe %d st    N=256  %6.1f cycles/MMA  %8.1f TFLOP/s  (%.3f ms, %s%s)\n", STAGES, mc / iters,
         2.0 * 2 * 128 * 64 * 256 * (double)iters * pairs / (ms * 1e-3) / 1e12, ms, cudaGetErrorString(err),
         bad ? ", a wait gave up" : "");
  cudaFree(d);
  cudaFree(src);
}

// The pair GEMM's main loop on 8192-row operands (4096 bytes of codes per
// row), tile order as the GEMM's (M fastest), no scales, no epilogue.
template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    bench_pair_tma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   long long* cycles, int iters, int num_m) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  __shared__ uint64_t bars[1 + 2 * STAGES];  // done | full[S] (leader) | empty[S]
  __shared__ uint32_t slot;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + STAGES;
  const uint32_t cta = ptx::cluster_ctarank();
  if (threadIdx.x == 0)
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
  const uint32_t tmem = setup<true>(sm, &slot, bars, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = iters / 4, pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (warp == 1 && lane == 0) {
    const uint32_t full_leader = ptx::mapa(ptx::smem_u32(&full[0]), 0);
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&empty[s], (uint32_t)(((k / STAGES) & 1) ^ 1), kLimit)) break;
      const int unit = pair + npairs * (k / 32), kt = k % 32;
      const int mt = unit % num_m, nt = (unit / num_m) % num_m;
      if (cta == 0) ptx::mbar_arrive_expect_tx(&full[s], 2u * 32768u);
      ptx::tma_load_2d_pair(sm + s * 32768, &tmA, kt * 128, mt * 256 + (int)cta * 128, full_leader + 8u * (uint32_t)s);
      ptx::tma_load_2d_pair(sm + s * 32768 + 16384, &tmB, kt * 128, nt * 256 + (int)cta * 128,
                            full_leader + 8u * (uint32_t)s);
    }
  } else if (warp == 0 && lane == 0 && cta == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (16u << 24);
    const long long t0 = clock64();
    bool ok = true;
    for (int k = 0; k < nk && ok; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&full[s], (uint32_t)((k / STAGES) & 1), kLimit)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a_s = ptx::smem_u32(sm + s * 32768), b_s = a_s + 16384u;
      for (int g = 0; g < 4; ++g) {
        const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, tmem + 256 + 4 * g, tmem + 272 + 8 * g, 1u);
      }
      ptx::tc_commit_pair(&empty[s], 0x3);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    if (!ptx::mbar_wait(&bars[0], 0, kLimit)) ok = false;
    cycles[pair] = ok ? clock64() - t0 : -1;
  }
  // every copy this CTA requested has been consumed by an MMA that completed
  // (leader) before the pair leaves: the follower waits in the cluster sync
  teardown<true>(tmem);
}

// SCALE 1: bulk-copied scales, four scale warps per CTA (tcgen05.st) and a
// cross-CTA arrival per stage; SCALE 2: scales by TMA on the stage barrier,
// tcgen05.cp from the MMA thread.
template <int STAGES, int SCALE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    bench_pair_sf(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmS, const uint8_t* sf_src, long long* cycles, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  uint8_t* sfs = sm + STAGES * 32768;  // per stage: A scales 2 KB | B scales 4 KB
  // done | full[S] | empty[S] | sf_loaded[S] | sf_full[S]
  __shared__ uint64_t bars[1 + 4 * STAGES];
  __shared__ uint32_t slot;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + STAGES;
  uint64_t* sf_loaded = empty + STAGES;
  uint64_t* sf_full = sf_loaded + STAGES;
  const uint32_t cta = ptx::cluster_ctarank();
  if (threadIdx.x == 0)
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&sf_loaded[s], 1);
      ptx::mbar_init(&sf_full[s], 8);
    }
  const uint32_t tmem = setup<true>(sm, &slot, bars, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = iters / 4, pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (warp == 1 && lane == 0) {
    const uint32_t full_leader = ptx::mapa(ptx::smem_u32(&full[0]), 0);
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&empty[s], (uint32_t)(((k / STAGES) & 1) ^ 1), kLimit)) break;
      const int unit = pair + npairs * (k / 32), kt = k % 32;
      const int mt = unit % 32, nt = (unit / 32) % 32;
      const int srow = ((pair * 2 + (int)cta) * 64 + (k % 64) * 48) % 4032;  // 16-row scale boxes, 3 per stage
      if (SCALE == 1) {
        ptx::mbar_arrive_expect_tx(&sf_loaded[s], 6144u);
        ptx::bulk_load(sfs + s * 6144, sf_src + (size_t)srow * 128, 2048u, &sf_loaded[s]);
        ptx::bulk_load(sfs + s * 6144 + 2048, sf_src + (size_t)(srow + 16) * 128, 4096u, &sf_loaded[s]);
      }
      if (cta == 0) ptx::mbar_arrive_expect_tx(&full[s], 2u * (32768u + (SCALE == 2 ? 6144u : 0u)));
      const uint32_t fb = full_leader + 8u * (uint32_t)s;
      ptx::tma_load_2d_pair(sm + s * 32768, &tmA, kt * 128, mt * 256 + (int)cta * 128, fb);
      ptx::tma_load_2d_pair(sm + s * 32768 + 16384, &tmB, kt * 128, nt * 256 + (int)cta * 128, fb);
      if (SCALE == 2) {
        ptx::tma_load_2d_pair(sfs + s * 6144, &tmS, 0, srow, fb);
        ptx::tma_load_2d_pair(sfs + s * 6144 + 2048, &tmS, 0, srow + 16, fb);
        ptx::tma_load_2d_pair(sfs + s * 6144 + 4096, &tmS, 0, srow + 32, fb);
      }
    }
  } else if (warp == 0 && lane == 0 && cta == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (16u << 24);
    const long long t0 = clock64();
    bool ok = true;
    for (int k = 0; k < nk && ok; ++k) {
      const int s = k % STAGES;
      const uint32_t par = (uint32_t)((k / STAGES) & 1);
      if (!ptx::mbar_wait(&full[s], par, kLimit) || (SCALE == 1 && !ptx::mbar_wait(&sf_full[s], par, kLimit))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sf_t = tmem + 256u + 48u * (uint32_t)(s & 3);
      if (SCALE == 2) {
        const uint32_t sa = ptx::smem_u32(sfs + s * 6144);
        for (int g = 0; g < 4; ++g) ptx::tc_cp_scales_pair(sf_t + 4u * g, ptx::smem_desc(sa + 512u * g, 128u, 128u, ptx::kSwizzleNone));
        for (int h = 0; h < 2; ++h)
          for (int g = 0; g < 4; ++g)
            ptx::tc_cp_scales_pair(sf_t + 16u + 8u * g + 4u * h,
                                   ptx::smem_desc(sa + 2048u + 2048u * h + 512u * g, 128u, 128u, ptx::kSwizzleNone));
      }
      const uint32_t a_s = ptx::smem_u32(sm + s * 32768), b_s = a_s + 16384u;
      for (int g = 0; g < 4; ++g) {
        const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
        ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf_t + 4 * g, sf_t + 16 + 8 * g, 1u);
      }
      ptx::tc_commit_pair(&empty[s], 0x3);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    if (!ptx::mbar_wait(&bars[0], 0, kLimit)) ok = false;
    cycles[pair] = ok ? clock64() - t0 : -1;
  } else if (SCALE == 1 && warp >= 4) {
    // scale warps: SMEM atoms -> TMEM (row i of an atom to lane 32 q + i), then
    // arrive on the leader's stage barrier; they also let every scale copy land
    const uint32_t q = (uint32_t)(warp & 3);
    const uint32_t sf_leader = ptx::mapa(ptx::smem_u32(&sf_full[0]), 0);
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      if (!ptx::mbar_wait(&sf_loaded[s], (uint32_t)((k / STAGES) & 1), kLimit)) break;
      const uint8_t* sa = sfs + s * 6144 + 16 * lane;
      uint32_t ra[16], rb[32];
      for (int g = 0; g < 4; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(sa + 512 * g);
        ra[4 * g] = v.x; ra[4 * g + 1] = v.y; ra[4 * g + 2] = v.z; ra[4 * g + 3] = v.w;
      }
      for (int h = 0; h < 2; ++h)
        for (int g = 0; g < 4; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(sa + 2048 + 2048 * h + 512 * g);
          const int o = 8 * g + 4 * h;
          rb[o] = v.x; rb[o + 1] = v.y; rb[o + 2] = v.z; rb[o + 3] = v.w;
        }
      const uint32_t t = tmem + ((q * 32u) << 16) + 256u + 48u * (uint32_t)(s & 3);
      ptx::tmem_st16(t, ra);
      ptx::tmem_st32(t + 16u, rb);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(sf_leader + 8u * (uint32_t)s);
    }
  }
  teardown<true>(tmem);
}

// Seeded pseudo-random bytes (an integer hash of the index); scales: E4M3
// codes 0x30..0x3F (0.5 .. 1.875), codes: any E2M1 pair.
__global__ void fill_random(uint8_t* p, size_t n, uint32_t seed, int scales) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    uint32_t h = (uint32_t)i * 0x9E3779B1u ^ seed;
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    p[i] = scales ? (uint8_t)(0x30u | (h & 15u)) : (uint8_t)h;
  }
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int STAGES>
void run_tma(int sms, int iters, bool rnd = false, size_t rows = 8192) {
  const int ctas = 2 * (sms / 2), pairs = ctas / 2;
  const int smem = STAGES * 32768 + 1024;
  const size_t row_bytes = 4096;
  const int num_m = (int)(rows / 256);
  long long* d = nullptr;
  uint8_t *a = nullptr, *b = nullptr;
  if (cudaMalloc(&d, pairs * sizeof(long long)) != cudaSuccess || cudaMalloc(&a, rows * row_bytes) != cudaSuccess ||
      cudaMalloc(&b, rows * row_bytes) != cudaSuccess)
    return;
  cudaMemset(a, 0x35, rows * row_bytes);
  cudaMemset(b, 0x53, rows * row_bytes);
  if (rnd) {
    fill_random<<<1024, 256>>>(a, rows * row_bytes, 1u, 0);
    fill_random<<<1024, 256>>>(b, rows * row_bytes, 2u, 0);
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      fn == nullptr)
    return;
  EncodeFn enc = reinterpret_cast<EncodeFn>(fn);
  CUtensorMap ma, mb;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return;
  cudaFuncSetAttribute(bench_pair_tma<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  bench_pair_tma<STAGES><<<ctas, 128, smem>>>(ma, mb, d, 64, num_m);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  bench_pair_tma<STAGES><<<ctas, 128, smem>>>(ma, mb, d, iters, num_m);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  long long h[256];
  cudaMemcpy(h, d, pairs * sizeof(long long), cudaMemcpyDeviceToHost);
  double mc = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) {
    if (h[i] < 0) ++bad;
    else mc += (double)h[i];
  }
  mc /= pairs;
  printf("tma %d st %s %4d MB  %6.1f cycles/MMA  %8.1f TFLOP/s  (%.3f ms, %s%s)\n", STAGES, rnd ? "rnd" : "   ",
         (int)(2 * rows * row_bytes >> 20), mc / iters,
         2.0 * 2 * 128 * 64 * 256 * (double)iters * pairs / (ms * 1e-3) / 1e12, ms, cudaGetErrorString(err),
         bad ? ", a wait gave up" : "");
  cudaFree(d);
  cudaFree(a);
  cudaFree(b);
}

template <int STAGES, int SCALE>
void run_sf(int sms, int iters, bool rnd = false) {
  const int ctas = 2 * (sms / 2), pairs = ctas / 2;
  const int smem = STAGES * (32768 + 6144) + 1024;
  const size_t rows = 8192, row_bytes = 4096, srows = 4096;
  long long* d = nullptr;
  uint8_t *a = nullptr, *b = nullptr, *sf = nullptr;
  if (cudaMalloc(&d, pairs * sizeof(long long)) != cudaSuccess || cudaMalloc(&a, rows * row_bytes) != cudaSuccess ||
      cudaMalloc(&b, rows * row_bytes) != cudaSuccess || cudaMalloc(&sf, srows * 128) != cudaSuccess)
    return;
  cudaMemset(a, 0x35, rows * row_bytes);
  cudaMemset(b, 0x53, rows * row_bytes);
  cudaMemset(sf, 0x38, srows * 128);
  if (rnd) {
    fill_random<<<1024, 256>>>(a, rows * row_bytes, 1u, 0);
    fill_random<<<1024, 256>>>(b, rows * row_bytes, 2u, 0);
    fill_random<<<1024, 256>>>(sf, srows * 128, 3u, 1);
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      fn == nullptr)
    return;
  EncodeFn enc = reinterpret_cast<EncodeFn>(fn);
  CUtensorMap ma, mb, ms;
  const cuuint64_t dims[2] = {row_bytes, rows}, sdims[2] = {128, srows};
  const cuuint64_t strides[1] = {row_bytes}, sstrides[1] = {128};
  const cuuint32_t box[2] = {128, 128}, sbox[2] = {128, 16};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, sf, sdims, sstrides, sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return;
  auto k = bench_pair_sf<STAGES, SCALE>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<ctas, 256, smem>>>(ma, mb, ms, sf, d, 64);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<ctas, 256, smem>>>(ma, mb, ms, sf, d, iters);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms_ = 0;
  cudaEventElapsedTime(&ms_, e0, e1);
  long long h[256];
  cudaMemcpy(h, d, pairs * sizeof(long long), cudaMemcpyDeviceToHost);
  double mc = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) {
    if (h[i] < 0) ++bad;
    else mc += (double)h[i];
  }
  mc /= pairs;
  printf("scales %s %d %s N=256 %6.1f cycles/MMA  %8.1f TFLOP/s  (%.3f ms, %s%s)\n", SCALE == 1 ? "st" : "cp", STAGES,
         rnd ? "rnd" : "   ", mc / iters, 2.0 * 2 * 128 * 64 * 256 * (double)iters * pairs / (ms_ * 1e-3) / 1e12, ms_,
         cudaGetErrorString(err), bad ? ", a wait gave up" : "");
  cudaFree(d);
  cudaFree(a);
  cudaFree(b);
  cudaFree(sf);
}

constexpr int kRing = 4 * 32768;
constexpr int kSmemCopy = 16384 + 32768 + kRing + 1024;

// Pair MMAs (MMA = true) and / or the bulk-copy stream; per CTA pair the
// leader's MMA cycles, per CTA the copy stream's cycles.
template <int N, bool MMA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    bench_pair_copy(long long* cycles, long long* copy_cycles, const uint8_t* src, int src_chunks, int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = aligned_smem(raw);
  __shared__ uint64_t bars[5];  // MMA end, ring slots
  __shared__ uint32_t slot;
  const uint32_t tmem = setup<true>(sm, &slot, bars, 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (MMA && ptx::cluster_ctarank() == 0 && threadIdx.x == 0) {
    const uint32_t a_s = ptx::smem_u32(sm), b_s = ptx::smem_u32(sm + 16384);
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (16u << 24);
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int g = i & 3;
      const uint64_t ad = ptx::smem_desc(a_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      const uint64_t bd = ptx::smem_desc(b_s + 32u * g, 16u, 1024u, ptx::kSwizzle128B);
      ptx::tc_mma_nvf4_pair(tmem, ad, bd, idesc, tmem + 256 + 4 * g, tmem + 272 + 8 * g, 1u);
    }
    ptx::tc_commit_pair(&bars[0], 0x1);
    const bool ok = ptx::mbar_wait(&bars[0], 0, kLimit);
    cycles[blockIdx.x >> 1] = ok ? clock64() - t0 : -1;
  }
  if (warp == 1 && lane == 0) {
    uint8_t* ring = sm + 16384 + 32768;
    const int ncopy = iters / 4;
    bool ok = true;
    const long long t0 = clock64();
    int i = 0;
    for (; i < ncopy; ++i) {
      const int s = i & 3;
      if (i >= 4 && !ptx::mbar_wait(&bars[1 + s], (uint32_t)(((i >> 2) - 1) & 1), kLimit)) {
        ok = false;
        break;
      }
      ptx::mbar_arrive_expect_tx(&bars[1 + s], 32768u);
      ptx::bulk_load(ring + s * 32768, src + (size_t)((blockIdx.x * 7 + i) % src_chunks) * 32768, 32768u, &bars[1 + s]);
    }
    // the copies still in flight land before the ring is given up (bounded)
    for (int j = i - 4 < 0 ? 0 : i - 4; j < i; ++j)
      if (!ptx::mbar_wait(&bars[1 + (j & 3)], (uint32_t)((j >> 2) & 1), kLimit)) ok = false;
    copy_cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
  }
  teardown<true>(tmem);
}

void run_copy(bool mma, int sms, int iters) {
  const int ctas = 2 * (sms / 2), pairs = ctas / 2, chunks = 256;
  long long *d_c = nullptr, *d_cc = nullptr;
  uint8_t* src = nullptr;
  if (cudaMalloc(&d_c, pairs * sizeof(long long)) != cudaSuccess ||
      cudaMalloc(&d_cc, ctas * sizeof(long long)) != cudaSuccess || cudaMalloc(&src, (size_t)chunks * 32768) != cudaSuccess)
    return;
  cudaMemset(src, 0x35, (size_t)chunks * 32768);
  cudaMemset(d_c, 0, pairs * sizeof(long long));
  auto k = mma ? bench_pair_copy<256, true> : bench_pair_copy<256, false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCopy);
  k<<<ctas, 128, kSmemCopy>>>(d_c, d_cc, src, chunks, 64);  // warm-up
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<ctas, 128, kSmemCopy>>>(d_c, d_cc, src, chunks, iters);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  long long hc[256], hcc[512];
  cudaMemcpy(hc, d_c, pairs * sizeof(long long), cudaMemcpyDeviceToHost);
  cudaMemcpy(hcc, d_cc, ctas * sizeof(long long), cudaMemcpyDeviceToHost);
  double mc = 0, cc = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) mc += (double)hc[i];
  for (int i = 0; i < ctas; ++i) {
    if (hcc[i] < 0) ++bad;
    else cc += (double)hcc[i];
  }
  mc /= pairs;
  cc /= ctas;
  const double bytes = (double)(iters / 4) * 32768.0;
  if (mma)
    printf("%-12s N=256  %6.1f cycles/MMA  copy %5.1f B/cycle per SM  %8.1f TFLOP/s  (%.3f ms, %s%s)\n", "pair+copy",
           mc / iters, bytes / cc, 2.0 * 2 * 128 * 64 * 256 * (double)iters * pairs / (ms * 1e-3) / 1e12, ms,
           cudaGetErrorString(err), bad ? ", a wait gave up" : "");
  else
    printf("%-12s        copy %5.1f B/cycle per SM, %6.1f GB/s over %d SMs  (%.3f ms, %s%s)\n", "copy alone", bytes / cc,
           bytes * ctas / (ms * 1e-3) / 1e9, ctas, ms, cudaGetErrorString(err), bad ? ", a wait gave up" : "");
  cudaFree(d_c);
  cudaFree(d_cc);
  cudaFree(src);
}

template <typename K>
double run(K kernel, const char* name, int n, double flop_per_mma, int ctas, int per_cycle_div, int iters) {
  long long* d = nullptr;
  if (cudaMalloc(&d, ctas * sizeof(long long)) != cudaSuccess) return -1;
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  kernel<<<ctas, 128, kSmem>>>(d, 64);  // warm-up
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  kernel<<<ctas, 128, kSmem>>>(d, iters);
  cudaEventRecord(e1);
  const cudaError_t err = cudaDeviceSynchronize();
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  const int timed = ctas / per_cycle_div;
  long long h[512];
  cudaMemcpy(h, d, timed * sizeof(long long), cudaMemcpyDeviceToHost);
  double cyc = 0;
  int bad = 0;
  for (int i = 0; i < timed; ++i) {
    if (h[i] < 0) ++bad;
    else cyc += (double)h[i];
  }
  cyc /= timed;
  const double tflops = flop_per_mma * iters * timed / (ms * 1e-3) / 1e12;
  printf("%-12s N=%3d  %6.1f cycles/MMA  %8.1f TFLOP/s  (%d CTAs, %.3f ms, %s%s)\n", name, n, cyc / iters, tflops, ctas,
         ms, cudaGetErrorString(err), bad ? ", a wait gave up" : "");
  cudaFree(d);
  return tflops;
}

}  // namespace

int main() {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms > 512) return 1;
  const int it = 20000;
  const double f4 = 2.0 * 128 * 64, bf = 2.0 * 128 * 16;
  run(bench_one<0, 256, 0>, "nvf4", 256, f4 * 256, 1, 1, it);
  run(bench_one<0, 256, 0>, "nvf4", 256, f4 * 256, sms, 1, it);
  run(bench_one<0, 128, 0>, "nvf4", 128, f4 * 128, sms, 1, it);
  run(bench_one<1, 256, 0>, "bf16", 256, bf * 256, sms, 1, it);
  run(bench_one<1, 128, 0>, "bf16", 128, bf * 128, sms, 1, it);
  run(bench_pair<256>, "nvf4 pair", 256, 2 * f4 * 256, 2 * (sms / 2), 2, it);
  run(bench_pair<128>, "nvf4 pair", 128, 2 * f4 * 128, 2 * (sms / 2), 2, it);
  run(bench_one<0, 256, 1>, "stage 1", 256, f4 * 256, sms, 1, it);
  run(bench_one<0, 256, 2>, "stage 2", 256, f4 * 256, sms, 1, it);
  run_st(false, sms, it);
  run_st(true, sms, it);
  run_copy(false, sms, it);
  run_copy(true, sms, it);
  run_pipe<4>(sms, it);
  run_pipe<6>(sms, it);
  run_tma<4>(sms, it);
  run_tma<6>(sms, it);
  run_sf<4, 1>(sms, it);
  run_sf<4, 2>(sms, it);
  run_tma<4>(sms, it, true);
  run_sf<4, 1>(sms, it, true);
  run_tma<4>(sms, it, true, 131072);
  run_tma<6>(sms, it, true, 131072);
  return 0;
}
