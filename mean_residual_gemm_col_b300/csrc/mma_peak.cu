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
  return 0;
}
