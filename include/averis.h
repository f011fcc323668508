/*
 * averis.h -- C ABI of libaveris.so: the Averis mean-residual split NVFP4
 * linear layer (forward and backward) on NVIDIA B300 (sm_103a).
 *
 * The method: "The Curse and Blessing of Mean Bias in FP4-Quantized LLM
 * Training" (arXiv 2603.10444).  Citations below use these keys:
 *
 *  [P1-method]   paper.rainbus.top summary "均值偏置的诅咒与祝福：FP4量化大语言模型训练",
 *                section 方法步骤详情 (method details): mu_X = (1/l) 1^T X,
 *                X_R = X - 1 mu_X, independent quantization of mu, X_R, W,
 *                Y = 1 (mu_X W) + X_R W; the same for the output gradient D:
 *                dX = 1 (mu_D W^T) + D_R W^T, dW = X_R^T D_R + l mu_X^T mu_D.
 *  [P1-quant]    same page, background 块量化 (blockwise quantization) and
 *                FP4量化 (NVFP4 uses E2M1 elements).
 *  [P1-hadamard] same page, background Hadamard变换: 16x16 Hadamard on
 *                [l, m/16, 16].
 *  [P2-method]   paperlayer.ai summary "The Curse and Blessing of Mean Bias in
 *                FP4-Quantized LLM Training", section 3 Method: the mean is
 *                broadcast over tokens, never materialised.
 *
 * NVFP4 reading (the pages fix only "E2M1, one shared scale per block"):
 * 16-element blocks along the GEMM's contraction axis, one E4M3 block scale,
 * one binary32 tensor scale s_g = fl32(amax / 2688); every rounding is
 * round-to-nearest-even with saturation.  Dequantized value =
 * e2m1(code) * e4m3(scale) * s_g.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device memory of the current CUDA device,
 *    allocated and owned by the caller.  The library makes no allocation.
 *    Every context that loads it holds two file-scope device objects: a
 *    4-byte error word and the AVERIS_NOALLOC_SCRATCH_BYTES scratch array of
 *    averis_quantize_noalloc.  Per device, the library caches the SM count,
 *    those objects' device addresses and the kernel attributes it set.  These
 *    caches are keyed by device ordinal and are not rebuilt, so do not keep
 *    using the library on a device after cudaDeviceReset.
 *  - All work is enqueued on `stream`; a call returns as soon as it is
 *    enqueued.  The status reports argument errors (nothing is enqueued then)
 *    and launch errors.  Device-side wait timeouts are reported through
 *    averis_last_device_error().
 *  - bf16 inputs are row-major and 16-byte aligned; every device pointer must
 *    be 16-byte aligned (256-byte for workspaces).
 *  - Workspaces: the first AVERIS_WORKSPACE_CTRL_BYTES bytes of every
 *    workspace are a control block (tickets and running maxima) that must be
 *    zero before the workspace is first used; its place does not depend on
 *    the sizes of a call, so one workspace serves calls of any shape.  Every
 *    call that runs to completion leaves it zero again, including a call
 *    whose device-side waits gave up (AVERIS_ERR_TIMEOUT).  So zero-fill the
 *    control block once when allocating a workspace, and again only after a
 *    call that returned AVERIS_ERR_CUDA, since then some of its kernels may
 *    not have run.  The rest of a workspace is scratch.
 *  - Calls that share a workspace or an output must not overlap in time.
 *  - Sizes: cols of every NVFP4 tensor and the m, n of a linear layer must be
 *    multiples of 16; the token count l may be any value >= 1 (a partial last
 *    16-block along l is zero-padded).
 */
#ifndef AVERIS_H
#define AVERIS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  AVERIS_OK = 0,
  AVERIS_ERR_INVALID_ARG = 1,        /* bad size, null or misaligned pointer */
  AVERIS_ERR_UNSUPPORTED_ARCH = 2,   /* current device is not sm_10x */
  AVERIS_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed */
  AVERIS_ERR_WORKSPACE_TOO_SMALL = 4,
  AVERIS_ERR_TIMEOUT = 5,            /* a device-side wait gave up (see averis_last_device_error) */
  AVERIS_ERR_OUT_OF_BOUNDS = 6       /* a debug build's bounds check skipped an access (ditto) */
} averis_status;

/* Size of the control block at the head of every workspace (zero at rest). */
#define AVERIS_WORKSPACE_CTRL_BYTES 4352
/* The same for the workspaces of the grouped (mixture-of-experts) calls. */
#define AVERIS_GROUPED_WORKSPACE_CTRL_BYTES 278528

/* flags */
#define AVERIS_MEAN_SPLIT 1u  /* subtract the column mean (Averis); clear = vanilla NVFP4 */
#define AVERIS_HADAMARD16 2u  /* rotate 16-blocks along each contraction axis by H16/4 ([P1-hadamard]) */
#define AVERIS_OUT_BF16   4u  /* write Y / dX (and averis_gemm's output) as bf16; default binary32 */

/*
 * An NVFP4 tensor of logical shape [rows, cols], blocked along cols
 * ([P1-quant]).  All pointers are device pointers owned by the caller.
 *  codes        rows * averis_nvfp4_ld(cols) bytes, row-major; byte j of a row
 *               holds element 2j in its low nibble and 2j+1 in its high nibble
 *               (E2M1 code: bit 3 sign, bits 2..0 magnitude index).
 *  scales       averis_nvfp4_scale_bytes(rows, cols) bytes of E4M3 block
 *               scales, tiled for the tensor cores: tile (rb, kc) covers rows
 *               128*rb .. +127 and blocks 4*kc .. +3; it sits at byte
 *               512*(rb*ceil(cols/64) + kc) and stores (row r, block k) at
 *               16*(r%32) + 4*((r%128)/32) + (k%4).  Padding entries are 0.
 *  tensor_scale one binary32 s_g.
 */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  float* tensor_scale;
  int64_t rows;
  int64_t cols;
} averis_nvfp4;

/* Bytes per row of an NVFP4 code buffer: round_up(cols, 64) / 2. */
int64_t averis_nvfp4_ld(int64_t cols);
/* rows * averis_nvfp4_ld(cols). */
size_t averis_nvfp4_code_bytes(int64_t rows, int64_t cols);
/* 512 * ceil(rows/128) * ceil(cols/64). */
size_t averis_nvfp4_scale_bytes(int64_t rows, int64_t cols);

/*
 * Forward state: what the forward pass produces and the backward pass reads.
 * All buffers device, caller-owned, sized for an l x m activation:
 *  x_row  X_R blocked along m, shape [l, m]  (operand of Y; may be scratch after fwd)
 *  x_col  X_R^T blocked along l, shape [m, l] (operand of dW, kept for bwd)
 *  mu_q   mu_X quantized along m, shape [1, m] (unused in vanilla mode)
 *  mu     [m] binary32 column mean (unused in vanilla mode)
 *  mu_hat [m] dequantized mean, unrotated basis (the dW outer product's left vector)
 */
typedef struct {
  averis_nvfp4 x_row;
  averis_nvfp4 x_col;
  averis_nvfp4 mu_q;
  float* mu;
  float* mu_hat;
} averis_fwd_state;

/* Scratch bytes needed by averis_quantize / averis_quantize_weight for a rows x cols input. */
size_t averis_quantize_workspace_bytes(int64_t rows, int64_t cols, unsigned flags);

/*
 * averis_quantize -- the fused mean-split quantize pass ([P1-method] steps
 * mu = (1/l) 1^T T, T_R = T - 1 mu, independent Q_b of mu and T_R).
 *  x         device bf16 [rows, cols] row-major (rows = tokens l, cols = features).
 *  flags     AVERIS_MEAN_SPLIT: subtract the column mean (else T_R = T, and mu,
 *            mu_q, mu_hat are ignored and may be NULL); AVERIS_HADAMARD16.
 *  mu        device [cols] binary32 column mean (output).
 *  mu_q      NVFP4 [1, cols] of the mean (output; rotated basis under HADAMARD16).
 *  mu_hat    device [cols] dequantized mean in the unrotated basis (output).
 *  out_row   NVFP4 [rows, cols] of T_R blocked along cols (output, NULL to skip).
 *  out_col   NVFP4 [cols, rows] of T_R^T blocked along rows (output, NULL to skip).
 *  workspace device scratch of averis_quantize_workspace_bytes() bytes.
 * Kernels: a column-statistics pass, then the quantize pass (plus a rotated-
 * maximum pass under HADAMARD16, which replaces the statistics pass when the
 * mean split is off: both layouts then take their scales from the rotated
 * maxima alone).  With the environment variable
 * AVERIS_SINGLE_READ_QUANTIZE=1 set when the library first sees the device,
 * an input of at most 1024 tiles of 128 x 128 whose tiles all fit the
 * resident CTAs' shared memory (two CTAs of three tiles per SM), without
 * HADAMARD16, takes one cooperative launch instead, which reads x once.  Its
 * mu may differ from the two-launch path's in the last bit (the compensated
 * column sums are added in another order), and on the B300 it is no faster at
 * the sizes measured, so it is off by default.
 * Errors: INVALID_ARG (cols % 16, shapes of the outputs, alignment),
 * WORKSPACE_TOO_SMALL, UNSUPPORTED_ARCH, CUDA.
 */
averis_status averis_quantize(const void* x, int64_t rows, int64_t cols, unsigned flags,
                              float* mu, const averis_nvfp4* mu_q, float* mu_hat,
                              const averis_nvfp4* out_row, const averis_nvfp4* out_col,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * averis_quantize_weight -- W_bar = Q_b(W) ([P1-method]); no mean split.
 *  w       device bf16 [m, n] row-major (Y = X W).
 *  w_n     NVFP4 [m, n] blocked along n: the B operand of dX = D W^T (output).
 *  w_m     NVFP4 [n, m] blocked along m: the B operand of Y = X W (output).
 *  flags   AVERIS_HADAMARD16 rotates along the blocking axis; MEAN_SPLIT is ignored.
 */
averis_status averis_quantize_weight(const void* w, int64_t m, int64_t n, unsigned flags,
                                     const averis_nvfp4* w_n, const averis_nvfp4* w_m,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * averis_quantize_weight_grouped -- averis_quantize_weight for the experts of
 * a mixture-of-experts layer, all in one launch chain (one statistics launch
 * and one quantize launch per 64 experts, plus the rotated-maximum launch
 * under HADAMARD16): W_bar_e = Q_b(W_e), each expert with its own tensor
 * scales, the same bits as num_experts calls of averis_quantize_weight.
 *  w          device bf16 [num_experts, m, n] row-major: expert e's [m, n]
 *             weight starts at element e * m * n.
 *  w_n, w_m   host arrays of num_experts NVFP4 descriptors (device buffers),
 *             expert e's outputs as in averis_quantize_weight; either array
 *             may be NULL to skip that layout (not both).
 *  workspace  averis_quantize_weight_grouped_workspace_bytes() bytes; its
 *             first AVERIS_GROUPED_WORKSPACE_CTRL_BYTES must be zero before
 *             first use, and every call leaves them zero.
 * Errors: INVALID_ARG (num_experts < 1, n % 16, an output's shape or
 * alignment), WORKSPACE_TOO_SMALL, UNSUPPORTED_ARCH, CUDA.
 */
size_t averis_quantize_weight_grouped_workspace_bytes(int64_t num_experts, int64_t m, int64_t n);
averis_status averis_quantize_weight_grouped(const void* w, int64_t num_experts, int64_t m, int64_t n,
                                             unsigned flags, const averis_nvfp4* w_n, const averis_nvfp4* w_m,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * averis_rank1 -- the rank-one row r = deq(mu_q) deq(w)^T ([P1-method]: the
 * mu_bar W_bar and mu_bar W_bar^T terms), binary32.
 *  mu_q  NVFP4 [1, K];  w  NVFP4 [N, K] blocked along K;  out  device [N].
 */
averis_status averis_rank1(const averis_nvfp4* mu_q, const averis_nvfp4* w, float* out,
                           cudaStream_t stream);

/*
 * averis_gemm -- block-scaled NVFP4 GEMM on the tcgen05 tensor cores with the
 * Averis epilogue:
 *   out[i][j] = s_a s_b sum_k a[i][k] b[j][k] + col_add[j] + outer_scale * row_vec[i] * col_vec[j]
 *  a        NVFP4 [M, K];  b  NVFP4 [N, K] (both blocked along K; K >= 1 need not
 *           be a multiple of 16: the last block's padding is zero in both).
 *  col_add  device [N] or NULL (the broadcast mean term of Y and dX).
 *  row_vec, col_vec  device [M], [N] or both NULL (the l mu_X^T mu_D term of dW).
 *  out      device [M, ldo] binary32, or bf16 with AVERIS_OUT_BF16; ldo >= N,
 *           ldo * element size a multiple of 16 bytes.
 */
averis_status averis_gemm(const averis_nvfp4* a, const averis_nvfp4* b,
                          const float* col_add, const float* row_vec, const float* col_vec,
                          float outer_scale, void* out, int64_t ldo, unsigned flags,
                          cudaStream_t stream);

/* Scratch bytes of averis_linear_fwd / averis_linear_bwd (and the nvfp4_ ones). */
size_t averis_linear_fwd_workspace_bytes(int64_t l, int64_t m, int64_t n, unsigned flags);
size_t averis_linear_bwd_workspace_bytes(int64_t l, int64_t m, int64_t n, unsigned flags);

/*
 * averis_linear_fwd -- Y = 1 (mu_bar_X W_bar) + X_bar_R W_bar ([P1-method]
 * forward equation; the mean term is added in the GEMM epilogue, never
 * materialised, [P2-method]).
 *  x      device bf16 [l, m];  w_m  NVFP4 [n, m] from averis_quantize_weight.
 *  y      device [l, n] binary32 (bf16 with AVERIS_OUT_BF16).
 *  state  forward state (outputs), see averis_fwd_state.
 *  flags  AVERIS_MEAN_SPLIT must be set (see nvfp4_linear_fwd for vanilla).
 */
averis_status averis_linear_fwd(const void* x, int64_t l, int64_t m, int64_t n,
                                const averis_nvfp4* w_m, unsigned flags, void* y,
                                const averis_fwd_state* state,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * averis_linear_bwd -- dX = 1 (mu_bar_D W_bar^T) + D_bar_R W_bar^T and
 * dW = X_bar_R^T D_bar_R + l mu_bar_X^T mu_bar_D ([P1-method] gradient
 * equations; cross terms dropped as written there).
 *  d      device bf16 [l, n];  w_n  NVFP4 [m, n] from averis_quantize_weight.
 *  state  the forward state of the same layer.
 *  dx     device [l, m] binary32 (bf16 with AVERIS_OUT_BF16);  dw  device [m, n] binary32.
 */
averis_status averis_linear_bwd(const void* d, int64_t l, int64_t m, int64_t n,
                                const averis_fwd_state* state, const averis_nvfp4* w_n,
                                unsigned flags, void* dx, float* dw,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Vanilla NVFP4 linear layer, the comparison path: Y = Q(X) Q(W),
 * dX = Q(D) Q(W)^T, dW = Q(X)^T Q(D).  Same arguments as the Averis calls;
 * AVERIS_MEAN_SPLIT is ignored, state.mu / mu_q / mu_hat are unused.
 */
averis_status nvfp4_linear_fwd(const void* x, int64_t l, int64_t m, int64_t n,
                               const averis_nvfp4* w_m, unsigned flags, void* y,
                               const averis_fwd_state* state,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);
averis_status nvfp4_linear_bwd(const void* d, int64_t l, int64_t m, int64_t n,
                               const averis_fwd_state* state, const averis_nvfp4* w_n,
                               unsigned flags, void* dx, float* dw,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Grouped (mixture-of-experts) linear layer: the same layer applied to each
 * expert's own tokens with the expert's own weights ([P1-method] per expert:
 * the means are taken over that expert's tokens).  The pages train a
 * Qwen3-7B-A1.5B MoE model with the method (paperlayer.ai summary, section 4
 * Experiments).
 *  x / d         device bf16 [L, m] / [L, n], rows grouped by expert: expert e
 *                owns rows offsets[e] .. offsets[e+1]-1 (L = offsets[E]).
 *  offsets       HOST array of E+1 non-decreasing row offsets, offsets[0] = 0;
 *                an expert with no rows is skipped (its state and dW untouched).
 *  w_m / w_n     HOST arrays of E NVFP4 descriptors (device buffers), as for
 *                averis_linear_fwd / averis_linear_bwd.
 *  states        HOST array of E forward states, expert e's sized for its rows.
 *  y / dx        device [L, n] / [L, m], the rows grouped like x;  dw  HOST
 *                array of E device pointers to binary32 [m, n].
 *  workspace     averis_grouped_linear_*_workspace_bytes() bytes; its first
 *                AVERIS_GROUPED_WORKSPACE_CTRL_BYTES bytes are its control
 *                block (zero before first use, left zero by every call).
 *                All experts are quantized together (one launch per pass for
 *                up to 64 experts) and their GEMMs run in one persistent
 *                launch per product (Y; dX; dW).
 *  flags         AVERIS_MEAN_SPLIT (clear: vanilla NVFP4), AVERIS_HADAMARD16,
 *                AVERIS_OUT_BF16.
 */
size_t averis_grouped_linear_fwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m,
                                                 int64_t n, unsigned flags);
size_t averis_grouped_linear_bwd_workspace_bytes(const int64_t* offsets, int64_t num_experts, int64_t m,
                                                 int64_t n, unsigned flags);
averis_status averis_grouped_linear_fwd(const void* x, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_nvfp4* w_m, unsigned flags, void* y,
                                        const averis_fwd_state* states, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);
averis_status averis_grouped_linear_bwd(const void* d, const int64_t* offsets, int64_t num_experts, int64_t m,
                                        int64_t n, const averis_fwd_state* states, const averis_nvfp4* w_n,
                                        unsigned flags, void* dx, float* const* dw, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);

/*
 * averis_quantize_noalloc -- averis_quantize without a caller-supplied
 * workspace.  The method has no counterpart of this call: it exists for
 * callers that cannot allocate device memory, such as plugin hosts that hand
 * an operator only its input and output buffers and own every other
 * allocation, or code that must not call cudaMalloc because it implicitly
 * synchronizes the device.
 *
 * Arguments, outputs and results are those of averis_quantize (same kernels,
 * same bits).  The scratch is one file-scope device array of
 * AVERIS_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.  The call allocates nothing.
 *  - The first call on a device looks up that array's device address (once per
 *    device, with the device current); make that first call before any stream
 *    capture.
 *  - Every call shares the one array, and it keeps the previous call's
 *    contents; the kernels clear the part that must start at zero.  Calls
 *    whose work overlaps on the GPU (other streams, other host threads) race
 *    on the array and give wrong results: order them on one stream.
 *  - Sizes whose scratch need, averis_quantize_workspace_bytes(rows, cols, flags),
 *    exceeds AVERIS_NOALLOC_SCRATCH_BYTES return AVERIS_ERR_WORKSPACE_TOO_SMALL
 *    and enqueue nothing.
 */
#define AVERIS_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
averis_status averis_quantize_noalloc(const void* x, int64_t rows, int64_t cols, unsigned flags,
                                      float* mu, const averis_nvfp4* mu_q, float* mu_hat,
                                      const averis_nvfp4* out_row, const averis_nvfp4* out_col,
                                      cudaStream_t stream);

/* Human-readable name of a status. */
const char* averis_status_string(averis_status status);

/*
 * Reads and clears the device error word that kernels set when a bounded
 * wait gives up (about one second of SM clock).  Synchronizes `stream`.
 * Returns AVERIS_OK or AVERIS_ERR_TIMEOUT; *where (if not NULL) receives the
 * code of the wait that gave up:
 *   1 GEMM TMA producer, 2 GEMM MMA issuer, 3 GEMM epilogue, 4 GEMM drain,
 *   5 quantize pass (an input box or tile never arrived), 6 GEMM scale feed,
 *   7 single-read quantize (a grid-wide wait for its other CTAs gave up).
 * In a library built with its bounds checks (averis_debug_checks() == 1) the
 * word can also hold 100 + site of the first access a check caught and
 * skipped; it then returns AVERIS_ERR_OUT_OF_BOUNDS.  Sites: 1-3 statistics
 * pass (partials, their combine, the mean), 4-6 mean CTAs (mean loads, NVFP4
 * mean, dequantized mean), 7-8 rank-one row (weights, output), 9-11 quantize
 * pass (row codes, column codes, scale atoms), 12 single-read quantize
 * partials, 13 GEMM epilogue vectors, 14 a TMA copy's inner coordinate off the
 * 16-byte rule, 15 averis_rank1's output.
 * The results of the calls that timed out are invalid.  When it reports a
 * timeout it also zeroes the control block of averis_quantize_noalloc's
 * scratch, whose callers cannot reach it.
 */
averis_status averis_last_device_error(cudaStream_t stream, int* where);

/*
 * averis_debug_starve_next_quantize -- diagnostics of the timeout path.  The
 * method has no counterpart of this call.  The next averis_quantize,
 * averis_quantize_weight or averis_quantize_noalloc call, or the next quantize
 * step of a linear call, from any host thread, runs its statistics pass without
 * requesting its input.  Every bounded wait of that pass for its input then
 * gives up after `wait_cycles` SM clock cycles.  That call's results are
 * invalid, and averis_last_device_error then reports AVERIS_ERR_TIMEOUT with
 * code 5.  The workspace's control block is left zero for the next call.  Only
 * a host-side switch: no copy is left in flight and nothing faults on the GPU.
 * wait_cycles must lie in [1e4, 2^31]; otherwise AVERIS_ERR_INVALID_ARG.
 */
averis_status averis_debug_starve_next_quantize(long long wait_cycles);

/* Library version, major*10000 + minor*100 + patch. */
int averis_version(void);

/*
 * averis_debug_checks -- whether the loaded library checks its kernels' memory
 * accesses.  The method has no counterpart of this call: it serves testing on
 * machines without a memory checker.  Built with -DAVERIS_DEBUG (the
 * libaveris_debug.so of the build script), every kernel checks each global
 * address it computes against the extent of its buffer, and the inner
 * coordinate of each TMA copy against the 16-byte rule; a failed check skips
 * the access and records its site (averis_last_device_error).  Returns 0 for
 * a release build (no checks compiled in).  In a debug build it first runs a
 * one-thread self-test on the current device -- the bounds predicate on
 * in-range and out-of-range (offset, extent) pairs, with no memory access,
 * and one recorded site read back and cleared -- and returns 1 if it passed,
 * -1 if not, or if an error was already pending (which it leaves in place)
 * or a CUDA call failed.  Synchronizes the device.
 */
int averis_debug_checks(void);

#ifdef __cplusplus
}
#endif
#endif /* AVERIS_H */
