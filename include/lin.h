/*
 * lin.h -- C ABI of the GB300 (sm_103a) forward linear-layer library.
 *
 * The operations are the forward kernels of the page
 * "matmul ve matmul_residual -- Tiled Matrix Multiply (Forward)"
 * (llm.istanbul/learn/tr/03_linear_forward):
 *
 *   lin_matmul                       Y = X @ W            ("Ne Yapar?")
 *   lin_matmul_residual              Y = X @ W + R        ("Ne Yapar?": residual
 *                                                          added in the epilogue)
 *   lin_matmul_residual_swiglu_a     Y = (silu(GATE) * UP) @ W + R
 *                                    ("Ne Yapar?" and "Onemli Optimizasyonlar" 3:
 *                                     the SwiGLU product is formed while the A tile
 *                                     is loaded; the [M, K] hidden matrix is never
 *                                     written to memory)
 *   lin_*_w16                        the same with W stored as IEEE binary16
 *                                    (the page's list of forward kernels:
 *                                     "f16 weight versiyonu")
 *
 * silu(x) = x * sigma(x) with the stable, sign-branched sigmoid of the page
 * "ffn_gelu_backward ve ffn_swiglu_backward" (09_backward_ffn), section "SiLU'".
 *
 * Argument order follows the pages' bind-group tables ("Bind Group ABI"):
 * inputs, then Y, then the dims (M, N, K), then the stream.
 *
 * Conventions shared by every compute entry point
 * -----------------------------------------------
 * Layout      All matrices are dense and row-major with no padding:
 *             X, GATE, UP are [M, K]; W is [K, N] (N contiguous, the pages'
 *             own convention); R and Y are [M, N].
 * Types       X, GATE, UP, R, Y and the f32 W are IEEE binary32. W16 holds
 *             IEEE binary16 bit patterns (uint16_t), so this header needs no
 *             CUDA half type.
 * Memory      Every pointer is device memory of the current CUDA device,
 *             owned by the caller. The library keeps no reference after the
 *             call returns. The w16 forms run a persistent launch; when its
 *             last round would leave SMs idle it splits that round along K
 *             and takes a workspace for the f32 partial tiles (at most
 *             128 KiB per SM, 19 MiB on a 152-SM GB300) from a memory pool
 *             the library creates on first use of each device. The workspace
 *             is allocated and freed in stream order on `stream`, so calls
 *             on different streams never share it; the pool keeps freed
 *             memory for reuse. On a stream that is being captured into a
 *             graph the workspace is a graph memory node (cudaMallocAsync /
 *             cudaFreeAsync), owned by that graph. If no workspace can be
 *             had the launch runs unsplit (the same results up to the order
 *             in which the tail's K ranges are summed). The f32 forms split
 *             K when a problem has too few 128 x 128 tiles to fill the SMs:
 *             the (at most 8) CTAs of a tile form a cluster and add their
 *             partial tiles through distributed shared memory, in K order;
 *             no workspace, one kernel.
 *             lin_matmul_w16 and lin_matmul_residual_w16 also place a
 *             binary16 copy of X (M*K*2 bytes) in the workspace, written by
 *             a first kernel, when each row block of X feeds several
 *             clusters of output tiles along N (N > 1024 on a GB300) and
 *             K % 8 == 0; without the memory they round X inside the GEMM
 *             instead (the same results).
 *             lin_last_launch_info() reports what a call used.
 * Stream      Work is enqueued on `stream` (a cudaStream_t; NULL means the
 *             legacy default stream) and the call returns without waiting.
 *             Inputs must stay valid, and Y must not be read, until the
 *             stream reaches the call.
 * Arithmetic  The f32 forms run the contraction on the tensor cores in TF32
 *             (operands keep their 10 explicit mantissa bits) with float32
 *             accumulation. The w16 forms round the A operand (X, or
 *             silu(GATE) * UP) to binary16, round-to-nearest-even, and
 *             multiply binary16 x binary16 with float32 accumulation. The
 *             residual is added once in float32. A split tail sums its K
 *             ranges' float32 partial tiles in K order, so every call with
 *             the same inputs, device and stream state gives the same bits.
 *             Results satisfy
 *             max |Y - Y_exact| / sum_k |A[i,k] W[k,j]| <= 4e-3.
 *             Values of A beyond the binary16 range (|A| > 65504) become
 *             +-inf in the w16 forms.
 *
 * Validation (synchronous, before anything is enqueued) and error behaviour
 * ------------------------------------------------------------------------
 *   M < 0, N < 0 or K < 0, or a required pointer NULL -> LIN_ERROR_INVALID_VALUE
 *   M == 0 or N == 0                        -> LIN_SUCCESS, nothing enqueued
 *                                              (pointers are not inspected)
 *   K == 0                                  -> Y = R (or Y = 0 without a residual);
 *                                              X/GATE/UP/W are not read and may be NULL
 *   K % 4 != 0 or N % 4 != 0                -> LIN_ERROR_UNSUPPORTED_SHAPE
 *                                              (the pages' vec4 rule, "Vec4 Tile Loads")
 *   w16 forms: N % 8 != 0                   -> LIN_ERROR_UNSUPPORTED_SHAPE
 *                                              (a binary16 W row must be a multiple of
 *                                              16 bytes for the tensor-memory copies)
 *   M, N or K > 2^31 - 1                    -> LIN_ERROR_UNSUPPORTED_SHAPE
 *   any pointer not 16-byte aligned         -> LIN_ERROR_MISALIGNED
 *   a buffer that is not device memory of the current device, or whose
 *   allocation is smaller than its extent   -> LIN_ERROR_INVALID_VALUE
 *   Y overlapping any input                 -> LIN_ERROR_ALIASING (in-place
 *                                              residual included; the pages forbid a
 *                                              buffer bound both read and read_write)
 *   current device not sm_103               -> LIN_ERROR_UNSUPPORTED_DEVICE
 *   a CUDA runtime/driver failure           -> LIN_ERROR_CUDA (lin_last_cuda_error()
 *                                              returns the cudaError_t value)
 * On any error nothing is enqueued and Y is untouched.
 *
 * Device-side failures. Every wait inside the kernels is bounded (about one
 * second by default). A wait that runs out records LIN_ERROR_TIMEOUT in a
 * per-device status word and the kernel exits cleanly; the next
 * lin_get_device_status() call reports and clears it. This is never expected
 * on a correct build; it exists so a scheduling bug cannot hang the GPU.
 *
 * Checked build. The same sources compiled with LIN_DEVICE_CHECKS=1 (the
 * library liblin_checked.so, built beside liblin.so) check, inside the
 * kernels, every shared-memory stage and buffer index, TMEM column range,
 * TMA coordinate alignment, cluster peer rank, and every global index that
 * is not a TMA access (partial tiles, row partials, transform and loss
 * loads) against its buffer. A failed check skips the access and records
 * LIN_ERROR_DEVICE_CHECK with the site and the offending value (a skipped
 * load then makes a bounded wait run out: the kernel still exits cleanly);
 * lin_get_device_status() reports it and lin_last_device_check() tells
 * which. In liblin.so the checks compile away.
 *
 * Thread safety: every entry point may be called from several host threads.
 */
#ifndef LIN_H
#define LIN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *lin_stream_t;

typedef enum lin_status {
  LIN_SUCCESS = 0,
  LIN_ERROR_INVALID_VALUE = 1,
  LIN_ERROR_UNSUPPORTED_SHAPE = 2,
  LIN_ERROR_MISALIGNED = 3,
  LIN_ERROR_ALIASING = 4,
  LIN_ERROR_UNSUPPORTED_DEVICE = 5,
  LIN_ERROR_CUDA = 6,
  LIN_ERROR_TIMEOUT = 7,
  LIN_ERROR_DEVICE_CHECK = 8
} lin_status;

/* Y[M,N] = X[M,K] @ W[K,N]; X, W, Y binary32.
 * 03_linear_forward, "Ne Yapar?"; bind group "matmul" (X, W, Y, dims). */
lin_status lin_matmul(const float *X, const float *W, float *Y,
                      int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* Y = X @ W + R; R[M,N] binary32, must not overlap Y.
 * 03_linear_forward, "Ne Yapar?"; bind group "matmul_residual". */
lin_status lin_matmul_residual(const float *X, const float *W, const float *R, float *Y,
                               int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* Y = (silu(GATE) * UP) @ W + R; GATE, UP [M,K], W [K,N] (W_down), R [M,N].
 * K is the FFN width (d_ff). The product silu(GATE) * UP is formed on chip and
 * never stored. 03_linear_forward, "Ne Yapar?" and "Onemli Optimizasyonlar" 3;
 * bind group "matmul_residual_swiglu_a" (GATE, UP, W, R, Y, dims). */
lin_status lin_matmul_residual_swiglu_a(const float *GATE, const float *UP, const float *W,
                                        const float *R, float *Y,
                                        int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* lin_matmul with binary16 weights W16[K,N] (bit patterns). N % 8 == 0.
 * 03_linear_forward, forward kernel list: "matmul_w16". */
lin_status lin_matmul_w16(const float *X, const uint16_t *W16, float *Y,
                          int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* lin_matmul_residual with binary16 weights. N % 8 == 0.
 * 03_linear_forward, forward kernel list: "matmul_residual_w16". */
lin_status lin_matmul_residual_w16(const float *X, const uint16_t *W16, const float *R,
                                   float *Y, int64_t M, int64_t N, int64_t K,
                                   lin_stream_t stream);

/* lin_matmul_residual_swiglu_a with binary16 W_down. N % 8 == 0.
 * 03_linear_forward, forward kernel list: "matmul_residual_swiglu_a_w16". */
lin_status lin_matmul_residual_swiglu_a_w16(const float *GATE, const float *UP,
                                            const uint16_t *W16, const float *R, float *Y,
                                            int64_t M, int64_t N, int64_t K,
                                            lin_stream_t stream);

/* lin_matmul_residual_swiglu_a_w16 that allocates no device memory. The pages
 * have no counterpart: their engine has no such constraint. It exists for
 * callers that must not allocate while a call runs, for example a serving
 * loop that reserves all of its device memory up front, or code for which
 * growing a memory pool (which maps new memory, can fail, and can take
 * milliseconds the first time) is not acceptable.
 *
 * Same arguments, layouts, validation, errors and results as
 * lin_matmul_residual_swiglu_a_w16 (bitwise, for the same device). The one
 * difference is where the workspace of a split tail lives: in a static
 * 19 MiB array on each device (152 SMs x 128 KiB), which the library loads
 * with the module that holds it, instead of the library's memory pool. The
 * call makes no cudaMalloc/cudaFree or pool allocation and never reports
 * workspace bytes in lin_last_launch_info.
 *   Limit     a problem whose split would need more than 19 MiB (possible
 *             only on a device with more than 152 SMs) is rejected with
 *             LIN_ERROR_UNSUPPORTED_SHAPE before anything is enqueued.
 *   Set-up    the first call on a device that passes validation looks up
 *             the array's address (cudaGetSymbolAddress, which loads its
 *             module); make that first call before capturing a stream.
 *             The address is kept for that device's context and looked up
 *             again once the context has changed (after cudaDeviceReset,
 *             for example). A failed look-up returns LIN_ERROR_CUDA and is
 *             not remembered: the next call tries again.
 *   Zeroing   nothing in the array needs to start at zero: a call writes
 *             every byte of it that it reads first.
 *   Races     every call on a device shares the one array. Calls whose
 *             execution can overlap (on different streams, or from threads
 *             that do not order their streams) corrupt each other's
 *             results; calls on a single stream are ordered and safe. */
lin_status lin_matmul_residual_swiglu_a_w16_noalloc(const float *GATE, const float *UP,
                                                    const uint16_t *W16, const float *R,
                                                    float *Y, int64_t M, int64_t N, int64_t K,
                                                    lin_stream_t stream);

/* Backward of the linear layer, input gradient: dX[M,K] = dY[M,N] @ W[K,N]^T
 * (dY, W, dX binary32; TF32 tensor cores, f32 accumulate). The pages' backward
 * linear page is not part of the material; the operation is the adjoint of
 * lin_matmul (03_linear_forward, "Ne Yapar?"): for every X,
 * sum(lin_matmul(X, W) * dY) == sum(X * dX). Same layout conventions (row
 * major, W as the forward stores it), validation and errors as lin_matmul:
 * K % 4 == 0 and N % 4 == 0; dX may overlap no input. */
lin_status lin_matmul_t(const float *DY, const float *W, float *DX,
                        int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* dX += dY @ W^T: dX is read and written in place (the accumulating form
 * of a gradient reaching X through several branches). */
lin_status lin_matmul_t_acc(const float *DY, const float *W, float *DX,
                            int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* lin_matmul_t with binary16 weights W16[K,N] (bit patterns); dY is rounded
 * to binary16 for the f16 tensor cores, as X is in lin_matmul_w16.
 * N % 8 == 0. */
lin_status lin_matmul_t_w16(const float *DY, const uint16_t *W16, float *DX,
                            int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* dX += dY @ W16^T (in place), binary16 weights. N % 8 == 0. */
lin_status lin_matmul_t_acc_w16(const float *DY, const uint16_t *W16, float *DX,
                                int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* Backward of the linear layer, weight gradient: dW[K,N] = X[M,K]^T @ dY[M,N]
 * (X, dY, dW binary32; TF32 tensor cores, f32 accumulate; the contraction
 * runs over the M tokens). Like lin_matmul_t it is defined as the adjoint of
 * the forward product, here with respect to W: for every W,
 * sum(lin_matmul(X, W) * dY) == sum(W * dW). K % 4 == 0 and N % 4 == 0
 * (the row strides of X, dY and dW); M is free. dW may overlap no input. */
lin_status lin_matmul_at(const float *X, const float *DY, float *DW,
                         int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* dW += X^T @ dY, dW read and written in place (gradient accumulation over
 * micro-batches). */
lin_status lin_matmul_at_acc(const float *X, const float *DY, float *DW,
                             int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* Weight gradient of the SwiGLU down projection: dW[K,N] =
 * (silu(GATE) * UP)^T @ dY, GATE and UP [M,K] (K = d_ff), dY [M,N], dW [K,N]
 * (W_down's shape). The product silu(GATE) * UP is recomputed on chip, as in
 * the forward lin_matmul_residual_swiglu_a, and never stored; TF32 tensor
 * cores. K % 4 == 0, N % 4 == 0; M is free. */
lin_status lin_matmul_at_swiglu_a(const float *GATE, const float *UP, const float *DY,
                                  float *DW, int64_t M, int64_t N, int64_t K,
                                  lin_stream_t stream);

/* dW += (silu(GATE) * UP)^T @ dY, dW in place. */
lin_status lin_matmul_at_swiglu_a_acc(const float *GATE, const float *UP, const float *DY,
                                      float *DW, int64_t M, int64_t N, int64_t K,
                                      lin_stream_t stream);

/* Backward of the SwiGLU FFN's down projection and of the SwiGLU itself in
 * one call: dA = dY[M,N] @ W[K,N]^T (the input gradient of
 * lin_matmul_residual_swiglu_a, K = d_ff) is formed on chip and never
 * stored; the epilogue applies ffn_swiglu_backward of page 09_backward_ffn
 * ("SwiGLU backward", "ffn_swiglu_backward") element by element:
 *   dGATE = nan_guard(dA * UP * silu'(GATE)),  dUP = nan_guard(dA * silu(GATE)),
 *   silu'(x) = s * (1 + x * (1 - s)), s = the stable sigmoid of x,
 * nan_guard(x) = x if x is finite (|x| < FLT_MAX), else 0 (the pages'
 * shared preamble). GATE, UP, DGATE, DUP are [M,K] binary32, 16-byte
 * aligned; DGATE and DUP overlap nothing. Same shape rules and errors as
 * lin_matmul_t. */
lin_status lin_matmul_t_swiglu_backward(const float *DY, const float *W, const float *GATE,
                                        const float *UP, float *DGATE, float *DUP,
                                        int64_t M, int64_t N, int64_t K, lin_stream_t stream);

/* The same with binary16 W_down (dY rounded to binary16). N % 8 == 0. */
lin_status lin_matmul_t_swiglu_backward_w16(const float *DY, const uint16_t *W16,
                                            const float *GATE, const float *UP, float *DGATE,
                                            float *DUP, int64_t M, int64_t N, int64_t K,
                                            lin_stream_t stream);

/* lm_head and the fused cross-entropy of page 07_loss ("cross_entropy ve
 * sum_losses -- Fused Loss + dLogits") in one call. The logits X[M,K] @
 * W16[K,V] (binary16 W, X rounded to binary16) are written to DLOGITS [M,V]
 * and then replaced in place by
 *   dLogits[s,v] = ((p[v] - target_dist[v]) + 2 beta LSE p[v]) * inv_norm,
 *   p = softmax of the row, target_dist = (1 - alpha) one_hot(targets[s]) + alpha / V,
 * losses[s] = LSE - (1 - alpha) l[t] - alpha mean(l) + beta LSE^2 with
 * LSE = max + log(max(sum exp(l - max), 1e-30)), and *loss_sum = the sum of
 * the M losses (a fixed-order, reproducible sum). A target outside [0, V)
 * (padding) gives loss 0 and a zero dLogits row. The GEMM's epilogue keeps
 * per-row partials (max, sum of exponentials and sum of the logits over each
 * 256 columns), so the loss kernel reads each logits row once instead of
 * three times. targets: int32 [M]; losses: f32 [M]; loss_sum: one f32.
 * V % 8 == 0, K % 4 == 0; DLOGITS, losses and loss_sum overlap no input or
 * each other. Kernels: the GEMM (and its binary16 pre-pass) and the loss,
 * whose last CTA adds the losses (a separate sum kernel only when the call
 * could not get its 16-byte-per-partial workspace). */
lin_status lin_lm_head_cross_entropy_w16(const float *X, const uint16_t *W16,
                                         const int32_t *targets, float *DLOGITS, float *losses,
                                         float *loss_sum, int64_t M, int64_t V, int64_t K,
                                         float alpha, float beta, float inv_norm,
                                         lin_stream_t stream);

/* The SwiGLU FFN's gate and up projections from one read of X: GATE[M,N] =
 * X[M,K] @ WG16[K,N] and UP[M,N] = X[M,K] @ WU16[K,N] (binary16 weights, X
 * rounded to binary16 once for both), the producer of lin_matmul_residual_swiglu_a's
 * GATE and UP (N = d_ff). The pages do not describe it (03_linear_forward
 * lists the forward GEMMs only); it is the two matmul_w16 products computed
 * from one read of X: one launch over both products' tiles, or, for shapes
 * that run as CTA pairs, the binary16 pre-pass and one launch per product
 * (the same rounding of X and the same K order as lin_matmul_w16 where that
 * runs without a split tail). N % 8 == 0, K % 4 == 0; GATE and UP overlap
 * nothing. */
lin_status lin_gate_up_w16(const float *X, const uint16_t *WG16, const uint16_t *WU16,
                           float *GATE, float *UP, int64_t M, int64_t N, int64_t K,
                           lin_stream_t stream);

/*
 * Host-operand forms
 * ------------------
 * lin_<form>_host: the six forward forms above with every operand (X or GATE
 * and UP, W or W16, R, Y) in HOST memory, same layouts, arithmetic, bound
 * and shape rules. The pages' engine binds device buffers only; these entry
 * points are the library's own, for callers whose activations live on the
 * host. The call copies the operands to the device and Y back itself, in
 * blocks of whole 128-row tiles (about 64 MiB of operands and result per
 * block; lin_set_host_block_bytes changes it): the copy of block c+1 to the
 * device and of block c-1 back run on two copy streams of the library's
 * while the caller's stream runs the device form on block c. Each block is
 * one call of the device form on its rows (its own split tail, if any), so
 * results satisfy the same bound but need not equal the device form's bits
 * where that splits differently.
 * Memory      Operands are host memory, pinned (cudaHostAlloc /
 *             cudaHostRegister: the copies then overlap the GEMMs) or
 *             pageable (correct, but the runtime stages each copy and the
 *             call is then largely synchronous). Device or managed memory
 *             -> LIN_ERROR_INVALID_VALUE. Staging memory on the device (W
 *             once, then three blocks' worth of each other operand) is one
 *             stream-ordered allocation from the library's pool, taken and
 *             given back on `stream`.
 * Stream      Enqueued work ends on `stream`, which waits for the last copy
 *             back: host inputs must stay unchanged, and Y must not be read,
 *             until `stream` gets there (cudaStreamSynchronize).
 * Errors      Validation as for the device forms, before anything is
 *             enqueued (Y overlapping an input -> LIN_ERROR_ALIASING; the
 *             16-byte alignment rule does not apply to host operands);
 *             `stream` under graph capture -> LIN_ERROR_INVALID_VALUE. A
 *             CUDA failure part-way returns LIN_ERROR_CUDA after the blocks
 *             already enqueued; Y is then partly written.
 * lin_last_launch_info reports the kernels of all blocks and the staging
 * plus the largest per-block workspace.
 */
lin_status lin_matmul_host(const float *X, const float *W, float *Y,
                           int64_t M, int64_t N, int64_t K, lin_stream_t stream);
lin_status lin_matmul_residual_host(const float *X, const float *W, const float *R, float *Y,
                                    int64_t M, int64_t N, int64_t K, lin_stream_t stream);
lin_status lin_matmul_residual_swiglu_a_host(const float *GATE, const float *UP, const float *W,
                                             const float *R, float *Y,
                                             int64_t M, int64_t N, int64_t K,
                                             lin_stream_t stream);
lin_status lin_matmul_w16_host(const float *X, const uint16_t *W16, float *Y,
                               int64_t M, int64_t N, int64_t K, lin_stream_t stream);
lin_status lin_matmul_residual_w16_host(const float *X, const uint16_t *W16, const float *R,
                                        float *Y, int64_t M, int64_t N, int64_t K,
                                        lin_stream_t stream);
lin_status lin_matmul_residual_swiglu_a_w16_host(const float *GATE, const float *UP,
                                                 const uint16_t *W16, const float *R, float *Y,
                                                 int64_t M, int64_t N, int64_t K,
                                                 lin_stream_t stream);

/* Operand-plus-result bytes per block of the host-operand forms (rounded
 * down to whole 128-row tiles, at least one tile); 0 restores the default
 * (64 MiB). Process-wide; values from 1 to 65535 -> LIN_ERROR_INVALID_VALUE. */
lin_status lin_set_host_block_bytes(uint64_t bytes);

/* Static, NUL-terminated name of a status code ("LIN_SUCCESS", ...). Never NULL. */
const char *lin_status_string(lin_status status);

/* The cudaError_t value behind the calling thread's last LIN_ERROR_CUDA (0 if none). */
int lin_last_cuda_error(void);

/* What the last compute call made on the calling thread enqueued: the number
 * of kernels it launched (the GEMM, plus the binary16 pre-pass of X and the
 * split-tail sum where those run, plus the loss kernels of the lm_head form;
 * all blocks' kernels for a host-operand form; 0 if it enqueued none or
 * failed) and the workspace bytes it took from the library's pool. Either
 * pointer may be NULL. */
void lin_last_launch_info(int* kernels, uint64_t* workspace_bytes);

/* Waits for `stream`, then returns and clears the current device's status
 * word: LIN_SUCCESS, LIN_ERROR_TIMEOUT if a kernel gave up on a wait since
 * the last call, or LIN_ERROR_DEVICE_CHECK if a check of the checked build
 * failed first (the first failure is the one kept). Returns LIN_ERROR_CUDA if
 * the synchronisation itself fails. */
lin_status lin_get_device_status(lin_stream_t stream);

/* The check behind the calling thread's last LIN_ERROR_DEVICE_CHECK from
 * lin_get_device_status(): its site (1 TMA coordinate alignment, 2 operand
 * stage, 3 epilogue or staging buffer, 4 TMEM column, 5 partial-tile index,
 * 6 row-partial index, 7 other global index, 8 cluster peer rank, 9 barrier
 * slot, 99 the self-test) and the offending value; 0 and 0 if none. Either
 * pointer may be NULL. */
void lin_last_device_check(int *site, int64_t *value);

/* Self-test of the bounded waits: enqueues one small kernel whose data
 * producer is told never to start, so every consumer's wait runs out after
 * `timeout_us` microseconds (1 .. 10,000,000); the kernel records
 * LIN_ERROR_TIMEOUT and exits cleanly. Waits for `stream` and returns the
 * status word (then cleared): LIN_ERROR_TIMEOUT when the mechanism works.
 * No memory is touched. */
lin_status lin_selftest_wait_timeout(int64_t timeout_us, lin_stream_t stream);

/* Self-test of the device-check record: enqueues one single-thread kernel
 * that reports a failed check (site 99, value `value`) the way every check
 * of the checked build does, without touching any other memory. Waits for
 * `stream` and returns the status word (then cleared): LIN_ERROR_DEVICE_CHECK
 * when the mechanism works, after which lin_last_device_check() gives 99 and
 * `value`. Works in either build. */
lin_status lin_selftest_device_check(int64_t value, lin_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int lin_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIN_H */
