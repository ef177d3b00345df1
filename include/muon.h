/*
 * muon.h -- C ABI of libmuon.so: the Muon optimizer step on one GB300 GPU
 * (sm_103a).
 *
 * The method is the one the page "深入解析KellerJordan/modded-nanogpt中的训练架构
 * 与优化技术" (reposource.net) walks through:
 *   - section "Muon优化器：动量正交化技术": Muon = SGD momentum followed by
 *     orthogonalisation of the update with a Newton-Schulz iteration;
 *     constructor defaults lr = 0.02, momentum = 0.95, nesterov = True,
 *     ns_steps = 5; step(): momentum update, Newton-Schulz, parameter update.
 *   - section "Newton-Schulz正交化": zeropower_via_newtonschulz5(G, steps):
 *     X = G in bfloat16, then `steps` times A = X X^T, B = b A + c A A,
 *     X = a X + B X with (a, b, c) = (3.4445, -4.7750, 2.0315).
 * Readings of what that page leaves out (fixed here):
 *   - momentum: buf <- mu*buf + g; Nesterov: u <- g + mu*buf (new buf),
 *     otherwise u <- buf;
 *   - before iterating, X <- X / (||X||_F + 1e-7), the norm of the bfloat16 X,
 *     the quotient rounded to bfloat16;
 *   - a matrix with more rows than columns is transposed before iterating and
 *     transposed back after, so the Gram matrix A is min(R,C) square;
 *   - update: p <- p - lr * O (no weight decay, no shape-dependent lr).
 * Each of A, B and X is rounded once to bfloat16 (round to nearest even)
 * after its statement; products accumulate in fp32 on the tensor cores.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major and contiguous: element (i, j) of an R x C
 *     matrix is at offset i*C + j.
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps device memory between calls.  `stream`
 *     is a cudaStream_t (NULL = legacy default stream) owned by the caller.
 *   - Calls are asynchronous on `stream` and never synchronise, except
 *     muon_device_status().  A workspace must not be shared by calls that
 *     may overlap on the GPU.
 *   - Arguments are checked, and every launch is prepared (tensor maps
 *     encoded, grids sized), on the host before anything is enqueued: on
 *     any error code nothing has been enqueued and no buffer has been
 *     touched -- except when the CUDA runtime itself rejects a kernel launch
 *     (MUON_ERR_CUDA), after which earlier kernels of the same call may have
 *     been enqueued.
 *   - Device-side conditions (a non-finite norm, an expired bounded wait)
 *     are recorded in the workspace's status word and are read with
 *     muon_device_status().
 */
#ifndef MUON_H
#define MUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum muon_status {
  MUON_OK = 0,
  MUON_WARN_NONFINITE = 1,          /* a matrix had a non-finite norm; values propagate */
  MUON_ERR_INVALID_ARG = -1,        /* null pointer, size <= 0, bad dtype, ns_steps < 0 */
  MUON_ERR_MISALIGNED = -2,         /* a data pointer is not 16-byte aligned */
  MUON_ERR_ALIASING = -3,           /* byte ranges that are written overlap another operand */
  MUON_ERR_WORKSPACE_TOO_SMALL = -4,
  MUON_ERR_CUDA = -5,               /* a CUDA runtime call or launch failed */
  MUON_ERR_DEVICE_TIMEOUT = -6,     /* a bounded on-device wait expired (results invalid) */
  MUON_ERR_UNSUPPORTED_DEVICE = -7, /* the current device is not compute capability 10.3 */
  MUON_ERR_TOO_LARGE = -8,          /* a dimension exceeds 2^31-1 elements per row/matrix */
  MUON_ERR_SCRATCH_LIMIT = -9       /* ns5_noalloc: the call needs more than its static scratch */
} muon_status_t;

typedef enum muon_dtype { MUON_BF16 = 0, MUON_F32 = 1 } muon_dtype_t;

/* One 2-D weight matrix of a bank (the unit the Muon class's step() updates). */
typedef struct muon_mat_desc {
  float* param;        /* R x C fp32, updated in place: p <- p - lr * O */
  const void* grad;    /* R x C gradient, read only, dtype = grad_dtype */
  float* buf;          /* R x C fp32 momentum buffer, updated in place */
  int64_t rows, cols;  /* R, C > 0 */
  int32_t grad_dtype;  /* muon_dtype_t */
  int32_t reserved;    /* must be 0 */
} muon_mat_desc;

/* Bytes of device workspace muon_step needs for this bank (0 on invalid
 * arguments).  Depends only on the shapes. */
size_t muon_workspace_size(const muon_mat_desc* mats, int n_mats);

/* One Muon step on a bank of matrices (page above, section "Muon优化器：
 * 动量正交化技术", step(): momentum, Newton-Schulz, update).
 *   mats      host array of n_mats descriptors (read during the call only);
 *             param/grad/buf must be 16-byte aligned and must not overlap
 *             each other or another matrix's param/buf.
 *   lr, momentum, nesterov   as in the Muon constructor (nesterov 0 or 1).
 *   ns_steps  Newton-Schulz steps (>= 0; 0 gives O = X0).
 *   workspace device memory of at least muon_workspace_size() bytes,
 *             256-byte aligned; its contents on entry do not matter.
 * Matrices of equal (min(R,C), max(R,C)) form one shape class; each
 * Newton-Schulz phase runs as one persistent launch over all classes. */
muon_status_t muon_step(const muon_mat_desc* mats, int n_mats, float lr, float momentum,
                        int nesterov, int ns_steps, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Bytes of device workspace ns5 needs. */
size_t ns5_workspace_size(int batch, int64_t rows, int64_t cols);

/* zeropower_via_newtonschulz5 (page above, section "Newton-Schulz正交化") on a
 * strided batch: G is batch x rows x cols (dtype g_dtype), O is the same
 * shape in bfloat16 (written).  No momentum.  G and O must be 16-byte aligned
 * and must not overlap. */
muon_status_t ns5(const void* G, int g_dtype, void* O, int batch, int64_t rows, int64_t cols,
                  int ns_steps, void* workspace, size_t workspace_bytes, void* stream);

/* Same as ns5 for a list of differently shaped matrices G[i] -> O[i]
 * (rows[i] x cols[i]); one launch per phase for the whole list. */
muon_status_t ns5_bank(const void* const* G, const int32_t* g_dtype, void* const* O,
                       const int64_t* rows, const int64_t* cols, int n_mats, int ns_steps,
                       void* workspace, size_t workspace_bytes, void* stream);
size_t ns5_bank_workspace_size(const int64_t* rows, const int64_t* cols, int n_mats);

/* Synchronises `stream`, then reads the status word of `workspace` left by
 * the last call that used it: MUON_OK, MUON_WARN_NONFINITE or
 * MUON_ERR_DEVICE_TIMEOUT (MUON_ERR_CUDA if the synchronisation failed).
 * The word lives in the caller's workspace, so the workspace names the call
 * whose status is read (calls on one stream may use different workspaces). */
muon_status_t muon_device_status(const void* workspace, void* stream);

/* Prepared calls.  muon_step, ns5, ns5_bank and ns5_noalloc keep the
 * prepared launches of recent calls in host memory (at most 32; the least
 * recently used is dropped), keyed by the current device, the entry point,
 * ns_steps, the workspace address and every pointer and shape argument.
 * lr, momentum and nesterov are not part of the key.  A call with a known
 * key only checks workspace_bytes and enqueues: the planning, the checks
 * that depend on the key alone, the tensor-map encoding and the occupancy
 * queries are skipped.  A prepared call depends on nothing but its key, so
 * it stays valid when the caller frees memory and allocates it again at the
 * same addresses.  muon_plan_cache_clear() drops every prepared call (for
 * example to return the host memory); it is never needed for correctness.
 * Thread-safe. */
void muon_plan_cache_clear(void);

/* Static description of a status code. */
const char* muon_status_str(muon_status_t status);

/* Where ns5 keeps its bfloat16 buffers inside the workspace (for tests and
 * inspection): byte offsets of the two X buffers, of A and of B, the row
 * pitches in elements, and m = min(rows, cols), n = max(rows, cols).  After
 * ns5 with ns_steps = k >= 1: A and B hold step k's A and B (for m <= 768
 * only their 256 x 256 blocks on and above the diagonal: both are symmetric
 * and blocks below the diagonal are not written; wider ones whole), and X
 * buffer (k % 2) holds step k's X (m x n, transposed for tall input); with
 * k = 0, X buffer 0 holds X0. */
typedef struct muon_ws_layout {
  size_t x_offset[2];
  size_t a_offset;
  size_t b_offset;
  int64_t ldx, lda;
  int64_t m, n;
} muon_ws_layout;
muon_status_t ns5_workspace_layout(int batch, int64_t rows, int64_t cols, muon_ws_layout* out);

/* Process-wide knobs for tests and diagnostics.  Keys:
 *   "wait_budget_cycles"  clock64 cycles a kernel waits on one barrier
 *                         before giving up (default 4e9, about 2 s);
 *   "inject_stall"        1: the Newton-Schulz kernels' MMA warp issues
 *                         nothing, so their waits expire (tests the bounded
 *                         wait path; combine with a small budget);
 *   "wait_profile_buffer" device address of a zeroed int64 array of
 *                         3 x 256 x 8 entries, or 0 to switch off:
 *                         each Newton-Schulz kernel CTA adds clock64 cycles
 *                         spent waiting per role (producer for free stages,
 *                         MMA issuer for operands / for a drained
 *                         accumulator, epilogue for an accumulator), the
 *                         epilogue's busy cycles, the whole kernel's cycles,
 *                         its tile count and the MMA loop's cycles, in that
 *                         order, at ((kind x 256) + CTA index) x 8 with kind
 *                         0 Gram, 1 polynomial, 2 update;
 *   "record_kernel_events" 1: every kernel launch is bracketed by a pair of
 *                         CUDA events recorded on the caller's stream (read
 *                         with muon_kernel_times; not for use under stream
 *                         capture);
 *   "fail_tensor_map_encode" 1: every tensor-map encoding fails, and no
 *                         prepared call is used or kept (tests that a
 *                         failure while preparing enqueues nothing).
 * Returns 0 on success, -1 for an unknown key. */
int muon_set_debug(const char* key, long long value);

/* Device-side checks of the debug build (libmuon_debug.so, compiled with
 * MUON_DEBUG): its kernels check the ranges of their raw-pointer accesses
 * and the alignment of their TMA coordinates; a failed check skips the
 * access (a skipped copy makes the kernel's bounded wait expire) and is
 * counted instead of trapping.  Synchronises the device, writes the number
 * of failed checks since the last call to *failures and clears the
 * counters.  Returns 0 in the debug build, -1 in the release build (which
 * has no checks; *failures = 0) or for a null argument, -2 if reading the
 * counters failed. */
int muon_debug_check_failures(long long* failures);

/* Waits for the events recorded since the last call (see
 * "record_kernel_events") and returns, per kernel kind, the summed
 * milliseconds and the launch count: kind 0 momentum_cast, 1 normalise,
 * 2 Gram (A = X X^T), 3 polynomial (B = b A + c A A), 4 update
 * (X = a X + B X), 5 apply (O written by ns5, or p <- p - lr O for a step
 * with no iteration), 6 muon_step's last update (X = a X + B X with
 * p <- p - lr O applied in place of storing X), 7 fp8_mm's quantise pass,
 * 8 fp8_mm's product, 9 fp8_mm_backward's quantise-and-transpose pass,
 * 10 its two products (one launch), 11 its split-K reduction.  ms and launches are host
 * arrays of n_kinds entries; kinds at or above n_kinds are not reported.
 * Returns 0, or -1 on a bad argument or a failed event query. */
int muon_kernel_times(double* ms, int* launches, int n_kinds);

/* Size of the static device scratch array used by ns5_noalloc. */
#define MUON_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* ns5 without a workspace argument, for callers that cannot allocate device
 * memory: code hosted by a framework whose allocator owns the whole GPU and
 * forbids side allocations, or code on a latency-critical path where
 * cudaMalloc/cudaFree may synchronise the device.  The pages describe no
 * counterpart; this is a convenience of this library.
 *   G, g_dtype, O, batch, rows, cols, ns_steps, stream: exactly as in ns5;
 *   the caller still provides G and O.
 * The scratch ns5 would take from a workspace comes instead from one
 * file-scope device array of MUON_NOALLOC_SCRATCH_BYTES (64 MiB).  That array
 * occupies device memory on every GPU where the library's device code is
 * loaded until the process exits.  CUDA loads the library's device code
 * lazily: the first call made on a device loads it and reserves the array
 * there, which can fail with MUON_ERR_CUDA when the device is full, so make
 * one call at initialisation, before any stream capture on that device.
 * The array's address is looked up on every call with the caller's device
 * current (it can move after cudaDeviceReset); a device other than compute
 * capability 10.3 gets MUON_ERR_UNSUPPORTED_DEVICE before anything is
 * loaded.  Calls whose workspace need
 * (ns5_workspace_size(batch, rows, cols)) exceeds the array return
 * MUON_ERR_SCRATCH_LIMIT without launching anything; for example one 2048 x
 * 2048 matrix or up to seven 1024 x 1024 matrices fit.  Every call shares the
 * array and finds the previous call's contents in it (the call clears what
 * must start at zero); calls that may overlap on the GPU -- on different
 * streams or different host threads -- race on it and must be serialised by
 * the caller.  Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine.  The device status word lives inside the private array:
 * read it with ns5_noalloc_status, not muon_device_status. */
muon_status_t ns5_noalloc(const void* G, int g_dtype, void* O, int batch, int64_t rows,
                          int64_t cols, int ns_steps, void* stream);

/* Device status of the last ns5_noalloc call on the current device, as
 * muon_device_status reports a workspace's: synchronises `stream` (the
 * stream of that call), then returns MUON_OK, MUON_WARN_NONFINITE (a matrix
 * had a non-finite norm) or MUON_ERR_DEVICE_TIMEOUT (a bounded wait
 * expired, O is not valid).  MUON_ERR_UNSUPPORTED_DEVICE or MUON_ERR_CUDA
 * when the array cannot be found.  Allocates nothing (the word is copied
 * into a host variable). */
muon_status_t ns5_noalloc_status(void* stream);

/* One tensor of an Adam step: caller-owned DEVICE memory, contiguous. */
typedef struct adam_tensor_desc {
  float* param;        /* numel fp32 values, updated in place */
  const void* grad;    /* numel values of grad_dtype, read only */
  float* exp_avg;      /* first moment m, numel fp32, updated in place */
  float* exp_avg_sq;   /* second moment v, numel fp32, updated in place */
  int64_t numel;       /* > 0 */
  int32_t grad_dtype;  /* MUON_BF16 or MUON_F32 */
  int32_t reserved;
} adam_tensor_desc;

/* Adam step with cautious weight decay over a list of tensors: the
 * optimizer of the embedding-type parameters (bigram table, value
 * embeddings) that the page on the modded-nanogpt record
 * "2026-06-11_RecursiveFromBest" (lqnn.cn, news/184262), section "3.3 bigram
 * 与 value-embedding 银行上的 C-Optim / 谨慎 Adam", pairs with Muon: decay is
 * applied only where the update and the parameter agree in sign.  Adam is
 * the textbook algorithm.  Per element, t = step, bc1 = 1 - beta1^t,
 * bc2 = 1 - beta2^t:
 *   m <- beta1 m + (1 - beta1) g;   v <- beta2 v + (1 - beta2) g^2
 *   u  = (m / bc1) / (sqrt(v / bc2) + eps)
 *   p <- p - lr (u + weight_decay * p * mask)
 * with mask = (u > 0 and p > 0) or (u < 0 and p < 0) when `cautious` is
 * non-zero, mask = 1 otherwise (plain decoupled decay).  Arithmetic: float32,
 * each operation one IEEE-rounded operation in the order above, no fused
 * multiply-add; (1 - beta), bc1 and bc2 are formed in double from the float
 * arguments and rounded once to float.  Updates are independent per element,
 * so the result does not depend on the launch configuration.
 *   tensors, n_tensors  host array of descriptors (n_tensors = 0: no-op);
 *   step                1 for the first step (>= 1);
 *   beta1, beta2 in [0, 1); eps >= 0; lr, weight_decay finite.
 * Errors (nothing enqueued): MUON_ERR_INVALID_ARG (null pointer, numel <= 0,
 * bad dtype, step < 1, hyper-parameter out of range, beta^step rounding to
 * 1), MUON_ERR_MISALIGNED (a pointer not 16-byte aligned),
 * MUON_ERR_ALIASING (a written array overlaps another written array or a
 * gradient), MUON_ERR_TOO_LARGE, MUON_ERR_CUDA (launch failure).  Non-finite
 * values propagate.  Asynchronous on `stream` (a cudaStream_t); one launch
 * per 64 tensors; needs no workspace. */
muon_status_t adam_step(const adam_tensor_desc* tensors, int n_tensors, float lr, float beta1, float beta2,
                        float eps, float weight_decay, int step, int cautious, void* stream);

/* FP8 scaled matrix product, the forward of the page's FP8 matmul
 * (walk-through page, section "自定义FP8矩阵乘法实现"):
 *   x_f8 = E4M3(bf16(x / x_s)),  w_f8 = E4M3(bf16(w / w_s)),
 *   out  = bf16(x_s * w_s * (x_f8 . w_f8^T)), accumulated in fp32.
 * x: M x K bfloat16, w: N x K bfloat16, row-major, read only.  out: M x N
 * bfloat16; x_f8: M x K and w_f8: N x K E4M3 bytes (1 sign, 4 exponent, 3
 * fraction bits, no infinities; 0x7F / 0xFF are NaN), all row-major and
 * written.  The quotient is rounded once to bfloat16, then to E4M3 to
 * nearest even; a quotient past E4M3's rounding range (|q| > 464) becomes
 * NaN.  x_s and w_s: finite and positive.
 * Limits: K a positive multiple of 16 and N a multiple of 8 (16-byte rows
 * for the copy engine); M, N, K at most INT_MAX.  M = 0 or N = 0 is a no-op.
 * All pointers 16-byte aligned; outputs overlap neither each other nor the
 * inputs.  workspace: at least 256 bytes, 256-byte aligned, holding the
 * device status word (muon_device_status).  Asynchronous on `stream`;
 * nothing is allocated.
 * Returns MUON_OK, MUON_ERR_INVALID_ARG, MUON_ERR_MISALIGNED,
 * MUON_ERR_ALIASING, MUON_ERR_WORKSPACE_TOO_SMALL, MUON_ERR_TOO_LARGE,
 * MUON_ERR_UNSUPPORTED_DEVICE or MUON_ERR_CUDA. */
muon_status_t fp8_mm(const void* x, const void* w, float x_s, float w_s, void* out, void* x_f8, void* w_f8,
                     int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace fp8_mm_backward needs for these sizes (0 on invalid
 * sizes, 256 when a size is 0). */
size_t fp8_mm_backward_workspace_size(int64_t M, int64_t N, int64_t K);

/* Backward of the FP8 scaled product (walk-through page, section
 * "自定义FP8矩阵乘法实现", subsection "反向传播优化"): the output gradient is
 * cast to E5M2, which keeps a wider range than E4M3, and multiplied with the
 * forward's E4M3 operands:
 *   g_f8   = E5M2(bf16(g / grad_s)),
 *   grad_x = bf16(grad_s * w_s * (g_f8 . w_f8)),      M x K,
 *   grad_w = bf16(grad_s * x_s * (g_f8^T . x_f8)),    N x K,
 * products accumulated in fp32.  As on the page, the products read
 * transposed copies of g_f8, x_f8 and w_f8 (made in the workspace by one
 * pass that also quantises g), so both operands of every product are
 * K-major; the E5M2 x E4M3 products run on the tensor cores.  When the
 * grad_w product has few output tiles, its contraction over the M rows is
 * split into slices whose fp32 partial sums are added in slice order.
 * g: M x N bfloat16; x_f8: M x K and w_f8: N x K E4M3 codes (as fp8_mm
 * writes them), read only.  grad_x: M x K and grad_w: N x K bfloat16, and
 * g_f8: M x N E5M2 codes (1 sign, 5 exponent, 2 fraction bits; 0x7C / 0xFC
 * are infinities, 0x7D-0x7F / 0xFD-0xFF NaN), written.  The quotient is
 * rounded once to bfloat16, then to E5M2 to nearest even; from 61440 in
 * magnitude on (the midpoint between 57344 and 2^16) it becomes an infinity
 * of its sign.  x_s, w_s, grad_s: finite and positive.
 * Limits: M, N, K multiples of 16 (16-byte rows of every operand and copy),
 * at most INT_MAX.  K = 0 is a no-op; M = 0 or N = 0 writes zeros to the
 * other gradient (an empty sum).  All pointers 16-byte aligned; outputs
 * overlap neither each other, the inputs nor the workspace.  workspace:
 * fp8_mm_backward_workspace_size(M, N, K) bytes, 256-byte aligned (status
 * word, the transposed copies, the partial sums).  Asynchronous on
 * `stream`; nothing is allocated.
 * Returns MUON_OK, MUON_ERR_INVALID_ARG, MUON_ERR_MISALIGNED,
 * MUON_ERR_ALIASING, MUON_ERR_WORKSPACE_TOO_SMALL, MUON_ERR_TOO_LARGE,
 * MUON_ERR_UNSUPPORTED_DEVICE or MUON_ERR_CUDA. */
muon_status_t fp8_mm_backward(const void* g, const void* x_f8, const void* w_f8, float x_s, float w_s, float grad_s,
                              void* grad_x, void* grad_w, void* g_f8, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Assigns each matrix of a bank to one of `world` ranks, for running the
 * step on several GPUs, one process per GPU, each updating only the matrices
 * it owns (every matrix's step depends on that matrix alone, so no data is
 * exchanged during the step).  The page's own multi-GPU variant (section
 * "Muon优化器：动量正交化技术") gives each rank a slice of every size group;
 * here the split balances the Newton-Schulz work instead: matrices are taken
 * from the heaviest down (work of an R x C matrix, m = min, n = max:
 * m(m+1)n + m^2(m+1) + 2 m^2 n) and each goes to the rank with the least work
 * so far (lowest rank on ties).  Among matrices of equal work, identical
 * shapes are taken together (more rows first, then more columns, then bank
 * order), so each shape group is dealt out evenly.  No rank gets more than
 * one matrix's work above the mean.
 *   rows, cols  host arrays of n_mats dimensions (> 0);
 *   world       number of ranks (> 0);
 *   owner       host array of n_mats entries, written with ranks 0..world-1.
 * The result depends only on the arguments: every rank computes the same
 * assignment without communicating.  Host only: touches no GPU.  Returns
 * MUON_OK (also for n_mats == 0) or MUON_ERR_INVALID_ARG (n_mats < 0,
 * world <= 0, a null array, a dimension <= 0), in which case owner is not
 * written. */
muon_status_t muon_partition(const int64_t* rows, const int64_t* cols, int n_mats, int world, int* owner);

#ifdef __cplusplus
}
#endif

#endif /* MUON_H */
