/*
 * ttc — tiled tensor-core GEMM for GB300 (sm_103a), C ABI.
 *
 * Computes  D = act(alpha * A * B + beta * C + bias)  on one GPU.
 *
 * Sources the operation follows (CUTLASS / CuTe tutorial pages):
 *   - "CUTLASS tutorial: from hand-written GEMM to CuTe / Tensor Core kernels"
 *     (hpc.payai.win/cutlass), section 1: the GEMM C[M,N] = A[M,K] x B[K,N]
 *     mapped onto CTA tiles, and its Epilogue box (alpha/beta, then
 *     bias/activation, then store);
 *   - same page, section 2: device::Gemm is the host entry point and behaves
 *     like cuBLAS (alpha scales A*B, beta scales the existing C);
 *   - PitchLinearStripminedThreadMap source walkthrough (lpnh.cn/news/2469163),
 *     sections 4.1 and 6.3: an element's address is its row times the pitch
 *     plus its column, with the pitch taken from the tensor's layout.
 *
 * Storage.  A is M x K, B is K x N (logical).  TTC_ROW_MAJOR places element
 * (i, j) at i * ld + j; TTC_COL_MAJOR places it at i + j * ld.  C and D are
 * M x N, row-major, with leading dimensions ldc and ldd.  For TTC_F16 and
 * TTC_BF16, C and D have the input type and the product is accumulated in
 * fp32.  For TTC_I8, A and B are int8 and C and D are int32; the result is
 * exact.  bias is fp32[N] (added per output column) or NULL.  Only D's M x N
 * elements are written: the pitch padding of its rows (columns N .. ldd - 1)
 * and any memory between batches keep their contents.
 *
 * Ownership.  Every pointer is caller-owned device memory.  The library keeps
 * no reference to any of it after the call returns and allocates no device
 * memory; ttc_gemm_ws uses only the workspace its caller passes.
 *
 * Asynchrony.  ttc_gemm only enqueues work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and returns.  Calls on different host threads
 * are safe.  Work on one stream keeps stream order: the kernels are launched
 * with programmatic dependent launch (TTC_KNOB_PDL), so a kernel may begin
 * its set-up while the previous kernel on the stream finishes, but it reads
 * and writes global memory only after that kernel has completed.  The calls
 * may be captured into a CUDA graph: run each kind of call once outside a
 * capture first, since the first use of a kernel variant on a device sets its
 * shared-memory attribute and caches its occupancy.
 *
 * Errors.  Every entry point returns a status; none aborts or throws.
 *   TTC_ERR_INVALID_ARG: negative sizes; a leading dimension below the
 *     contiguous extent (A row-major lda < K, column-major lda < M; B
 *     row-major ldb < N, column-major ldb < K; ldc < N when C is read;
 *     ldd < N); NULL A or B when M*N*K > 0; NULL D when M*N > 0; NULL C with
 *     beta != 0; D overlapping C other than exactly in place (D == C and
 *     ldd == ldc); an unknown enum value.
 *   TTC_ERR_UNSUPPORTED: TTC_I8 with bias, act != NONE, alpha != 1 or beta
 *     not in {0, 1}; a size or leading dimension beyond 2^31 - 2^24 elements.
 *   TTC_ERR_CUDA: a CUDA runtime or driver call failed (launch, device query).
 *   TTC_ERR_TIMEOUT: returned by ttc_get_device_error when a kernel's bounded
 *     wait ran out; the kernel then ended early and D is undefined.
 *   TTC_ERR_SCRATCH_TOO_SMALL: ttc_gemm_static_scratch only: the operands need
 *     more scratch than its fixed array holds.
 * M == 0 or N == 0 is a no-op returning TTC_OK.  K == 0 gives
 * D = act(beta * C + bias).  beta == 0 never reads C (NaNs in C do not
 * propagate).
 */
#ifndef TTC_H_
#define TTC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TTC_OK = 0,
  TTC_ERR_INVALID_ARG = 1,
  TTC_ERR_UNSUPPORTED = 2,
  TTC_ERR_CUDA = 3,
  TTC_ERR_TIMEOUT = 4,
  TTC_ERR_SCRATCH_TOO_SMALL = 5
} ttc_status;

typedef enum { TTC_ROW_MAJOR = 0, TTC_COL_MAJOR = 1 } ttc_layout;

typedef enum { TTC_ACT_NONE = 0, TTC_ACT_RELU = 1, TTC_ACT_GELU_TANH = 2 } ttc_act;

typedef enum { TTC_F16 = 0, TTC_BF16 = 1, TTC_I8 = 2 } ttc_dtype;

/*
 * D = act(alpha * A * B + beta * C + bias).  See the file comment for the
 * meaning, layout, ownership and error behaviour of every argument.
 * act: NONE, RELU = max(v, 0), GELU_TANH = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))).
 * stream: a cudaStream_t passed as void*.
 */
ttc_status ttc_gemm(int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda, ttc_layout layoutA,
                    const void* B, int64_t ldb, ttc_layout layoutB,
                    const void* C, int64_t ldc,
                    void* D, int64_t ldd,
                    float alpha, float beta, const float* bias,
                    ttc_act act, ttc_dtype dtype, void* stream);

/*
 * Strided batched GEMM: for b in [0, batch),
 *   D_b = act(alpha * A_b * B_b + beta * C_b + bias)
 * where operand X_b starts strideX elements after X_0 (X = A, B, C, D) and
 * every matrix has the layout and leading dimension given, as in ttc_gemm.
 * A stride of 0 shares that operand among all batches (e.g. one B for every
 * A_b); bias is shared.  The batches form one launch: their tiles are walked
 * together by the persistent kernels.  The pages name batched layouts as a
 * use of layout composition ("Advanced CUTLASS Architecture and Kernel
 * Optimization", Functional Composition: a layout for matrices composed with
 * one for how matrices are batched).
 * Errors as ttc_gemm, plus TTC_ERR_INVALID_ARG for a negative batch or stride,
 * or (batch > 1) a strideD below (M - 1) * ldd + N so that D batches would
 * overlap; a C that aliases D in place needs strideC == strideD.  batch == 0
 * is a no-op.  batch > 65535 is TTC_ERR_UNSUPPORTED.
 */
ttc_status ttc_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                    const void* A, int64_t lda, int64_t strideA, ttc_layout layoutA,
                                    const void* B, int64_t ldb, int64_t strideB, ttc_layout layoutB,
                                    const void* C, int64_t ldc, int64_t strideC,
                                    void* D, int64_t ldd, int64_t strideD,
                                    float alpha, float beta, const float* bias,
                                    ttc_act act, ttc_dtype dtype, void* stream);

/*
 * Implicit-GEMM 2-D convolution, forward: the convolution run as a GEMM whose
 * rows are output pixels and whose reduction runs over filter tap x channel,
 * the A operand gathered from the input on the fly and never stored (the
 * implicit-GEMM view described in section 5.2 of the
 * PitchLinearStripminedThreadMap walkthrough, lpnh.cn/news/2469163).  With
 *   P = (H + 2 pad_h - dil_h (R - 1) - 1) / stride_h + 1   (Q likewise)
 * and m = (n P + p) Q + q it computes, for every m < N P Q and k < K,
 *   D[m ldd + k] = act(alpha acc + beta Cm[m ldc + k] + bias[k]),
 *   acc = sum over r < R, s < S, c < C of
 *         X[n, p stride_h - pad_h + r dil_h, q stride_w - pad_w + s dil_w, c] * Wt[k, r, s, c]
 * (cross-correlation; taps outside the H x W input count as zero).
 * Layouts: X is N x H x W x C (NHWC) and Wt is K x R x S x C (KRSC), both tightly
 * packed; Cm and D are (N P Q) x K row-major with pitches ldc, ldd >= K (the
 * NPQK output).  fp16 or bf16 in and out, fp32 accumulation; bias fp32[K] or
 * NULL; Cm read only when beta != 0 (it may equal D with ldc == ldd).
 * Asynchronous on `stream`; allocates nothing; the caller owns every buffer.
 * TTC_ERR_INVALID_ARG for negative sizes, zero strides or dilations, a filter
 * larger than the padded input, NULL or misaligned pointers, pitches below K,
 * D overlapping X or Cm; TTC_ERR_UNSUPPORTED for int8 or extents beyond int
 * range.  N == 0 or K == 0 is a no-op; C == 0 leaves the epilogue of a zero
 * sum.
 */
ttc_status ttc_conv2d_fprop(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K,
                            int64_t R, int64_t S, int64_t pad_h, int64_t pad_w,
                            int64_t stride_h, int64_t stride_w, int64_t dil_h, int64_t dil_w,
                            const void* X, const void* Wt, const void* Cm, int64_t ldc,
                            void* D, int64_t ldd, float alpha, float beta, const float* bias,
                            ttc_act act, ttc_dtype dtype, void* stream);

/*
 * Out-of-place transpose: dst (cols x rows, row-major, pitch ldd) = src
 * (rows x cols, row-major, pitch lds)^T, for elements of elem_bytes = 1, 2,
 * 4 or 8 bytes (bit copies).  The layout-only transpose kernel of "4.21 What
 * is CuTe?" (gpu-glossary-zh): a tile split among a row-major (8, 32) thread
 * grid and written back through the transposed view.  Asynchronous on
 * `stream`; allocates nothing.  TTC_ERR_INVALID_ARG for negative sizes, an
 * unsupported element size, NULL pointers, lds < cols, ldd < rows, pointers
 * not aligned to the element size, or overlapping source and destination.
 * rows == 0 or cols == 0 is a no-op.
 */
ttc_status ttc_transpose(int64_t rows, int64_t cols, const void* src, int64_t lds,
                         void* dst, int64_t ldd, int elem_bytes, void* stream);

/*
 * As ttc_gemm, with caller-provided device workspace.  An operand that TMA
 * cannot read (a base not 16-byte aligned, or a pitch in bytes that is not a
 * multiple of 16: the tight leading dimensions of odd-sized matrices) is first
 * copied into the workspace with a padded pitch, on `stream`, so the GEMM runs
 * on the TMA-staged path.  The workspace must be 256-byte aligned, at least
 * ttc_gemm_workspace_size() bytes, and not touched by anything else until the
 * work enqueued on `stream` has finished; its contents are scratch.  With a
 * NULL, misaligned or too small workspace the call behaves exactly like
 * ttc_gemm (operands TMA cannot read are then loaded with plain loads inside
 * the GEMM kernel, which is correct but slower).
 * The repacking follows the pitch rule of the PitchLinearStripminedThreadMap
 * walkthrough (lpnh.cn/news/2469163), sections 4.4 and 6.3: 16-byte vector
 * access needs a 16-byte-aligned start, so the pitch is padded.
 */
ttc_status ttc_gemm_ws(int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, ttc_layout layoutA,
                       const void* B, int64_t ldb, ttc_layout layoutB,
                       const void* C, int64_t ldc,
                       void* D, int64_t ldd,
                       float alpha, float beta, const float* bias,
                       ttc_act act, ttc_dtype dtype,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes ttc_gemm_ws uses for these operands: 0 when TMA can read
 * both, for matrix-vector problems (one output row or column, fp16/bf16, with
 * the matrix operand's reduction or its outputs contiguous, the latter from
 * 1024 outputs or for K up to 8192: their kernels read the operands with
 * plain loads and need no workspace), and for invalid or empty arguments.
 * Pure host computation.
 */
size_t ttc_gemm_workspace_size(int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, ttc_layout layoutA,
                               const void* B, int64_t ldb, ttc_layout layoutB,
                               ttc_dtype dtype);

/*
 * Workspace bytes for ttc_gemm_ws's fastest path: ttc_gemm_workspace_size's
 * operand repack plus, for an int32 D (int8 problems) whose rows cannot be
 * written as 16-byte vectors (ldd times 4, or D itself, not a multiple of 16
 * bytes), an aligned copy of D placed after it.  Given a workspace at least
 * this large, ttc_gemm_ws copies C (when beta != 0) into that copy, runs the
 * GEMM on it in place and copies the result to D, all on `stream`; with less
 * it behaves as with ttc_gemm_workspace_size bytes.  The result is the same
 * either way.  fp16/bf16 outputs need no copy: the GEMM writes rows at any
 * 2-byte boundary itself.  0 for invalid or empty arguments and for
 * matrix-vector problems (which use no workspace).
 * int8 problems of at least 64 tiles of 256 x 256 (TTC_KNOB_I8_WIDE) whose
 * operands TMA can read as int8 and whose D it can write as int32 instead
 * get fp16 copies of A and B (2 bytes per element, rows padded to 16
 * elements): given that much, ttc_gemm_ws widens the operands into them and
 * runs the product on the CTA-pair kernel, exactly as before (int8 values
 * and products are exact in fp16 and fp32, and the kernel adds 1024-deep
 * partial sums as int32).  Pure host computation.
 */
size_t ttc_gemm_workspace_size_staged(int64_t M, int64_t N, int64_t K,
                                      const void* A, int64_t lda, ttc_layout layoutA,
                                      const void* B, int64_t ldb, ttc_layout layoutB,
                                      const void* D, int64_t ldd, ttc_dtype dtype);

/*
 * Size of the fixed device scratch array ttc_gemm_static_scratch uses: 16 MiB.
 */
#define TTC_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * ttc_gemm_ws for callers that cannot allocate device memory.  The pages this
 * library follows have no counterpart of this entry point.
 *
 * Who needs it: code that may not call cudaMalloc at all, for example a plugin
 * running inside a host application or framework that has reserved the
 * device's memory for its own pool, or a latency-critical path where the
 * implicit device-wide synchronisation of cudaMalloc/cudaFree is not
 * acceptable.  Such a caller cannot hand ttc_gemm_ws a workspace.
 *
 * What it does: exactly ttc_gemm_ws, with the workspace taken from a fixed
 * array of TTC_STATIC_SCRATCH_BYTES in device memory that the library
 * declares statically.  That array exists on every GPU that loads the library
 * and stays allocated until the process exits.  This call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *
 * Limit: a problem whose operands need more scratch than
 * TTC_STATIC_SCRATCH_BYTES (ttc_gemm_workspace_size() tells how much) is
 * rejected with TTC_ERR_SCRATCH_TOO_SMALL before any work is enqueued; operands
 * TMA can read need no scratch at all.
 *
 * Set-up: the first call on a device looks up the array's device address on
 * that device (with that device current) and caches it; make that first call
 * before any stream capture on the device.
 *
 * Sharing: every call uses the same array, which keeps whatever the previous
 * call left there; nothing in it has to start at zero (each call overwrites
 * all the scratch it reads).  Calls whose work overlaps on the GPU (concurrent
 * streams, or another host thread) race on the array: order them, for example
 * by issuing them on one stream.
 */
ttc_status ttc_gemm_static_scratch(int64_t M, int64_t N, int64_t K,
                                   const void* A, int64_t lda, ttc_layout layoutA,
                                   const void* B, int64_t ldb, ttc_layout layoutB,
                                   const void* C, int64_t ldc,
                                   void* D, int64_t ldd,
                                   float alpha, float beta, const float* bias,
                                   ttc_act act, ttc_dtype dtype, void* stream);

/*
 * Synchronizes `stream`, then returns and clears the device error word that
 * the library's kernels set when a bounded wait runs out (TTC_ERR_TIMEOUT), or
 * TTC_OK.  A CUDA error seen while synchronizing is returned as TTC_ERR_CUDA.
 * The word is per device, shared by all streams.
 */
ttc_status ttc_get_device_error(void* stream);

/* A static, human-readable name for a status code. */
const char* ttc_status_string(ttc_status status);

/*
 * Debug and test knobs (not needed for normal use).  Process-wide; read at
 * every ttc_gemm call.
 *   TTC_KNOB_TIMEOUT_NS: budget of every in-kernel barrier wait (default
 *     2e9 ns); values <= 0 restore the default.
 *   TTC_KNOB_INJECT_STALL: when 1, the next kernels make their tensor-core
 *     issuer wait on a barrier that nothing arrives at, so every wait runs
 *     out; used to test that a stalled pipeline ends with TTC_ERR_TIMEOUT
 *     instead of hanging.
 *   TTC_KNOB_FORCE_GENERIC_LOAD: when 1, operands are staged with plain
 *     loads even when TMA could describe them.
 *   TTC_KNOB_FORCE_GENERIC_STORE: when 1, results are written with plain
 *     predicated stores even when TMA could describe D.
 *   TTC_KNOB_TILE_N: force the CTA tile width (256, 128, 64, 32 or 16); 0
 *     lets the planner choose.
 *   TTC_KNOB_PAIR: 0 lets the planner choose between the single-CTA kernel and
 *     the CTA-pair (2-SM, 256 x 256 tile) kernel; 1 uses the pair kernel
 *     whenever it applies (fp16/bf16 operands TMA can describe); 2 never.
 *   TTC_KNOB_SWAP_AB: 0 lets the planner choose whether to compute D or
 *     D^T = B^T A^T (for skinny problems); 1 always D^T; 2 always D.
 *   TTC_KNOB_GROUP_M: tile rasterization: consecutive tiles walk this many
 *     tile rows per column of tiles (0: 16 for single CTAs, 8 for pairs).
 *   TTC_KNOB_PAIR_TILE_N: 0 lets the planner choose the CTA-pair tile width;
 *     256, 224, 192 or 128 forces it (224 and 192 only with a column-major B).
 *   TTC_KNOB_GEMV: 0 (default) runs matrix-vector problems (fp16/bf16,
 *     K > 0, not batched) on the CUDA-core matrix-vector kernels: M == 1 with
 *     a column-major B or N == 1 with a row-major A (the reduction
 *     contiguous), and M == 1 with a row-major B or N == 1 with a
 *     column-major A (the outputs contiguous; from 1024 outputs, or K up to
 *     8192); 1 sends them to the tensor-core kernels like any other shape.
 *   TTC_KNOB_PAIR_TAIL: 0 (default) lets the CTA-pair kernels run a last,
 *     partial wave of tiles (or a problem of at most half a wave) as half
 *     tiles on twice as many pairs; 1 keeps whole tiles.
 *   TTC_KNOB_CONV_HALO: 0 (default) runs a unit-stride convolution that
 *     qualifies (see ttc_conv2d_fprop) on the halo-tile kernel; 1 does the
 *     same whatever the problem's size; 2 never uses it (im2col loads or
 *     plain loads instead).
 *   TTC_KNOB_SPLIT_K: 0 lets the planner choose; 1..8 splits every tile's K
 *     range across that many CTAs of a cluster (fp16/bf16 only), whose
 *     partial sums are added through distributed shared memory.
 *   TTC_KNOB_PDL: 0 (default) launches the GEMM, convolution and
 *     matrix-vector kernels with programmatic dependent launch: a kernel may
 *     start its prologue (barrier set-up, tensor-memory allocation) while the
 *     previous kernel on the stream finishes, and touches global memory only
 *     once that kernel has completed; 1 launches them in plain stream order.
 *   TTC_KNOB_I8_WIDE: 0 (default) lets ttc_gemm_ws run int8 problems of at
 *     least 64 tiles of 256 x 256 on the CTA-pair kernel when its workspace
 *     holds fp16 copies of A and B (ttc_gemm_workspace_size_staged); 1 does
 *     so from one tile up; 2 never (the single-CTA int8 kernels, which widen
 *     the operands in shared memory, take every int8 problem).
 *   TTC_KNOB_PAIR_EPI_WARPS: 0 (default) lets the CTA-pair kernel drain
 *     256-wide tiles whose output rows TMA cannot store with twelve
 *     epilogue warps (three per TMEM lane quarter) and all others with
 *     eight; 8 keeps eight everywhere; 12 is the default's choice.
 * Returns TTC_ERR_INVALID_ARG for an unknown knob or value.
 */
typedef enum {
  TTC_KNOB_TIMEOUT_NS = 0,
  TTC_KNOB_INJECT_STALL = 1,
  TTC_KNOB_FORCE_GENERIC_LOAD = 2,
  TTC_KNOB_FORCE_GENERIC_STORE = 3,
  TTC_KNOB_TILE_N = 4,
  TTC_KNOB_PAIR = 5,
  TTC_KNOB_SWAP_AB = 6,
  TTC_KNOB_SPLIT_K = 7,
  TTC_KNOB_PAIR_TILE_N = 8,
  TTC_KNOB_GROUP_M = 9,
  TTC_KNOB_GEMV = 10,
  TTC_KNOB_CONV_HALO = 11,
  TTC_KNOB_PAIR_TAIL = 12,
  TTC_KNOB_PDL = 13,
  TTC_KNOB_I8_WIDE = 14,
  TTC_KNOB_PAIR_EPI_WARPS = 15
} ttc_knob;

ttc_status ttc_set_knob(ttc_knob knob, int64_t value);

/* Number of kernel launches ttc_gemm has enqueued in this process. */
int64_t ttc_launch_count(void);

/*
 * Planning aid for tests and tuning: runs the planner of ttc_gemm_ws and
 * ttc_gemm_strided_batched (batch = 1 and workspace NULL describe ttc_gemm)
 * as if on a GB300-class device with `sm_count` SMs (2 .. 4096), without
 * touching any GPU: the pointers are only inspected for alignment and
 * overlap, nothing is read, no tensor map is encoded and nothing is
 * launched.  Writes the launches the call would make, as "kernel key=value
 * ..." items separated by "; ", to `out` (NUL-terminated, cut to out_len - 1
 * bytes; out may be NULL when out_len is 0), and returns the status the call
 * would return.  Knobs set with ttc_set_knob apply as they do to real calls.
 * Calls on other threads are unaffected while one thread plans.
 * TTC_ERR_INVALID_ARG: sm_count out of range, or out NULL with out_len > 0.
 */
ttc_status ttc_gemm_plan(int64_t batch, int64_t M, int64_t N, int64_t K,
                         const void* A, int64_t lda, int64_t strideA, ttc_layout layoutA,
                         const void* B, int64_t ldb, int64_t strideB, ttc_layout layoutB,
                         const void* C, int64_t ldc, int64_t strideC,
                         void* D, int64_t ldd, int64_t strideD,
                         float alpha, float beta, const float* bias,
                         ttc_act act, ttc_dtype dtype, void* workspace, size_t workspace_bytes,
                         int sm_count, char* out, size_t out_len);

#ifdef __cplusplus
}
#endif

#endif /* TTC_H_ */
