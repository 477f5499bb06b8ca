/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library, libgemm_gb300.so.
 *
 * The library computes
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * over row-major matrices: full SGEMM as defined in the Introduction sidenote of
 * "Optimizing GEMM on Apple's M5 from scratch, Part 1: Basics" (the pages fix
 * alpha = 1, beta = 0 for their benchmark; the library takes both), for
 *   - fp32 operands and result (the SGEMM of that page and of "Part 2"), and
 *   - fp16 operands, fp32 accumulation and an fp16 result, the regime of
 *     "Metal GEMM Kernels for LoRA Training on Apple Silicon", section 1 (table
 *     of operand/accumulator types) and section 2 (output converted from the
 *     fp32 accumulator on the way out), and the same with bfloat16,
 * in the transpose variants of that page's section 2 variant table:
 *     nn  A[M,K]   @ B[K,N]
 *     tn  A[K,M]^T @ B[K,N]
 *     nt  A[M,K]   @ B[N,K]^T
 * (tt, both transposed, is not on the pages; it falls out of the same operand
 * descriptors and is accepted.)
 *
 * Conventions (all entry points):
 *   - Row-major storage; every leading dimension (lda, ldb, ldc) is in
 *     ELEMENTS and is the distance between consecutive stored rows.
 *   - op(A) is M x K: A is stored M x K (lda >= K) when transA == 0, and
 *     K x M (lda >= M) when transA == 1.  op(B) is K x N: B is stored K x N
 *     (ldb >= N) when transB == 0, N x K (ldb >= K) when transB == 1.
 *     C is M x N, ldc >= N.  A sub-matrix is passed as a pointer at its first
 *     element plus the parent's leading dimension (the row-offset entry of the
 *     LoRA page, section 7).
 *   - alpha and beta are fp32 for both dtypes.  beta == 0 makes C write-only:
 *     it is not read, so NaN or garbage in C does not reach the result.
 *   - M == 0 or N == 0 returns GEMM_OK without touching the GPU.  K == 0 sets
 *     C = beta * C (zero when beta == 0).
 *   - Pointers passed to gemm() are DEVICE pointers (cudaMalloc, the stream-
 *     ordered allocator or a torch CUDA tensor's storage), aligned to the
 *     element size.  The caller owns every buffer; the library never frees
 *     caller memory.  C must not overlap A or B (GEMM_ERR_ALIAS).
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *     may be made from several host threads.  Scratch space the library needs
 *     (split-K partial sums; zero-padded copies of operands whose rows are not
 *     16-byte aligned; on large problems an aligned working copy of a C whose
 *     rows are not, copied into place at the end) is taken in stream order on
 *     `stream` from a memory pool the library creates once per device, and
 *     released on the same stream; the pool keeps released memory for reuse
 *     until the process exits.
 *   - The library's kernels are launched with programmatic stream
 *     serialization: each may start its set-up while the previous work on the
 *     stream is finishing, and waits for that work to complete before reading
 *     or writing any buffer.  Stream order is therefore kept exactly as for
 *     ordinary launches (environment GEMM_GB300_PDL=0 turns the overlap off).
 *   - Argument errors are returned synchronously, before anything is
 *     launched.  Launch failures return GEMM_ERR_CUDA.  A kernel whose
 *     internal wait exceeds its time limit records the fact in a per-device
 *     status word and exits early; gemm_check_device_status() reports it.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* gemm_stream_t;

typedef enum {
    GEMM_F32 = 0,         /* A, B, C fp32; fp32 FMA accumulation */
    GEMM_F16_F32ACC = 1,  /* A, B, C fp16 (IEEE binary16); fp32 accumulation;
                             result rounded to fp16 round-to-nearest-even */
    GEMM_BF16_F32ACC = 2, /* A, B, C bfloat16; fp32 accumulation; result
                             rounded to bfloat16 round-to-nearest-even (the
                             bfloat16 row of the LoRA page's section 1 type
                             table, native on these tensor cores) */
    GEMM_F32_TF32 = 3,    /* OPT-IN reduced precision: A, B, C fp32, but the
                             products use only the TF32 part of each operand
                             (sign, 8 exponent and the top 10 fraction bits)
                             on the tensor cores; fp32 accumulation.  Error up
                             to ~2^-9 * sum|a*b|, against ~K * 2^-24 for
                             GEMM_F32.  The counterpart of the relaxed-
                             precision switch of "Optimizing GEMM on Apple's
                             M5 from scratch, Part 2"; never chosen for you.
                             Not accepted by gemm_splitk_noalloc. */
    GEMM_F32_3XTF32 = 4   /* OPT-IN: A, B, C fp32 on the tensor cores at about
                             fp32 accuracy.  Each operand is split into its
                             TF32 part hi (low 13 fraction bits cleared) and
                             the rest lo = x - hi (exact), and the products are
                             formed as hi*hi + hi*lo + lo*hi in one fp32
                             accumulation: the dropped lo*lo term and the TF32
                             reading of lo leave an error of about 2^-19 *
                             sum|a*b|, within GEMM_F32's tolerance.  Inputs
                             must be finite (an infinity in one operand meets a
                             zero lo of the other).  Takes scratch for the
                             split planes (2 x 4 bytes x (M + N) x K); not
                             accepted by gemm_splitk_noalloc. */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* bad dimension, leading dimension, pointer, flag or dtype */
    GEMM_ERR_UNSUPPORTED = 2, /* valid but not handled (e.g. a dimension >= 2^31) */
    GEMM_ERR_ALIAS = 3,       /* C overlaps A or B */
    GEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
    GEMM_ERR_NO_MEMORY = 5,   /* scratch allocation failed */
    GEMM_ERR_TIMEOUT = 6      /* a kernel's bounded internal wait expired */
} gemm_status_t;

/*
 * gemm -- C = alpha * op(A) * op(B) + beta * C on the GPU.
 *
 * transA, transB: 0 or 1 (see above).  M, N, K >= 0 and < 2^31.
 * dtype: a gemm_dtype_t.  A, B, C: device pointers, element-aligned.
 * lda, ldb, ldc: leading dimensions in elements (see above).
 * stream: the CUDA stream to run on.
 * Returns a gemm_status_t.  Nothing is launched unless it returns GEMM_OK.
 */
int gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
         float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
         int64_t ldc, gemm_stream_t stream);

/*
 * gemm_ex -- gemm() with a fused epilogue ("From a C loop to a GPU kernel",
 * section "Fusion": add the bias and apply the activation while the tile is
 * still in registers, write the result once):
 *
 *     C = act(alpha * op(A) * op(B) + beta * C + bias[j])
 *
 * bias: DEVICE pointer to N elements of the output type (fp32 for GEMM_F32,
 *   fp16 / bf16 otherwise), one per output column (the per-output offset), or
 *   NULL for none; element-aligned; must not overlap C (GEMM_ERR_ALIAS).
 * act: a gemm_act_t.  GEMM_ACT_GELU is the exact v * Phi(v) =
 *   v/2 * (1 + erf(v / sqrt 2)), evaluated in fp32 with CUDA's erff.
 * Everything else as gemm(); with bias == NULL and GEMM_ACT_NONE it is gemm().
 * The bias and activation are applied in fp32 before the output rounding, in
 * every path (split-K: by the reduction; K == 0: act(beta * C + bias)).
 */
typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,  /* max(v, 0) */
    GEMM_ACT_GELU = 2   /* v * Phi(v), Phi the standard normal distribution function */
} gemm_act_t;

int gemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
            float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
            int64_t ldc, const void* bias, int act, gemm_stream_t stream);

/*
 * gemm_host -- the same product on HOST buffers: copies A, B (and C when
 * beta != 0) to device memory taken from the stream-ordered allocator, runs
 * gemm() on `stream`, copies C back and synchronises `stream` before it
 * returns.  Problems of at least 2^30 multiply-adds are cut into 2 to 4 row
 * panels of C whose copies run on two library-owned copy streams (one per
 * direction, per device), ordered by events against the GEMMs on `stream`, so
 * that copies overlap computation; the call still returns only when C is
 * complete in host memory.  A, B, C are host pointers with the same layout rules as gemm();
 * page-locked (pinned) memory gives asynchronous DMA copies, pageable memory
 * works but is staged by the driver.  The device copies are packed (ld equal
 * to the row length) and freed before return.
 */
int gemm_host(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
              float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
              int64_t ldc, gemm_stream_t stream);

/*
 * gemm_splitk_noalloc -- gemm() for callers that must not allocate device
 * memory: code running under an allocator that already owns the whole GPU
 * (a framework's caching allocator), or a process that forbids runtime
 * allocation once it is serving.  It never calls cudaMalloc, cudaFree or any
 * other allocating routine.  (No page of the method describes this entry
 * point; it is a property of this library.)
 *
 * Same arguments, rules and results as gemm(), with gemm()'s kernels and
 * choice of tile and schedule.  The partial sums that gemm() keeps in scratch
 * from the stream-ordered allocator -- the fp32 kernel's K slices, and the
 * tensor-core kernel's shared (stream-K) tiles with their arrival counters --
 * live in one fixed array of 8 MiB compiled into the library, which every
 * GPU that loads the library holds until the process exits.  Differences and
 * limits:
 *   - an fp32 problem whose K slices (splits x M x N x 4 bytes) exceed 8 MiB
 *     returns GEMM_ERR_UNSUPPORTED without launching anything;
 *   - a tensor-core problem whose shared tiles would not fit the array runs
 *     with whole tiles only (no scratch needed);
 *   - gemm()'s scratch-based steps are left out: the fp32 operand packing and
 *     persistent stream-K launch on large problems (where gemm() shares the K
 *     steps of fewer tiles than SMs in one launch, this call keeps the K
 *     slices and their reduction), and the aligned working copy of an
 *     unaligned fp16 C (the kernel stores such a C row by row);
 *   - fp16/bf16 operands must have 16-byte aligned bases and row pitches (lda,
 *     ldb multiples of 8), else GEMM_ERR_UNSUPPORTED (padding them would need
 *     scratch); GEMM_F32_TF32 and GEMM_F32_3XTF32 are not accepted.
 * The first call on a device looks up the array's device address (a CUDA
 * runtime query, done once per device with that device current); make that
 * first call before any stream capture.  All calls share the array: calls
 * whose kernels can overlap on the GPU (e.g. on two unordered streams) race
 * on it, so order them on one stream or with events.  A call writes every
 * partial sum it reads, and clears the counters that must start at zero
 * (cudaMemsetAsync on `stream`, which allocates nothing) before its launch.
 */
int gemm_splitk_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                        float alpha, float beta, const void* A, int64_t lda, const void* B,
                        int64_t ldb, void* C, int64_t ldc, gemm_stream_t stream);

/*
 * gemm_strided_batched -- `batch` independent products of one shape,
 *
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   b = 0 .. batch-1,
 *
 * with A_b = A + b*strideA, B_b = B + b*strideB, C_b = C + b*strideC (pitches
 * in ELEMENTS).  This is the per-head GEMM of "Metal GEMM Kernels for LoRA
 * Training on Apple Silicon", section 8 (Attention): Q, K, V stored head-major
 * [H, N, d_h], so head h is a contiguous matrix at offset h*N*d_h and the six
 * attention products are the nn/tn/nt variants entered at a head offset.  The
 * page issues one GEMM per head; here the whole batch is one launch.
 *
 * Arguments as gemm(), plus:
 *   strideA, strideB, strideC >= 0.  A pitch of 0 shares one matrix across
 *     the batch (A or B only).  The C matrices must not overlap one another
 *     (strideC >= (M-1)*ldc + N when batch > 1), else GEMM_ERR_ALIAS.
 *   batch >= 0 and < 2^31; batch == 0 returns GEMM_OK without touching the
 *     GPU.  batch == 1 is gemm().
 * Aliasing is checked over whole extents: the span C .. C_{batch-1} must not
 * overlap the span of A's or B's matrices (GEMM_ERR_ALIAS), even where the
 * entries themselves would interleave without touching.
 * One launch covers the batch (gemm_last_path() GEMM_PATH_FFMA_BATCHED or
 * GEMM_PATH_TC_BATCHED) when the operands allow: fp32 always, in groups of
 * 65535 entries; fp16/bf16 when A and B have 16-byte aligned bases, row
 * pitches and batch pitches (lda, ldb, strideA, strideB multiples of 8).
 * Otherwise each entry runs as its own gemm() in stream order
 * (GEMM_PATH_PER_ENTRY).  No split-K within a batch.
 */
int gemm_strided_batched(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                         float alpha, float beta, const void* A, int64_t lda, int64_t strideA,
                         const void* B, int64_t ldb, int64_t strideB, void* C, int64_t ldc,
                         int64_t strideC, int64_t batch, gemm_stream_t stream);

/*
 * gemm_check_device_status -- synchronises `stream`, then reads and clears
 * the current device's status word.  Returns GEMM_ERR_TIMEOUT if a kernel
 * gave up on a wait since the last check, GEMM_ERR_CUDA if the stream
 * reported an error, GEMM_OK otherwise.
 */
int gemm_check_device_status(gemm_stream_t stream);

/* Human-readable name of a gemm_status_t (a static string). */
const char* gemm_status_string(int status);

/* Library version, (major << 16) | minor. */
int gemm_version(void);

/*
 * Diagnostics, per calling host thread: the kernel path the last successful
 * gemm() call on this thread launched (a gemm_path_t), and the number of
 * kernels it launched.  gemm_total_launches() counts kernels launched by the
 * library in this process since it was loaded (all threads).
 */
typedef enum {
    GEMM_PATH_NONE = 0,        /* nothing launched (empty problem or error) */
    GEMM_PATH_SCALE = 1,       /* K == 0: C = beta * C */
    GEMM_PATH_FFMA = 2,        /* fp32 FFMA tiled kernel */
    GEMM_PATH_FFMA_SPLITK = 3, /* fp32 FFMA kernel over K slices + reduction */
    GEMM_PATH_TC = 4,          /* fp16/bf16 tcgen05 kernel, fused epilogue */
    GEMM_PATH_TC_SPLITK = 5,   /* tcgen05 kernel whose persistent grid shares the K steps
                                  of some tiles (stream-K); partial sums combined inside
                                  the kernel */
    GEMM_PATH_FFMA_BATCHED = 6, /* strided batch: fp32 FFMA kernel, batch on the grid */
    GEMM_PATH_TC_BATCHED = 7,  /* strided batch: one persistent tcgen05 launch */
    GEMM_PATH_PER_ENTRY = 8    /* strided batch run entry by entry (unaligned operands) */
} gemm_path_t;

int gemm_last_path(void);
int gemm_last_launches(void);
int64_t gemm_total_launches(void);
/* Blocks in the grid of the last main GEMM kernel gemm() launched on this
 * thread (the persistent fp16 kernel sizes its grid to the resident blocks). */
int gemm_last_grid(void);

/*
 * Diagnostics: kernel timing.  With two CUDA events (cudaEvent_t, created by
 * the caller), every later gemm(), gemm_splitk_noalloc() and
 * gemm_strided_batched() call made from this host thread records `start` on
 * its stream immediately before its main GEMM kernel and `end` immediately
 * after it -- not around pre-passes (operand packing or padding) or the
 * split-K reduction -- so cudaEventElapsedTime(start, end) is that kernel's
 * device time for the latest call.  Passing NULL for either turns it off.  The
 * events stay owned by the caller and must outlive their use.
 */
void gemm_set_kernel_events(void* start, void* end);

/*
 * Diagnostics: scratch use.  Returns the largest number of bytes that were in
 * use at once, on the current device, from the stream-ordered memory pool the
 * library takes its scratch from, since the previous reset (0 if the pool has
 * not been created yet, -1 on a CUDA error); a nonzero `reset` then sets the
 * mark back to zero.  A stretch of calls that leaves the mark at zero took no
 * scratch from the pool.
 */
int64_t gemm_scratch_high_water(int reset);

/*
 * Test hook: the time limit, in nanoseconds, of every bounded wait inside the
 * kernels launched afterwards by this process (default 2e9, i.e. 2 s; values
 * <= 0 restore the default).  A wait that runs out sets the device status
 * word, releases what its block holds and returns.
 */
void gemm_set_wait_timeout_ns(int64_t ns);

/*
 * Test hook for failure detection: mode 1 makes the fp16 kernel's operand
 * producer skip its first load (no copy, no arrival), so the consumer's
 * bounded wait runs out and the kernel reports GEMM_ERR_TIMEOUT through
 * gemm_check_device_status() instead of hanging.  Mode 0 (the default) turns
 * it off.  Process-wide; not for production use.
 */
void gemm_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
