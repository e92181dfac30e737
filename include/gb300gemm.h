/*
 * gb300gemm.h -- C ABI of the GB300 (sm_103a) dense matrix multiply.
 *
 * Operation: C = A x B, overwriting C, with
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * for A of M x K, B of K x N and C of M x N ("Tensor cores and matrix
 * operations", section "Traditional Approach: Element-by-Element").  The
 * fixed entry points (gemm_f16f32, gemm_bf16f32, sgemm_f32) take row-major
 * A, B and C and no scaling; gemm_ex and its host and no-alloc forms add,
 * through gemm_options_t, C = alpha * A x B + beta * C, transposed storage of
 * A and/or B, and a 16-bit C.  The _bt entry points take B stored as its
 * transpose.  A leading dimension is the row stride of the full matrix as
 * stored, in elements, not of a tile ("04-wmma-matmul" code example, comment
 * on load_matrix_sync): for row-major A element (i, k) is A[i * lda + k] and
 * lda >= K, ldb >= N, ldc >= N.
 *
 * Arithmetic: the 16-bit entry points multiply FP16 or BF16 inputs and
 * accumulate in FP32 ("CUDA-Practice 09", the sections on mixed precision:
 * 16-bit inputs halve the bytes moved, FP32 accumulation avoids the rounding
 * of long 16-bit sums).  The FP32 entry point computes in FP32 on the CUDA
 * cores ("matmul_registers.cu", the register-tiled SGEMM it builds up).  The
 * TF32 and FP8 entry points use the tensor cores' TF32 and 8-bit modes with
 * FP32 accumulation.  Summation order inside a sum is unspecified; FP16,
 * BF16, FP32 and FP8 results meet max|C - C_exact| <= 1e-3 sqrt(K) max|A|
 * max|B| and a relative Frobenius error <= 1e-4, and are bit-exact whenever
 * every product and partial sum is an integer below 2^24 (TF32: see its
 * entry point).  A 16-bit C holds that FP32 result rounded once to nearest
 * even.
 *
 * Memory and ownership: A, B and C are DEVICE pointers owned by the caller
 * on the current CUDA device; the library never allocates, frees or copies
 * them.  C must not overlap A or B.  The library owns a small per-device,
 * per-stream split-K workspace (partial tiles + tile counters) that it
 * allocates on first use and grows as needed; gemm_release_workspace() frees
 * it.  Its caches remember the CUDA context they were made in: after a
 * cudaDeviceReset the next call starts afresh instead of using pointers of
 * the destroyed context.
 *
 * Streams: every call enqueues its kernels on `stream` (NULL = the legacy
 * default stream) and returns without synchronising.  A fault in a kernel
 * surfaces at the caller's next synchronisation; a pipeline wait that ran out
 * of time (see gemm_device_error) is recorded on the device instead of
 * hanging it.  Calls may be captured into a CUDA graph: the plan is fixed at
 * capture time and the graph replays the same kernels.  A plan with split-K
 * or stream-K allocates its workspace on its first call, which must
 * therefore run before the capture (or use gemm_ex_noalloc).
 *
 * Errors: every function returns a gemm_status_t and never prints or exits.
 * Argument errors are found on the host before anything is enqueued.
 *
 * Thread safety: calls from several host threads are safe.  Calls on
 * different streams of one device each use their own workspace.
 */
#ifndef GB300GEMM_H
#define GB300GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL selects the default stream. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* null pointer with M, N > 0; negative dim; ld too small;
                                        a dimension above 2^31 - 1                       */
    GEMM_ERR_OVERLAP = 2,            /* C's span overlaps A's or B's                      */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3     */
    GEMM_ERR_LAUNCH = 4,             /* a kernel launch failed (see gemm_last_cuda_error) */
    GEMM_ERR_DEVICE_TIMEOUT = 5,     /* a pipeline wait in a kernel gave up (device flag) */
    GEMM_ERR_CUDA = 6,               /* another CUDA runtime call failed                  */
    GEMM_ERR_OUT_OF_MEMORY = 7       /* the split-K workspace could not be allocated       */
} gemm_status_t;

/*
 * gemm_f16f32 -- C (FP32) = A (FP16) x B (FP16), FP32 accumulate, tensor cores.
 *
 * A: const __half*, M x K, row stride lda.  B: const __half*, K x N, row
 * stride ldb.  C: float*, M x N, row stride ldc.
 * Path: when A and B start on 16-byte boundaries and lda, ldb are multiples of
 * 8, a TMA + tcgen05.mma kernel (accumulators in tensor memory); otherwise a
 * CUDA-core kernel with the same FP32 accumulation.  Shapes that are not a
 * whole number of tiles are handled by the kernels' edge paths.
 * M == 0 or N == 0: nothing is enqueued.  K == 0: C is filled with zeros (the
 * empty sum).
 */
gemm_status_t gemm_f16f32(const void *A, const void *B, float *C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc,
                          gemm_stream_t stream);

/* gemm_bf16f32 -- as gemm_f16f32, with BF16 (__nv_bfloat16) A and B. */
gemm_status_t gemm_bf16f32(const void *A, const void *B, float *C,
                           int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldc,
                           gemm_stream_t stream);

/*
 * sgemm_f32 -- C = A x B, all FP32, FP32 fused multiply-add on the CUDA
 * cores (no TF32).  Layout, ownership, streams and degenerate shapes as
 * gemm_f16f32.  Path: a register-tiled kernel (8 x 8 outputs per thread,
 * float4 global loads, A staged transposed in shared memory) when A, B and C
 * start on 16-byte boundaries and lda, ldb, ldc are multiples of 4; a guarded
 * scalar kernel otherwise.  Never returns an alignment error.
 */
gemm_status_t sgemm_f32(const float *A, const float *B, float *C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc,
                        gemm_stream_t stream);

/*
 * gemm_tf32f32_bt -- C (FP32) = A x B with FP32 A and B read by the tensor
 * cores as TF32 (10 fraction bits; the pages' "TF32 path", which changes
 * results more than any kernel edit -- "matmul_registers.cu", the note on
 * CUBLAS_COMPUTE_32F), FP32 accumulation.  B is passed TRANSPOSED: Bt is
 * N x K row-major (ldb >= K), because the tensor cores read TF32 operands
 * only K-contiguous.  A: M x K row-major.  A and Bt must start on 16-byte
 * boundaries with lda, ldb multiples of 4; otherwise GEMM_ERR_INVALID_VALUE.
 * Results stay within (2^-9 + 2^-20) * sum_k |A[i][k]| |B[k][j]| of the exact
 * product of the FP32 inputs.
 */
gemm_status_t gemm_tf32f32_bt(const float *A, const float *Bt, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream);

/*
 * gemm_e4m3f32_bt / gemm_e5m2f32_bt -- C (FP32) = A x B with 8-bit floating
 * point A and B (E4M3: 4 exponent bits, 3 fraction bits, largest 448; E5M2:
 * 5 and 2, largest 57344) on the tensor cores, FP32 accumulation.  The
 * 8-bit tensor-core modes are the next step the pages point to after 16-bit
 * inputs ("Tensor cores and matrix operations", "Connections": quantisation
 * and the 8-bit tensor-core modes).  As for TF32, B is passed TRANSPOSED
 * (Bt N x K row-major, ldb >= K) and A is M x K row-major; both must start on
 * 16-byte boundaries with lda, ldb multiples of 16.  Use gemm_ex's alpha for
 * a scale.
 */
gemm_status_t gemm_e4m3f32_bt(const void *A, const void *Bt, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream);
gemm_status_t gemm_e5m2f32_bt(const void *A, const void *Bt, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream);

/*
 * Options for gemm_ex.  Zero-initialise and set what you need; a zero field
 * means "let the planner choose".
 *   dtype     0 = FP16, 1 = BF16, 2 = FP32 (sgemm_f32's kernels), 3 = TF32
 *             (FP32 storage on the tensor cores), 4 = E4M3, 5 = E5M2.  Types
 *             3-5 need trans_a = 0 and trans_b = 1 (both operands
 *             K-contiguous) and TMA-legal alignment.
 *   tile_n    dtype 0/1: tensor-core tile width along the MMA's N side: 16,
 *             32, 64, 128 or 256 (16..64 only with swap_ab = 1; 64..256
 *             without).  dtype 2: 256 -> 128x128 SGEMM tiles with 8x16
 *             outputs per thread (128 threads), 128 -> 128x128 with 8x8
 *             (256 threads), 64 -> 128x64, 32 -> 64x64.
 *   split_k   number of K slices, each reduced in a fixed order (1..64).
 *   swap_ab   -1 = planner, 0 = never, 1 = compute C^T = B^T A^T so that N
 *             runs along the 128-row MMA side (for small M).  The planner
 *             never swaps when cta_pair = 2.
 *   generic   1 = force the CUDA-core kernel (any alignment).
 *   group_m   tiles per raster group along the MMA's M side (0 = planner).
 *   cta_pair  0 = planner, 1 = one CTA per 128-row tile, 2 = CTA pairs
 *             (clusters of two SMs sharing a 256-row tile; tile_n 128 or
 *             256, no swap, no split-K).
 *   store_mode 0 = planner (tensor-core results leave through TMA stores
 *             when C's base, ldc and N allow it), 1 = plain stores.
 *   stream_k  0 = planner, 1 = off, 2 = stream-K, 3 = tail split
 *             (tensor-core kernels only).  Stream-K keeps whole tiles while
 *             whole waves last and shares the remaining tiles' K range
 *             evenly over all CTAs (CTA pairs); tail split keeps whole tiles
 *             for every whole wave and cuts each leftover tile into
 *             floor(CTAs / leftover tiles) equal K pieces, one per CTA (CTA
 *             pair).  A tile cut into pieces is summed in a fixed order.  For
 *             the tensor-core kernels the planner uses tail split for the
 *             CTA-pair kernel with at least 8 whole waves (it measured about
 *             1 % faster at 8192^3 and slower with fewer waves) and never
 *             stream-K (at the power cap, idle clusters in a partial last
 *             wave let the busy ones clock higher, which the measured shapes
 *             favour over the partial sums' traffic).  For the FP32 SGEMM it
 *             turns stream-K on when there are fewer than three waves of
 *             128 x 128 tiles (M > 64), choosing the tile from the K steps
 *             each persistent CTA gets; from three waves on it runs whole
 *             waves of 128 x 128 tiles with 8x16 outputs per thread (N > 64).
 *             Ignored with split_k > 0.
 *   epilogue  0 = C = A x B (alpha and beta ignored); 1 = C = alpha * (A x B)
 *             + beta * C, the accumulate-onto-C form of the tensor-core
 *             operation ("04-wmma-matmul", header comment: D = A*B + C).  The
 *             product is accumulated in FP32, then scaled and added in FP32.
 *             With beta == 0, C is not read (it may hold anything, NaN
 *             included).  With K == 0 the result is beta * C.
 *   trans_a   0 = A is op(A), stored M x K (lda >= K); 1 = A is stored as its
 *             transpose, K x M row-major (lda >= M), and the product uses Aᵀ.
 *   trans_b   0 = B stored K x N (ldb >= N); 1 = B stored as its transpose,
 *             N x K (ldb >= K).  Together: C = op(A) x op(B), the row-major
 *             reading of the transposition the pages use to call a
 *             column-major library ("matmul_registers.cu", the cuBLAS call).
 *             The tensor-core kernels read either layout directly (TMA boxes
 *             and MMA descriptors per layout); FP32 with a transpose runs the
 *             guarded CUDA-core kernel.  gemm_ex_host honours both flags.
 *   c_dtype   element type of C: 0 = FP32, 1 = FP16, 2 = BF16.  The product
 *             (and alpha * AB + beta * C) is formed in FP32 as always, then
 *             rounded once to nearest, ties to even, into the 16-bit C -- the
 *             16-bit form of the accumulate-onto-C operation the pages
 *             describe ("Tensor cores and matrix operations": FP16 or FP32
 *             C and D).  With beta != 0 the old 16-bit C is read and widened
 *             exactly.  ldc counts elements of C's type; a 16-bit C needs
 *             only 2-byte alignment (TMA stores are used when its base is
 *             16-byte aligned and ldc and N are multiples of 8).  Every
 *             kernel path and gemm_ex_host honour it.
 * Invalid combinations return GEMM_ERR_INVALID_VALUE.
 */
typedef struct {
    int32_t dtype;
    int32_t tile_n;
    int32_t split_k;
    int32_t swap_ab;
    int32_t generic;
    int32_t group_m;
    int32_t cta_pair;
    int32_t store_mode;
    int32_t stream_k;
    float alpha;
    float beta;
    int32_t epilogue;
    int32_t trans_a;
    int32_t trans_b;
    int32_t c_dtype;
    int32_t reserved;
} gemm_options_t;

/*
 * gemm_ex -- the operation with explicit options (gemm_options_t above):
 * input type, plan, alpha/beta epilogue, transposed storage, C's type.  C is
 * void* because its element type is options->c_dtype; A and B follow
 * options->dtype and the trans_* flags.  options must not be NULL.
 */
gemm_status_t gemm_ex(const void *A, const void *B, void *C,
                      int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc,
                      const gemm_options_t *options, gemm_stream_t stream);

/*
 * gemm_plan_describe -- the plan gemm_ex would use for these arguments and
 * options on the current device (options NULL: the plan of the fixed entry
 * point for `dtype`), as text written to buf (always NUL-terminated when
 * size > 0).  Pointers are not dereferenced; only their alignment is read.
 * Returns the status the call would return from argument checking and
 * planning.
 */
gemm_status_t gemm_plan_describe(int32_t dtype, const void *A, const void *B, const void *C,
                                 int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc,
                                 const gemm_options_t *options, char *buf, int64_t size);

/*
 * gemm_device_error -- synchronises `stream`, then reads and clears the
 * current device's error flag.  Returns GEMM_ERR_DEVICE_TIMEOUT if any
 * kernel since the last call gave up a pipeline wait (it then wrote no
 * trustworthy output), GEMM_ERR_CUDA if the synchronisation failed, else
 * GEMM_OK.  A kernel that gives up may leave split-K tile counters part-way;
 * on GEMM_ERR_DEVICE_TIMEOUT every split-K workspace of the device is
 * therefore marked, and each clears its counters (an asynchronous memset on
 * its stream) before it is next used, so later calls are correct again.
 */
gemm_status_t gemm_device_error(gemm_stream_t stream);

/*
 * gemm_watchdog_selftest -- checks the failure path of the kernels' pipeline
 * waits.  Enqueues on `stream` one small kernel whose single wait can never
 * be satisfied; the wait gives up after limit_ms (1..2000) milliseconds,
 * through the same bounded wait the GEMM kernels use, and records the fact
 * in the device error word.  A following gemm_device_error(stream) returns
 * GEMM_ERR_DEVICE_TIMEOUT (and clears the word); the context stays usable.
 * No GEMM is affected.  (A testing aid of this library; the pages have no
 * counterpart.)
 */
gemm_status_t gemm_watchdog_selftest(int32_t limit_ms, gemm_stream_t stream);

/*
 * gemm_ex_stall_selftest -- checks the GEMM kernels' own failure path.  Runs
 * the tensor-core plan gemm_ex would run for these arguments (other plans:
 * GEMM_ERR_INVALID_VALUE) with two changes: every pipeline wait gives up
 * after limit_ms (1..2000) milliseconds, and the TMA producer of CTA
 * `stall_cta` (for the CTA-pair kernel: of both CTAs of cluster `stall_cta`)
 * withholds the copies of its pipeline stage number `stall_fill` (0 = the
 * first stage it fills).  The MMA thread's wait for that stage then runs
 * out; the CTA (pair) records GEMM_ERR_DEVICE_TIMEOUT in the device error
 * word, leaves its loops, waits (bounded) for its copies and MMAs in flight,
 * frees its tensor memory and exits, while the other CTAs finish normally.
 * Nothing faults, traps or hangs; the context stays usable.  C is then
 * unspecified (the stalled CTA's tiles are missing).  stall_cta must be below
 * the plan's CTA (cluster) count; a CTA with fewer than stall_fill + 1 stage
 * fills runs normally.  (A testing aid of this library; the pages have no
 * counterpart.)
 */
gemm_status_t gemm_ex_stall_selftest(const void *A, const void *B, void *C,
                                     int64_t M, int64_t N, int64_t K,
                                     int64_t lda, int64_t ldb, int64_t ldc,
                                     const gemm_options_t *options, int32_t limit_ms,
                                     int32_t stall_cta, int32_t stall_fill,
                                     gemm_stream_t stream);

/* gemm_release_workspace -- frees the split-K workspaces of the current
 * device after synchronising the device.  Later calls allocate again. */
gemm_status_t gemm_release_workspace(void);

/*
 * gemm_ex_host -- the same operation with A, B and C in HOST memory.
 *
 * The library cuts C into blocks of A row panels by B column panels (up to
 * four of each).  It copies the first two A panels in interleaved with the
 * B panels (A0, B0, A1, B1, B2, ...), the later A panels one by one, runs
 * each block's product as soon as its panels are in (the kernels of
 * gemm_ex, on `stream`) and copies each C block back as soon as it is done,
 * on two internal copy streams, so the two copy directions overlap each
 * other and the products.
 * With epilogue 1 and beta != 0, each C block is also copied in before its
 * product (on `stream`).
 * For the copies to overlap, A, B and C must be page-locked (cudaHostAlloc /
 * cudaHostRegister); pageable memory works but serialises.  Leading
 * dimensions are those of the host arrays.  With trans_a, an A panel is a
 * column block of the stored K x M matrix; with trans_b, a B panel is a row
 * block of the stored N x K matrix (so TF32 and the 8-bit types, which take
 * B transposed, run from host buffers too).  The device copies keep each
 * operand's storage order with row strides rounded up to 16 elements, so
 * every panel suits the TMA kernels whatever the host leading dimensions
 * are (the rules on lda and ldb above apply to the host arrays only).
 *
 * The call returns after enqueueing; C is complete when `stream` reaches
 * this point (synchronise `stream` before reading C).  Work already queued on
 * `stream` finishes before the copies start.  Device staging buffers (B, two
 * A panels, two C panels), the copy streams and events belong to the library,
 * one set per (device, stream), allocated on first use and grown as needed;
 * gemm_release_workspace() does not free them.
 */
gemm_status_t gemm_ex_host(const void *A, const void *B, void *C,
                           int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldc,
                           const gemm_options_t *options, gemm_stream_t stream);

/*
 * gemm_ex_noalloc -- gemm_ex for callers that cannot allocate device memory.
 * (An addition of this library; the pages have no counterpart.)
 *
 * Who needs it: applications that give the GPU's memory to their own pool at
 * start-up and account for every byte, and latency-critical loops in which a
 * cudaMalloc or cudaFree -- which can synchronise the whole device -- is not
 * acceptable.  gemm_ex may allocate its split-K workspace on first use; this
 * entry point never calls cudaMalloc, cudaFree or any other allocating
 * routine.  The caller still passes A, B and C.
 *
 * Scratch: every plan that splits tiles along K keeps its partial tiles and
 * arrival counters in one static device array of GEMM_NOALLOC_SCRATCH_BYTES
 * (8 MiB: the first 64 KiB hold counters for up to 4096 tiles, the rest
 * holds partial tiles) -- the split-K, stream-K and tail-split plans of the
 * tensor-core kernels (one CTA or CTA pairs) and the split-K and stream-K
 * plans of the FP32 SGEMM.  When the planner's own choice (stream_k = 0) is
 * a stream-K SGEMM or a tail split whose pieces do not fit, this entry point
 * plans the product without them (split-K waves or whole tiles) instead.
 * Every GPU that loads the library holds this array until the process exits.
 * A plan whose scratch does not fit returns GEMM_ERR_INVALID_VALUE, and
 * gemm_last_cuda_error() says how much it needed.  Plans that do not split
 * tiles use no scratch at all.  The results are bit-identical to gemm_ex's
 * for the same plan.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Under CUDA's lazy module loading (the default)
 * the library's device code, and with it this array, is placed in device
 * memory when it is first used -- by the first call of each kind.  A caller
 * that must not allocate later should make one call of each plan kind it
 * will use at start-up, before it hands the remaining memory to its pool
 * (or run with CUDA_MODULE_LOADING=EAGER).
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; each call clears the counters it needs (an asynchronous
 * memset on `stream`) before its kernel runs.  Calls whose kernels overlap on
 * the GPU -- for example on two streams at once -- race on the array and give
 * wrong results: serialise them.
 *
 * Arguments, options, layout, errors and results are those of gemm_ex.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (8u << 20)

gemm_status_t gemm_ex_noalloc(const void *A, const void *B, void *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              const gemm_options_t *options, gemm_stream_t stream);

/* Text for a status code (static storage). */
const char *gemm_status_string(gemm_status_t status);

/* Text of the last CUDA error seen by this host thread inside the library
 * (static thread-local storage; "" if none). */
const char *gemm_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t gemm_version(void);

/* Number of kernel launches this host thread has enqueued through the library
 * since it loaded (monotonic counter, for accounting in benchmarks). */
int64_t gemm_launch_count(void);

/* Number of device allocations (cudaMalloc) the library has made since it
 * loaded, over all threads and devices: split-K workspaces and gemm_ex_host's
 * staging buffers (monotonic counter; gemm_ex_noalloc never adds to it). */
int64_t gemm_alloc_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_H */
