/*
 * gemm.h -- C ABI of libgemm.so, the GB300 (sm_103a) software-pipelined GEMM.
 *
 * Operation (every gemm* entry point below; pipelined_copy, mma_rate and
 * the hooks document their own):
 *
 *     C = alpha * A * B + beta * C
 *
 * The problem is the tiled GEMM of "CUTLASS-CuTe 初步(6)" (hxf0223.github.io),
 * section 2 "Thread Block Tile": each thread block owns one tile of C and loops
 * over K, accumulating the product of an A tile and a B tile per step.  The
 * page's own formula was lost; the BLAS form with alpha and beta is used.
 * What the library adds is the mainloop the four pages describe: the next K
 * tile's global-to-shared copy overlaps the current tile's multiply-accumulate
 * through a ring of `stages` shared-memory buffers ("learn-kernels.com,
 * Matrix multiplication", the paragraph "Overlap needs stages"; "Software
 * Pipelining and Double Buffering", sections "Double buffering with shared
 * memory" and "Multi-stage pipelines").  stages = 1 is the single buffer with
 * a load phase and a compute phase per K tile, stages = 2 is double
 * buffering, stages >= 3 is a multi-stage ring.  The stage count changes
 * timing only: for one dtype and tile, every stage count gives bit-identical C.
 * A tensor-core stage holds a K slice of 64 of both operands on every tile
 * (one 128-byte swizzle row of 16-bit data): 4 tcgen05.mma instructions per
 * ring wait (8 on the 256 x 512 tile, two N = 256 MMAs per K step).
 *
 * Layout (all row-major, leading dimensions in elements):
 *   A  M x K, element (i,k) at A[i*lda + k], lda >= K
 *   B  K x N, row-major: element (k,j) at B[k*ldb + j], ldb >= N
 *           column-major (gemm_ex, b_col_major = 1): B[j*ldb + k], ldb >= K
 *   C  M x N, element (i,j) at C[i*ldc + j], ldc >= N
 *
 * Types (`dtype`, input -> output; accumulation is always fp32):
 *   GEMM_F32        fp32 A, B, C      CUDA-core SIMT sgemm, stages 1..4
 *   GEMM_F16_F32    fp16 A, B; fp32 C tcgen05 tensor cores, stages 1..6
 *   GEMM_BF16_F32   bf16 A, B; fp32 C tcgen05 tensor cores, stages 1..6
 *   GEMM_BF16_BF16  bf16 A, B, C      tcgen05 tensor cores, stages 1..6
 *                                     (1..4 on two tiles, see gemm_tile_t);
 *                                     fp32 result rounded to nearest even
 *   alpha and beta are fp32.  alpha is applied to the fp32 sum, then beta*C
 *   is added (one fp32 multiply-add per element).
 *
 * Memory: A, B and C are device pointers owned by the caller (except in
 * gemm_host, which takes host pointers).  The library keeps no pointer after
 * a call returns.  Two schedules keep fp32 partial tiles in a workspace the
 * library allocates (cudaMalloc) on first use, one per (device, stream), and
 * keeps until gemm_host_release: the SIMT path's split tail (used when the
 * last wave of 128 x 64 tiles -- 3 per SM -- is partial, also when it is the
 * only one: its tiles are cut along K into 2..8 pieces; at most 3 x SMs x
 * 32 KB, 14.9 MB on GB300) and
 * the tensor-core stream-K tail (gemm_schedule_set mode 2).  Every other call
 * allocates nothing.  A call that would allocate cannot run inside a stream
 * capture: make the first such call on each (device, stream) before capturing
 * (a larger shape later may grow the workspace again).
 *
 * Alignment (GEMM_ERR_ALIGN otherwise): A, B and C start on 16-byte
 * boundaries and lda*size, ldb*size and ldc*size are multiples of 16 bytes
 * (size = element size of that operand).  These are the tensor-copy (TMA)
 * and 16-byte cp.async rules; there is no slower fallback path.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 * gemm and gemm_ex enqueue work and return without synchronising.
 *
 * Degenerate sizes: M == 0 or N == 0 does nothing.  K == 0 or alpha == 0
 * gives C = beta*C without reading A or B.  beta == 0 never reads C (so NaN
 * in C does not propagate), following the BLAS convention.
 *
 * Error behaviour: every entry point returns a gemm_status_t.  Argument
 * checks happen on the host before anything is enqueued.  Inside the
 * tensor-core kernel every wait on a pipeline barrier is bounded in time; a
 * wait that runs out records GEMM_ERR_TIMEOUT in a device status word and the
 * kernel returns early (its output is then undefined).  gemm and gemm_ex do
 * not look at that word (they would have to synchronise); gemm_checked does.
 */
#ifndef SSP_GEMM_H
#define SSP_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_F32 = 0,
    GEMM_F16_F32 = 1,
    GEMM_BF16_F32 = 2,
    GEMM_BF16_BF16 = 3
} gemm_dtype_t;

/* Tensor-core tile (gemm_ex's `tile`).  The 2-SM tiles run on a cluster of
 * two CTAs with tcgen05.mma.cta_group::2: each CTA stages 128 rows of A and
 * 128 (256 on the 512-wide tile) columns of B per K step and holds 128 rows
 * of the result.
 * The stage limits are what fits in 227 KB of shared memory per CTA. */
typedef enum {
    GEMM_TILE_AUTO = 0,          /* 256x256 on a CTA pair if M > 128 and N > 128
                                    (128x128 if the pair tiles would number at
                                    most a quarter of the SMs, 128x256 if at
                                    most half and K <= 4096, 256x512 if
                                    K >= 8192 and the 256x512 tiles fill at
                                    least one round of pairs), else 128x128
                                    (N <= 128) or 128x256.  With stages 5 or 6
                                    the 128x256 and 256x512 choices become
                                    256x256 on a pair (128x128 when M or N is
                                    a single tile), whose rings hold 6.
                                    gemm_resolve_tile tells which */
    GEMM_TILE_128x128 = 128,     /* one CTA, stages 1..6 (32 KB each) */
    GEMM_TILE_128x256 = 256,     /* one CTA, stages 1..4 (48 KB each) */
    GEMM_TILE_256x256_2SM = 512, /* a CTA pair, stages 1..6 (32 KB each per CTA) */
    GEMM_TILE_256x512_2SM = 1024 /* a CTA pair, stages 1..4
                                    (48 KB each per CTA): two N = 256 MMAs share
                                    each A stage (a quarter fewer operand bytes
                                    per FLOP), one 512-column accumulator
                                    released in halves; bit-identical to the
                                    256x256 pair tile */
} gemm_tile_t;

/* Register-fragment scheme of the SIMT sgemm (gemm_ex's `tile` when dtype
 * is GEMM_F32): fragments double-buffered in registers (the warp-scope
 * double buffer, the default) or a single fragment set. */
typedef enum {
    GEMM_SIMT_FRAGMENTS_DOUBLE = 0,
    GEMM_SIMT_FRAGMENTS_SINGLE = 1
} gemm_simt_fragments_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_ARG = -1,          /* bad size, leading dimension, pointer, dtype or stages */
    GEMM_ERR_UNSUPPORTED = -2,  /* a valid request the library does not implement */
    GEMM_ERR_ALIGN = -3,        /* a 16-byte alignment rule above is broken */
    GEMM_ERR_LAUNCH = -4,       /* the CUDA launch (or tensor-map encode) failed */
    GEMM_ERR_TIMEOUT = -5,      /* a pipeline wait ran out (gemm_checked only) */
    GEMM_ERR_CUDA = -6,         /* another CUDA runtime call failed (copies, sync, device) */
    GEMM_ERR_SCRATCH = -7       /* gemm_noalloc: needs more scratch than its fixed array */
} gemm_status_t;

/*
 * gemm -- C = alpha*A*B + beta*C with row-major B, asynchronous on `stream`.
 *   M, N, K    problem size (>= 0)
 *   A, lda     device pointer and leading dimension of A (M x K)
 *   B, ldb     device pointer and leading dimension of B (K x N, row-major)
 *   C, ldc     device pointer and leading dimension of C (M x N), read when
 *              beta != 0 and written
 *   dtype      a gemm_dtype_t
 *   stages     depth of the shared-memory ring, each stage a K slice of 64:
 *              1..6 on the tensor-core path, 1..4 on the SIMT path (32 of K
 *              per stage); anything else is GEMM_ERR_ARG
 *   stream     cudaStream_t
 * The tensor-core tile is GEMM_TILE_AUTO's choice for these sizes and this
 * stage count (every stage count 1..6 has a tile that holds it).
 */
int gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
         void* C, int64_t ldc, float alpha, float beta, int dtype, int stages, void* stream);

/*
 * gemm_ex -- gemm with two more choices.
 *   b_col_major  0: B row-major (as gemm); 1: B column-major (element (k,j)
 *                at B[j*ldb + k], ldb >= K).  Column-major B is implemented on
 *                the tensor-core path only (GEMM_ERR_UNSUPPORTED for GEMM_F32).
 *   tile         tensor-core path: a gemm_tile_t; a stage count in 1..6 above
 *                an explicit tile's limit (5 or 6 on GEMM_TILE_128x256 or
 *                GEMM_TILE_256x512_2SM) gives GEMM_ERR_UNSUPPORTED.  SIMT path
 *                (tile 128 x 64): a gemm_simt_fragments_t.
 */
int gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
            int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
            int b_col_major, int tile, void* stream);

/*
 * gemm_checked -- gemm_ex, then synchronise `stream` and read (and clear) the
 * device status word.  Returns GEMM_ERR_TIMEOUT if a pipeline wait ran out,
 * GEMM_ERR_CUDA if the stream reported an error, otherwise gemm_ex's status.
 * Meant for tests and debugging; it blocks the calling thread.
 */
int gemm_checked(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype,
                 int stages, int b_col_major, int tile, void* stream);

/*
 * gemm_host -- the same operation on HOST buffers: copies A, B (and C when
 * beta != 0) to the device, runs gemm_ex, copies C back and synchronises.
 * The copies are pipelined with the computation: B goes first, then M is cut
 * into up to 16 row panels (whole 256-row tiles); panel p's rows of A and C
 * are copied in on an internal stream while panel p-1 is computed on
 * `stream` and earlier panels' C rows are copied back on a second internal
 * stream.  Every panel gives the same bits as one gemm_ex over all of M.
 * Work queued on `stream` before the call runs first.  Device staging
 * buffers, the two streams and their events are created on first use and
 * cached per device (buffers grow when a larger problem arrives); pinned
 * host memory makes the copies asynchronous DMA.  Leading dimensions are kept
 * as given.  Calls from several threads run one at a time.
 */
int gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
              int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
              int b_col_major, int tile, void* stream);

/* Frees what the library caches on the current device: gemm_host's staging
 * buffers, copy streams and events, the SIMT split-tail workspaces and the
 * stream-K workspaces (gemm_schedule_set mode 2).  Call it when no GEMM of
 * this library is running on the device; later calls create them again as
 * needed. */
int gemm_host_release(void);

/* Human-readable name of a gemm_status_t (static storage). */
const char* gemm_status_string(int status);

/* Largest `stages` value accepted for a dtype and tile (as in gemm_ex; 6 for
 * GEMM_TILE_AUTO), or GEMM_ERR_ARG for an unknown combination. */
int gemm_max_stages(int dtype, int tile);

/*
 * gemm_resolve_tile -- the gemm_tile_t that gemm_ex uses for these sizes and
 * this stage count on the current device when passed `tile` (GEMM_TILE_AUTO
 * resolves to a tile code; an explicit tile comes back unchanged).
 * GEMM_ERR_ARG for a dtype of the SIMT path, a negative size, stages outside
 * 1..6 or an unknown tile code.
 */
int gemm_resolve_tile(int64_t M, int64_t N, int64_t K, int dtype, int tile, int stages);

/*
 * gemm_plan -- the launch gemm_ex would make for these sizes, without making
 * it: CTAs in the grid, CTAs per cluster (2 for the pair tile) and dynamic
 * shared memory per CTA.  Needs a current CUDA device (it asks the runtime
 * how many CTA pairs can be resident).  M == 0, N == 0 or K == 0 plans no
 * GEMM kernel (grid 0).  Returns a gemm_status_t; outputs may be NULL.
 */
int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int stages, int b_col_major, int tile,
              int* grid, int* cluster, int* smem_bytes);

/*
 * gemm_schedule_set -- how the tensor-core kernel spreads output tiles over
 * its persistent CTAs (or CTA pairs), for the calls that follow from this
 * process (not thread-safe):
 *   0  automatic (default): currently the same as 1 (measured faster on
 *      GB300 for every workload of this library).
 *   1  whole tiles, round-robin over the units; no workspace.
 *   2  stream-K tail: when the last round of whole tiles would leave units
 *      idle, the leftover tiles are cut along K into segments spread evenly
 *      over all units; the unit holding a tile's first K segment adds the
 *      others' fp32 partials (in a fixed order) and writes C.  The partials
 *      go to a workspace the library allocates with cudaMalloc on first use,
 *      one per (device, stream), of at most one tile per unit (about 20 MB on
 *      GB300).  Calls that overlap on the GPU must use different streams.
 * Results are within the same tolerances for every schedule and, for one
 * schedule, bit-identical for every stage count.  Returns GEMM_ERR_ARG for
 * another value.
 */
int gemm_schedule_set(int schedule);

/*
 * gemm_noalloc -- gemm_ex on the tensor-core path with the stream-K tail
 * schedule (gemm_schedule_set's mode 2), for callers that must not allocate
 * device memory.  (This entry point has no counterpart on the pages: it is a
 * packaging of the same kernel.)
 *
 * Who needs it: code that cannot call cudaMalloc at the point where it runs
 * the GEMM -- for example a caller whose device memory is all owned by its
 * own pool or arena allocator, a latency-sensitive loop that must not hit the
 * implicit device synchronisation of cudaMalloc/cudaFree, or a process that
 * has handed out its free device memory.  gemm_ex's stream-K schedule
 * allocates its workspace on first use; this entry point instead keeps the
 * fp32 partial tiles and their flags in a fixed 20 MiB array inside the
 * library's device image (held by every GPU that loads the library, until the
 * process exits), and calls no allocating routine at all.
 *
 * Arguments, layout, alignment and return codes: as gemm_ex, tensor-core
 * dtypes only (GEMM_F32 gives GEMM_ERR_UNSUPPORTED).  The workspace is one
 * 128 x tile-width fp32 partial per CTA, plus flags: 19.9 MB for the 256-wide
 * tiles on 152 SMs.  GEMM_TILE_256x512_2SM asked for by name is refused with
 * GEMM_ERR_SCRATCH for every shape (its partials would take 38 MB); any
 * other launch whose workspace exceeds 20 MiB (a GPU with more SMs) is
 * refused the same way.  Both checks come before anything is enqueued.
 * Where GEMM_TILE_AUTO would pick the 256 x 512 tile, this entry point runs
 * GEMM_TILE_256x256_2SM instead, with the same `stages` and the same bits.
 *
 * Every call shares the one array (per GPU).  Each call clears the flags it
 * uses with cudaMemsetAsync on `stream` before its kernel (the array keeps
 * the previous call's contents).  Calls that overlap on the GPU -- on
 * different streams, or from different threads -- race on the array: order
 * them on one stream.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) and sets the kernel's shared-memory
 * limit; make that first call before any stream capture on that device.  The
 * address is then kept until the process exits: resetting the device
 * (cudaDeviceReset) and calling this entry point again is not supported.
 */
int gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
                 int b_col_major, int tile, void* stream);

/*
 * pipelined_copy -- dst[0 .. n_bytes) = src[0 .. n_bytes), streamed through a
 * ring of `stages` shared-memory slots of 8 KB per CTA (one bulk tensor-engine
 * copy into a slot and one out of it per chunk, full/empty mbarriers as in
 * the GEMM's ring, chunks walked grid-stride), asynchronous on `stream`.
 *
 * This is the bandwidth-bound counter-example to the GEMM: a copy has no
 * arithmetic to hide a load behind, which "Software Pipelining and Double
 * Buffering" ("When it pays"), the CUDA Handbook ("Asynchronous data
 * movement", closing rule) and the copy example after "Overlap needs stages"
 * on "learn-kernels.com, Matrix multiplication" name as the case where extra
 * stages do not pay.  Its stage sweep is measured by bench.py.  A ring wait
 * that runs out (2 s) leaves dst incomplete; nothing is reported.
 *   dst, src   device pointers, 16-byte aligned, ranges must not overlap
 *              (GEMM_ERR_ARG), owned by the caller
 *   n_bytes    >= 0, a multiple of 16 (GEMM_ERR_ALIGN otherwise); 0 is a no-op
 *   stages     1..8 (GEMM_ERR_ARG otherwise)
 */
int pipelined_copy(void* dst, const void* src, int64_t n_bytes, int stages, void* stream);

/*
 * mma_rate -- the tensor pipe's dense bf16 rate on this GPU, in SM clocks:
 * the per-SM factor of the GEMM's compute roofline (SMs x FLOP per SM per
 * clock x clock), measured rather than taken from a data sheet.
 *
 * `ctas` CTAs (at most one per SM) each fill a 128 x 64 and a 256 x 64 bf16
 * operand tile in shared memory, then issue n_mma back-to-back tcgen05.mma
 * (cta_group::1, kind::f16, M = 128, N = 256, K = 16, fp32 accumulate in
 * TMEM) from one thread; no global memory is read in between.  Each CTA reads
 * its SM clock (clock64) before the first issue and after the commit of the
 * last MMA has arrived.  FLOP per SM per clock = n_mma * 2*128*256*16 /
 * cycles[i].
 *   n_mma        1 .. 2^20 MMAs per CTA (GEMM_ERR_ARG otherwise)
 *   ctas         1 .. the device's SM count (GEMM_ERR_ARG otherwise)
 *   cycles       host array of `ctas` entries, written: SM clocks per CTA
 *   elapsed_ms   host pointer, written: CUDA-event time of the launch
 * Runs on the current device's legacy default stream and returns when the
 * kernel has finished (synchronous).  A CTA whose wait for its MMAs runs out
 * (2 s) writes -1 and the call returns GEMM_ERR_TIMEOUT.
 */
int mma_rate(int n_mma, int ctas, long long* cycles, float* elapsed_ms);

/*
 * mma_rate_pair -- mma_rate for the CTA-pair instruction the 256-row tiles
 * issue: `pairs` clusters of two CTAs (on two SMs each) allocate TMEM across
 * the pair, and each leader issues n_mma tcgen05.mma.cta_group::2 (M = 256,
 * N = 256, K = 16; each CTA supplies 128 rows of A and 128 columns of B),
 * timing them on its SM clock.  Per SM this is again 2*128*256*16 FLOP per
 * instruction.
 *   n_mma        1 .. 2^20 MMAs per pair (GEMM_ERR_ARG otherwise)
 *   pairs        1 .. half the device's SM count (GEMM_ERR_ARG otherwise)
 *   cycles       host array of `pairs` entries, written: each leader's SM clocks
 *   elapsed_ms   host pointer, written: CUDA-event time of the launch
 * Synchronous, on the legacy default stream; GEMM_ERR_TIMEOUT as mma_rate.
 */
int mma_rate_pair(int n_mma, int pairs, long long* cycles, float* elapsed_ms);

/*
 * gemm_debug_set -- test hook for the bounded waits (not thread-safe; affects
 * later launches of the tensor-core kernel from this process).
 *   wait_limit_ns      time a pipeline wait may spin before it gives up
 *                      (<= 0 restores the default of 2 s)
 *   withhold_arrive    -1: normal.  k >= 0: block 0's producer skips the
 *                      copy and the barrier arrive of its k-th K tile, so the
 *                      MMA warp's wait on that stage runs out.  Used to check
 *                      that a stuck pipeline ends with GEMM_ERR_TIMEOUT
 *                      instead of a hang.
 */
int gemm_debug_set(int64_t wait_limit_ns, int withhold_arrive);

/*
 * gemm_clock_log -- measurement hook (not thread-safe; affects later launches
 * of the tensor-core and SIMT kernels from this process).  With dev_buf
 * non-null, CTA 0 of every later launch adds, when it exits, its SM clock
 * ticks (clock64) to dev_buf[0] and its wall-clock nanoseconds (globaltimer)
 * to dev_buf[1], both counted from the point where it may first touch global
 * memory (the SIMT kernel: from the start of its tile).
 * dev_buf[0] * 1000 / dev_buf[1] is then the launches' mean SM clock in MHz.
 *   dev_buf   device pointer to two zeroed 64-bit unsigned integers, owned by
 *             the caller, live until every launch made while it was set has
 *             finished; NULL turns the hook off (the default)
 */
int gemm_clock_log(void* dev_buf);

#ifdef __cplusplus
}
#endif

#endif /* SSP_GEMM_H */
