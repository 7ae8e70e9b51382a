// gemm_tc_sm103a.cu -- warp-specialised tcgen05 GEMM with an N-stage TMA ring.
//
// C = alpha * A * B + beta * C, fp16/bf16 inputs, fp32 accumulation in tensor
// memory (TMEM), fp32 or bf16 output.
//
// The mainloop is the multi-stage pipeline of "learn-kernels.com, Matrix
// multiplication" (paragraph "Overlap needs stages": submit N stages of
// copies, wait for the oldest, compute on it, release it, submit the next)
// with the two roles given to different warps, the form the same page's last
// paragraph describes for Hopper: a producer waits for a buffer to be
// signalled empty and issues a TMA load into it, the TMA updates that stage's
// barrier on completion, a consumer waits on that barrier, runs the
// tensor-core MMAs and releases the buffer.  "Software Pipelining and Double
// Buffering", section "TMA-based pipelines", gives the single-thread bulk
// tensor copy and mbarrier wait this uses.  What changes on sm_103a:
//   * the consumer is one MMA warp in which a single elected thread issues
//     each tcgen05.mma (128 x BN x 16 per instruction), reading both
//     operands straight from shared memory and accumulating in TMEM, so
//     there is no shared->register stage at all;
//   * the release is tcgen05.commit, which arrives on the stage's "empty"
//     barrier once the MMAs reading it have finished;
//   * the CTA is persistent and keeps two accumulators in TMEM, so the
//     epilogue of one output tile overlaps the mainloop of the next (the
//     256 x 512 tile has room for one, and releases it in halves);
//   * a stage is one 64-deep K slice of both operands (one 128-byte swizzle
//     row of 16-bit data) on every tile, so the stage count alone sets the
//     ring's depth: 1..6 stages on the 128 x 128 and 256 x 256 tiles (32 KB
//     per CTA each), 1..4 on the 128 x 256 and 256 x 512 tiles (48 KB);
//   * the epilogue moves C with tensor copies (and, for beta = 1 with fp32 C,
//     adds into C at L2 with tensor reduces), and consecutive GEMMs on a
//     stream overlap their prologue through programmatic dependent launch.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and
// TMEM owner (the whole warp with an elected issuing lane; lane 0 of the
// leader alone on the 256 x 512 tile), warps 2..5 = epilogue (warp w reads
// TMEM lanes 32*(w%4)...).
//
// Ring protocol (slot s = i mod S, n = i div S for the i-th K tile a CTA
// handles): the producer waits empty[s] for parity (n&1)^1, arms full[s] with
// the stage's byte count and issues the copies; the MMA issuer waits full[s]
// for parity n&1, issues the stage's MMAs (K = 64 per stage, 16 per MMA)
// and commits to empty[s].  With S = 1 the producer's next copy waits for the
// MMAs of the same slot: the page's single buffer with a load phase and a
// compute phase.
//
// Every wait is bounded (wait_limit_ns, %globaltimer).  A wait that runs out
// records the failure in g_gemm_status, raises a shared abort flag that the
// other roles poll, and the CTA drains what it has in flight (its issued TMA
// copies and MMAs), frees TMEM and returns.  Nothing traps.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {

__device__ GemmDeviceStatus g_gemm_status;

namespace {

constexpr int BM = 128;                 // tile rows = TMEM lanes = UMMA M
constexpr int BK = 64;                  // K of one swizzle atom: 64 x 2 bytes = one 128-byte row
constexpr int UMMA_K = 16;              // K per tcgen05.mma (kind::f16)
constexpr int NUM_THREADS = 192;
constexpr int A_ATOM_BYTES = BM * BK * 2;  // 16 KB
constexpr int EPI_BOX_BYTES = 4096;         // one output box: 32 rows x 128 bytes
constexpr int kEpiMaxBufs = 4;              // output boxes per epilogue warp, at most
constexpr int kTcMaxSmem = 227 * 1024;      // dynamic shared memory a CTA may opt in to
constexpr int ROLE_PRODUCER = 0, ROLE_MMA = 1, ROLE_EPILOGUE = 2;

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, k_tiles;
    int group_m;
    int stages;
    int bn;           // tile width (columns of C per tile)
    int b_mn_major;
    int b_chunked;    // row-major B through a 3-D map: one copy per stage for all 64-column chunks
    int out_bf16;
    uint32_t idesc;
    float alpha, beta;
    void* C;
    long long ldc;
    unsigned long long wait_limit_ns;
    int withhold;
    // Stream-K tail: tiles [dp_tiles, num_tiles) are cut into K segments
    // spread evenly over the persistent units (sk_iters = their k-tiles).
    int dp_tiles;
    long long sk_iters;
    int epi_bufs;           // output boxes per epilogue warp (2..kEpiMaxBufs)
    float* ws;              // one partial tile per unit (per CTA: 128 x bn fp32)
    unsigned long long* clock_log;  // null, or [2]: CTA 0 adds its SM clocks and ns
    unsigned int* ws_flag;  // per unit and CTA rank: 1 = partial published
};

// One piece of work of a persistent unit: k-tiles [kb, ke) of a tile.
//   FULL     the whole K range: the epilogue writes C
//   PARTIAL  a later K segment of a stream-K tile: the epilogue publishes the
//            fp32 partial in the unit's workspace slot
//   FINISH   the K segment that starts at k = 0: the epilogue adds the
//            partials of units [slot_lo, slot_hi) in order, then writes C
enum JobRole { JOB_FULL = 0, JOB_PARTIAL = 1, JOB_FINISH = 2 };
struct Job {
    int tile, kb, ke, role, slot_lo, slot_hi;
};

struct SharedCtl {
    // full[S], empty[S], tmem_full[2], tmem_empty[2], drain (on the 256 x 512
    // tile: tmem_full[0] for the one accumulator, tmem_empty[h] for its halves)
    unsigned long long bar[2 * kTcMaxStages + 5];
    unsigned long long cbar[4 * kEpiMaxBufs];  // C box copies, per epilogue warp and box
    uint32_t tmem_base;
    int abort;
    int epi_ok[2];  // the epilogue's per-job go/abort decision, by job parity
};

// Shared-memory matrix descriptor for tcgen05 with 128-byte swizzle:
// start address, leading and stride byte offsets (16-byte units), the
// descriptor version bit (46) and the swizzle mode (61..63 = 2: 128 B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void record_timeout(int role, int iter) {
    if (atomicCAS(&g_gemm_status.code, 0, GEMM_ERR_TIMEOUT) == 0) {
        g_gemm_status.block = blockIdx.x;
        g_gemm_status.role = role;
        g_gemm_status.iter = iter;
        __threadfence();
    }
}

// Raise the abort flag of this CTA and, for a CTA pair, of the peer CTA.
template <bool PAIR>
__device__ __forceinline__ void raise_abort(volatile int* abort, uint32_t peer_rank) {
    *abort = 1;
    if constexpr (PAIR) {
        st_cluster_u32(mapa_shared(smem_addr(const_cast<int*>(abort)), peer_rank), 1u);
    }
}

// Wait for the phase of `bar` with parity `parity`; give up after
// limit_ns or when another role has raised the abort flag.
template <bool PAIR>
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                             unsigned long long limit_ns, int role, int iter,
                                             uint32_t peer_rank) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                record_timeout(role, iter);
                raise_abort<PAIR>(abort, peer_rank);
                return false;
            }
        }
    }
}

// Drain wait used after an abort: no abort check, still bounded.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity,
                                           unsigned long long limit_ns) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return;
    }
}

// Output tile of persistent work item t: groups of group_m tile rows are
// walked column by column so that CTAs running at the same time share A rows
// and B columns in L2.  Every other group walks its columns backwards, so
// that a group starts on the B columns the previous one has just read
// (measured on the 256 x 512 tile: 2.5 % fewer DRAM bytes, time level).
__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& tm, int& tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
    if (g & 1) tn = p.tiles_n - 1 - tn;
}

// First stream-K iteration of unit u: floor(u * W / U).
__device__ __forceinline__ long long sk_begin(const TcParams& p, int u, int U) {
    return static_cast<long long>(u) * p.sk_iters / U;
}

// The unit whose stream-K range holds iteration g.
__device__ __forceinline__ int sk_unit_of(const TcParams& p, long long g, int U) {
    int u = static_cast<int>((g * U) / p.sk_iters);
    while (u + 1 < U && sk_begin(p, u + 1, U) <= g) ++u;
    while (u > 0 && sk_begin(p, u, U) > g) --u;
    return u;
}

// The j-th job of unit u (false when it has no more).  Full tiles first (data
// parallel, tile u + i*U), then at most two stream-K segments.  A unit's range
// is shorter than one tile's K, so it touches at most two tiles; its
// non-finishing segment (if any) comes first, so no unit waits before it has
// published its own partial.
__device__ bool next_job(const TcParams& p, int u, int U, int j, Job& job) {
    const int n_dp = p.dp_tiles > u ? (p.dp_tiles - u + U - 1) / U : 0;
    if (j < n_dp) {
        job = {u + j * U, 0, p.k_tiles, JOB_FULL, 0, 0};
        return true;
    }
    if (p.sk_iters == 0) return false;
    const long long g0 = sk_begin(p, u, U), g1 = sk_begin(p, u + 1, U);
    if (g0 == g1) return false;
    const int KT = p.k_tiles;
    const long long ta = g0 / KT, tb = (g1 - 1) / KT;
    int js = j - n_dp;
    if (ta != tb) {  // tail of tile ta (published), then head of tile tb (finished)
        if (js == 0) {
            job = {p.dp_tiles + static_cast<int>(ta), static_cast<int>(g0 % KT), KT, JOB_PARTIAL,
                   0, 0};
            return true;
        }
        js -= 1;
        if (js != 0) return false;
        const int ke = static_cast<int>((g1 - 1) % KT) + 1;
        const int last = sk_unit_of(p, (tb + 1) * KT - 1, U);
        job = {p.dp_tiles + static_cast<int>(tb), 0, ke, JOB_FINISH, u + 1, last + 1};
        return true;
    }
    if (js != 0) return false;
    const int kb = static_cast<int>(g0 % KT), ke = static_cast<int>((g1 - 1) % KT) + 1;
    if (kb != 0) {
        job = {p.dp_tiles + static_cast<int>(ta), kb, ke, JOB_PARTIAL, 0, 0};
    } else {
        const int last = sk_unit_of(p, (ta + 1) * KT - 1, U);
        job = {p.dp_tiles + static_cast<int>(ta), 0, ke, JOB_FINISH, u + 1, last + 1};
    }
    return true;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Epilogue of whole output boxes [ci0, ci1) of one tile for this warp's 32
// TMEM lanes: each box of 32 rows x 128 bytes (CW = 32 fp32 or 64 bf16
// columns) is read from TMEM, scaled by alpha, written 128-byte swizzled into
// the warp's ring of nb boxes and sent by one tensor store, or for REDUCE by
// one tensor reduce-add into C.  The box width, the output type and the kind
// of write-back are compile-time, so the loop has no per-box branches: the
// general loop below, with its runtime tests for edges, stream-K partials and
// C read-back, issues about twice the instructions per box.
template <int CW, bool REDUCE>
__device__ __forceinline__ void epilogue_boxes(const CUtensorMap* tmC, uint32_t t_row,
                                               uint32_t epi_buf0, int nb, int ci0, int ci1,
                                               int col0, int row_base, float alpha, int lane) {
    for (int ci = ci0; ci < ci1; ++ci) {
        const uint32_t buf = epi_buf0 + static_cast<uint32_t>(ci % nb) * 4096u;
        // The store that last used this box has read it.
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint32_t r[CW];
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(ci * CW),
                           *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        if constexpr (CW == 64)
            tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(ci * CW + 32),
                               *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            uint4 u;
            if constexpr (CW == 32) {
                u = make_uint4(__float_as_uint(alpha * __uint_as_float(r[4 * jj])),
                               __float_as_uint(alpha * __uint_as_float(r[4 * jj + 1])),
                               __float_as_uint(alpha * __uint_as_float(r[4 * jj + 2])),
                               __float_as_uint(alpha * __uint_as_float(r[4 * jj + 3])));
            } else {
                __nv_bfloat162 h[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    h[e] = __floats2bfloat162_rn(alpha * __uint_as_float(r[8 * jj + 2 * e]),
                                                 alpha * __uint_as_float(r[8 * jj + 2 * e + 1]));
                u = *reinterpret_cast<const uint4*>(h);
            }
            st_shared_v4(buf + lane * 128 + ((jj ^ (lane & 7)) << 4), u);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            if constexpr (REDUCE) tma_reduce_add_2d(tmC, buf, col0 + ci * CW, row_base);
            else tma_store_2d(tmC, buf, col0 + ci * CW, row_base);
            bulk_commit_group();
        }
    }
}

// Named barrier over the four epilogue warps (128 threads).
__device__ __forceinline__ void epilogue_bar_sync() {
    asm volatile("barrier.sync 1, 128;" ::: "memory");
}

// PAIR = false: one CTA computes a 128 x bn tile with tcgen05.mma.cta_group::1.
// PAIR = true: a cluster of two CTAs computes a 256 x bn tile with
// tcgen05.mma.cta_group::2: CTA rank r stages rows 128r..128r+127 of the A
// tile and columns (bn/2)r..(bn/2)r+bn/2-1 of the B tile, the leader (rank 0)
// issues every MMA, and each CTA's TMEM receives its own 128 rows of C.
// Both CTAs' copies of a stage complete on the LEADER's full[s], which the
// leader arms with the pair's byte count; the MMA's commit frees the slot in
// both CTAs (multicast), and both epilogues release the accumulator to the
// leader.  (Relaying the peer's stage through a thread instead costs one
// remote round trip per stage and capped the pair at ~60 % of the MMA rate.)
//
// A stage is K = 64 (4 MMAs of K = 16 between two ring waits; 8 on the
// 256 x 512 tile).  Each stage costs the MMA issuer one wait and one commit;
// with the descriptors advanced by plain adds and the pair's peer copies
// completing on the leader's barrier directly, those stay off the tensor
// pipe's critical path (measured: six stages of K = 64 run level with three
// of K = 128 and give the same bits).
//
// WIDE (a pair): the 256 x 512 tile.  Each K = 16 step is two
// N = 256 MMAs that share the A operand, so a stage carries a quarter fewer
// operand bytes per FLOP than two 256 x 256 tiles would.  CTA rank r stages
// two 128-column pieces of B, tile columns 128r.. and 256 + 128r.., so that
// MMA h writes tile columns 256h..256h+255 into TMEM columns 256h.. of one
// 512-column accumulator.  With no second accumulator the epilogue cannot
// overlap the next tile's whole mainloop, so the accumulator is released in
// halves: the epilogue frees columns 0..255 first, the next tile's h = 0 MMAs
// start at once, and each stage's h = 1 MMAs (with the stage's release) wait
// until columns 256..511 are free too, at most S stages behind.  Both halves
// still see their K steps in order, so C is bit-identical to the 256-wide
// pair tile's.
template <bool PAIR, bool WIDE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Swizzled TMA destinations and UMMA operands want 1024-byte alignment.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    static_assert(!WIDE || PAIR, "the 256 x 512 tile is a CTA pair");
    constexpr int TILE_M = PAIR ? 2 * BM : BM;
    constexpr int A_STAGE_BYTES = A_ATOM_BYTES;        // 128 rows x K = 64
    constexpr int B_CHUNK_BYTES = 64 * BK * 2;         // MN-major B: one 64-column chunk of a stage
    const int S = p.stages;
    const int b_cols = PAIR ? p.bn / 2 : p.bn;   // B columns staged by this CTA
    const int b_stage_bytes = b_cols * BK * 2;   // this CTA's B columns x K = 64
    uint8_t* a_ring = smem;
    uint8_t* b_ring = smem + S * A_STAGE_BYTES;
    uint8_t* epi_ring = b_ring + S * b_stage_bytes;  // 4 warps x epi_bufs output boxes
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(epi_ring + 4 * p.epi_bufs * EPI_BOX_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? (cluster_ctarank() & 1u) : 0u;
    const uint32_t peer_rank = rank ^ 1u;
    const bool leader = rank == 0;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int num_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    const uint32_t bar0 = smem_addr(&ctl->bar[0]);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    volatile int* abort_flag = &ctl->abort;
    // Two accumulators of bn columns (256 or 512 in all), or one of 512 (WIDE).
    const uint32_t tmem_cols = WIDE ? 512u : 2u * p.bn;
    constexpr uint16_t kPairMask = 0x3;

    if (threadIdx.x == 0) {
        // The tensor maps are kernel parameters, not data an earlier grid
        // writes: fetch them into the descriptor cache before waiting on it.
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), PAIR ? 8 : 4);  // one arrive per epilogue warp (both CTAs)
        }
        mbar_init(drain_bar, 1);
        for (int b = 0; b < 4 * kEpiMaxBufs; ++b) mbar_init(smem_addr(&ctl->cbar[b]), 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_addr(&ctl->tmem_base), tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(&ctl->tmem_base), tmem_cols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    // The grid is launched with programmatic stream serialization: the next
    // GEMM on the stream may be scheduled as soon as every CTA of this one has
    // got here, so its CTAs take the SMs this grid's last round leaves idle
    // and run their prologue early.  Nothing above touches global memory;
    // nothing below does before the previous grid has completed.
    griddep_launch_dependents();
    griddep_wait();
    // SM clock of this launch (measurement hook): CTA 0's clock ticks and
    // wall-clock nanoseconds from here to its exit.
    const bool log_clock = p.clock_log != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
    long long clk0 = 0;
    unsigned long long ns0 = 0;
    if (log_clock) {
        clk0 = clock64();
        ns0 = globaltimer_ns();
    }

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t stage_bytes = A_STAGE_BYTES + b_stage_bytes;
            // The leader's full[s] counts the bytes of both CTAs of a pair.
            const uint32_t armed_bytes = PAIR ? 2u * stage_bytes : stage_bytes;
            const uint32_t leader_full0 = PAIR ? mapa_shared(full_bar(0), 0u) : full_bar(0);
            // A panels are reused by the next round of tiles (tiles are walked
            // in groups of tile rows): ask L2 to keep them over B and C lines.
            const uint64_t a_policy = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            Job job;
            for (int j = 0; ok && next_job(p, unit, num_units, j, job); ++j) {
                int tm, tn;
                tile_coords(p, job.tile, tm, tn);
                const int a_row = tm * TILE_M + static_cast<int>(rank) * BM;
                const int b_col = tn * p.bn + static_cast<int>(rank) * b_cols;
                // B pieces of this CTA: one of b_cols columns, or (WIDE) two of
                // 128 columns, tile columns 128r and 256 + 128r.
                constexpr int NPIECES = WIDE ? 2 : 1;
                const int pw = b_cols / NPIECES;
                for (int kt = job.kb; kt < job.ke; ++kt) {
                    if (!bounded_wait<PAIR>(empty_bar(s), ph ^ 1u, abort_flag, p.wait_limit_ns,
                                            ROLE_PRODUCER, it, peer_rank)) {
                        ok = false;
                        break;
                    }
                    if (!(it == p.withhold && blockIdx.x == 0)) {
                        const uint32_t a_dst = smem_addr(a_ring + s * A_STAGE_BYTES);
                        const uint32_t b_dst = smem_addr(b_ring + s * b_stage_bytes);
                        if (leader) mbar_arrive_expect_tx(full_bar(s), armed_bytes);
                        // A: one 64 (K) x 128 (rows) box; B: one copy per piece
                        // (MN-major: all 64-column chunks at once through the 3-D
                        // map, or one per chunk; K-major: one 64 x pw box).
                        const int k0 = kt * BK;
                        if (PAIR && !leader) {
                            const uint32_t bar = leader_full0 + 8u * s;
                            tma_load_2d_pair_hint(a_dst, &tmA, bar, k0, a_row, a_policy);
#pragma unroll
                            for (int pc = 0; pc < NPIECES; ++pc) {
                                const int bc = WIDE ? tn * p.bn + pc * 256 + static_cast<int>(rank) * pw : b_col;
                                const uint32_t bd = b_dst + static_cast<uint32_t>(
                                    pc * (p.b_mn_major ? (pw / 64) * B_CHUNK_BYTES : pw * 128));
                                if (p.b_chunked) {
                                    tma_load_3d_pair(bd, &tmB, bar, 0, k0, bc / 64);
                                } else if (p.b_mn_major) {
                                    for (int j = 0; j < pw / 64; ++j)
                                        tma_load_2d_pair(bd + j * B_CHUNK_BYTES, &tmB, bar, bc + 64 * j,
                                                         k0);
                                } else {
                                    tma_load_2d_pair(bd, &tmB, bar, k0, bc);
                                }
                            }
                        } else {
                            tma_load_2d_hint(a_dst, &tmA, full_bar(s), k0, a_row, a_policy);
#pragma unroll
                            for (int pc = 0; pc < NPIECES; ++pc) {
                                const int bc = WIDE ? tn * p.bn + pc * 256 + static_cast<int>(rank) * pw : b_col;
                                const uint32_t bd = b_dst + static_cast<uint32_t>(
                                    pc * (p.b_mn_major ? (pw / 64) * B_CHUNK_BYTES : pw * 128));
                                if (p.b_chunked) {
                                    tma_load_3d(bd, &tmB, full_bar(s), 0, k0, bc / 64);
                                } else if (p.b_mn_major) {
                                    for (int j = 0; j < pw / 64; ++j)
                                        tma_load_2d(bd + j * B_CHUNK_BYTES, &tmB, full_bar(s),
                                                    bc + 64 * j, k0);
                                } else {
                                    tma_load_2d(bd, &tmB, full_bar(s), k0, bc);
                                }
                            }
                        }
                    }
                    ++it;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    // Let every copy this CTA armed land before the CTA exits (for
                    // a pair this also covers the peer's copies of those stages).
                    const int first = it - S > 0 ? it - S : 0;
                    for (int j = first; j < it; ++j) {
                        if (j == p.withhold && blockIdx.x == 0) continue;
                        drain_wait(full_bar(j % S), static_cast<uint32_t>((j / S) & 1),
                                   p.wait_limit_ns);
                    }
                } else {
                    // The peer's copies complete on the leader's barriers, which this
                    // CTA cannot wait on: give them a bounded grace period (a stage
                    // lands within microseconds), then the closing cluster barrier
                    // keeps this CTA alive until the leader has drained as well.
                    const unsigned long long grace =
                        p.wait_limit_ns < 200000ull ? p.wait_limit_ns : 200000ull;
                    const unsigned long long t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < grace) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // With 4 MMAs per stage the whole warp runs the issue loop (on a CTA
        // pair, the leader's warp): every lane polls the ring's barriers and
        // elect.sync picks the lane that issues each MMA and commit.  A lone
        // issuing lane that stops for a barrier poll every 4 MMAs leaves the
        // tensor pipe idle for part of the poll; the convergent warp does not
        // (measured, the same bits: +6.5 % on the 128 x 128 tile at 6 stages,
        // +1.5 % on the 128 x 256 tile of fp16 2048^3, +1 to 2 % on the
        // 256 x 256 pair tile).  The 256 x 512 tile, with 8 MMAs per stage and
        // the held-back second half, keeps the leader's lane 0 alone, which
        // measured level or better there.
        if ((!WIDE || lane == 0) && leader) {
            // -------------------------------------------------------- MMA issuer
            // K-major operands: 128-byte rows (the stage's K = 64), 8-row groups
            // 1024 bytes apart; one K=16 step is 32 bytes along the row.
            // MN-major B: 64-column chunks B_CHUNK_BYTES
            // apart (leading offset), 8-row K groups 1024 bytes apart; one K=16
            // step is 16 rows = 2048 bytes.
            // The descriptors of stage 0's first MMA; every other MMA of the
            // ring only moves the start address (the low 14 bits, in 16-byte
            // units), which stays below 2^14 for any shared-memory address.
            const uint64_t a_desc0 = smem_desc(smem_addr(a_ring), 16u, 1024u);
            const uint64_t b_desc0 =
                smem_desc(smem_addr(b_ring), p.b_mn_major ? B_CHUNK_BYTES : 16u, 1024u);
            const uint32_t a_lo = static_cast<uint32_t>(a_desc0);
            const uint32_t a_hi = static_cast<uint32_t>(a_desc0 >> 32);
            const uint32_t b_lo = static_cast<uint32_t>(b_desc0);
            const uint32_t b_hi = static_cast<uint32_t>(b_desc0 >> 32);
            // B start-address step (16-byte units) per K = 16.
            const uint32_t b_k16 = p.b_mn_major ? 2048u / 16u : 32u / 16u;
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            int lt = 0;
            bool ok = true;
            Job job;
            // A bounded ring wait; in the convergent loop every lane waits and
            // the warp goes on only if all of them saw the phase complete.
            auto mma_wait = [&](uint32_t bar, uint32_t parity, int itx) -> bool {
                const bool r = bounded_wait<PAIR>(bar, parity, abort_flag, p.wait_limit_ns, ROLE_MMA,
                                                  itx, peer_rank);
                if constexpr (WIDE) return r;
                else return __all_sync(0xffffffffu, r) != 0;
            };
            if constexpr (WIDE) {
                // One accumulator in two halves: tmem_empty[h] is released by the
                // epilogue once it has read columns 256h..256h+255.
                int dq_s[kTcMaxStagesWide], dq_kt[kTcMaxStagesWide];  // stages whose h = 1 MMAs wait
                for (int j = 0; ok && next_job(p, unit, num_units, j, job); ++j, ++lt) {
                    const uint32_t tph = static_cast<uint32_t>(lt & 1) ^ 1u;
                    if (!bounded_wait<PAIR>(tempty_bar(0), tph, abort_flag, p.wait_limit_ns, ROLE_MMA,
                                            it, peer_rank)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    bool d1 = mbar_try_wait(tempty_bar(1), tph);
                    if (d1) tc_fence_after();
                    int nd = 0;
                    // The stage's MMAs into half h: N = 256, B from piece h (16 KB on).
                    auto issue_half = [&](int h, int ss, int kt_) {
                        const uint32_t a_s = a_lo + static_cast<uint32_t>(ss * A_STAGE_BYTES) / 16u;
                        const uint32_t b_s = b_lo + static_cast<uint32_t>(ss * b_stage_bytes) / 16u +
                                             static_cast<uint32_t>(h) * (16384u / 16u);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint64_t ad = (static_cast<uint64_t>(a_hi) << 32) |
                                                (a_s + static_cast<uint32_t>(kk) * 2u);
                            const uint64_t bd = (static_cast<uint64_t>(b_hi) << 32) |
                                                (b_s + static_cast<uint32_t>(kk) * b_k16);
                            const uint32_t accum = (kt_ != job.kb || kk != 0) ? 1u : 0u;
                            umma_f16_pair(tmem_base + static_cast<uint32_t>(h) * 256u, ad, bd, p.idesc,
                                          accum);
                        }
                    };
                    // Catch up the waiting stages' h = 1 MMAs, in K order, and free their slots.
                    auto flush = [&]() {
                        for (int i = 0; i < nd; ++i) {
                            issue_half(1, dq_s[i], dq_kt[i]);
                            umma_commit_pair_multicast(empty_bar(dq_s[i]), kPairMask);
                        }
                        nd = 0;
                    };
                    for (int kt = job.kb; kt < job.ke; ++kt) {
                        if (!bounded_wait<PAIR>(full_bar(s), ph, abort_flag, p.wait_limit_ns,
                                                ROLE_MMA, it, peer_rank)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_half(0, s, kt);
                        if (!d1) {
                            d1 = mbar_try_wait(tempty_bar(1), tph);
                            if (d1) tc_fence_after();
                        }
                        if (d1) {
                            flush();
                            issue_half(1, s, kt);
                            umma_commit_pair_multicast(empty_bar(s), kPairMask);
                        } else {
                            dq_s[nd] = s;
                            dq_kt[nd] = kt;
                            if (++nd == S) {  // every slot is held: wait for the second half
                                if (!bounded_wait<PAIR>(tempty_bar(1), tph, abort_flag,
                                                        p.wait_limit_ns, ROLE_MMA, it, peer_rank)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                d1 = true;
                                flush();
                            }
                        }
                        ++it;
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (!d1) {
                        if (!bounded_wait<PAIR>(tempty_bar(1), tph, abort_flag, p.wait_limit_ns,
                                                ROLE_MMA, it, peer_rank)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    flush();
                    // accumulator ready for the epilogue (of both CTAs)
                    umma_commit_pair_multicast(tfull_bar(0), kPairMask);
                }
            } else {
            for (int j = 0; ok && next_job(p, unit, num_units, j, job); ++j, ++lt) {
                const int acc = lt & 1;
                const uint32_t acc_ph = static_cast<uint32_t>((lt >> 1) & 1);
                if (!mma_wait(tempty_bar(acc), acc_ph ^ 1u, it)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.bn);
                for (int kt = job.kb; kt < job.ke; ++kt) {
                    if (!mma_wait(full_bar(s), ph, it)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = a_lo + static_cast<uint32_t>(s * A_STAGE_BYTES) / 16u;
                    const uint32_t b_s = b_lo + static_cast<uint32_t>(s * b_stage_bytes) / 16u;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t ad = (static_cast<uint64_t>(a_hi) << 32) |
                                            (a_s + static_cast<uint32_t>(kk) * 2u);
                        const uint64_t bd = (static_cast<uint64_t>(b_hi) << 32) |
                                            (b_s + static_cast<uint32_t>(kk) * b_k16);
                        const uint32_t accum = (kt != job.kb || kk != 0) ? 1u : 0u;
                        if (elect_one_sync()) {
                            if constexpr (PAIR) umma_f16_pair(d_tmem, ad, bd, p.idesc, accum);
                            else umma_f16(d_tmem, ad, bd, p.idesc, accum);
                        }
                        __syncwarp();
                    }
                    // slot s is free (in both CTAs) once these MMAs finish
                    if (elect_one_sync()) {
                        if constexpr (PAIR) umma_commit_pair_multicast(empty_bar(s), kPairMask);
                        else umma_commit(empty_bar(s));
                    }
                    __syncwarp();
                    ++it;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator ready for the epilogue (of both CTAs)
                if (elect_one_sync()) {
                    if constexpr (PAIR) umma_commit_pair_multicast(tfull_bar(acc), kPairMask);
                    else umma_commit(tfull_bar(acc));
                }
                __syncwarp();
            }
            }
            if (!ok) {
                // Wait for every MMA this warp issued before TMEM is freed.
                if constexpr (WIDE) umma_commit_pair_multicast(drain_bar, 0x1);
                else {
                    if (elect_one_sync()) {
                        if constexpr (PAIR) umma_commit_pair_multicast(drain_bar, 0x1);
                        else umma_commit(drain_bar);
                    }
                    __syncwarp();
                }
                if (lane == 0) drain_wait(drain_bar, 0u, p.wait_limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t tempty_leader0 = PAIR ? mapa_shared(tempty_bar(0), 0u) : tempty_bar(0);
        const int ctas_per_unit = PAIR ? 2 : 1;
        const size_t slot_floats = static_cast<size_t>(BM) * p.bn;  // one CTA's partial
        volatile int* epi_ok = ctl->epi_ok;
        // Output boxes of 32 rows x 128 bytes: 32 fp32 or 64 bf16 columns.
        const int cw = p.out_bf16 ? 64 : 32;
        // This warp's ring of nb output boxes (32 rows x 128 bytes, 4 KB),
        // each written back by one tensor copy: a store, or for beta = 1 with
        // fp32 C a reduce-add at L2.  For other beta != 0 the box is first
        // filled with C by a tensor copy (issued up to nb boxes ahead, the
        // first ones before the accumulator is ready) and updated in place.
        const int nb = p.epi_bufs;
        const uint32_t epi_buf0 = smem_addr(epi_ring) + static_cast<uint32_t>(q * nb) * 4096u;
        const uint32_t cbar0 = smem_addr(&ctl->cbar[q * kEpiMaxBufs]);
        const bool load_c = p.beta != 0.0f;
        // beta = 1 with fp32 C: the box of alpha*acc is added into C at L2 by
        // a tensor reduce instead of C being read in (one fp32 add per
        // element, the same value as fmaf(1, C, alpha*acc)).
        const bool reduce_c = p.beta == 1.0f && !p.out_bf16;
        uint32_t c_phase = 0;    // bit b: parity of the next C copy into box b
        uint32_t c_pending = 0;  // bit b: a C copy into box b is issued and not yet consumed
        int lt = 0;
        Job job;
        for (int j = 0; next_job(p, unit, num_units, j, job); ++j, ++lt) {
            const int acc = WIDE ? 0 : (lt & 1);
            const uint32_t acc_ph = static_cast<uint32_t>(WIDE ? (lt & 1) : ((lt >> 1) & 1));
            int tm, tn;
            tile_coords(p, job.tile, tm, tn);
            const int row_base = tm * TILE_M + static_cast<int>(rank) * BM + 32 * q;  // this warp's rows
            const int col0 = tn * p.bn;
            const int nchunks = p.bn / cw;
            // A box goes through the tensor copies when it lies inside M x N
            // but for rows past M (the copies fill and clip whole rows); a box
            // across the N edge is read and written by each thread for its row.
            auto tma_box = [&](int ci) {
                return row_base < p.M && col0 + (ci + 1) * cw <= p.N;
            };
            auto issue_c = [&](int ci) {  // lane 0: copy C box ci into box ci % nb
                const int b = ci % nb;
                mbar_arrive_expect_tx(cbar0 + 8u * b, 4096u);
                tma_load_2d(epi_buf0 + static_cast<uint32_t>(b) * 4096u, &tmC, cbar0 + 8u * b,
                            col0 + ci * cw, row_base);
            };
            const bool job_loads_c = load_c && !reduce_c && job.role != JOB_PARTIAL;
            // The previous job's stores have read their boxes (issued before
            // this job's accumulator wait, this costs nothing in steady state).
            if (lane == 0) bulk_wait_group_read<0>();
            if (job_loads_c && !*abort_flag) {
                // Prefetch the first C boxes.
                for (int ci = 0; ci < nchunks && ci < nb; ++ci) {
                    if (!tma_box(ci)) continue;
                    if (lane == 0) issue_c(ci);
                    c_pending |= 1u << (ci % nb);
                }
            }
            // One thread waits (for the accumulator and, when finishing a
            // stream-K tile, for the other segments' partials) and tells the
            // other 127 through shared memory: every epilogue thread takes the
            // same path, so the named barriers below always fill.
            if (warp == 2 && lane == 0) {
                bool ok = bounded_wait<PAIR>(tfull_bar(acc), acc_ph, abort_flag, p.wait_limit_ns,
                                             ROLE_EPILOGUE, lt, peer_rank);
                if (ok && job.role == JOB_FINISH) {
                    for (int u2 = job.slot_lo; ok && u2 < job.slot_hi; ++u2) {
                        const unsigned int* f = p.ws_flag + u2 * ctas_per_unit + rank;
                        const unsigned long long t0 = globaltimer_ns();
                        while (ld_acquire_gpu(f) == 0u) {
                            if (*abort_flag) {
                                ok = false;
                                break;
                            }
                            if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                                record_timeout(ROLE_EPILOGUE, lt);
                                raise_abort<PAIR>(abort_flag, peer_rank);
                                ok = false;
                                break;
                            }
                        }
                    }
                }
                epi_ok[j & 1] = ok ? 1 : 0;
            }
            __syncwarp();
            epilogue_bar_sync();
            if (!epi_ok[j & 1]) break;
            if (job.role == JOB_FINISH) __threadfence();  // read the partials after the flags
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(acc * p.bn);
            // Partials are kept in the order the threads produce them: float4
            // i of chunk ci of warp q's lane l at ((q * nchunks + ci) * cw/4 + i) * 32 + l,
            // so that each warp access is 512 contiguous bytes.
            const size_t my_slot_off = (static_cast<size_t>(unit) * ctas_per_unit + rank) * slot_floats;
            // Whole tile, nothing read back: the branch-free box loop.
            const bool fast = job.role == JOB_FULL && !job_loads_c && row_base < p.M &&
                              col0 + p.bn <= p.N;
            if (fast) {
                auto boxes = [&](int c0, int c1) {
                    if (p.out_bf16)
                        epilogue_boxes<64, false>(&tmC, t_row, epi_buf0, nb, c0, c1, col0, row_base,
                                                  p.alpha, lane);
                    else if (reduce_c)
                        epilogue_boxes<32, true>(&tmC, t_row, epi_buf0, nb, c0, c1, col0, row_base,
                                                 p.alpha, lane);
                    else
                        epilogue_boxes<32, false>(&tmC, t_row, epi_buf0, nb, c0, c1, col0, row_base,
                                                  p.alpha, lane);
                };
                const int nh = WIDE ? nchunks / 2 : nchunks;
                boxes(0, nh);
                if constexpr (WIDE) {
                    // Columns 0..255 are read: the next tile's first half may start.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader0);
                }
                boxes(nh, nchunks);
            }
            for (int ci = 0; !fast && ci < nchunks; ++ci) {
                const int c = ci * cw;
                const int col_base = col0 + c;
                const int b = ci % nb;
                const uint32_t buf = epi_buf0 + static_cast<uint32_t>(b) * 4096u;
                const bool via_tma = tma_box(ci);
                if (!job_loads_c) {
                    // The store that last used this box has read it.
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                }
                float f[64];
                {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(r[i]);
                    if (cw == 64) {
                        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c + 32), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) f[32 + i] = __uint_as_float(r[i]);
                    }
                }
                const size_t part_off = static_cast<size_t>((q * nchunks + ci) * (cw / 4)) * 32 + lane;
                if (job.role == JOB_PARTIAL) {
                    // Publish this segment's fp32 partial (rows past M too: the
                    // slot is private to this unit).
                    float4* dst = reinterpret_cast<float4*>(p.ws + my_slot_off) + part_off;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i < cw / 4)
                            dst[32 * i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
                    continue;
                }
                if (job.role == JOB_FINISH) {
                    // acc(k from 0) + partial(unit lo) + ... in unit order.
                    for (int u2 = job.slot_lo; u2 < job.slot_hi; ++u2) {
                        const float4* src = reinterpret_cast<const float4*>(
                            p.ws + (static_cast<size_t>(u2) * ctas_per_unit + rank) * slot_floats) +
                                            part_off;
                        float4 v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < cw / 4) v[i] = __ldcg(src + 32 * i);  // written by another SM: read L2
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (i < cw / 4) {
                                f[4 * i + 0] += v[i].x;
                                f[4 * i + 1] += v[i].y;
                                f[4 * i + 2] += v[i].z;
                                f[4 * i + 3] += v[i].w;
                            }
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 64; ++i) f[i] *= p.alpha;
                if (!via_tma) {
                    // A box across the N edge (or past M): each thread reads
                    // and writes the columns of its own row that lie below N.
                    const int row = row_base + lane;
                    if (row < p.M && col_base < p.N) {
                        if (p.out_bf16) {
                            __nv_bfloat16* cp = static_cast<__nv_bfloat16*>(p.C) +
                                                static_cast<long long>(row) * p.ldc + col_base;
#pragma unroll
                            for (int i = 0; i < 64; ++i) {
                                if (i < cw && col_base + i < p.N) {
                                    float o = f[i];
                                    if (load_c) o = fmaf(p.beta, __bfloat162float(cp[i]), o);
                                    cp[i] = __float2bfloat16_rn(o);
                                }
                            }
                        } else {
                            float* cp = static_cast<float*>(p.C) +
                                        static_cast<long long>(row) * p.ldc + col_base;
#pragma unroll
                            for (int i = 0; i < 64; ++i) {
                                if (i < cw && col_base + i < p.N) {
                                    float o = f[i];
                                    if (load_c) o = fmaf(p.beta, cp[i], o);
                                    cp[i] = o;
                                }
                            }
                        }
                    }
                    continue;
                }
                if (job_loads_c) {
                    // out = alpha*acc + beta*C, C from this thread's row of the box.
                    bounded_wait<PAIR>(cbar0 + 8u * b, (c_phase >> b) & 1u, abort_flag,
                                       p.wait_limit_ns, ROLE_EPILOGUE, lt, peer_rank);
                    c_phase ^= 1u << b;
                    c_pending &= ~(1u << b);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const uint4 u = ld_shared_v4(buf + lane * 128 + ((jj ^ (lane & 7)) << 4));
                        if (cw == 32) {
                            f[4 * jj + 0] = fmaf(p.beta, __uint_as_float(u.x), f[4 * jj + 0]);
                            f[4 * jj + 1] = fmaf(p.beta, __uint_as_float(u.y), f[4 * jj + 1]);
                            f[4 * jj + 2] = fmaf(p.beta, __uint_as_float(u.z), f[4 * jj + 2]);
                            f[4 * jj + 3] = fmaf(p.beta, __uint_as_float(u.w), f[4 * jj + 3]);
                        } else {
                            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 fc = __bfloat1622float2(h[e]);
                                f[8 * jj + 2 * e] = fmaf(p.beta, fc.x, f[8 * jj + 2 * e]);
                                f[8 * jj + 2 * e + 1] = fmaf(p.beta, fc.y, f[8 * jj + 2 * e + 1]);
                            }
                        }
                    }
                }
                // This thread's row of the box, 128-byte swizzled as the tensor
                // store expects, then one lane stores the 32-row box.
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    uint4 u;
                    if (cw == 32) {
                        u = make_uint4(__float_as_uint(f[4 * jj]), __float_as_uint(f[4 * jj + 1]),
                                       __float_as_uint(f[4 * jj + 2]), __float_as_uint(f[4 * jj + 3]));
                    } else {
                        __nv_bfloat162 h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            h[e] = __floats2bfloat162_rn(f[8 * jj + 2 * e], f[8 * jj + 2 * e + 1]);
                        u = *reinterpret_cast<const uint4*>(h);
                    }
                    st_shared_v4(buf + lane * 128 + ((jj ^ (lane & 7)) << 4), u);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    if (reduce_c) tma_reduce_add_2d(&tmC, buf, col_base, row_base);
                    else tma_store_2d(&tmC, buf, col_base, row_base);
                    bulk_commit_group();
                }
                // Refill the box the previous chunk's store used with C box
                // ci + nb - 1 once that store has read it.
                const int nxt = ci + nb - 1;
                if (job_loads_c && ci >= 1 && nxt < nchunks && tma_box(nxt) && !*abort_flag) {
                    if (lane == 0) {
                        bulk_wait_group_read<1>();
                        issue_c(nxt);
                    }
                    c_pending |= 1u << (nxt % nb);
                }
            }
            tc_fence_before();
            if (job.role == JOB_PARTIAL) {
                __threadfence();
                epilogue_bar_sync();  // all 128 rows of this CTA's partial are written
                if (warp == 2 && lane == 0)
                    st_release_gpu(p.ws_flag + unit * ctas_per_unit + rank, 1u);
            } else if (job.role == JOB_FINISH && job.slot_lo < job.slot_hi) {
                epilogue_bar_sync();  // every row has read the partials: re-arm the flags
                if (warp == 2 && lane == 0)
                    for (int u2 = job.slot_lo; u2 < job.slot_hi; ++u2)
                        p.ws_flag[u2 * ctas_per_unit + rank] = 0u;
            }
            __syncwarp();
            if (lane == 0) {
                if constexpr (WIDE) {
                    if (!fast) mbar_arrive_cluster(tempty_leader0);  // both halves at once
                    mbar_arrive_cluster(tempty_leader0 + 8u);
                } else if constexpr (PAIR) {
                    mbar_arrive_cluster(tempty_leader0 + 8u * acc);
                } else {
                    mbar_arrive(tempty_bar(acc));
                }
            }
        }
        // C copies still in flight after an abort land before the CTA exits.
        if (lane == 0)
            for (int b = 0; b < nb; ++b)
                if ((c_pending >> b) & 1u)
                    drain_wait(cbar0 + 8u * b, (c_phase >> b) & 1u, p.wait_limit_ns);
    }

    if (warp >= 2 && lane == 0) bulk_wait_group_all();  // this warp's C stores are done
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // no remote arrive or multicast is still pending
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, tmem_cols);
        else tmem_dealloc(tmem_base, tmem_cols);
    }
    if (log_clock) {
        atomicAdd(p.clock_log, static_cast<unsigned long long>(clock64() - clk0));
        atomicAdd(p.clock_log + 1, globaltimer_ns() - ns0);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tensor map over a row-major (rows x cols) matrix with leading dimension
// ld (elements), 16-bit elements, box (box_cols x box_rows), 128-byte swizzle,
// zero fill outside the matrix.
bool encode_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t rows, uint64_t cols,
               uint64_t ld, uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major B (K x N, N a multiple of 64) as a 3-D tensor: 64 columns
// (contiguous), K rows (stride ld elements), N/64 chunks (stride 64 elements).
// A box (64, bks, chunks) then lands chunk after chunk, each chunk's bks rows
// (the K of one stage) of 128 bytes contiguous and 128-byte swizzled: the
// MN-major operand layout the MMA reads, filled by one copy instead of one
// per chunk.
bool encode_b_chunked(CUtensorMap* map, const void* base, bool bf16, uint64_t K, uint64_t N,
                      uint64_t ld, uint32_t chunks, uint32_t bks) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, K, N / 64};
    cuuint64_t strides[2] = {ld * 2, 128};
    cuuint32_t box[3] = {64, bks, chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over C (rows x cols, leading dimension ld elements) for the
// epilogue's box stores: 32 rows x 128 bytes (32 fp32 or 64 bf16 columns),
// 128-byte swizzle.
bool encode_c(CUtensorMap* map, void* base, bool bf16, uint64_t rows, uint64_t cols, uint64_t ld) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * es};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int device_sms(int dev) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return cache[dev];
}

using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const TcParams);

// The kernel instance for a tile (wide: the 256 x 512 pair tile).
TcKernel kernel_for(bool pair, bool wide) {
    if (pair) return wide ? gemm_tc_kernel<true, true> : gemm_tc_kernel<true, false>;
    return gemm_tc_kernel<false, false>;
}

// The kernels' dynamic shared-memory limit is a per-device attribute.
bool smem_attribute(int dev, bool pair, bool wide) {
    static std::mutex mu;
    static bool done[64][2][2] = {};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return false;
    if (!done[dev][pair][wide]) {
        const cudaError_t e = cudaFuncSetAttribute(
            kernel_for(pair, wide), cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
        done[dev][pair][wide] = e == cudaSuccess;
    }
    return done[dev][pair][wide];
}

// Launch configuration: clusters of `cluster` CTAs (2 for the pair tile),
// and, for a real launch, programmatic stream serialization (see the kernel's
// griddepcontrol).  attr must hold two entries.
void launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, int cluster,
                   size_t smem, cudaStream_t stream, bool programmatic) {
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (programmatic) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(grid);
    cfg->blockDim = dim3(NUM_THREADS);
    cfg->dynamicSmemBytes = smem;
    cfg->stream = stream;
    cfg->attrs = attr;
    cfg->numAttrs = static_cast<unsigned>(n);
}

// Number of CTA pairs that can be resident at once for a given shared-memory
// size (cached per device and size).
int max_resident_pairs(int dev, size_t smem, bool wide) {
    static std::mutex mu;
    static size_t key_smem[64][2][8] = {};
    static int val[64][2][8] = {};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return 0;
    for (int i = 0; i < 8; ++i)
        if (key_smem[dev][wide][i] == smem && val[dev][wide][i] > 0) return val[dev][wide][i];
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    launch_config(&cfg, attr, 2, 2, smem, nullptr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel_for(true, wide), &cfg) !=
        cudaSuccess)
        n = 0;
    for (int i = 0; i < 8; ++i)
        if (key_smem[dev][wide][i] == 0 || i == 7) {
            key_smem[dev][wide][i] = smem;
            val[dev][wide][i] = n;
            break;
        }
    return n;
}

struct Geometry {
    int grid = 0;      // CTAs launched
    int cluster = 1;   // CTAs per cluster
    size_t smem = 0;   // dynamic shared memory per CTA
    int units = 0;     // persistent workers (CTAs, or CTA pairs)
    bool wide = false; // the 256 x 512 pair tile
    size_t ws_bytes = 0;  // stream-K workspace (partials + flags), 0 if unused
};

// Stream-K workspace layout: the flags first (one per unit and CTA rank),
// then one fp32 partial tile per unit and CTA.  The flags keep their place
// whatever the tile, so a workspace that a call with another tile reuses
// never has old partial data where this call's flags are.
constexpr size_t kWsFlagBytes = 4096;  // room for 1024 flags

// Stream-K workspaces, one per (device, stream): calls on one stream are
// ordered, so they never share a workspace concurrently.
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int workspace_for(int dev, cudaStream_t stream, size_t bytes, void** out) {
    std::lock_guard<std::mutex> g(g_ws_mu);
    Workspace& w = g_ws[{dev, stream}];
    if (w.bytes < bytes) {
        if (w.ptr) cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaMemset(w.ptr, 0, bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        w.bytes = bytes;
    }
    *out = w.ptr;
    return GEMM_OK;
}

// Parameters and launch geometry of one call (no launch).
int plan(const TcLaunch& L, TcParams& p, Geometry& geo) {
    const bool pair = L.pair != 0;
    const int bn = L.tile_n;
    const int S = L.stages;
    const int b_cols = pair ? bn / 2 : bn;
    const int tile_m = pair ? 2 * BM : BM;
    p.M = static_cast<int>(L.M);
    p.N = static_cast<int>(L.N);
    p.K = static_cast<int>(L.K);
    p.tiles_m = static_cast<int>((L.M + tile_m - 1) / tile_m);
    p.tiles_n = static_cast<int>((L.N + bn - 1) / bn);
    p.num_tiles = p.tiles_m * p.tiles_n;
    const bool wide = pair && bn == 512;
    geo.wide = wide;
    p.k_tiles = static_cast<int>((L.K + BK - 1) / BK);
    // Tile rows per raster group.  The tiles running at once should touch as
    // few A rows and B columns as possible, and a group's A panel should stay
    // in L2 while the group walks its columns.  On the 256 x 512 tile a round
    // of 76 pairs spans about 12 rows and 6 columns of tiles (measured: 4 %
    // fewer DRAM bytes than groups of 8, and level or slightly faster).  On
    // the 256 x 256 tile the group holds about 32 MB of A: 16 tile rows at
    // K = 4096 (+1.7 % in long runs on 8191 x 28672 x 4096 against 8), 8 at
    // K = 8192 (16 lost 2 % there).
    int pair_group = static_cast<int>((32ll << 20) / (2ll * tile_m * (L.K > 0 ? L.K : 1)));
    pair_group = pair_group < 8 ? 8 : (pair_group > 16 ? 16 : pair_group);
    p.group_m = pair ? (wide ? 12 : pair_group) : 16;
    p.stages = S;
    p.bn = bn;
    p.b_mn_major = L.b_col_major ? 0 : 1;
    p.b_chunked = 0;
    p.out_bf16 = L.out_bf16;
    // Instruction descriptor (kind::f16): D fp32 (bit 4), A and B type
    // (bits 7..9, 10..12: 0 fp16, 1 bf16), A K-major (bit 15 = 0), B major
    // (bit 16: 1 = MN-major), N >> 3 at bits 17..22, M >> 4 at bits 24..28
    // (M = 256 across a CTA pair; N = 256 per MMA on the 512-wide tile).
    const uint32_t fmt = L.in_bf16 ? 1u : 0u;
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(p.b_mn_major) << 16) |
              (static_cast<uint32_t>((bn > 256 ? 256 : bn) >> 3) << 17) |
              (static_cast<uint32_t>(tile_m >> 4) << 24);
    p.alpha = L.alpha;
    p.beta = L.beta;
    p.C = L.C;
    p.ldc = L.ldc;
    p.wait_limit_ns = static_cast<unsigned long long>(L.wait_limit_ns);
    p.withhold = L.withhold_arrive;
    p.clock_log = L.clock_log;
    p.dp_tiles = p.num_tiles;
    p.sk_iters = 0;
    p.ws = nullptr;
    p.ws_flag = nullptr;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    const int sms = device_sms(dev);
    if (sms <= 0) return GEMM_ERR_CUDA;
    if (!smem_attribute(dev, pair, wide)) return GEMM_ERR_LAUNCH;

    // The operand ring, then as many output boxes per epilogue warp (up to
    // kEpiMaxBufs) as the 227 KB of shared memory leave room for.
    const size_t base = 1024 + static_cast<size_t>(S) * (A_ATOM_BYTES + b_cols * BK * 2) +
                        sizeof(SharedCtl);
    const size_t max_smem = kTcMaxSmem;
    int nb = base < max_smem ? static_cast<int>((max_smem - base) / (4 * EPI_BOX_BYTES)) : 0;
    if (nb > kEpiMaxBufs) nb = kEpiMaxBufs;
    if (nb < 2) return GEMM_ERR_UNSUPPORTED;
    p.epi_bufs = nb;
    size_t smem = base + static_cast<size_t>(4 * nb) * EPI_BOX_BYTES;
    // One CTA per SM: a 256-wide tile uses all 512 TMEM columns, and a
    // stream-K finisher must never wait on a unit that is itself waiting for
    // TMEM held by another CTA of the same SM.
    if (smem < 120 * 1024) smem = 120 * 1024;
    geo.smem = smem;
    int max_units = sms;
    if (pair) {
        max_units = max_resident_pairs(dev, smem, wide);
        if (max_units <= 0) return GEMM_ERR_LAUNCH;
    }
    // Stream-K tail: when the last round of full tiles would leave units idle,
    // cut the leftover tiles into K segments over all units (each unit's share
    // is under one tile, so it touches at most two tiles).
    const int T = p.num_tiles, KT = p.k_tiles, U = max_units;
    const int rem = T % U;
    const int sk_tiles = T < U ? T : rem;
    // Automatic scheduling uses whole tiles: measured on GB300 the stream-K
    // fix-up (a second epilogue per unit that publishes, then reduces its
    // partial through the workspace) gains nothing over the idle tail it
    // removes under the power cap (8192^3: 1622-1624 vs 1628-1629 TFLOP/s in
    // 2000-step runs) and loses where every tile is split (2048^3).
    const bool use_sk = L.schedule == 2 && rem != 0 && static_cast<long long>(sk_tiles) * KT >= U;
    if (use_sk) {
        p.dp_tiles = T - sk_tiles;
        p.sk_iters = static_cast<long long>(sk_tiles) * KT;
        geo.units = U;
        const int cpu = pair ? 2 : 1;
        geo.ws_bytes = kWsFlagBytes + static_cast<size_t>(U) * cpu * BM * bn * sizeof(float);
    } else {
        geo.units = T < U ? T : U;
    }
    geo.cluster = pair ? 2 : 1;
    geo.grid = geo.cluster * geo.units;
    return GEMM_OK;
}

// Tensor maps of one call.  A: M x K row-major, boxes of 64 (K) x 128 (M).
// B column-major (N x K row-major): boxes of 64 (K) x b_cols (N).  B
// row-major: one 3-D box of b_cols/64 chunks per stage when N is a multiple
// of 64 and `chunked` is allowed, else boxes of 64 (N) x 64 (K), b_cols/64
// of them per stage.
bool encode_maps(const TcLaunch& L, bool chunked, CUtensorMap* tmA, CUtensorMap* tmB,
                 CUtensorMap* tmC, int* b_chunked) {
    // Columns per B box: the CTA's half of the tile, or a 128-column piece of
    // it on the 512-wide tile.
    const int b_cols = L.pair ? (L.tile_n >= 512 ? 128 : L.tile_n / 2) : L.tile_n;
    if (!encode_c(tmC, L.C, L.out_bf16, L.M, L.N, L.ldc)) return false;
    if (!encode_2d(tmA, L.A, L.in_bf16, L.M, L.K, L.lda, BK, BM)) return false;
    *b_chunked = (chunked && !L.b_col_major && L.N % 64 == 0) ? 1 : 0;
    if (L.b_col_major) return encode_2d(tmB, L.B, L.in_bf16, L.N, L.K, L.ldb, BK, b_cols);
    if (*b_chunked) return encode_b_chunked(tmB, L.B, L.in_bf16, L.K, L.N, L.ldb, b_cols / 64, BK);
    return encode_2d(tmB, L.B, L.in_bf16, L.K, L.N, L.ldb, 64, BK);
}

int launch_kernel(const Geometry& geo, bool pair, const CUtensorMap& tmA, const CUtensorMap& tmB,
                  const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    launch_config(&cfg, attr, geo.grid, geo.cluster, geo.smem, stream, true);
    if (cudaLaunchKernelEx(&cfg, kernel_for(pair, geo.wide), tmA, tmB, tmC, p) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace

int tc_launch(const TcLaunch& L, cudaStream_t stream) {
    const bool pair = L.pair != 0;
    TcParams p;
    Geometry geo;
    int st = plan(L, p, geo);
    if (st != GEMM_OK) return st;
    CUtensorMap tmA, tmB, tmC;
    if (!encode_maps(L, true, &tmA, &tmB, &tmC, &p.b_chunked)) return GEMM_ERR_LAUNCH;
    if (geo.ws_bytes) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
        void* ws = nullptr;
        st = workspace_for(dev, stream, geo.ws_bytes, &ws);
        if (st != GEMM_OK) return st;
        p.ws_flag = static_cast<unsigned int*>(ws);
        p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsFlagBytes);
    }
    return launch_kernel(geo, pair, tmA, tmB, tmC, p, stream);
}

// ---------------------------------------------------------------- allocation-free variant
// The stream-K workspace of gemm_noalloc: a fixed array in the library's own
// device memory, so that launching needs no cudaMalloc.  Every GPU that loads
// this module holds it until the process exits.  In host code the name is a
// stand-in for the device array: the kernel receives the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Device address of g_noalloc_scratch on `dev` (which must be current),
// looked up once per device.
int noalloc_scratch_address(int dev, void** out) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    if (addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return GEMM_ERR_CUDA;
        addr[dev] = ptr;
    }
    *out = addr[dev];
    return GEMM_OK;
}
}  // namespace

int tc_launch_noalloc(const TcLaunch& L, cudaStream_t stream) {
    const bool pair = L.pair != 0;
    TcParams p;
    Geometry geo;
    int st = plan(L, p, geo);
    if (st != GEMM_OK) return st;
    CUtensorMap tmA, tmB, tmC;
    if (!encode_maps(L, false, &tmA, &tmB, &tmC, &p.b_chunked)) return GEMM_ERR_LAUNCH;
    if (geo.ws_bytes) {
        if (geo.ws_bytes > kNoAllocScratchBytes) return GEMM_ERR_SCRATCH;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
        void* ws = nullptr;
        st = noalloc_scratch_address(dev, &ws);
        if (st != GEMM_OK) return st;
        // The array keeps the previous call's contents: the flags must start at 0.
        if (cudaMemsetAsync(ws, 0, kWsFlagBytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        p.ws_flag = static_cast<unsigned int*>(ws);
        p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsFlagBytes);
    }
    return launch_kernel(geo, pair, tmA, tmB, tmC, p, stream);
}

int tc_current_device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return device_sms(dev);
}

int tc_plan(const TcLaunch& L, int* grid, int* cluster, int* smem_bytes) {
    TcParams p;
    Geometry geo;
    const int st = plan(L, p, geo);
    if (st != GEMM_OK) return st;
    if (grid) *grid = geo.grid;
    if (cluster) *cluster = geo.cluster;
    if (smem_bytes) *smem_bytes = static_cast<int>(geo.smem);
    return GEMM_OK;
}

// Free the stream-K workspaces of the current device (the caller makes sure
// no launch that uses them is still running).
int tc_release_workspaces() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_ws_mu);
    for (auto it = g_ws.begin(); it != g_ws.end();) {
        if (it->first.first == dev) {
            if (it->second.ptr) cudaFree(it->second.ptr);
            it = g_ws.erase(it);
        } else {
            ++it;
        }
    }
    return GEMM_OK;
}

// After a run that gave up, a finisher may have left contributors' flags
// set: clear the flags of every workspace of the current device.
int tc_clear_workspace_flags() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_ws_mu);
    for (auto& kv : g_ws)
        if (kv.first.first == dev && kv.second.ptr)
            if (cudaMemset(kv.second.ptr, 0, kv.second.bytes) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}

int tc_read_and_clear_status(GemmDeviceStatus* out) {
    GemmDeviceStatus zero = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(GemmDeviceStatus)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(GemmDeviceStatus)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

}  // namespace ssp
