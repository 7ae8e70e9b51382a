// pipelined_copy.cu -- a streaming copy through an S-slot shared-memory ring.
//
// The bandwidth-bound counter-example to the GEMM.  The pages state when an
// asynchronous multi-stage ring pays: when a load's latency can hide behind
// arithmetic on data already staged ("Software Pipelining and Double
// Buffering", section "When it pays"; the CUDA Handbook, closing rule of
// "Asynchronous data movement"; the copy example that follows "Overlap needs
// stages" on "learn-kernels.com, Matrix multiplication").  A copy has no
// arithmetic: moving the bytes is the whole job, so once enough bytes are in
// flight to cover the memory latency, more stages cannot make it faster.
// The stage sweep of this kernel measures that claim on GB300 against the HBM
// copy bandwidth.
//
// Form (the GEMM's own ring, without the MMA): each CTA walks 8 KB chunks of
// the buffer, grid-stride.  One thread is the producer: it waits until slot
// s = i mod S is empty, arms the slot's "full" mbarrier with the chunk's byte
// count and issues one untiled bulk copy (TMA) global -> shared.  A second
// thread is the storer: it waits on "full", issues one bulk copy shared ->
// global, and releases a slot to the producer once the store that used it has
// read it (with S = 1 at once, the single buffer: load, store, load ...;
// with S >= 2 one store behind, so that a store and up to S - 1 loads are in
// flight at once).  The grid is one full wave at the occupancy the ring's
// shared memory allows, so a deeper ring means fewer CTAs per SM: the bytes in
// flight per SM stay about the same, which is the page's point -- depth and
// parallelism are two ways of covering the same latency.
//
// Every mbarrier wait is bounded (2 s on %globaltimer).  A wait that runs out
// sets g_copy_timeout and a shared abort flag; the producer then waits
// (bounded) for the loads it issued, the storer for its stores, and the CTA
// returns.  dst is then incomplete.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {

// Set to 1 by a copy-ring wait that ran out.
__device__ int g_copy_timeout;

namespace {

constexpr int COPY_THREADS = 64;      // warp 0 lane 0: producer; warp 1 lane 0: storer
constexpr int COPY_SLOT = 8192;       // bytes per ring slot (one chunk)
constexpr unsigned long long kCopyWaitLimitNs = 2000000000ull;

// Bytes of chunk c (the last one may be short; always a multiple of 16).
__device__ __forceinline__ uint32_t chunk_bytes(long long n, long long c) {
    const long long left = n - c * COPY_SLOT;
    return static_cast<uint32_t>(left < COPY_SLOT ? left : COPY_SLOT);
}

__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kCopyWaitLimitNs) {
                atomicExch(&g_copy_timeout, 1);
                *abort = 1;
                return false;
            }
        }
    }
}

template <int S>
__global__ void __launch_bounds__(COPY_THREADS)
    pipelined_copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, long long n) {
    extern __shared__ __align__(128) uint8_t ring[];  // S slots, then 2S mbarriers, then a flag
    unsigned long long* bars = reinterpret_cast<unsigned long long*>(ring + S * COPY_SLOT);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * S);
    const uint32_t slot0 = smem_addr(ring);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = full0 + 8u * S;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const long long chunks = (n + COPY_SLOT - 1) / COPY_SLOT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        long long i = 0;  // chunks issued by this CTA
        for (long long c = blockIdx.x; c < chunks; c += gridDim.x, ++i) {
            const int s = static_cast<int>(i % S);
            if (!ring_wait(empty0 + 8u * s, static_cast<uint32_t>((i / S) & 1) ^ 1u, abort)) break;
            const uint32_t bytes = chunk_bytes(n, c);
            mbar_arrive_expect_tx(full0 + 8u * s, bytes);
            bulk_load(slot0 + s * COPY_SLOT, src + c * COPY_SLOT, bytes, full0 + 8u * s);
        }
        if (*abort) {
            // The loads of the last S chunks issued land before the CTA exits
            // (a consumed one's phase has already completed).
            for (long long j = i - S > 0 ? i - S : 0; j < i; ++j) {
                const uint32_t bar = full0 + 8u * static_cast<uint32_t>(j % S);
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_try_wait(bar, static_cast<uint32_t>((j / S) & 1)) &&
                       globaltimer_ns() - t0 < kCopyWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        long long i = 0;  // chunks stored by this CTA
        for (long long c = blockIdx.x; c < chunks; c += gridDim.x, ++i) {
            const int s = static_cast<int>(i % S);
            if (!ring_wait(full0 + 8u * s, static_cast<uint32_t>((i / S) & 1), abort)) break;
            const uint32_t bytes = chunk_bytes(n, c);
            bulk_store(dst + c * COPY_SLOT, slot0 + s * COPY_SLOT, bytes);
            bulk_commit_group();
            if constexpr (S == 1) {
                bulk_wait_group_read<0>();  // this store has read the only slot
                mbar_arrive(empty0);
            } else {
                bulk_wait_group_read<1>();  // the previous store has read its slot
                if (i > 0) mbar_arrive(empty0 + 8u * static_cast<uint32_t>((i - 1) % S));
            }
        }
        bulk_wait_group_all();  // every store has landed in global memory
    }
    __syncthreads();
}

size_t ring_bytes(int S) { return static_cast<size_t>(S) * COPY_SLOT + 16u * S + 16u; }

template <int S>
int launch(uint8_t* dst, const uint8_t* src, long long n, cudaStream_t stream) {
    static std::mutex mu;
    static int blocks_per_sm[64] = {0};
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    const size_t smem = ring_bytes(S);
    {
        std::lock_guard<std::mutex> g(mu);
        if (blocks_per_sm[dev] == 0) {
            if (smem > 48 * 1024 &&
                cudaFuncSetAttribute(pipelined_copy_kernel<S>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &blocks_per_sm[dev], pipelined_copy_kernel<S>, COPY_THREADS, smem) !=
                    cudaSuccess ||
                blocks_per_sm[dev] <= 0) {
                blocks_per_sm[dev] = 0;
                return GEMM_ERR_CUDA;
            }
        }
    }
    // One full wave of resident CTAs, each walking the chunks grid-stride.
    long long grid = static_cast<long long>(sms[dev]) * blocks_per_sm[dev];
    const long long chunks = (n + COPY_SLOT - 1) / COPY_SLOT;
    if (grid > chunks) grid = chunks;
    pipelined_copy_kernel<S><<<static_cast<unsigned>(grid), COPY_THREADS, smem, stream>>>(dst, src, n);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace

int copy_launch(void* dst, const void* src, int64_t n_bytes, int stages, cudaStream_t stream) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    switch (stages) {
        case 1: return launch<1>(d, s, n_bytes, stream);
        case 2: return launch<2>(d, s, n_bytes, stream);
        case 3: return launch<3>(d, s, n_bytes, stream);
        case 4: return launch<4>(d, s, n_bytes, stream);
        case 5: return launch<5>(d, s, n_bytes, stream);
        case 6: return launch<6>(d, s, n_bytes, stream);
        case 7: return launch<7>(d, s, n_bytes, stream);
        case 8: return launch<8>(d, s, n_bytes, stream);
        default: return GEMM_ERR_ARG;
    }
}

}  // namespace ssp
