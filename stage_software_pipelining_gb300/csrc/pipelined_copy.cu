// pipelined_copy.cu -- a streaming copy through an N-stage shared-memory ring.
//
// The bandwidth-bound counter-example to the GEMM: the grid-stride copy of
// "learn-kernels.com, Matrix multiplication" (the `cuda::pipeline` listing
// after "Overlap needs stages"), where each thread stages its element of the
// next stage into shared memory with an asynchronous copy while it writes out
// the element of the current stage.  "Software Pipelining and Double
// Buffering", section "When it pays", and the CUDA Handbook's closing rule in
// "Asynchronous data movement" say that such a kernel gains nothing from the
// extra stages: streaming the data is the work, there is no arithmetic to
// hide the transfer behind.  The stage sweep of this kernel measures that
// claim on GB300 against the HBM copy bandwidth.
//
// GB300 form: 16-byte cp.async per thread per stage (the 16-byte LDGSTS form
// bypasses L1), a ring of S slots per thread, S stages committed before the
// loop and one committed per iteration (also when it copies nothing) so that
// "wait until at most S-1 groups are pending" always means "the oldest stage
// landed".  Each thread reads back only its own slot, so, as the page notes,
// no block barrier is needed.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {
namespace {

constexpr int COPY_THREADS = 256;

template <int S>
__global__ void __launch_bounds__(COPY_THREADS)
    pipelined_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, long long n16) {
    __shared__ uint4 ring[S][COPY_THREADS];
    const long long stride = static_cast<long long>(gridDim.x) * COPY_THREADS;
    const long long first = static_cast<long long>(blockIdx.x) * COPY_THREADS + threadIdx.x;
    const uint32_t slot0 = smem_addr(&ring[0][threadIdx.x]);
    constexpr uint32_t kSlotStride = COPY_THREADS * sizeof(uint4);

#pragma unroll
    for (int s = 0; s < S; ++s) {
        const long long idx = first + s * stride;
        const bool in = idx < n16;
        cp_async_16(slot0 + s * kSlotStride, in ? src + idx : src, in ? 16u : 0u);
        cp_async_commit();
    }
    int s = 0;
    for (long long i = first; i < n16; i += stride) {
        cp_async_wait<S - 1>();  // the oldest stage (element i) has landed
        dst[i] = ring[s][threadIdx.x];
        const long long nxt = i + S * stride;
        const bool in = nxt < n16;
        cp_async_16(slot0 + s * kSlotStride, in ? src + nxt : src, in ? 16u : 0u);
        cp_async_commit();
        s = (s + 1 == S) ? 0 : s + 1;
    }
    cp_async_wait<0>();
}

template <int S>
int launch(uint4* dst, const uint4* src, long long n16, cudaStream_t stream) {
    static std::mutex mu;
    static int blocks_per_sm[64] = {0};
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(mu);
        if (blocks_per_sm[dev] == 0) {
            if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &blocks_per_sm[dev], pipelined_copy_kernel<S>, COPY_THREADS, 0) != cudaSuccess ||
                blocks_per_sm[dev] <= 0) {
                blocks_per_sm[dev] = 0;
                return GEMM_ERR_CUDA;
            }
        }
    }
    // One full wave of resident blocks, each walking the array grid-stride.
    long long grid = static_cast<long long>(sms[dev]) * blocks_per_sm[dev];
    const long long needed = (n16 + COPY_THREADS - 1) / COPY_THREADS;
    if (grid > needed) grid = needed;
    pipelined_copy_kernel<S><<<static_cast<unsigned>(grid), COPY_THREADS, 0, stream>>>(dst, src, n16);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace

int copy_launch(void* dst, const void* src, int64_t n_bytes, int stages, cudaStream_t stream) {
    uint4* d = static_cast<uint4*>(dst);
    const uint4* s = static_cast<const uint4*>(src);
    const long long n16 = n_bytes / 16;
    switch (stages) {
        case 1: return launch<1>(d, s, n16, stream);
        case 2: return launch<2>(d, s, n16, stream);
        case 3: return launch<3>(d, s, n16, stream);
        case 4: return launch<4>(d, s, n16, stream);
        case 5: return launch<5>(d, s, n16, stream);
        case 6: return launch<6>(d, s, n16, stream);
        case 7: return launch<7>(d, s, n16, stream);
        case 8: return launch<8>(d, s, n16, stream);
        default: return GEMM_ERR_ARG;
    }
}

}  // namespace ssp
