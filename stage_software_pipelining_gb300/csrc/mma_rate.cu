// mma_rate.cu -- the tensor pipe's own rate, measured in SM clocks.
//
// The GEMM's roofline has a compute bound of (SMs x dense bf16 FLOP per SM
// per clock x clock).  This kernel measures the middle factor on the GPU it
// runs on, with no memory traffic: every CTA (one per SM) fills its operand
// tiles in shared memory once, then one thread issues n back-to-back
// tcgen05.mma (cta_group::1, kind::f16, bf16 operands, fp32 accumulate into
// TMEM, M = 128, N = 256, K = 16) and reads the SM clock before the first
// issue and after the commit of the last MMA has arrived on its mbarrier.
// FLOP per clock per SM = n * 2*128*256*16 / cycles, independent of the
// clock the GPU happened to run at.
//
// The pair form measures the instruction the CTA-pair tiles issue: a cluster
// of two CTAs, TMEM allocated across the pair, and the leader issuing
// tcgen05.mma.cta_group::2 with M = 256 and N = 256, each CTA supplying 128
// rows of A and 128 columns of B.  Per SM that is the same 2*128*256*16 FLOP
// per instruction.
#include <cuda_runtime.h>

#include <vector>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {
namespace {

constexpr int kRateThreads = 128;
constexpr int kRateM = 128;
constexpr int kRateN = 256;
constexpr int kRateAtomRowBytes = 128;                       // one 64-deep bf16 K atom per row
constexpr int kRateABytes = kRateM * kRateAtomRowBytes;      // 16 KB
constexpr int kRateBBytes = kRateN * kRateAtomRowBytes;      // 32 KB
// The operands need 1 KB + 48 KB; asking for 120 KB keeps one CTA per SM, so
// that each CTA has its SM's tensor pipe to itself and the two CTAs of a
// pair sit on two SMs, as cta_group::2 requires.
constexpr int kRateSmem = 120 * 1024;
static_assert(kRateSmem >= 1024 + kRateABytes + kRateBBytes, "operands must fit");
constexpr unsigned long long kRateWaitNs = 2000000000ull;

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: rows
// of 128 bytes, 8-row groups 1024 bytes apart (stride offset), version 1
// (bit 46), layout type 2 (bits 61..63).
__device__ __forceinline__ uint64_t rate_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1u) << 16) |
           (static_cast<uint64_t>(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

template <bool PAIR>
__global__ void __launch_bounds__(kRateThreads, 1)
    mma_rate_kernel(int n_mma, long long* __restrict__ cycles, int* __restrict__ timed_out) {
    extern __shared__ uint8_t rate_smem[];
    __shared__ uint64_t done_bar;
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = smem_addr(rate_smem);
    const uint32_t a_addr = (raw + 1023u) & ~1023u;  // the swizzle atoms want 1024-byte alignment
    const uint32_t b_addr = a_addr + kRateABytes;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = PAIR ? (cluster_ctarank() & 1u) : 0u;

    // Operands: every bf16 element 1.0 (0x3F80); the rate does not depend on
    // the values.  Written by the generic proxy, read by the tensor core
    // through the async proxy: fence between the two.
    const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    for (int i = threadIdx.x; i < (kRateABytes + kRateBBytes) / 16; i += kRateThreads)
        st_shared_v4(a_addr + 16u * static_cast<uint32_t>(i), ones);
    fence_proxy_async_shared();
    if (warp == 0) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_addr(&tmem_slot), kRateN);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(&tmem_slot), kRateN);
            tmem_relinquish();
        }
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&done_bar), 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // the peer's operands and barrier are ready
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0) {
        long long t0 = 0;
        if (rank == 0) {
            // D fp32 (bit 4), A and B bf16 (bits 7..9, 10..12), both K-major,
            // N >> 3 at bits 17..22, M >> 4 at bits 24..28 (256 across a pair).
            constexpr int M = PAIR ? 2 * kRateM : kRateM;
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                   (static_cast<uint32_t>(kRateN >> 3) << 17) |
                                   (static_cast<uint32_t>(M >> 4) << 24);
            const uint64_t a0 = rate_desc(a_addr), b0 = rate_desc(b_addr);
            t0 = clock64();
            for (int i = 0; i < n_mma; ++i) {
                // Walk the four K = 16 slices of the atom (32 bytes = 2 units each).
                const uint64_t k = static_cast<uint64_t>(i & 3) * 2u;
                if constexpr (PAIR) umma_f16_pair(tmem, a0 + k, b0 + k, idesc, i > 0 ? 1u : 0u);
                else umma_f16(tmem, a0 + k, b0 + k, idesc, i > 0 ? 1u : 0u);
            }
            if constexpr (PAIR) umma_commit_pair_multicast(smem_addr(&done_bar), 0x3);
            else umma_commit(smem_addr(&done_bar));
        }
        const unsigned long long w0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(smem_addr(&done_bar), 0u)) {
            if (globaltimer_ns() - w0 > kRateWaitNs) {
                ok = false;
                break;
            }
        }
        const long long t1 = clock64();
        cycles[blockIdx.x] = !ok ? -1 : rank == 0 ? t1 - t0 : 0;  // a pair's peer only waits
        if (!ok) atomicExch(timed_out, 1);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // neither CTA frees TMEM while the pair still uses it
    tc_fence_after();
    if (warp == 0) {
        if constexpr (PAIR) tmem_dealloc_pair(tmem, kRateN);
        else tmem_dealloc(tmem, kRateN);
    }
}

}  // namespace
}  // namespace ssp

extern "C" int mma_rate(int n_mma, int ctas, long long* cycles, float* elapsed_ms) {
    if (n_mma < 1 || n_mma > (1 << 20) || ctas < 1 || !cycles || !elapsed_ms) return GEMM_ERR_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (ctas > sms) return GEMM_ERR_ARG;
    if (cudaFuncSetAttribute(ssp::mma_rate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ssp::kRateSmem) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    long long* d_cycles = nullptr;
    int* d_flag = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int st = GEMM_OK;
    if (cudaMalloc(&d_cycles, sizeof(long long) * ctas) != cudaSuccess ||
        cudaMalloc(&d_flag, sizeof(int)) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
        cudaEventCreate(&e1) != cudaSuccess || cudaMemset(d_flag, 0, sizeof(int)) != cudaSuccess) {
        st = GEMM_ERR_CUDA;
    } else {
        cudaEventRecord(e0, nullptr);
        ssp::mma_rate_kernel<false><<<ctas, ssp::kRateThreads, ssp::kRateSmem>>>(n_mma, d_cycles, d_flag);
        if (cudaGetLastError() != cudaSuccess) st = GEMM_ERR_LAUNCH;
        cudaEventRecord(e1, nullptr);
        int flag = 0;
        if (st == GEMM_OK &&
            (cudaEventSynchronize(e1) != cudaSuccess ||
             cudaEventElapsedTime(elapsed_ms, e0, e1) != cudaSuccess ||
             cudaMemcpy(cycles, d_cycles, sizeof(long long) * ctas, cudaMemcpyDeviceToHost) !=
                 cudaSuccess ||
             cudaMemcpy(&flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess))
            st = GEMM_ERR_CUDA;
        if (st == GEMM_OK && flag) st = GEMM_ERR_TIMEOUT;
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (d_cycles) cudaFree(d_cycles);
    if (d_flag) cudaFree(d_flag);
    return st;
}

extern "C" int mma_rate_pair(int n_mma, int pairs, long long* cycles, float* elapsed_ms) {
    if (n_mma < 1 || n_mma > (1 << 20) || pairs < 1 || !cycles || !elapsed_ms) return GEMM_ERR_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (2 * pairs > sms) return GEMM_ERR_ARG;
    if (cudaFuncSetAttribute(ssp::mma_rate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ssp::kRateSmem) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    const int ctas = 2 * pairs;
    long long* d_cycles = nullptr;
    int* d_flag = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int st = GEMM_OK;
    std::vector<long long> h(ctas);
    if (cudaMalloc(&d_cycles, sizeof(long long) * ctas) != cudaSuccess ||
        cudaMalloc(&d_flag, sizeof(int)) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
        cudaEventCreate(&e1) != cudaSuccess || cudaMemset(d_flag, 0, sizeof(int)) != cudaSuccess) {
        st = GEMM_ERR_CUDA;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(ctas));
        cfg.blockDim = dim3(ssp::kRateThreads);
        cfg.dynamicSmemBytes = ssp::kRateSmem;
        cfg.stream = nullptr;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaEventRecord(e0, nullptr);
        if (cudaLaunchKernelEx(&cfg, ssp::mma_rate_kernel<true>, n_mma, d_cycles, d_flag) !=
            cudaSuccess)
            st = GEMM_ERR_LAUNCH;
        cudaEventRecord(e1, nullptr);
        int flag = 0;
        if (st == GEMM_OK &&
            (cudaEventSynchronize(e1) != cudaSuccess ||
             cudaEventElapsedTime(elapsed_ms, e0, e1) != cudaSuccess ||
             cudaMemcpy(h.data(), d_cycles, sizeof(long long) * ctas, cudaMemcpyDeviceToHost) !=
                 cudaSuccess ||
             cudaMemcpy(&flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess))
            st = GEMM_ERR_CUDA;
        if (st == GEMM_OK && flag) st = GEMM_ERR_TIMEOUT;
        if (st == GEMM_OK)
            for (int i = 0; i < pairs; ++i) cycles[i] = h[2 * i];  // the leaders' clocks
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (d_cycles) cudaFree(d_cycles);
    if (d_flag) cudaFree(d_flag);
    return st;
}
