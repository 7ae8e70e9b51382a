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
//   * the consumer is ONE thread issuing tcgen05.mma (128 x BN x 16 per
//     instruction) that reads both operands straight from shared memory and
//     accumulates in TMEM, so there is no shared->register stage at all;
//   * the release is tcgen05.commit, which arrives on the stage's "empty"
//     barrier once the MMAs reading it have finished;
//   * the CTA is persistent and keeps two accumulators in TMEM, so the
//     epilogue of one output tile overlaps the mainloop of the next.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and
// TMEM owner, warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4)...).
//
// Ring protocol (slot s = i mod S, n = i div S for the i-th K tile a CTA
// handles): the producer waits empty[s] for parity (n&1)^1, arms full[s] with
// the stage's byte count and issues the copies; the MMA thread waits full[s]
// for parity n&1, issues BK/16 MMAs and commits to empty[s].  With S = 1 the
// producer's next copy waits for the MMAs of the same slot: the page's single
// buffer with a load phase and a compute phase.
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
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {

__device__ GemmDeviceStatus g_gemm_status;

namespace {

constexpr int BM = 128;                 // tile rows = TMEM lanes = UMMA M
constexpr int BK = 64;                  // 64 x 2 bytes = one 128-byte swizzle row
constexpr int UMMA_K = 16;              // K per tcgen05.mma (kind::f16)
constexpr int NUM_THREADS = 192;
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;     // one 64 x 64 box, 8 KB
constexpr int ROLE_PRODUCER = 0, ROLE_MMA = 1, ROLE_EPILOGUE = 2;

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, k_tiles;
    int group_m;
    int stages;
    int bn;
    int b_mn_major;
    int out_bf16;
    uint32_t idesc;
    float alpha, beta;
    void* C;
    long long ldc;
    unsigned long long wait_limit_ns;
    int withhold;
};

struct SharedCtl {
    unsigned long long bar[2 * kTcMaxStages128 + 5];  // full[S], empty[S], tfull[2], tempty[2], drain
    uint32_t tmem_base;
    int abort;
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

// Wait for the phase of `bar` with parity `parity`; give up after
// limit_ns or when another role has raised the abort flag.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                             unsigned long long limit_ns, int role, int iter) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                record_timeout(role, iter);
                *abort = 1;
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
// and B columns in L2.
__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& tm, int& tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

__device__ __forceinline__ void store_row_chunk(const TcParams& p, int row, int col0,
                                                const uint32_t (&r)[16]) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = p.alpha * __uint_as_float(r[i]);
    const bool full = col0 + 16 <= p.N;
    if (p.out_bf16) {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(p.C) + static_cast<long long>(row) * p.ldc + col0;
        if (p.beta != 0.0f) {
            if (full) {
                uint4 u[2];
                u[0] = *reinterpret_cast<const uint4*>(c);
                u[1] = *reinterpret_cast<const uint4*>(c + 8);
                const __nv_bfloat16* cb = reinterpret_cast<const __nv_bfloat16*>(u);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = fmaf(p.beta, __bfloat162float(cb[i]), v[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (col0 + i < p.N) v[i] = fmaf(p.beta, __bfloat162float(c[i]), v[i]);
            }
        }
        if (full) {
            uint4 u[2];
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(u);
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            *reinterpret_cast<uint4*>(c) = u[0];
            *reinterpret_cast<uint4*>(c + 8) = u[1];
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (col0 + i < p.N) c[i] = __float2bfloat16_rn(v[i]);
        }
    } else {
        float* c = static_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc + col0;
        if (p.beta != 0.0f) {
            if (full) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 o = *reinterpret_cast<const float4*>(c + 4 * q);
                    v[4 * q + 0] = fmaf(p.beta, o.x, v[4 * q + 0]);
                    v[4 * q + 1] = fmaf(p.beta, o.y, v[4 * q + 1]);
                    v[4 * q + 2] = fmaf(p.beta, o.z, v[4 * q + 2]);
                    v[4 * q + 3] = fmaf(p.beta, o.w, v[4 * q + 3]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (col0 + i < p.N) v[i] = fmaf(p.beta, c[i], v[i]);
            }
        }
        if (full) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4*>(c + 4 * q) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (col0 + i < p.N) c[i] = v[i];
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Swizzled TMA destinations and UMMA operands want 1024-byte alignment.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const int b_stage_bytes = p.bn * BK * 2;
    uint8_t* a_ring = smem;
    uint8_t* b_ring = smem + S * A_STAGE_BYTES;
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(b_ring + S * b_stage_bytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_addr(&ctl->bar[0]);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    volatile int* abort_flag = &ctl->abort;
    const uint32_t tmem_cols = 2u * p.bn;  // two accumulators: 256 or 512 columns

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4 * 32);
        }
        mbar_init(drain_bar, 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            const uint32_t stage_bytes = A_STAGE_BYTES + b_stage_bytes;
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
                int tm, tn;
                tile_coords(p, t, tm, tn);
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!bounded_wait(empty_bar(s), ph ^ 1u, abort_flag, p.wait_limit_ns,
                                      ROLE_PRODUCER, it)) {
                        ok = false;
                        break;
                    }
                    if (!(it == p.withhold && blockIdx.x == 0)) {
                        const uint32_t a_dst = smem_addr(a_ring + s * A_STAGE_BYTES);
                        const uint32_t b_dst = smem_addr(b_ring + s * b_stage_bytes);
                        mbar_arrive_expect_tx(full_bar(s), stage_bytes);
                        tma_load_2d(a_dst, &tmA, full_bar(s), kt * BK, tm * BM);
                        if (p.b_mn_major) {
                            for (int j = 0; j < p.bn / 64; ++j)
                                tma_load_2d(b_dst + j * B_BOX_BYTES, &tmB, full_bar(s),
                                            tn * p.bn + 64 * j, kt * BK);
                        } else {
                            tma_load_2d(b_dst, &tmB, full_bar(s), kt * BK, tn * p.bn);
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
                // Let every copy this thread issued land before the CTA exits.
                const int first = it - S > 0 ? it - S : 0;
                for (int j = first; j < it; ++j) {
                    if (j == p.withhold && blockIdx.x == 0) continue;
                    drain_wait(full_bar(j % S), static_cast<uint32_t>((j / S) & 1), p.wait_limit_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a_base = smem_addr(a_ring);
            const uint32_t b_base = smem_addr(b_ring);
            // K-major operands: 128-byte rows, 8-row groups 1024 bytes apart; one
            // K=16 step is 32 bytes along the row.  MN-major B: 64-column boxes
            // 8 KB apart (leading offset), 8-row K groups 1024 bytes apart; one
            // K=16 step is 16 rows = 2048 bytes.
            const uint32_t b_lbo = p.b_mn_major ? B_BOX_BYTES : 16u;
            const uint32_t b_kstep = p.b_mn_major ? 2048u : 32u;
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            int lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++lt) {
                const int acc = lt & 1;
                const uint32_t acc_ph = static_cast<uint32_t>((lt >> 1) & 1);
                if (!bounded_wait(tempty_bar(acc), acc_ph ^ 1u, abort_flag, p.wait_limit_ns,
                                  ROLE_MMA, it)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.bn);
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!bounded_wait(full_bar(s), ph, abort_flag, p.wait_limit_ns, ROLE_MMA, it)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = a_base + s * A_STAGE_BYTES;
                    const uint32_t b_s = b_base + s * b_stage_bytes;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t ad = smem_desc(a_s + kk * 32u, 16u, 1024u);
                        const uint64_t bd = smem_desc(b_s + kk * b_kstep, b_lbo, 1024u);
                        umma_f16(d_tmem, ad, bd, p.idesc, (kt | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty_bar(s));  // slot s is free once these MMAs finish
                    ++it;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull_bar(acc));  // accumulator ready for the epilogue
            }
            if (!ok) {
                // Wait for every MMA this thread issued before TMEM is freed.
                umma_commit(drain_bar);
                drain_wait(drain_bar, 0u, p.wait_limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_in_tile = 32 * q + lane;
        int lt = 0;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++lt) {
            const int acc = lt & 1;
            const uint32_t acc_ph = static_cast<uint32_t>((lt >> 1) & 1);
            if (!bounded_wait(tfull_bar(acc), acc_ph, abort_flag, p.wait_limit_ns, ROLE_EPILOGUE,
                              lt))
                break;
            tc_fence_after();
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int row = tm * BM + row_in_tile;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(acc * p.bn);
            for (int c = 0; c < p.bn; c += 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(t_row + static_cast<uint32_t>(c), r);
                tmem_ld_wait();
                const int col0 = tn * p.bn + c;
                if (row < p.M && col0 < p.N) store_row_chunk(p, row, col0, r);
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
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

// The kernel's dynamic shared-memory limit is a per-device attribute.
bool smem_attribute_set(int dev) {
    static std::mutex mu;
    static bool done[64] = {false};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return false;
    if (!done[dev])
        done[dev] = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024) == cudaSuccess;
    return done[dev];
}

int device_sms(int dev) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return cache[dev];
}

}  // namespace

int tc_launch(const TcLaunch& L, cudaStream_t stream) {
    const int bn = L.tile_n;
    const int S = L.stages;
    CUtensorMap tmA, tmB;
    // A: M x K row-major, boxes of 64 (K) x 128 (M).
    if (!encode_2d(&tmA, L.A, L.in_bf16, L.M, L.K, L.lda, BK, BM)) return GEMM_ERR_LAUNCH;
    if (L.b_col_major) {
        // B column-major = N x K row-major: boxes of 64 (K) x bn (N).
        if (!encode_2d(&tmB, L.B, L.in_bf16, L.N, L.K, L.ldb, BK, bn)) return GEMM_ERR_LAUNCH;
    } else {
        // B row-major K x N: boxes of 64 (N) x 64 (K); bn/64 boxes per stage.
        if (!encode_2d(&tmB, L.B, L.in_bf16, L.K, L.N, L.ldb, 64, BK)) return GEMM_ERR_LAUNCH;
    }

    TcParams p;
    p.M = static_cast<int>(L.M);
    p.N = static_cast<int>(L.N);
    p.K = static_cast<int>(L.K);
    p.tiles_m = static_cast<int>((L.M + BM - 1) / BM);
    p.tiles_n = static_cast<int>((L.N + bn - 1) / bn);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.k_tiles = static_cast<int>((L.K + BK - 1) / BK);
    p.group_m = 16;
    p.stages = S;
    p.bn = bn;
    p.b_mn_major = L.b_col_major ? 0 : 1;
    p.out_bf16 = L.out_bf16;
    // Instruction descriptor (kind::f16): D fp32 (bit 4), A and B type
    // (bits 7..9, 10..12: 0 fp16, 1 bf16), A K-major (bit 15 = 0), B major
    // (bit 16: 1 = MN-major), N >> 3 at bits 17..22, M >> 4 at bits 24..28.
    const uint32_t fmt = L.in_bf16 ? 1u : 0u;
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(p.b_mn_major) << 16) |
              (static_cast<uint32_t>(bn >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
    p.alpha = L.alpha;
    p.beta = L.beta;
    p.C = L.C;
    p.ldc = L.ldc;
    p.wait_limit_ns = static_cast<unsigned long long>(L.wait_limit_ns);
    p.withhold = L.withhold_arrive;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    const int sms = device_sms(dev);
    if (sms <= 0) return GEMM_ERR_CUDA;

    size_t smem = 1024 + static_cast<size_t>(S) * (A_STAGE_BYTES + bn * BK * 2) + sizeof(SharedCtl);
    // A 256-wide tile uses all 512 TMEM columns: keep one CTA per SM.
    if (bn == 256 && smem < 120 * 1024) smem = 120 * 1024;
    if (!smem_attribute_set(dev)) return GEMM_ERR_LAUNCH;

    const int grid = p.num_tiles < sms ? p.num_tiles : sms;
    gemm_tc_kernel<<<grid, NUM_THREADS, smem, stream>>>(tmA, tmB, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
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
