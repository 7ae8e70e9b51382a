// sgemm_simt.cu -- FP32 CUDA-core GEMM with cp.async staging, 1..4 stages.
//
// The register-blocked sgemm the pages treat as the FP32 path: a 128 x 64
// block tile, 128 threads, each thread accumulating an 8 x 8 tile of C as the
// outer product of an 8 x 1 A fragment and a 1 x 8 B fragment per k
// ("CUTLASS-CuTe 初步(6)", section 4 "Thread Tile"; the CUDA Handbook's
// chapter 17 register-blocked 128 x 64 kernel).  Tiles go global -> shared with
// 16-byte cp.async (no register staging, "learn-kernels.com, Matrix
// multiplication", paragraph on LDGSTS), one commit group per stage.
//
// A stage is a K slice of 32 (18 KB of A with its row padding, 8 KB of B):
// 32 outer products per barrier.  Measured against slices of 16: +2.0 % at
// 2048^3 and +2.6 % at 4096^3 with 2 stages, the same bits; 3 CTAs per SM
// still fit up to 2 stages.
//
// stages = 1 is the single-buffer loop with two barriers per K tile (load,
// barrier, compute, barrier: "CUTLASS-CuTe 初步(6)" section 6.2, first loop).
// stages >= 2 keeps S-1 tiles in flight: at the top of each iteration it
// waits until at most S-2 groups are pending, then one barrier (which both
// publishes the landed tile and proves every thread is done with the slot
// about to be refilled), then issues the copy S-1 tiles ahead and computes --
// one barrier per iteration, as the pages' double-buffered loops have.
// Out-of-range rows/columns are zero-filled by cp.async's source-size operand,
// so ragged M, N and K need no special path; stores are masked.
//
// Tail schedule: the tiles form one wave per 3 CTAs per SM (the occupancy
// this kernel has at 1 and 2 stages; 3 and 4 stages fit 2).  The plan keeps
// 3 at every stage count so that it, and the bits, never depend on the
// stage count.  When the last wave is partial, its
// tiles are cut along K into `parts` equal ranges of K tiles, so that the
// short pieces fill the SMs the whole tiles leave idle (a problem of less
// than one wave is all split: at 256^3 its 8 tiles run as 32 pieces, 1.3x
// faster; 512^3 1.85x).  Each piece stores
// its fp32 partial tile in a workspace and counts itself in on the tile's
// counter; the piece that arrives last adds the partials of parts 0, 1, ...
// in that order (the same bits whichever piece is last), writes C and resets
// the counter.  Nothing waits on anything, so no piece can hold up another.
// The plan depends only on the shape and the SM count, so every stage count
// gives the same bits.
//
// GB300 form of the outer product: the 64 multiply-adds of a k step are 32
// packed fp32 FMAs (fma.rn.f32x2, sm_100 and later).  Each lane of one is an
// ordinary fused multiply-add rounded once to nearest, so C is bit-for-bit
// what 64 scalar fmaf would give; the packed form halves the issue slots the
// FMAs take, which is what limits a register-blocked sgemm.  A thread keeps
// its 8 x 8 accumulators as 8 x 4 pairs of adjacent columns, reads its B
// fragment from shared memory directly as such pairs, and duplicates each A
// value into both halves of a pair.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssp {
namespace {

constexpr int BM = 128, BN = 64, BK = 32;
constexpr int THREADS = 128;
constexpr int A_LD = BK + 4;  // padded row (144 bytes): conflict-free fragment reads
constexpr int A_STAGE_FLOATS = BM * A_LD;
constexpr int B_STAGE_FLOATS = BK * BN;

constexpr int kSimtCtasPerSm = 3;  // the wave the tail schedule plans for
constexpr int kSimtMaxParts = 8;
constexpr int kSimtMinPartKTiles = 2;  // a piece spans at least 64 of K
constexpr size_t kSimtCounterBytes = 4096;

struct SimtParams {
    int M, N, K;
    const float* A;
    long long lda;
    const float* B;
    long long ldb;
    float* C;
    long long ldc;
    float alpha, beta;
    int tiles_n;              // tiles along N
    int dp_tiles;             // tiles [0, dp_tiles) run whole, one CTA each
    int parts;                // K pieces of each later tile (1: none)
    float* ws;                // split tiles: one 128 x 64 fp32 partial per piece
    unsigned int* counters;   // split tiles: pieces arrived so far
    unsigned long long* clock_log;  // null, or [2]: CTA 0 adds its SM clocks and ns
};

// Copy K tile kt into stage buffers (As, Bs).  A tile: 128 rows x 32 floats =
// 1024 16-byte chunks; B tile: 32 rows x 64 floats = 512 chunks.
__device__ __forceinline__ void load_tile(const SimtParams& p, int m0, int n0, int kt, float* As,
                                          float* Bs) {
    const int tid = threadIdx.x;
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = tid + THREADS * i;
        const int row = c >> 3;
        const int kc = (c & 7) * 4;
        const int gm = m0 + row, gk = k0 + kc;
        int valid = 0;
        const float* src = p.A;
        if (gm < p.M && gk < p.K) {
            valid = min(p.K - gk, 4) * 4;
            src = p.A + static_cast<long long>(gm) * p.lda + gk;
        }
        cp_async_16(smem_addr(As + row * A_LD + kc), src, static_cast<uint32_t>(valid));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = tid + THREADS * i;
        const int row = c >> 4;
        const int nc = (c & 15) * 4;
        const int gk = k0 + row, gn = n0 + nc;
        int valid = 0;
        const float* src = p.B;
        if (gk < p.K && gn < p.N) {
            valid = min(p.N - gn, 4) * 4;
            src = p.B + static_cast<long long>(gk) * p.ldb + gn;
        }
        cp_async_16(smem_addr(Bs + row * BN + nc), src, static_cast<uint32_t>(valid));
    }
}

// Two fp32 in one 64-bit register: the low half is the even column.
using Pair = unsigned long long;

__device__ __forceinline__ Pair dup2(float x) {
    Pair r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
    return r;
}

// c.lo = fma(a.lo, b.lo, c.lo); c.hi = fma(a.hi, b.hi, c.hi), each rounded once.
__device__ __forceinline__ void ffma2(Pair& c, Pair a, Pair b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(a), "l"(b));
}

// Both halves added in fp32, each rounded once.
__device__ __forceinline__ Pair add2(Pair a, Pair b) {
    Pair r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float lo32(Pair v) { return __uint_as_float(static_cast<unsigned>(v)); }
__device__ __forceinline__ float hi32(Pair v) {
    return __uint_as_float(static_cast<unsigned>(v >> 32));
}

// acc[r][q] += A[ty + 16 r][k] * B[k][cols of pair q] over the BK values of one
// stage (pair q: columns 4tx+2q, +1 for q < 2, 32+4tx+2(q-2), +1 for q >= 2).
// Thread rows are ty, ty+16, ..., ty+112; thread columns are 4tx..4tx+3 and
// 32+4tx..32+4tx+3, so a warp's fragment reads hit distinct banks.
// One fragment set: the A fragments of 4 consecutive k (8 float4) and the B
// fragment of one k (2 float4) are loaded, then used.
__device__ __forceinline__ void compute_tile_single(const float* As, const float* Bs, int ty,
                                                    int tx, Pair (&acc)[8][4]) {
#pragma unroll
    for (int kq = 0; kq < BK; kq += 4) {
        float4 a4[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            a4[r] = *reinterpret_cast<const float4*>(As + (ty + 16 * r) * A_LD + kq);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(Bs + (kq + kk) * BN + 4 * tx);
            const ulonglong2 b1 =
                *reinterpret_cast<const ulonglong2*>(Bs + (kq + kk) * BN + 32 + 4 * tx);
            const Pair b[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float a = kk == 0 ? a4[r].x : kk == 1 ? a4[r].y : kk == 2 ? a4[r].z : a4[r].w;
                const Pair a2 = dup2(a);
#pragma unroll
                for (int q = 0; q < 4; ++q) ffma2(acc[r][q], a2, b[q]);
            }
        }
    }
}

// Two fragment sets in registers (the warp-scope double buffer of
// "CUTLASS-CuTe 初步(6)" section 6 and of "learn-kernels.com, Matrix
// multiplication"): while the outer products of step k run, the B fragment of
// step k+1 and, at the first step of each group of 4, the A fragments of the
// next group are already being fetched from shared memory.
__device__ __forceinline__ void compute_tile_double(const float* As, const float* Bs, int ty,
                                                    int tx, Pair (&acc)[8][4]) {
    float4 a4[2][8];
    ulonglong2 bf[2][2];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        a4[0][r] = *reinterpret_cast<const float4*>(As + (ty + 16 * r) * A_LD);
    bf[0][0] = *reinterpret_cast<const ulonglong2*>(Bs + 4 * tx);
    bf[0][1] = *reinterpret_cast<const ulonglong2*>(Bs + 32 + 4 * tx);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
        const int kq = k >> 2, kk = k & 3;
        if (kk == 0 && k + 4 < BK) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
                a4[(kq + 1) & 1][r] =
                    *reinterpret_cast<const float4*>(As + (ty + 16 * r) * A_LD + k + 4);
        }
        if (k + 1 < BK) {
            bf[(k + 1) & 1][0] = *reinterpret_cast<const ulonglong2*>(Bs + (k + 1) * BN + 4 * tx);
            bf[(k + 1) & 1][1] =
                *reinterpret_cast<const ulonglong2*>(Bs + (k + 1) * BN + 32 + 4 * tx);
        }
        const Pair b[4] = {bf[k & 1][0].x, bf[k & 1][0].y, bf[k & 1][1].x, bf[k & 1][1].y};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float4 av = a4[kq & 1][r];
            const float a = kk == 0 ? av.x : kk == 1 ? av.y : kk == 2 ? av.z : av.w;
            const Pair a2 = dup2(a);
#pragma unroll
            for (int q = 0; q < 4; ++q) ffma2(acc[r][q], a2, b[q]);
        }
    }
}

template <bool FRAG_DB>
__device__ __forceinline__ void compute_tile(const float* As, const float* Bs, int ty, int tx,
                                             Pair (&acc)[8][4]) {
    if constexpr (FRAG_DB) compute_tile_double(As, Bs, ty, tx, acc);
    else compute_tile_single(As, Bs, ty, tx, acc);
}

// C = alpha*acc + beta*C for this thread's 8 x 8 outputs, masked at the M and N edges.
__device__ __forceinline__ void simt_epilogue(const SimtParams& p, int m0, int n0, int ty, int tx,
                                              const Pair (&acc)[8][4]) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int gm = m0 + ty + 16 * r;
        if (gm >= p.M) continue;
        float* crow = p.C + static_cast<long long>(gm) * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + 32 * h + 4 * tx;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const Pair pr = acc[r][2 * h + (j >> 1)];
                v[j] = p.alpha * ((j & 1) ? hi32(pr) : lo32(pr));
            }
            if (gn + 4 <= p.N) {
                float4* cp = reinterpret_cast<float4*>(crow + gn);
                if (p.beta != 0.0f) {
                    const float4 o = *cp;
                    v[0] = fmaf(p.beta, o.x, v[0]);
                    v[1] = fmaf(p.beta, o.y, v[1]);
                    v[2] = fmaf(p.beta, o.z, v[2]);
                    v[3] = fmaf(p.beta, o.w, v[3]);
                }
                *cp = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (gn + j < p.N) {
                        float o = v[j];
                        if (p.beta != 0.0f) o = fmaf(p.beta, crow[gn + j], o);
                        crow[gn + j] = o;
                    }
                }
            }
        }
    }
}

template <int STAGES, bool FRAG_DB>
__global__ void __launch_bounds__(THREADS) sgemm_simt_kernel(const SimtParams p) {
    extern __shared__ __align__(16) float smem[];
    float* As = smem;                              // [STAGES][BM][A_LD]
    float* Bs = smem + STAGES * A_STAGE_FLOATS;    // [STAGES][BK][BN]
    __shared__ int last_piece;
    const int tid = threadIdx.x;
    const int ty = tid >> 3, tx = tid & 7;
    const int KT = (p.K + BK - 1) / BK;
    // Whole tile, or piece `part` of a split tile: K tiles [kt0, kt1).
    int tile = blockIdx.x, part = -1, kt0 = 0, kt1 = KT;
    if (tile >= p.dp_tiles) {
        const int u = tile - p.dp_tiles;
        part = u % p.parts;
        tile = p.dp_tiles + u / p.parts;
        kt0 = static_cast<int>(static_cast<long long>(part) * KT / p.parts);
        kt1 = static_cast<int>(static_cast<long long>(part + 1) * KT / p.parts);
    }
    const int m0 = (tile / p.tiles_n) * BM, n0 = (tile % p.tiles_n) * BN;
    const int NK = kt1 - kt0;
    // SM clock of this launch (measurement hook): CTA 0, from here to its exit.
    const bool log_clock = p.clock_log != nullptr && blockIdx.x == 0 && tid == 0;
    long long clk0 = 0;
    unsigned long long ns0 = 0;
    if (log_clock) {
        clk0 = clock64();
        ns0 = globaltimer_ns();
    }
    auto log_exit = [&]() {
        if (log_clock) {
            atomicAdd(p.clock_log, static_cast<unsigned long long>(clock64() - clk0));
            atomicAdd(p.clock_log + 1, globaltimer_ns() - ns0);
        }
    };

    Pair acc[8][4];  // acc[r][q]: columns 2q, 2q+1 of the thread's 8 (bits of +0.0f: zero)
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = 0ull;

    if constexpr (STAGES == 1) {
        for (int i = 0; i < NK; ++i) {
            load_tile(p, m0, n0, kt0 + i, As, Bs);
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();  // read after write: every thread's copies landed
            compute_tile<FRAG_DB>(As, Bs, ty, tx, acc);
            __syncthreads();  // write after read: nobody still reads the buffer
        }
    } else {
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s) {
            if (s < NK)
                load_tile(p, m0, n0, kt0 + s, As + s * A_STAGE_FLOATS, Bs + s * B_STAGE_FLOATS);
            cp_async_commit();  // always commit: a fixed number of groups stays in flight
        }
        for (int i = 0; i < NK; ++i) {
            cp_async_wait<STAGES - 2>();  // this thread's copies of tile i landed
            __syncthreads();              // ... everyone's, and slot (i-1) % S is free
            const int nk = i + STAGES - 1;
            if (nk < NK) {
                const int ns = nk % STAGES;
                load_tile(p, m0, n0, kt0 + nk, As + ns * A_STAGE_FLOATS, Bs + ns * B_STAGE_FLOATS);
            }
            cp_async_commit();
            const int cs = i % STAGES;
            compute_tile<FRAG_DB>(As + cs * A_STAGE_FLOATS, Bs + cs * B_STAGE_FLOATS, ty, tx, acc);
        }
        cp_async_wait<0>();
    }

    if (part < 0) {
        simt_epilogue(p, m0, n0, ty, tx, acc);
        log_exit();
        return;
    }
    // A piece of a split tile: publish the partial (thread-ordered, so that
    // each warp access is 512 contiguous bytes), count in, and let the last
    // piece to arrive finish the tile.
    const int split = tile - p.dp_tiles;
    ulonglong2* mine = reinterpret_cast<ulonglong2*>(
        p.ws + static_cast<size_t>(split * p.parts + part) * (BM * BN));
#pragma unroll
    for (int j = 0; j < 16; ++j)
        mine[j * THREADS + tid] = make_ulonglong2(acc[j >> 1][(j & 1) * 2], acc[j >> 1][(j & 1) * 2 + 1]);
    __threadfence();
    __syncthreads();
    if (tid == 0) last_piece = atomicAdd(p.counters + split, 1u) == static_cast<unsigned>(p.parts - 1);
    __syncthreads();
    if (!last_piece) {
        log_exit();
        return;
    }
    __threadfence();  // the other pieces' partials are visible after their count
    for (int q = 0; q < p.parts; ++q) {
        const ulonglong2* src = reinterpret_cast<const ulonglong2*>(
            p.ws + static_cast<size_t>(split * p.parts + q) * (BM * BN));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const ulonglong2 v = __ldcg(src + j * THREADS + tid);  // written by other SMs: read L2
            Pair& a0 = acc[j >> 1][(j & 1) * 2];
            Pair& a1 = acc[j >> 1][(j & 1) * 2 + 1];
            if (q == 0) {
                a0 = v.x;
                a1 = v.y;
            } else {
                a0 = add2(a0, v.x);
                a1 = add2(a1, v.y);
            }
        }
    }
    simt_epilogue(p, m0, n0, ty, tx, acc);
    if (tid == 0) p.counters[split] = 0u;  // ready for the next launch
    log_exit();
}

int simt_tiles(int M, int N) { return ((M + BM - 1) / BM) * ((N + BN - 1) / BN); }

template <int S, bool FRAG_DB>
int launch_stages(const SimtParams& p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(S) * (A_STAGE_FLOATS + B_STAGE_FLOATS) * sizeof(float);
    if (smem > 48 * 1024) {
        // A per-device attribute: set it once on each device used.
        static std::mutex mu;
        static bool done[64] = {false};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
        std::lock_guard<std::mutex> g(mu);
        if (!done[dev]) {
            if (cudaFuncSetAttribute(sgemm_simt_kernel<S, FRAG_DB>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return GEMM_ERR_LAUNCH;
            done[dev] = true;
        }
    }
    const int grid = p.dp_tiles + (simt_tiles(p.M, p.N) - p.dp_tiles) * p.parts;
    sgemm_simt_kernel<S, FRAG_DB><<<grid, THREADS, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// Split-tail workspaces, one per (device, stream): launches on one stream are
// ordered, so they never use a workspace at the same time.  Counters first
// (zeroed once; every finished tile resets its own), then the partials.
struct SimtWorkspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_simt_ws_mu;
std::map<std::pair<int, cudaStream_t>, SimtWorkspace> g_simt_ws;

int simt_workspace(int dev, cudaStream_t stream, size_t bytes, void** out) {
    std::lock_guard<std::mutex> g(g_simt_ws_mu);
    SimtWorkspace& w = g_simt_ws[{dev, stream}];
    if (w.bytes < bytes) {
        if (w.ptr) cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaMemset(w.ptr, 0, kSimtCounterBytes) != cudaSuccess) return GEMM_ERR_CUDA;
        w.bytes = bytes;
    }
    *out = w.ptr;
    return GEMM_OK;
}

__global__ void scale_kernel(long long M, long long N, void* C, long long ldc, int out_bf16,
                             float beta) {
    const long long total = M * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long i = idx / N, j = idx - i * N;
        if (out_bf16) {
            __nv_bfloat16* c = static_cast<__nv_bfloat16*>(C) + i * ldc + j;
            *c = beta == 0.0f ? __float2bfloat16_rn(0.0f) : __float2bfloat16_rn(beta * __bfloat162float(*c));
        } else {
            float* c = static_cast<float*>(C) + i * ldc + j;
            *c = beta == 0.0f ? 0.0f : beta * *c;
        }
    }
}

}  // namespace

SimtPlan simt_plan(int64_t M, int64_t N, int64_t K, int sms) {
    SimtPlan pl;
    const long long T64 = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (T64 * kSimtMaxParts > 0x7fffffffLL) return pl;  // too many tiles: simt_launch refuses
    const int T = static_cast<int>(T64);
    const int KT = static_cast<int>((K + BK - 1) / BK);
    const int W = sms * kSimtCtasPerSm;
    pl.dp_tiles = T;
    pl.parts = 1;
    const int R = W > 0 ? T % W : 0;
    if (W > 0 && R > 0) {  // also when all the tiles fit in one partial wave
        int parts = W / R;
        if (parts > kSimtMaxParts) parts = kSimtMaxParts;
        if (parts > KT / kSimtMinPartKTiles) parts = KT / kSimtMinPartKTiles;
        if (parts >= 2 && R <= static_cast<int>(kSimtCounterBytes / sizeof(unsigned int))) {
            pl.dp_tiles = T - R;
            pl.parts = parts;
            pl.ws_bytes = kSimtCounterBytes + static_cast<size_t>(R) * parts * BM * BN * sizeof(float);
        }
    }
    pl.grid = pl.dp_tiles + (T - pl.dp_tiles) * pl.parts;
    return pl;
}

int simt_launch(const SimtLaunch& L, cudaStream_t stream) {
    SimtParams p;
    p.M = static_cast<int>(L.M);
    p.N = static_cast<int>(L.N);
    p.K = static_cast<int>(L.K);
    p.A = L.A;
    p.lda = L.lda;
    p.B = L.B;
    p.ldb = L.ldb;
    p.C = L.C;
    p.ldc = L.ldc;
    p.alpha = L.alpha;
    p.beta = L.beta;
    p.tiles_n = (p.N + BN - 1) / BN;
    // The grid is 1-D: tiles (and their pieces) must number below 2^31.
    if (((L.M + BM - 1) / BM) * ((L.N + BN - 1) / BN) * kSimtMaxParts > 0x7fffffffLL)
        return GEMM_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    SimtPlan pl = simt_plan(L.M, L.N, L.K, sms);
    if (L.split_from >= 0) {
        // The caller's schedule: the same pieces a larger call would cut.
        const int T = simt_tiles(p.M, p.N);
        pl.dp_tiles = L.split_from < T ? L.split_from : T;
        pl.parts = pl.dp_tiles < T ? L.split_parts : 1;
        if (pl.parts < 2) {
            pl.dp_tiles = T;
            pl.parts = 1;
        }
        if (T - pl.dp_tiles > static_cast<int>(kSimtCounterBytes / sizeof(unsigned int)))
            return GEMM_ERR_UNSUPPORTED;
        pl.ws_bytes = pl.parts > 1 ? kSimtCounterBytes + static_cast<size_t>(T - pl.dp_tiles) *
                                                             pl.parts * BM * BN * sizeof(float)
                                   : 0;
        pl.grid = pl.dp_tiles + (T - pl.dp_tiles) * pl.parts;
    }
    p.dp_tiles = pl.dp_tiles;
    p.parts = pl.parts;
    p.ws = nullptr;
    p.counters = nullptr;
    p.clock_log = L.clock_log;
    if (pl.ws_bytes) {
        void* ws = nullptr;
        const int st = simt_workspace(dev, stream, pl.ws_bytes, &ws);
        if (st != GEMM_OK) return st;
        p.counters = static_cast<unsigned int*>(ws);
        p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kSimtCounterBytes);
    }
    if (L.single_fragments) {
        switch (L.stages) {
            case 1: return launch_stages<1, false>(p, stream);
            case 2: return launch_stages<2, false>(p, stream);
            case 3: return launch_stages<3, false>(p, stream);
            case 4: return launch_stages<4, false>(p, stream);
            default: return GEMM_ERR_ARG;
        }
    }
    switch (L.stages) {
        case 1: return launch_stages<1, true>(p, stream);
        case 2: return launch_stages<2, true>(p, stream);
        case 3: return launch_stages<3, true>(p, stream);
        case 4: return launch_stages<4, true>(p, stream);
        default: return GEMM_ERR_ARG;
    }
}

int simt_release_workspaces() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_simt_ws_mu);
    for (auto it = g_simt_ws.begin(); it != g_simt_ws.end();) {
        if (it->first.first == dev) {
            if (it->second.ptr) cudaFree(it->second.ptr);
            it = g_simt_ws.erase(it);
        } else {
            ++it;
        }
    }
    return GEMM_OK;
}

int scale_launch(int64_t M, int64_t N, void* C, int64_t ldc, int out_bf16, float beta,
                 cudaStream_t stream) {
    const long long total = M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    if (blocks < 1) blocks = 1;
    scale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, C, ldc, out_bf16, beta);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace ssp
