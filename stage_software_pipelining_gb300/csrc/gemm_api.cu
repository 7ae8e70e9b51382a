// gemm_api.cu -- the C ABI of libgemm.so (declared in include/gemm.h):
// argument checks, dispatch to the tensor-core or SIMT kernel, the checked
// and host-buffer entry points, and status strings.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"

namespace {

int64_t g_wait_limit_ns = 2000000000LL;  // 2 s per pipeline wait
int g_withhold_arrive = -1;
unsigned long long* g_clock_log = nullptr;  // gemm_clock_log
int g_schedule = 0;  // tensor-core tile schedule (gemm_schedule_set)

bool is_tc(int dtype) {
    return dtype == GEMM_F16_F32 || dtype == GEMM_BF16_F32 || dtype == GEMM_BF16_BF16;
}

int in_size(int dtype) { return dtype == GEMM_F32 ? 4 : 2; }
int out_size(int dtype) { return dtype == GEMM_BF16_BF16 ? 2 : 4; }

int tile_max_stages(int tile) {
    switch (tile) {
        case GEMM_TILE_128x128: return ssp::kTcMaxStages128;
        case GEMM_TILE_128x256: return ssp::kTcMaxStages256;
        case GEMM_TILE_256x256_2SM: return ssp::kTcMaxStagesPair;
        case GEMM_TILE_256x512_2SM: return ssp::kTcMaxStagesWide;
        default: return 0;
    }
}

// Tensor-core tile for a request (0 = invalid tile code).  An explicit tile
// comes back unchanged.  The automatic choice is the 256 x 256 tile on a CTA
// pair unless M or N is a single 128-wide tile, or the pair tiles make one
// partial round (measured on GB300, bf16):
//   * at most a quarter of the SMs busy: 128 x 128 tiles (four per pair
//     tile, one SM each) still fit in one round and finish in about half the
//     time (1024^2 x 4096: 459 vs 316 TFLOP/s);
//   * at most half of them busy and K <= 4096: the one-CTA 128 x 256 tile
//     (the same work per SM in the same single round) runs 4-9 % faster
//     (2048^2 x 1024 / 2048 / 4096); at K = 8192 the pair stays ahead.
// A ring deeper than the chosen tile holds (5 or 6 stages on the 128 x 256
// or 256 x 512 tile) takes the tile of the same rows per SM that holds it:
// the 256 x 256 pair tile (128 x 128 when M or N is a single tile).
int resolve_tile(int64_t M, int64_t N, int64_t K, int tile, int stages) {
    if (tile == GEMM_TILE_128x128 || tile == GEMM_TILE_128x256 || tile == GEMM_TILE_256x256_2SM ||
        tile == GEMM_TILE_256x512_2SM)
        return tile;
    if (tile != GEMM_TILE_AUTO) return 0;
    int t;
    const bool two_d = M > 128 && N > 128;
    if (two_d) {
        const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
        const int sms = ssp::tc_current_device_sms();
        const int64_t wide_tiles = ((M + 255) / 256) * ((N + 511) / 512);
        if (pair_tiles * 4 <= sms) t = GEMM_TILE_128x128;
        else if (pair_tiles * 2 <= sms && K <= 4096) t = GEMM_TILE_128x256;
        // The 512-wide tile carries a quarter fewer operand bytes per FLOP,
        // but its epilogue only half overlaps the next tile: it pays once the
        // mainloop is long (K >= 8192, measured +3-4 %; K = 4096 is even or
        // worse) and there is at least a full round of wide tiles.
        else if (K >= 8192 && wide_tiles * 2 >= sms) t = GEMM_TILE_256x512_2SM;
        else t = GEMM_TILE_256x256_2SM;
    } else {
        t = N <= 128 ? GEMM_TILE_128x128 : GEMM_TILE_128x256;
    }
    if (stages > tile_max_stages(t))
        t = two_d ? GEMM_TILE_256x256_2SM : GEMM_TILE_128x128;
    return t;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Checked {
    int status;
    int tile;  // resolved gemm_tile_t (tensor-core path)
};

// With a single row in memory an operand's leading dimension is never used;
// it is normalised to the row length rounded up to 16 bytes so that the
// alignment rule (and the tensor map's stride rule) holds.
int64_t single_row_ld(int64_t ld, int64_t cols, int size) {
    const int64_t m = 16 / size;
    const int64_t c = ld > cols ? ld : cols;
    return (c + m - 1) / m * m;
}

Checked validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t& lda, const void* B,
                 int64_t& ldb, void* C, int64_t& ldc, int dtype, int stages, int b_col_major,
                 int tile) {
    Checked r{GEMM_OK, 0};
    if (dtype < GEMM_F32 || dtype > GEMM_BF16_BF16) return {GEMM_ERR_ARG, 0};
    if (M < 0 || N < 0 || K < 0) return {GEMM_ERR_ARG, 0};
    if (b_col_major != 0 && b_col_major != 1) return {GEMM_ERR_ARG, 0};
    if (is_tc(dtype)) {
        if (stages < 1 || stages > ssp::kTcMaxStages) return {GEMM_ERR_ARG, 0};
        r.tile = resolve_tile(M, N, K, tile, stages);
        if (r.tile == 0) return {GEMM_ERR_ARG, 0};
        if (stages > tile_max_stages(r.tile)) return {GEMM_ERR_UNSUPPORTED, 0};
    } else {
        if (tile != GEMM_SIMT_FRAGMENTS_DOUBLE && tile != GEMM_SIMT_FRAGMENTS_SINGLE)
            return {GEMM_ERR_ARG, 0};
        if (stages < 1 || stages > ssp::kSimtMaxStages) return {GEMM_ERR_ARG, 0};
    }
    const bool use_a = M > 0 && K > 0;
    const bool use_b = N > 0 && K > 0;
    const bool use_c = M > 0 && N > 0;
    if (use_a && (A == nullptr || lda < K)) return {GEMM_ERR_ARG, 0};
    if (use_b && (B == nullptr || ldb < (b_col_major ? K : N))) return {GEMM_ERR_ARG, 0};
    if (use_c && (C == nullptr || ldc < N)) return {GEMM_ERR_ARG, 0};
    if (!is_tc(dtype) && b_col_major) return {GEMM_ERR_UNSUPPORTED, 0};
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return {GEMM_ERR_UNSUPPORTED, 0};
    const int si = in_size(dtype), so = out_size(dtype);
    if (M <= 1) lda = single_row_ld(lda, K, si);
    if ((b_col_major ? N : K) <= 1) ldb = single_row_ld(ldb, b_col_major ? K : N, si);
    if (M <= 1) ldc = single_row_ld(ldc, N, so);
    if (use_a && (!aligned16(A) || (lda * si) % 16 != 0)) return {GEMM_ERR_ALIGN, 0};
    if (use_b && (!aligned16(B) || (ldb * si) % 16 != 0)) return {GEMM_ERR_ALIGN, 0};
    if (use_c && (!aligned16(C) || (ldc * so) % 16 != 0)) return {GEMM_ERR_ALIGN, 0};
    return r;
}

ssp::TcLaunch tc_request(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, void* C, int64_t ldc, float alpha, float beta,
                         int dtype, int stages, int b_col_major, int tile) {
    ssp::TcLaunch L;
    L.M = M;
    L.N = N;
    L.K = K;
    L.A = A;
    L.lda = lda;
    L.B = B;
    L.ldb = ldb;
    L.C = C;
    L.ldc = ldc;
    L.alpha = alpha;
    L.beta = beta;
    L.in_bf16 = dtype != GEMM_F16_F32;
    L.out_bf16 = dtype == GEMM_BF16_BF16;
    L.b_col_major = b_col_major;
    L.stages = stages;
    L.tile_n = tile == GEMM_TILE_128x128 ? 128 : tile == GEMM_TILE_256x512_2SM ? 512 : 256;
    L.pair = tile == GEMM_TILE_256x256_2SM || tile == GEMM_TILE_256x512_2SM;
    L.wait_limit_ns = g_wait_limit_ns;
    L.withhold_arrive = g_withhold_arrive;
    L.clock_log = g_clock_log;
    L.schedule = g_schedule;
    return L;
}

// simt_split_from / simt_split_parts: the SIMT tile schedule to use instead
// of the one planned for these sizes (gemm_host's panels; -1: plan).
int run(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
        void* C, int64_t ldc, float alpha, float beta, int dtype, int stages, int b_col_major,
        int tile, cudaStream_t stream, int simt_split_from = -1, int simt_split_parts = 0) {
    Checked v = validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, stages, b_col_major, tile);
    if (v.status != GEMM_OK) return v.status;
    if (M == 0 || N == 0) return GEMM_OK;
    if (K == 0 || alpha == 0.0f)
        return ssp::scale_launch(M, N, C, ldc, dtype == GEMM_BF16_BF16, beta, stream);
    if (dtype == GEMM_F32) {
        ssp::SimtLaunch L{M, N, K, static_cast<const float*>(A), lda,
                          static_cast<const float*>(B), ldb, static_cast<float*>(C), ldc,
                          alpha, beta, stages, tile == GEMM_SIMT_FRAGMENTS_SINGLE, g_clock_log,
                          simt_split_from, simt_split_parts};
        return ssp::simt_launch(L, stream);
    }
    const ssp::TcLaunch L = tc_request(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype,
                                       stages, b_col_major, v.tile);
    return ssp::tc_launch(L, stream);
}

// ---- gemm_host staging buffers, cached per device
struct Staging {
    void* ptr[3] = {nullptr, nullptr, nullptr};
    size_t cap[3] = {0, 0, 0};
};
std::mutex g_staging_mu;
Staging g_staging[64];

// gemm_host's copy streams and events, created on first use per device.
constexpr int kHostPanels = 16;  // row panels a large gemm_host call is cut into
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;  // host->device and device->host copies
    cudaEvent_t start = nullptr, b_done = nullptr, done = nullptr;
    cudaEvent_t in_done[kHostPanels] = {}, gemm_done[kHostPanels] = {};
};
HostPipe g_pipe[64];

int host_pipe(int dev, HostPipe** out) {
    HostPipe& p = g_pipe[dev];
    if (!p.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.b_done, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.done, ef) != cudaSuccess)
            return GEMM_ERR_CUDA;
        for (int i = 0; i < kHostPanels; ++i)
            if (cudaEventCreateWithFlags(&p.in_done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.gemm_done[i], ef) != cudaSuccess)
                return GEMM_ERR_CUDA;
        p.ready = true;
    }
    *out = &p;
    return GEMM_OK;
}

void host_pipe_release(int dev) {
    HostPipe& p = g_pipe[dev];
    if (!p.ready) return;
    cudaStreamSynchronize(p.in);
    cudaStreamSynchronize(p.out);
    cudaStreamDestroy(p.in);
    cudaStreamDestroy(p.out);
    for (cudaEvent_t e : {p.start, p.b_done, p.done}) cudaEventDestroy(e);
    for (int i = 0; i < kHostPanels; ++i) {
        cudaEventDestroy(p.in_done[i]);
        cudaEventDestroy(p.gemm_done[i]);
    }
    p = HostPipe{};
}

int staging_get(int dev, int which, size_t bytes, void** out) {
    Staging& s = g_staging[dev];
    if (s.cap[which] < bytes) {
        if (s.ptr[which]) cudaFree(s.ptr[which]);
        s.ptr[which] = nullptr;
        s.cap[which] = 0;
        if (cudaMalloc(&s.ptr[which], bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        s.cap[which] = bytes;
    }
    *out = s.ptr[which];
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
         void* C, int64_t ldc, float alpha, float beta, int dtype, int stages, void* stream) {
    return run(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, 0, 0,
               static_cast<cudaStream_t>(stream));
}

int gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
            int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
            int b_col_major, int tile, void* stream) {
    return run(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, b_col_major, tile,
               static_cast<cudaStream_t>(stream));
}

int gemm_checked(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype,
                 int stages, int b_col_major, int tile, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = run(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, b_col_major, tile,
                 s);
    if (st != GEMM_OK) return st;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
    ssp::GemmDeviceStatus ds;
    st = ssp::tc_read_and_clear_status(&ds);
    if (st != GEMM_OK) return st;
    if (ds.code != 0) {
        ssp::tc_clear_workspace_flags();  // a run that gave up may leave flags set
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

int gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
              int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
              int b_col_major, int tile, void* stream) {
    Checked v = validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, stages, b_col_major, tile);
    if (v.status != GEMM_OK) return v.status;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    const size_t si = in_size(dtype), so = out_size(dtype);
    const bool need_ab = K > 0 && alpha != 0.0f;
    const size_t b_bytes =
        need_ab ? (b_col_major ? static_cast<size_t>(N - 1) * ldb + K
                               : static_cast<size_t>(K - 1) * ldb + N) * si
                : 0;
    // Bytes of rows [r0, r1) of a row-major operand with leading dimension ld.
    auto rows_bytes = [](int64_t r0, int64_t r1, int64_t ld, int64_t cols, size_t size) {
        return (static_cast<size_t>(r1 - r0 - 1) * ld + cols) * size;
    };
    const size_t a_bytes = need_ab ? rows_bytes(0, M, lda, K, si) : 0;
    const size_t c_bytes = rows_bytes(0, M, ldc, N, so);
    std::lock_guard<std::mutex> g(g_staging_mu);
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    int st;
    if (a_bytes && (st = staging_get(dev, 0, a_bytes, &dA)) != GEMM_OK) return st;
    if (b_bytes && (st = staging_get(dev, 1, b_bytes, &dB)) != GEMM_OK) return st;
    if ((st = staging_get(dev, 2, c_bytes, &dC)) != GEMM_OK) return st;
    HostPipe* hp = nullptr;
    if ((st = host_pipe(dev, &hp)) != GEMM_OK) return st;

    // The copies themselves are pipelined with the GEMM: B goes over first,
    // then M is cut into row panels; panel p's A and C rows are copied in on
    // one stream while panel p-1 is computed on the caller's stream and the
    // C rows of earlier panels are copied back on a third.  Host->device and
    // device->host copies use the link in both directions at once.  Each
    // panel is a whole number of 256-row tiles.
    const int64_t panel_rows = std::max<int64_t>(256, (M + kHostPanels - 1) / kHostPanels + 255) / 256 * 256;
    const int panels = static_cast<int>((M + panel_rows - 1) / panel_rows);
    // The SIMT path cuts the tiles of a partial last wave along K: each panel
    // cuts exactly the tiles the whole call would, so the bits match.
    const ssp::SimtPlan simt_whole =
        dtype == GEMM_F32 ? ssp::simt_plan(M, N, K, ssp::tc_current_device_sms()) : ssp::SimtPlan{};
    auto fail = [&]() {
        cudaStreamSynchronize(hp->in);
        cudaStreamSynchronize(s);
        cudaStreamSynchronize(hp->out);
        return GEMM_ERR_CUDA;
    };
    // Work already queued on the caller's stream comes first.
    if (cudaEventRecord(hp->start, s) != cudaSuccess ||
        cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
        return fail();
    if (b_bytes && cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
        return fail();
    for (int pi = 0; pi < panels; ++pi) {
        const int64_t r0 = pi * panel_rows, r1 = std::min<int64_t>(M, r0 + panel_rows);
        char* pA = static_cast<char*>(dA) + static_cast<size_t>(r0) * lda * si;
        char* pC = static_cast<char*>(dC) + static_cast<size_t>(r0) * ldc * so;
        const char* hA = static_cast<const char*>(A) + static_cast<size_t>(r0) * lda * si;
        char* hC = static_cast<char*>(C) + static_cast<size_t>(r0) * ldc * so;
        const size_t pc_bytes = rows_bytes(r0, r1, ldc, N, so);
        if (need_ab && cudaMemcpyAsync(pA, hA, rows_bytes(r0, r1, lda, K, si),
                                       cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
            return fail();
        if (beta != 0.0f &&
            cudaMemcpyAsync(pC, hC, pc_bytes, cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
            return fail();
        if (cudaEventRecord(hp->in_done[pi], hp->in) != cudaSuccess ||
            cudaStreamWaitEvent(s, hp->in_done[pi], 0) != cudaSuccess)
            return fail();
        // Every panel uses the tile chosen for the whole of M, so that the
        // panels compute exactly what one call over all of M would.  The one
        // exception gives the same bits: a panel too short to fill a round of
        // 256 x 512 tiles runs the 256 x 256 pair tile, whose MMAs take every
        // K step of every output in the same order (and whose ring holds any
        // depth the wide tile's does).
        int ptile = is_tc(dtype) ? v.tile : tile;
        if (ptile == GEMM_TILE_256x512_2SM &&
            resolve_tile(r1 - r0, N, K, GEMM_TILE_AUTO, stages) != GEMM_TILE_256x512_2SM)
            ptile = GEMM_TILE_256x256_2SM;
        int split_from = -1;
        if (dtype == GEMM_F32) {
            const int64_t first_tile = (r0 / 128) * ((N + 63) / 64);
            split_from = static_cast<int>(std::max<int64_t>(0, simt_whole.dp_tiles - first_tile));
        }
        st = run(r1 - r0, N, K, need_ab ? pA : hA, lda, need_ab ? dB : B, ldb, pC, ldc, alpha,
                 beta, dtype, stages, b_col_major, ptile, s, split_from, simt_whole.parts);
        if (st != GEMM_OK) {
            fail();
            return st;
        }
        if (cudaEventRecord(hp->gemm_done[pi], s) != cudaSuccess ||
            cudaStreamWaitEvent(hp->out, hp->gemm_done[pi], 0) != cudaSuccess ||
            cudaMemcpyAsync(hC, pC, pc_bytes, cudaMemcpyDeviceToHost, hp->out) != cudaSuccess)
            return fail();
    }
    // The caller's stream ends after the last copy back.
    if (cudaEventRecord(hp->done, hp->out) != cudaSuccess ||
        cudaStreamWaitEvent(s, hp->done, 0) != cudaSuccess)
        return fail();
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail();
    return GEMM_OK;
}

int gemm_host_release(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(g_staging_mu);
        Staging& s = g_staging[dev];
        for (int i = 0; i < 3; ++i) {
            if (s.ptr[i]) cudaFree(s.ptr[i]);
            s.ptr[i] = nullptr;
            s.cap[i] = 0;
        }
        host_pipe_release(dev);
    }
    const int st = ssp::simt_release_workspaces();
    if (st != GEMM_OK) return st;
    return ssp::tc_release_workspaces();
}

const char* gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_ARG: return "GEMM_ERR_ARG: invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: combination not implemented";
        case GEMM_ERR_ALIGN: return "GEMM_ERR_ALIGN: pointer or leading dimension not 16-byte aligned";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch or tensor-map encode failed";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a pipeline wait ran out";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA runtime call failed";
        case GEMM_ERR_SCRATCH:
            return "GEMM_ERR_SCRATCH: the launch needs more scratch than gemm_noalloc's fixed array";
        default: return "unknown gemm status";
    }
}

int gemm_max_stages(int dtype, int tile) {
    if (dtype == GEMM_F32)
        return (tile == GEMM_SIMT_FRAGMENTS_DOUBLE || tile == GEMM_SIMT_FRAGMENTS_SINGLE)
                   ? ssp::kSimtMaxStages
                   : GEMM_ERR_ARG;
    if (!is_tc(dtype)) return GEMM_ERR_ARG;
    if (tile == GEMM_TILE_AUTO) return ssp::kTcMaxStages;
    const int m = tile_max_stages(tile);
    return m > 0 ? m : GEMM_ERR_ARG;
}

int gemm_resolve_tile(int64_t M, int64_t N, int64_t K, int dtype, int tile, int stages) {
    if (!is_tc(dtype) || M < 0 || N < 0 || K < 0) return GEMM_ERR_ARG;
    if (stages < 1 || stages > ssp::kTcMaxStages) return GEMM_ERR_ARG;
    const int t = resolve_tile(M, N, K, tile, stages);
    return t != 0 ? t : GEMM_ERR_ARG;
}

int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int stages, int b_col_major, int tile,
              int* grid, int* cluster, int* smem_bytes) {
    // Validation with placeholder (aligned, non-null) pointers: only the
    // sizes, types, stages and tile are being planned.
    const void* P = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    const int si = in_size(dtype >= GEMM_F32 && dtype <= GEMM_BF16_BF16 ? dtype : 0);
    const int so = out_size(dtype);
    auto pad = [](int64_t x, int64_t size) { return (x + 16 / size - 1) / (16 / size) * (16 / size); };
    int64_t lda = pad(K > 0 ? K : 1, si), ldb = pad(b_col_major ? K : N, si), ldc = pad(N > 0 ? N : 1, so);
    if (ldb < 1) ldb = 16 / si;
    Checked v = validate(M, N, K, P, lda, P, ldb, const_cast<void*>(P), ldc, dtype, stages,
                         b_col_major, tile);
    if (v.status != GEMM_OK) return v.status;
    if (M == 0 || N == 0 || K == 0) {
        if (grid) *grid = 0;
        if (cluster) *cluster = 1;
        if (smem_bytes) *smem_bytes = 0;
        return GEMM_OK;
    }
    if (dtype == GEMM_F32) {
        if (grid) *grid = ssp::simt_plan(M, N, K, ssp::tc_current_device_sms()).grid;
        if (cluster) *cluster = 1;
        if (smem_bytes) *smem_bytes = stages * (128 * 20 + 16 * 64) * 4;
        return GEMM_OK;
    }
    const ssp::TcLaunch L = tc_request(M, N, K, P, lda, P, ldb, const_cast<void*>(P), ldc, 1.0f,
                                       0.0f, dtype, stages, b_col_major, v.tile);
    return ssp::tc_plan(L, grid, cluster, smem_bytes);
}

int pipelined_copy(void* dst, const void* src, int64_t n_bytes, int stages, void* stream) {
    if (n_bytes < 0 || stages < 1 || stages > ssp::kCopyMaxStages) return GEMM_ERR_ARG;
    if (n_bytes == 0) return GEMM_OK;
    if (dst == nullptr || src == nullptr) return GEMM_ERR_ARG;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + static_cast<uintptr_t>(n_bytes) && s < d + static_cast<uintptr_t>(n_bytes))
        return GEMM_ERR_ARG;  // overlapping ranges
    if (!aligned16(dst) || !aligned16(src) || n_bytes % 16 != 0) return GEMM_ERR_ALIGN;
    return ssp::copy_launch(dst, src, n_bytes, stages, static_cast<cudaStream_t>(stream));
}

int gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
                 int b_col_major, int tile, void* stream) {
    Checked v = validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, stages, b_col_major, tile);
    if (v.status != GEMM_OK) return v.status;
    if (!is_tc(dtype)) return GEMM_ERR_UNSUPPORTED;  // the SIMT kernel has no scratch variant
    // One 128 x 512 fp32 partial per CTA of the 256 x 512 tile (256 KB, 38 MB
    // over 152 SMs) does not fit the fixed array: that tile is refused when
    // asked for by name, whatever the shape, before anything is enqueued.
    if (tile == GEMM_TILE_256x512_2SM) return GEMM_ERR_SCRATCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0) return GEMM_OK;
    if (K == 0 || alpha == 0.0f)
        return ssp::scale_launch(M, N, C, ldc, dtype == GEMM_BF16_BF16, beta, s);
    // Where the automatic choice is the 256 x 512 tile, the 256 x 256 pair
    // tile runs instead: it gives the same bits, and its ring holds any depth
    // the wide tile's does.
    const int t = v.tile == GEMM_TILE_256x512_2SM ? GEMM_TILE_256x256_2SM : v.tile;
    ssp::TcLaunch L = tc_request(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages,
                                 b_col_major, t);
    L.schedule = 2;  // stream-K tail, its partials in the fixed array
    return ssp::tc_launch_noalloc(L, s);
}

int gemm_schedule_set(int schedule) {
    if (schedule < 0 || schedule > 2) return GEMM_ERR_ARG;
    g_schedule = schedule;
    return GEMM_OK;
}

int gemm_debug_set(int64_t wait_limit_ns, int withhold_arrive) {
    g_wait_limit_ns = wait_limit_ns > 0 ? wait_limit_ns : 2000000000LL;
    g_withhold_arrive = withhold_arrive < 0 ? -1 : withhold_arrive;
    return GEMM_OK;
}

int gemm_clock_log(void* dev_buf) {
    g_clock_log = static_cast<unsigned long long*>(dev_buf);
    return GEMM_OK;
}

}  // extern "C"
