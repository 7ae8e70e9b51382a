// gemm_api.cu -- the C ABI of libgemm.so (declared in include/gemm.h):
// argument checks, dispatch to the tensor-core or SIMT kernel, the checked
// and host-buffer entry points, and status strings.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"

namespace {

int64_t g_wait_limit_ns = 2000000000LL;  // 2 s per pipeline wait
int g_withhold_arrive = -1;

bool is_tc(int dtype) {
    return dtype == GEMM_F16_F32 || dtype == GEMM_BF16_F32 || dtype == GEMM_BF16_BF16;
}

int in_size(int dtype) { return dtype == GEMM_F32 ? 4 : 2; }
int out_size(int dtype) { return dtype == GEMM_BF16_BF16 ? 2 : 4; }

// Tensor-core tile width for a request (0 = invalid).
int resolve_tile_n(int64_t N, int stages, int tile_n) {
    if (tile_n == 128 || tile_n == 256) return tile_n;
    if (tile_n != 0) return 0;
    if (stages > ssp::kTcMaxStages256 || N <= 128) return 128;
    return 256;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Checked {
    int status;
    int tile_n;
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
                 int tile_n) {
    Checked r{GEMM_OK, 0};
    if (dtype < GEMM_F32 || dtype > GEMM_BF16_BF16) return {GEMM_ERR_ARG, 0};
    if (M < 0 || N < 0 || K < 0) return {GEMM_ERR_ARG, 0};
    if (b_col_major != 0 && b_col_major != 1) return {GEMM_ERR_ARG, 0};
    if (is_tc(dtype)) {
        r.tile_n = resolve_tile_n(N, stages, tile_n);
        if (r.tile_n == 0) return {GEMM_ERR_ARG, 0};
        const int max_s = r.tile_n == 256 ? ssp::kTcMaxStages256 : ssp::kTcMaxStages128;
        if (stages < 1 || stages > ssp::kTcMaxStages128) return {GEMM_ERR_ARG, 0};
        if (stages > max_s) return {GEMM_ERR_UNSUPPORTED, 0};
    } else {
        if (tile_n != 0) return {GEMM_ERR_ARG, 0};
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

int run(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
        void* C, int64_t ldc, float alpha, float beta, int dtype, int stages, int b_col_major,
        int tile_n, cudaStream_t stream) {
    Checked v = validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, stages, b_col_major, tile_n);
    if (v.status != GEMM_OK) return v.status;
    if (M == 0 || N == 0) return GEMM_OK;
    if (K == 0 || alpha == 0.0f)
        return ssp::scale_launch(M, N, C, ldc, dtype == GEMM_BF16_BF16, beta, stream);
    if (dtype == GEMM_F32) {
        ssp::SimtLaunch L{M, N, K, static_cast<const float*>(A), lda,
                          static_cast<const float*>(B), ldb, static_cast<float*>(C), ldc,
                          alpha, beta, stages};
        return ssp::simt_launch(L, stream);
    }
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
    L.tile_n = v.tile_n;
    L.wait_limit_ns = g_wait_limit_ns;
    L.withhold_arrive = g_withhold_arrive;
    return ssp::tc_launch(L, stream);
}

// ---- gemm_host staging buffers, cached per device
struct Staging {
    void* ptr[3] = {nullptr, nullptr, nullptr};
    size_t cap[3] = {0, 0, 0};
};
std::mutex g_staging_mu;
Staging g_staging[64];

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
            int b_col_major, int tile_n, void* stream) {
    return run(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, b_col_major, tile_n,
               static_cast<cudaStream_t>(stream));
}

int gemm_checked(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                 int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype,
                 int stages, int b_col_major, int tile_n, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = run(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, b_col_major, tile_n,
                 s);
    if (st != GEMM_OK) return st;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
    ssp::GemmDeviceStatus ds;
    st = ssp::tc_read_and_clear_status(&ds);
    if (st != GEMM_OK) return st;
    return ds.code != 0 ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

int gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
              int64_t ldb, void* C, int64_t ldc, float alpha, float beta, int dtype, int stages,
              int b_col_major, int tile_n, void* stream) {
    Checked v = validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, stages, b_col_major, tile_n);
    if (v.status != GEMM_OK) return v.status;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    const size_t si = in_size(dtype), so = out_size(dtype);
    const bool need_ab = K > 0 && alpha != 0.0f;
    const size_t a_bytes = need_ab ? (static_cast<size_t>(M - 1) * lda + K) * si : 0;
    const size_t b_bytes =
        need_ab ? (b_col_major ? static_cast<size_t>(N - 1) * ldb + K
                               : static_cast<size_t>(K - 1) * ldb + N) * si
                : 0;
    const size_t c_bytes = (static_cast<size_t>(M - 1) * ldc + N) * so;
    std::lock_guard<std::mutex> g(g_staging_mu);
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    int st;
    if (a_bytes && (st = staging_get(dev, 0, a_bytes, &dA)) != GEMM_OK) return st;
    if (b_bytes && (st = staging_get(dev, 1, b_bytes, &dB)) != GEMM_OK) return st;
    if ((st = staging_get(dev, 2, c_bytes, &dC)) != GEMM_OK) return st;
    if (a_bytes && cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (b_bytes && cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (beta != 0.0f && cudaMemcpyAsync(dC, C, c_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    st = run(M, N, K, need_ab ? dA : A, lda, need_ab ? dB : B, ldb, dC, ldc, alpha, beta, dtype,
             stages, b_col_major, tile_n, s);
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}

int gemm_host_release(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_staging_mu);
    Staging& s = g_staging[dev];
    for (int i = 0; i < 3; ++i) {
        if (s.ptr[i]) cudaFree(s.ptr[i]);
        s.ptr[i] = nullptr;
        s.cap[i] = 0;
    }
    return GEMM_OK;
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
        default: return "unknown gemm status";
    }
}

int gemm_max_stages(int dtype, int tile_n) {
    if (dtype == GEMM_F32) return tile_n == 0 ? ssp::kSimtMaxStages : GEMM_ERR_ARG;
    if (!is_tc(dtype)) return GEMM_ERR_ARG;
    if (tile_n == 256) return ssp::kTcMaxStages256;
    if (tile_n == 128 || tile_n == 0) return ssp::kTcMaxStages128;
    return GEMM_ERR_ARG;
}

int gemm_debug_set(int64_t wait_limit_ns, int withhold_arrive) {
    g_wait_limit_ns = wait_limit_ns > 0 ? wait_limit_ns : 2000000000LL;
    g_withhold_arrive = withhold_arrive < 0 ? -1 : withhold_arrive;
    return GEMM_OK;
}

}  // extern "C"
