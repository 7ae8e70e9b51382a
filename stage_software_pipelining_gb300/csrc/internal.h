// internal.h -- launcher interfaces shared by the C ABI (gemm_api.cu) and the
// two kernels (gemm_tc_sm103a.cu, sgemm_simt.cu).  Not installed; the public
// interface is include/gemm.h.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace ssp {

// Device status word written by a pipeline wait that ran out.
struct GemmDeviceStatus {
    int code;   // 0 = fine, else GEMM_ERR_TIMEOUT
    int block;  // blockIdx.x of the first CTA that gave up
    int role;   // 0 producer, 1 MMA issuer, 2 epilogue
    int iter;   // the K-tile iteration (producer/MMA) or tile count (epilogue)
};

struct TcLaunch {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    void* C;
    int64_t ldc;
    float alpha, beta;
    int in_bf16;      // 0 fp16 inputs, 1 bf16 inputs
    int out_bf16;     // 0 fp32 output, 1 bf16 output
    int b_col_major;  // 0 B row-major (N contiguous), 1 B column-major (K contiguous)
    int stages;       // ring depth (1..6, or 1..4 for the 128 x 256 and 256 x 512 tiles)
    int tile_n;       // tile width: 128, 256 or (pair only) 512
    int pair;         // 1: 256-row tile on a CTA pair (cta_group::2), tile_n = 256 or 512
    int schedule;     // 0 auto, 1 full tiles only, 2 stream-K tail whenever a round is partial
    int64_t wait_limit_ns;
    int withhold_arrive;
    unsigned long long* clock_log;  // device [2] or null: CTA 0's SM clocks and ns
};

struct SimtLaunch {
    int64_t M, N, K;
    const float* A;
    int64_t lda;
    const float* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
    float alpha, beta;
    int stages;            // 1..4
    int single_fragments;  // 1: one register fragment set; 0: two (double-buffered)
    unsigned long long* clock_log;  // device [2] or null: CTA 0's SM clocks and ns
    // Tile schedule imposed by the caller (gemm_host's row panels follow the
    // whole call's): split_from < 0 lets simt_launch plan; otherwise tiles
    // [split_from, ...) of this launch run as split_parts K pieces.
    int split_from;
    int split_parts;
};

// Enqueue the tensor-core GEMM (K > 0, M > 0, N > 0, alpha != 0).  Returns a
// gemm_status_t.
int tc_launch(const TcLaunch& L, cudaStream_t stream);
// Size of the fixed stream-K workspace of gemm_noalloc (20 MiB: one 128 x 256
// fp32 partial per CTA for 152 CTAs, plus flags).
constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;
// tc_launch with the stream-K tail schedule and its workspace in that fixed
// array: no allocation.  GEMM_ERR_SCRATCH if the launch needs more.
int tc_launch_noalloc(const TcLaunch& L, cudaStream_t stream);

// Launch geometry tc_launch would use (CTAs, CTAs per cluster, dynamic
// shared memory per CTA), without launching.
int tc_plan(const TcLaunch& L, int* grid, int* cluster, int* smem_bytes);
// Free the stream-K workspaces of the current device.
int tc_release_workspaces();

// SM count of the current device (0 when it cannot be queried).
int tc_current_device_sms();
// Zero the stream-K flags of every workspace of the current device (after a
// run that gave up; synchronous).
int tc_clear_workspace_flags();
// Read the device status word of the tensor-core kernel on the current device
// and reset it to zero (synchronous).
int tc_read_and_clear_status(GemmDeviceStatus* out);

int simt_launch(const SimtLaunch& L, cudaStream_t stream);
// Tile schedule of the SIMT kernel for a shape on a GPU with `sms` SMs: tiles
// [0, dp_tiles) run whole; each later tile (those of a partial last wave) runs
// as `parts` pieces along K, combined through a workspace of ws_bytes.
struct SimtPlan {
    int dp_tiles = 0;
    int parts = 1;
    int grid = 0;
    size_t ws_bytes = 0;
};
SimtPlan simt_plan(int64_t M, int64_t N, int64_t K, int sms);
// Free the split-tail workspaces of the current device.
int simt_release_workspaces();

// C = beta*C over an M x N block (K == 0 or alpha == 0); elem_bytes 4 (fp32) or 2 (bf16).
int scale_launch(int64_t M, int64_t N, void* C, int64_t ldc, int out_bf16, float beta,
                 cudaStream_t stream);

// Streaming copy of n_bytes (a multiple of 16) through a ring of `stages`
// shared-memory slots per thread (1..8).
int copy_launch(void* dst, const void* src, int64_t n_bytes, int stages, cudaStream_t stream);
constexpr int kCopyMaxStages = 8;

// Tensor-core ring depth limits.  A stage holds K = 64 of both operands on
// every tile; the limit is what fits in 227 KB of shared memory next to the
// epilogue's output boxes.
constexpr int kTcMaxStages128 = 6;   // 128 x 128 x 64 tile: 32 KB per stage
constexpr int kTcMaxStages256 = 4;   // 128 x 256 x 64 tile: 48 KB per stage
constexpr int kTcMaxStagesPair = 6;  // 256 x 256 x 64 tile on a CTA pair: 32 KB per stage per CTA
constexpr int kTcMaxStagesWide = 4;  // 256 x 512 x 64 tile on a CTA pair: 48 KB per stage per CTA
constexpr int kTcMaxStages = 6;      // the largest of the four
constexpr int kSimtMaxStages = 4;

}  // namespace ssp
