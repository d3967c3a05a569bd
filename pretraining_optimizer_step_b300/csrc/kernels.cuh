// kernels.cuh -- launch parameters shared by the host planner (muon_api.cu) and
// the device kernels (momentum_norm.cu, ns_gemm.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace muon {

// Device status word bits (latched with atomicOr, read by muon_get_status).
enum : unsigned int {
    STATUS_TIMEOUT = 1u,
    STATUS_BOUNDS = 2u,
};

// ------------------------------------------------------------------ momentum + norm
// One launch handles up to kMomentumMaxMats matrices (by value in the params).
constexpr int kMomentumMaxMats = 192;
constexpr int kMomTile = 64;       // 64 x 64 stored elements per CTA
constexpr int kMomThreads = 256;

struct MomentumMat {
    const float* g;
    float* mom;
    float* p;             // published to p_table for the fused final update
    __nv_bfloat16* x0;    // oriented X0 (unscaled u), m x n
    int rows, cols;       // stored shape
    int transposed;       // rows > cols: X0 = u^T
    int tiles_x;          // ceil(cols / 64)
    int tile_begin;       // first CTA of this matrix in the launch
    int ntiles;
    int gidx;             // index of the matrix in the step
};

struct MomentumParams {
    MomentumMat mats[kMomentumMaxMats];
    int nmats;
    int total_tiles;
    float beta;
    int nesterov;
    int mode;             // 0: m' = beta m + g ; 1: m' = beta m + (1 - beta) g
    float eps;
    float* partials;      // one float per CTA of the launch
    unsigned int* counters;  // per step matrix; reset to 0 by the last CTA
    float* inv_norm;      // per step matrix: 1 / (||u|| + eps)
    float* norms;         // per step matrix: ||u||
    float** p_table;      // per step matrix
};

// ------------------------------------------------------------------ weight update without NS
struct UpdateParams {
    MomentumMat mats[kMomentumMaxMats];  // reuses the per-matrix geometry of the momentum pass
    int nmats;
    int total_tiles;
    const float* inv_norm;
    const float* aspect;  // per step matrix: sqrt(max(1, rows/cols))
    float lr;
    float* const* dbg_O;  // per step matrix or nullptr
};

// ------------------------------------------------------------------ Newton-Schulz GEMM
constexpr int kBM = 128;             // tile rows (TMEM lanes)
constexpr int kBN = 256;             // tile columns (fp32 TMEM columns per accumulator)
constexpr int kBK = 64;              // K slice per pipeline stage (128 B of bf16)
constexpr int kStages = 4;
constexpr int kAStageBytes = kBM * kBK * 2;   // 16 KiB
constexpr int kBStageBytes = kBN * kBK * 2;   // 32 KiB
constexpr int kStageBytes = kAStageBytes + kBStageBytes;
constexpr int kTmemCols = 512;       // two 256-column accumulators
constexpr int kGemmThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kGemmSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
constexpr int kMaxClasses = 8;

enum GemmMode : int {
    MODE_GRAM = 0,        // A = s^2 X X^T (upper tiles, mirrored)
    MODE_POLY = 1,        // B = b A + c A A (upper tiles, mirrored)
    MODE_AXPY = 2,        // X' = s (a X + B X)
    MODE_AXPY_FINAL = 3,  // O = s (a X + B X); p -= scale O
};

struct GemmClass {
    int m, n;             // oriented X is m x n (m <= n)
    int nmats;
    int tile_begin;
    int tiles_per_mat;
    int k_blocks;         // ceil(K / 64)
    int row_blocks;       // ceil(m / 128)
    int col_tiles;        // axpy: ceil(n / 256)
    int transposed;       // stored matrix is n x m
    int mat_base;         // step index of the class's first matrix
    const __nv_bfloat16* aux;  // poly: A ; axpy: X_in
    __nv_bfloat16* out;        // gram: A ; poly: B ; axpy: X_out
};

struct GemmParams {
    CUtensorMap tmA[kMaxClasses];  // M-side operand, K-major, box 64 x 128
    CUtensorMap tmB[kMaxClasses];  // N-side operand: K-major box 64 x 128, or MN-major box 64 x 64 (axpy)
    GemmClass cls[kMaxClasses];
    int nclasses;
    int total_tiles;
    int mode;
    int first_iter;       // fold 1/||u|| (X0 is stored unscaled)
    float ca, cb, cc;
    const float* inv_norm;     // per step matrix
    const float* aspect;       // per step matrix: sqrt(max(1, rows/cols))
    float lr;
    float* const* p_table;     // per step matrix
    float* const* dbg_O;       // per step matrix or nullptr
    unsigned int* status;
    unsigned long long timeout_ns;
    int inject_lost_load;      // test hook (see MUON_DEBUG_INJECT_LOST_LOAD)
};

// Launchers (return the launch error, if any).
cudaError_t launch_momentum_norm(const MomentumParams& p, cudaStream_t s);
cudaError_t launch_update(const UpdateParams& p, cudaStream_t s);
cudaError_t launch_ns_gemm(const GemmParams& p, int grid, cudaStream_t s);
cudaError_t ns_gemm_prepare();  // one-time kernel attribute setup

}  // namespace muon
