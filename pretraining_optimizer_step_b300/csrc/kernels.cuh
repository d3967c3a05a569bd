// kernels.cuh -- launch parameters shared by the host planner (muon_api.cu) and
// the device kernels (momentum_norm.cu, ns_pair.cu, normuon.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace muon {

// Device status word bits (latched with atomicOr, read by muon_get_status).
enum : unsigned int {
    STATUS_TIMEOUT = 1u,
    STATUS_BOUNDS = 2u,     // a launch's tile list did not match its classes (no tile was run)
};

// ------------------------------------------------------------------ momentum + norm
// One launch handles up to kMomentumMaxMats matrices (by value in the params).
constexpr int kMomentumMaxMats = 192;
constexpr int kMomTile = 64;       // 64 x 64 stored elements per CTA
constexpr int kMomThreads = 256;

struct MomentumMat {
    const float* g;
    float* mom;
    float* p;             // weights (read by the standalone update only)
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

// ------------------------------------------------------------------ Newton-Schulz GEMM tiling
constexpr int kBM = 128;             // row block of the symmetric products (TMEM lanes per CTA)
constexpr int kBN = 256;             // axpy column tile (fp32 TMEM columns per accumulator)
constexpr int kBK = 64;              // K width of one 128B-swizzled operand panel (128 B of bf16)
constexpr int kTmemCols = 512;       // two 256-column accumulators
constexpr int kGemmThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kMaxClasses = 8;

// Symmetric results (A, B) are computed on tiles on and above the diagonal and stored as
// their upper 128 x 128 blocks; a I is folded into B, so the axpy modes compute s B' X with
// B' = B + a I.
enum GemmMode : int {
    MODE_GRAM = 0,        // A = s^2 X X^T
    MODE_POLY = 1,        // B' = b A + c A A + a I
    MODE_AXPY = 2,        // X' = s B' X
    MODE_AXPY_FINAL = 3,  // O = s B' X; p -= scale O
    MODE_AXPY_O = 4,      // O = s B' X written in bf16 (stored layout) for the NorMuon pass
};

// ------------------------------------------------------------------ NorMuon scaling
// Per stored row i of O (fp32, stored r x c): v_mean = mean_j O_ij^2, V_i <- b2 V_i + (1 - b2) v_mean,
// step_i = 1 / sqrt(V_i + eps); per matrix: ratio = sqrt(sum v_mean) / max(sqrt(sum v_mean step^2), 1e-10).
// Then p_ij -= lr aspect step_i ratio O_ij.
constexpr int kNormWarps = 8;                // 256 threads
constexpr int kNormRowsPerWarp = 4;
constexpr int kNormRowsPerCta = kNormWarps * kNormRowsPerWarp;
struct NormuonMat {
    const __nv_bfloat16* O;  // stored rows x cols, bf16 (workspace)
    float* V;             // caller-owned second moments, rows floats
    float* p;             // weights
    float* dbg;           // O' (stored layout) when the debug copy is kept, else nullptr
    int rows, cols;
    int cta_begin;        // rows kernel: first CTA of this matrix
    int nctas;            // rows kernel: CTAs of this matrix (ceil(rows / 8))
    int tile_begin;       // update kernel: first 64 x 64 tile of this matrix
    int tiles_x;          // update kernel: ceil(cols / 64)
    int pos;              // step position (aspect, ratio, counters)
};
struct NormuonParams {
    NormuonMat mats[kMomentumMaxMats];
    int nmats;
    int total;            // CTAs (rows kernel) or tiles (update kernel)
    float beta2, eps;
    float lr;
    const float* aspect;  // per position
    float* step;          // per matrix row block: step_i, indexed by a per-matrix offset (row_base[pos] + i)
    const int* row_base;  // per position: offset of the matrix's rows in `step`
    double* partials;     // rows kernel: two doubles per CTA (sum v_mean, sum v_mean step^2)
    unsigned int* counters;  // per position
    float* ratio;         // per position
};
cudaError_t launch_normuon_rows(const NormuonParams& p, cudaStream_t s);
cudaError_t launch_normuon_update(const NormuonParams& p, cudaStream_t s);

// Launchers (return the launch error, if any).
cudaError_t launch_momentum_norm(const MomentumParams& p, cudaStream_t s);
cudaError_t launch_update(const UpdateParams& p, cudaStream_t s);

// ------------------------------------------------------------------ Newton-Schulz GEMM on CTA pairs
// A cluster of two CTAs computes a 256 x N tile (N = 256, or 128 for a ragged
// last column tile) with tcgen05.mma.cta_group::2: each CTA holds 128 rows of
// the A operand and N/2 rows of the B operand per pipeline stage, and receives
// its 128 rows of the accumulator in its own TMEM.  A row pair whose second
// block does not exist runs as a 128 x N tile (M = 128: 64 rows per CTA).
// Each pipeline stage covers 128 of K (8 MMAs of K 16): per CTA two 16 KiB
// panels of A (128 rows x 64 K, 128B-swizzled) and two of its B half.  Fewer,
// deeper stages amortise the per-stage barrier round trip of the MMA issuer.
constexpr int kPairBK = 128;
constexpr int kPairPanelBytes = 128 * 64 * 2;               // 16 KiB
constexpr int kPairStageBytes = 4 * kPairPanelBytes;         // 64 KiB
constexpr int kPairMaxStages = 3;
// Shared memory by mode: every launch uses 3 stages + 8 KiB of epilogue slots per warp,
// except a final launch that also stores the debug copy of O: 2 stages + 24 KiB per warp.
constexpr int kPairSmemBytes = 224 * 1024 + 1024;
static_assert(3 * kPairStageBytes + 4 * 8192 <= 224 * 1024, "stage + epilogue layout");
static_assert(2 * kPairStageBytes + 4 * 24576 <= 224 * 1024, "stage + epilogue layout (final, debug O)");

struct PairClass {
    int m, n;             // oriented X is m x n (m <= n)
    int nmats;
    int tile_begin;       // first pair tile of this class in the launch
    int tiles_per_mat;    // pair tiles per matrix
    int k_blocks;         // ceil(K / 128)
    int row_blocks;       // ceil(m / 128)
    int col_groups;       // Gram/poly: ceil(row_blocks / 2) column pairs; axpy: ceil(n / 256) column tiles
    int transposed;       // stored matrix is n x m
    int mat_base;         // step position of the class's first matrix
};

struct PairParams {
    CUtensorMap tmA[kMaxClasses];    // A side, K-major, box 64 (K) x 128 rows, 128B swizzle
    CUtensorMap tmB[kMaxClasses];    // B side: Gram/poly K-major box 64 x 64 (N = 128 tiles; N = 256 tiles
                                     // use tmA); axpy MN-major box 64 cols x 128 K
    CUtensorMap tmIn[kMaxClasses];   // epilogue input (poly: A), bf16 box 32 rows x 64 columns, 128B swizzle
    CUtensorMap tmOut[kMaxClasses];  // epilogue output (gram: A, poly: B', axpy: X'), bf16 box 32 x 64, 128B swizzle
    CUtensorMap tmA64[kMaxClasses];  // A side of a half tile (M = 128): K-major box 64 (K) x 64 rows
    PairClass cls[kMaxClasses];
    int nclasses;
    int total_tiles;      // pair tiles
    int mode;             // GemmMode
    int first_iter;
    float ca, cb, cc;
    const float* inv_norm;
    const float* aspect;
    float lr;
    const CUtensorMap* p_maps;    // per step position: fp32 weights (stored layout), box 32 x 32, 128B swizzle
    const CUtensorMap* dbg_maps;  // per step position (O, stored layout) or nullptr
    const CUtensorMap* o_maps;    // MODE_AXPY_O: per step position, the bf16 O buffer (stored layout), box 32 x 32,
                                  // 64B swizzle
    unsigned int* status;
    unsigned long long timeout_ns;
    int inject_lost_load;
};

cudaError_t launch_ns_pair(const PairParams& p, int clusters, cudaStream_t s);
cudaError_t ns_pair_prepare(int* max_clusters);  // kernel attributes; co-resident clusters of two


}  // namespace muon
