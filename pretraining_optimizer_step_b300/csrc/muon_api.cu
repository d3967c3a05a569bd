// muon_api.cu -- the C ABI of libmuon.so (declared in include/muon.h) and the
// host-side planner: argument checks, grouping of the step's matrices into
// oriented shape classes, one workspace arena per shape list, TMA tensor maps,
// and the launch sequence
//   momentum_norm  ->  K x { Gram -> polynomial -> axpy (the last one fused with
//   the weight update) }     (or the standalone update when K = 0).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/muon.h"
#include "kernels.cuh"

using namespace muon;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kKinds = 8;  // momentum, gram, poly, axpy, axpy+update, update, axpy writing O, NorMuon
constexpr int kMaxCoeffRows = 16;
constexpr int kMaxPlans = 8;  // workspaces kept, one per distinct shape list (least recently used dropped)

struct ClassPlan {
    int m = 0, n = 0, transposed = 0;
    std::vector<int> mats;  // step indices, in step order
    __nv_bfloat16* X[2] = {nullptr, nullptr};
    __nv_bfloat16* A = nullptr;
    __nv_bfloat16* B = nullptr;
    // A-side K-major maps (box 64 x 128), B-side K-major maps (box 64 x 64), the MN-major X map
    // of the axpy B operand (box 64 x 128), and epilogue subtile maps (bf16 32 x 32)
    CUtensorMap tmXk[2], tmAk, tmBk;
    CUtensorMap tmXk64[2], tmAk64, tmBk64, tmXmn128[2], epiX64[2], epiA64, epiB64;
    int row_blocks = 0, col_tiles = 0;
    int col_pairs = 0, sym_pair_tiles = 0, axpy_pair_tiles = 0;
};

struct Plan {
    std::vector<muon_shape> shapes;
    std::vector<ClassPlan> classes;
    std::vector<int> mat_class, mat_slot;
    // class-ordered step index: matrices of class 0 first, then class 1, ...
    std::vector<int> order;         // position -> step matrix
    std::vector<int> position;      // step matrix -> position
    char* arena = nullptr;
    size_t arena_bytes = 0;
    float* inv_norm = nullptr;
    float* norms = nullptr;
    float* aspect = nullptr;
    unsigned int* counters = nullptr;
    float** dbg_table = nullptr;    // device array of per-matrix O buffers (KEEP_O)
    float* partials = nullptr;
    size_t workspace_bf16_bytes = 0;
    char* workspace_bf16 = nullptr;
    std::vector<float*> dbg_O;      // host copies of the O buffer pointers
    CUtensorMap* p_maps = nullptr;  // device: fp32 weight maps per position (refreshed when params change)
    CUtensorMap* dbg_maps = nullptr;  // device: O maps per position (KEEP_O)
    std::vector<float*> mapped_p;   // params the device p_maps describe, by step index
    // NorMuon resources (allocated by the first muon_step_normuon on this plan)
    char* nm_arena = nullptr;
    std::vector<__nv_bfloat16*> o_bufs;  // bf16 O per matrix (stored layout), by step index
    CUtensorMap* o_maps = nullptr;  // device, by position
    float* nm_step = nullptr;       // step_i of every stored row, matrices at row_base
    int* nm_row_base = nullptr;     // device, by position
    std::vector<int> row_base;      // host copy
    double* nm_partials = nullptr;
    unsigned int* nm_counters = nullptr;
    float* nm_ratio = nullptr;
    double ns_flops_per_iter = 0.0;
    double elem_bytes = 0.0;
};

struct PendingTime {
    int kind;
    cudaEvent_t a, b;
};

struct Context {
    int device = -1;
    int sm_count = 0;
    int max_clusters = 0;           // co-resident CTA pairs of the pair kernel
    std::vector<double> coeffs;
    int n_rows = 0;
    double eps = 1e-7;
    int momentum_mode = 0;
    int debug = 0;
    unsigned long long timeout_ns = 5000000000ull;
    EncodeTiledFn encode = nullptr;
    unsigned int* status = nullptr;
    std::vector<Plan*> plans;       // most recently used first
    Plan* last = nullptr;           // the plan of the last step (debug copies)
    muon_step_info info{};
    std::vector<cudaEvent_t> event_pool;
    std::vector<PendingTime> pending;
    double kind_ms[kKinds] = {0};
    int kind_launches[kKinds] = {0};
    bool injected = false;
    bool injected_bad = false;
};

Context* g_ctx = nullptr;

// An NVTX range for the lifetime of a scope (header-only NVTX: a no-op unless a profiler
// attaches).  The step, its momentum pass, every Newton-Schulz iteration and the NorMuon pass
// show up as named ranges on the host timeline.
struct NvtxScope {
    explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope&) = delete;
    NvtxScope& operator=(const NvtxScope&) = delete;
};
const char* const kIterRange[kMaxCoeffRows] = {
    "muon NS iteration 1",  "muon NS iteration 2",  "muon NS iteration 3",  "muon NS iteration 4",
    "muon NS iteration 5",  "muon NS iteration 6",  "muon NS iteration 7",  "muon NS iteration 8",
    "muon NS iteration 9",  "muon NS iteration 10", "muon NS iteration 11", "muon NS iteration 12",
    "muon NS iteration 13", "muon NS iteration 14", "muon NS iteration 15", "muon NS iteration 16"};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void free_plan(Plan* p) {
    if (!p) return;
    if (p->arena) cudaFree(p->arena);
    if (p->nm_arena) cudaFree(p->nm_arena);
    delete p;
}

muon_status encode_map(EncodeTiledFn enc, CUtensorMap* map, void* base, int cols, int rows, int depth,
                       int box_cols, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                             static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MUON_OK : MUON_ERR_CUDA;
}

muon_status encode_map_ex(EncodeTiledFn enc, CUtensorMap* map, CUtensorMapDataType dtype, int esize, void* base,
                          int cols, int rows, int depth, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    const cuuint32_t rank = depth > 0 ? 3 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(depth > 0 ? depth : 1)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esize,
                             static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows) * esize};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MUON_OK : MUON_ERR_CUDA;
}

// fp32 weight (or O) matrix in its stored r x c layout, 32 x 32 boxes, 128B swizzle.
muon_status encode_f32_map(EncodeTiledFn enc, CUtensorMap* map, float* base, int rows, int cols) {
    return encode_map_ex(enc, map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, rows, 0, 32, 32,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

// CTA-pair tiling: Gram/poly tiles per matrix (column steps q, row pairs 0..q) and their
// executed flops; axpy tiles per matrix (row pairs x 256-column tiles).  Gram/poly with an even
// block count: 256 x 256 tiles, the diagonal ones included.  With an odd count: 256 x 256 tiles
// off the diagonal (row pair rp x column blocks 2q-1, 2q) and each even diagonal block as an
// M = 128, N = 128 tile.  An axpy row pair whose second block does not exist (odd row_blocks,
// last pair) runs as M = 128 tiles.
int pair_col_pairs(int row_blocks) { return (row_blocks + 1) / 2; }
int pair_sym_tiles(int row_blocks) {
    const int Q = pair_col_pairs(row_blocks);
    return Q * (Q + 1) / 2;
}
double pair_rows(int row_blocks, int rp) { return 2 * rp + 1 < row_blocks ? 256.0 : 128.0; }
double pair_sym_exec_flops(int row_blocks, int K) {
    double f = 0.0;
    const bool odd = (row_blocks & 1) != 0;
    for (int q = 0; q < pair_col_pairs(row_blocks); ++q)
        for (int rp = 0; rp <= q; ++rp) f += (odd && rp == q ? 2.0 * 128 * 128 : 2.0 * 256 * 256) * K;
    return f;
}
double pair_axpy_exec_flops(int row_blocks, int n, int K) {
    double f = 0.0;
    for (int c0 = 0; c0 < n; c0 += 256) {
        const int ncols = (n - c0 > 128) ? 256 : 128;
        for (int rp = 0; rp < pair_col_pairs(row_blocks); ++rp) f += 2.0 * pair_rows(row_blocks, rp) * ncols * K;
    }
    return f;
}

// Host-only part of planning: shape classes, arena layout, tile counts.
struct Layout {
    std::vector<size_t> offX0, offX1, offA, offB, off_dbg;
    size_t off_pmaps = 0, off_dmaps = 0;
    size_t bf16_end = 0, off_inv = 0, off_nrm = 0, off_asp = 0, off_cnt = 0, off_dt = 0,
           off_part = 0, total = 0;
    int momentum_ctas = 0;
    long long sym_tiles = 0, axpy_tiles = 0;
    double ns_exec_flops_per_iter = 0.0;
};

void compute_layout(Plan* P, const muon_shape* shapes, int n, bool keep_o, Layout* L) {
    P->shapes.assign(shapes, shapes + n);
    P->mat_class.resize(n);
    P->mat_slot.resize(n);
    for (int i = 0; i < n; ++i) {
        const int r = shapes[i].rows, c = shapes[i].cols;
        const int tr = r > c ? 1 : 0;
        const int m = tr ? c : r, nn = tr ? r : c;
        int ci = -1;
        for (size_t k = 0; k < P->classes.size(); ++k)
            if (P->classes[k].m == m && P->classes[k].n == nn && P->classes[k].transposed == tr) {
                ci = static_cast<int>(k);
                break;
            }
        if (ci < 0) {
            ClassPlan cp;
            cp.m = m;
            cp.n = nn;
            cp.transposed = tr;
            P->classes.push_back(cp);
            ci = static_cast<int>(P->classes.size()) - 1;
        }
        P->mat_class[i] = ci;
        P->mat_slot[i] = static_cast<int>(P->classes[ci].mats.size());
        P->classes[ci].mats.push_back(i);
    }
    for (auto& cp : P->classes)
        for (int i : cp.mats) P->order.push_back(i);
    P->position.resize(n);
    for (int k = 0; k < n; ++k) P->position[P->order[k]] = k;

    size_t off = 0;
    for (auto& cp : P->classes) {
        const size_t G = cp.mats.size();
        const size_t xb = G * static_cast<size_t>(cp.m) * cp.n * 2;
        const size_t ab = G * static_cast<size_t>(cp.m) * cp.m * 2;
        L->offX0.push_back(off); off = align_up(off + xb, 1024);
        L->offX1.push_back(off); off = align_up(off + xb, 1024);
        L->offA.push_back(off); off = align_up(off + ab, 1024);
        L->offB.push_back(off); off = align_up(off + ab, 1024);
        cp.row_blocks = (cp.m + kBM - 1) / kBM;
        cp.col_tiles = (cp.n + kBN - 1) / kBN;
        cp.col_pairs = pair_col_pairs(cp.row_blocks);
        cp.sym_pair_tiles = pair_sym_tiles(cp.row_blocks);
        cp.axpy_pair_tiles = cp.col_pairs * cp.col_tiles;
        const double m = cp.m, nn = cp.n;
        P->ns_flops_per_iter += static_cast<double>(G) * (3.0 * m * m * nn + m * m * m);
        L->ns_exec_flops_per_iter += static_cast<double>(G) *
            (pair_sym_exec_flops(cp.row_blocks, cp.n) + pair_sym_exec_flops(cp.row_blocks, cp.m) +
             pair_axpy_exec_flops(cp.row_blocks, cp.n, cp.m));
        L->sym_tiles += static_cast<long long>(G) * cp.sym_pair_tiles;
        L->axpy_tiles += static_cast<long long>(G) * cp.axpy_pair_tiles;
        P->elem_bytes += static_cast<double>(G) * m * nn * 22.0;
    }
    L->bf16_end = off;
    L->off_inv = off; off = align_up(off + n * sizeof(float), 256);
    L->off_nrm = off; off = align_up(off + n * sizeof(float), 256);
    L->off_asp = off; off = align_up(off + n * sizeof(float), 256);
    L->off_cnt = off; off = align_up(off + n * sizeof(unsigned int), 256);
    L->off_dt = off; off = align_up(off + n * sizeof(float*), 256);
    L->off_pmaps = off; off = align_up(off + n * sizeof(CUtensorMap), 256);
    L->off_dmaps = off; off = align_up(off + n * sizeof(CUtensorMap), 256);
    // one partial per momentum CTA of the largest launch chunk
    size_t max_tiles = 0, chunk_tiles = 0;
    for (int k = 0; k < n; ++k) {
        if (k % kMomentumMaxMats == 0) chunk_tiles = 0;
        const muon_shape& s = shapes[P->order[k]];
        const size_t t = static_cast<size_t>((s.rows + kMomTile - 1) / kMomTile) *
                         ((s.cols + kMomTile - 1) / kMomTile);
        chunk_tiles += t;
        L->momentum_ctas += static_cast<int>(t);
        if (chunk_tiles > max_tiles) max_tiles = chunk_tiles;
    }
    L->off_part = off; off = align_up(off + max_tiles * sizeof(float), 256);
    if (keep_o) {
        for (int i = 0; i < n; ++i) {
            L->off_dbg.push_back(off);
            off = align_up(off + static_cast<size_t>(shapes[i].rows) * shapes[i].cols * sizeof(float), 256);
        }
    }
    L->total = off;
}

int launches_for(const Plan* P, int ns_steps) {
    const int n = static_cast<int>(P->shapes.size());
    const int chunks = (n + kMomentumMaxMats - 1) / kMomentumMaxMats;
    const int groups = (static_cast<int>(P->classes.size()) + kMaxClasses - 1) / kMaxClasses;
    return ns_steps == 0 ? 2 * chunks : chunks + 3 * ns_steps * groups;
}

muon_status build_plan(Context* ctx, const muon_shape* shapes, int n, Plan** out) {
    Plan* P = new Plan();
    Layout L;
    compute_layout(P, shapes, n, (ctx->debug & MUON_DEBUG_KEEP_O) != 0, &L);
    P->arena_bytes = L.total;
    if (cudaMalloc(&P->arena, L.total) != cudaSuccess) {
        cudaGetLastError();
        P->arena = nullptr;
        free_plan(P);
        return MUON_ERR_OUT_OF_MEMORY;
    }
    char* a = P->arena;
    P->workspace_bf16 = a;
    P->workspace_bf16_bytes = L.bf16_end;
    for (size_t k = 0; k < P->classes.size(); ++k) {
        ClassPlan& cp = P->classes[k];
        cp.X[0] = reinterpret_cast<__nv_bfloat16*>(a + L.offX0[k]);
        cp.X[1] = reinterpret_cast<__nv_bfloat16*>(a + L.offX1[k]);
        cp.A = reinterpret_cast<__nv_bfloat16*>(a + L.offA[k]);
        cp.B = reinterpret_cast<__nv_bfloat16*>(a + L.offB[k]);
        const int G = static_cast<int>(cp.mats.size());
        muon_status st = MUON_OK;
        for (int pp = 0; pp < 2 && st == MUON_OK; ++pp) {
            st = encode_map(ctx->encode, &cp.tmXk[pp], cp.X[pp], cp.n, cp.m, G, kBK, kBM);
        }
        if (st == MUON_OK) st = encode_map(ctx->encode, &cp.tmAk, cp.A, cp.m, cp.m, G, kBK, kBM);
        if (st == MUON_OK) st = encode_map(ctx->encode, &cp.tmBk, cp.B, cp.m, cp.m, G, kBK, kBM);
        const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        for (int pp = 0; pp < 2 && st == MUON_OK; ++pp) {
            st = encode_map_ex(ctx->encode, &cp.tmXk64[pp], bf, 2, cp.X[pp], cp.n, cp.m, G, kBK, 64,
                               CU_TENSOR_MAP_SWIZZLE_128B);
            if (st == MUON_OK)
                st = encode_map_ex(ctx->encode, &cp.tmXmn128[pp], bf, 2, cp.X[pp], cp.n, cp.m, G, 64, kPairBK,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
            if (st == MUON_OK)
                st = encode_map_ex(ctx->encode, &cp.epiX64[pp], bf, 2, cp.X[pp], cp.n, cp.m, G, 64, 32,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (st == MUON_OK)
            st = encode_map_ex(ctx->encode, &cp.tmAk64, bf, 2, cp.A, cp.m, cp.m, G, kBK, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st == MUON_OK)
            st = encode_map_ex(ctx->encode, &cp.tmBk64, bf, 2, cp.B, cp.m, cp.m, G, kBK, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st == MUON_OK)
            st = encode_map_ex(ctx->encode, &cp.epiA64, bf, 2, cp.A, cp.m, cp.m, G, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st == MUON_OK)
            st = encode_map_ex(ctx->encode, &cp.epiB64, bf, 2, cp.B, cp.m, cp.m, G, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != MUON_OK) {
            free_plan(P);
            return st;
        }
    }
    P->inv_norm = reinterpret_cast<float*>(a + L.off_inv);
    P->norms = reinterpret_cast<float*>(a + L.off_nrm);
    P->aspect = reinterpret_cast<float*>(a + L.off_asp);
    P->counters = reinterpret_cast<unsigned int*>(a + L.off_cnt);
    P->dbg_table = reinterpret_cast<float**>(a + L.off_dt);
    P->partials = reinterpret_cast<float*>(a + L.off_part);

    // per-matrix constants, indexed by class-ordered position
    std::vector<float> asp(n);
    std::vector<float*> dbg(n, nullptr);
    for (int k = 0; k < n; ++k) {
        const muon_shape& s = shapes[P->order[k]];
        const double ratio = static_cast<double>(s.rows) / s.cols;
        asp[k] = static_cast<float>(std::sqrt(ratio > 1.0 ? ratio : 1.0));
        if (!L.off_dbg.empty()) dbg[k] = reinterpret_cast<float*>(a + L.off_dbg[P->order[k]]);
    }
    P->dbg_O.assign(n, nullptr);
    for (int i = 0; i < n; ++i)
        if (!L.off_dbg.empty()) P->dbg_O[i] = reinterpret_cast<float*>(a + L.off_dbg[i]);
    P->p_maps = reinterpret_cast<CUtensorMap*>(a + L.off_pmaps);
    P->mapped_p.assign(n, nullptr);
    if (!L.off_dbg.empty()) {
        P->dbg_maps = reinterpret_cast<CUtensorMap*>(a + L.off_dmaps);
        std::vector<CUtensorMap> dm(n);
        for (int k = 0; k < n; ++k) {
            const int i = P->order[k];
            if (encode_f32_map(ctx->encode, &dm[k], P->dbg_O[i], shapes[i].rows, shapes[i].cols) != MUON_OK) {
                free_plan(P);
                return MUON_ERR_CUDA;
            }
        }
        if (cudaMemcpy(P->dbg_maps, dm.data(), n * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess) {
            free_plan(P);
            return MUON_ERR_CUDA;
        }
    }
    bool ok = cudaMemcpy(P->aspect, asp.data(), n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(P->dbg_table, dbg.data(), n * sizeof(float*), cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(P->counters, 0, n * sizeof(unsigned int)) == cudaSuccess;
    ok = ok && cudaMemset(P->inv_norm, 0, n * sizeof(float)) == cudaSuccess;
    ok = ok && cudaMemset(P->norms, 0, n * sizeof(float)) == cudaSuccess;
    if (!ok) {
        free_plan(P);
        return MUON_ERR_CUDA;
    }
    *out = P;
    return MUON_OK;
}

// Workspace of the NorMuon pass: bf16 O per matrix, their tensor maps, the per-row
// step sizes and the per-matrix reduction state.  Built once per plan.
muon_status ensure_normuon(Context* ctx, Plan* P) {
    if (P->nm_arena) return MUON_OK;
    const int n = static_cast<int>(P->shapes.size());
    std::vector<size_t> off_o(n);
    size_t off = 0;
    long long total_rows = 0;
    size_t max_ctas = 0, chunk_ctas = 0;
    P->row_base.assign(n, 0);
    for (int k = 0; k < n; ++k) {
        const muon_shape& s = P->shapes[P->order[k]];
        P->row_base[k] = static_cast<int>(total_rows);
        total_rows += s.rows;
        if (k % kMomentumMaxMats == 0) chunk_ctas = 0;
        chunk_ctas += (s.rows + kNormRowsPerCta - 1) / kNormRowsPerCta;
        if (chunk_ctas > max_ctas) max_ctas = chunk_ctas;
    }
    for (int i = 0; i < n; ++i) {
        off_o[i] = off;
        off = align_up(off + static_cast<size_t>(P->shapes[i].rows) * P->shapes[i].cols * sizeof(__nv_bfloat16), 1024);
    }
    const size_t off_maps = off; off = align_up(off + n * sizeof(CUtensorMap), 256);
    const size_t off_step = off; off = align_up(off + static_cast<size_t>(total_rows) * sizeof(float), 256);
    const size_t off_rb = off; off = align_up(off + n * sizeof(int), 256);
    const size_t off_part = off; off = align_up(off + max_ctas * 2 * sizeof(double), 256);
    const size_t off_cnt = off; off = align_up(off + n * sizeof(unsigned int), 256);
    const size_t off_ratio = off; off = align_up(off + n * sizeof(float), 256);
    char* a = nullptr;
    if (cudaMalloc(&a, off) != cudaSuccess) {
        cudaGetLastError();
        return MUON_ERR_OUT_OF_MEMORY;
    }
    P->o_bufs.resize(n);
    for (int i = 0; i < n; ++i) P->o_bufs[i] = reinterpret_cast<__nv_bfloat16*>(a + off_o[i]);
    P->o_maps = reinterpret_cast<CUtensorMap*>(a + off_maps);
    P->nm_step = reinterpret_cast<float*>(a + off_step);
    P->nm_row_base = reinterpret_cast<int*>(a + off_rb);
    P->nm_partials = reinterpret_cast<double*>(a + off_part);
    P->nm_counters = reinterpret_cast<unsigned int*>(a + off_cnt);
    P->nm_ratio = reinterpret_cast<float*>(a + off_ratio);
    std::vector<CUtensorMap> om(n);
    for (int k = 0; k < n; ++k) {
        const int i = P->order[k];
        if (encode_map_ex(ctx->encode, &om[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P->o_bufs[i], P->shapes[i].cols,
                          P->shapes[i].rows, 0, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) != MUON_OK) {
            cudaFree(a);
            return MUON_ERR_CUDA;
        }
    }
    bool ok = cudaMemcpy(P->o_maps, om.data(), n * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(P->nm_row_base, P->row_base.data(), n * sizeof(int), cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(P->nm_counters, 0, n * sizeof(unsigned int)) == cudaSuccess;
    if (!ok) {
        cudaFree(a);
        return MUON_ERR_CUDA;
    }
    P->nm_arena = a;
    return MUON_OK;
}

// The NorMuon arguments of a step (nullptr for a plain Muon step).
struct NormuonCall {
    float* const* second_moments;  // by step index
    float beta2, eps;
};

muon_status check_shapes(const muon_shape* shapes, int n) {
    for (int i = 0; i < n; ++i) {
        const int r = shapes[i].rows, c = shapes[i].cols;
        if (r < 8 || c < 8 || (r % 8) != 0 || (c % 8) != 0 || r > 65536 || c > 65536)
            return MUON_ERR_UNSUPPORTED_SHAPE;
    }
    return MUON_OK;
}

bool same_shapes(const Plan* P, const muon_shape* shapes, int n) {
    if (!P || static_cast<int>(P->shapes.size()) != n) return false;
    for (int i = 0; i < n; ++i)
        if (P->shapes[i].rows != shapes[i].rows || P->shapes[i].cols != shapes[i].cols) return false;
    return true;
}

cudaEvent_t take_event(Context* ctx) {
    if (!ctx->event_pool.empty()) {
        cudaEvent_t e = ctx->event_pool.back();
        ctx->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Runs `launch` on `stream`, bracketed by timing events when enabled.
template <typename F>
muon_status timed_launch(Context* ctx, int kind, cudaStream_t stream, F&& launch) {
    cudaEvent_t a = nullptr, b = nullptr;
    const bool timing = (ctx->debug & MUON_DEBUG_TIME_KERNELS) != 0;
    if (timing) {
        a = take_event(ctx);
        b = take_event(ctx);
        cudaEventRecord(a, stream);
    }
    const cudaError_t e = launch();
    if (timing) {
        cudaEventRecord(b, stream);
        ctx->pending.push_back({kind, a, b});
    }
    ctx->info.launches += 1;
    return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

void fill_momentum_mat(const Plan* P, int pos, float* const params[], const float* const grads[],
                       float* const moms[], int tile_begin, MomentumMat* M) {
    const int i = P->order[pos];
    const ClassPlan& cp = P->classes[P->mat_class[i]];
    M->g = grads[i];
    M->mom = moms[i];
    M->p = params[i];
    M->x0 = cp.X[0] + static_cast<size_t>(P->mat_slot[i]) * cp.m * cp.n;
    M->rows = P->shapes[i].rows;
    M->cols = P->shapes[i].cols;
    M->transposed = cp.transposed;
    M->tiles_x = (M->cols + kMomTile - 1) / kMomTile;
    M->ntiles = M->tiles_x * ((M->rows + kMomTile - 1) / kMomTile);
    M->tile_begin = tile_begin;
    M->gidx = pos;
}

}  // namespace

extern "C" {

const char* muon_status_string(muon_status s) {
    switch (s) {
        case MUON_OK: return "ok";
        case MUON_ERR_INVALID_ARG: return "invalid argument";
        case MUON_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (rows and cols must be >= 8 and multiples of 8)";
        case MUON_ERR_MISALIGNED: return "matrix pointer not 16-byte aligned";
        case MUON_ERR_NOT_INITIALIZED: return "muon_init has not succeeded";
        case MUON_ERR_CUDA: return "CUDA call failed";
        case MUON_ERR_OUT_OF_MEMORY: return "workspace allocation failed";
        case MUON_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
        case MUON_ERR_DEVICE_BOUNDS: return "a kernel refused a tile list that does not match its classes";
        case MUON_ERR_UNSUPPORTED_DEVICE: return "no sm_103 CUDA device";
        case MUON_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of muon_momentum_norm_noalloc";
    }
    return "unknown status";
}

muon_status muon_destroy(void) {
    if (!g_ctx) return MUON_OK;
    cudaDeviceSynchronize();
    for (Plan* P : g_ctx->plans) free_plan(P);
    for (auto& pt : g_ctx->pending) {
        cudaEventDestroy(pt.a);
        cudaEventDestroy(pt.b);
    }
    for (auto e : g_ctx->event_pool) cudaEventDestroy(e);
    if (g_ctx->status) cudaFree(g_ctx->status);
    delete g_ctx;
    g_ctx = nullptr;
    return MUON_OK;
}

muon_status muon_init(const muon_config* cfg) {
    // validate the configuration before touching the device
    std::vector<double> coeffs;
    if (cfg && cfg->coeffs) {
        if (cfg->n_coeff_rows < 1 || cfg->n_coeff_rows > kMaxCoeffRows) return MUON_ERR_INVALID_ARG;
        coeffs.assign(cfg->coeffs, cfg->coeffs + 3 * cfg->n_coeff_rows);
        for (double v : coeffs)
            if (!std::isfinite(v)) return MUON_ERR_INVALID_ARG;
    } else {
        for (int k = 0; k < 5; ++k) {
            coeffs.push_back(3.4445);
            coeffs.push_back(-4.7750);
            coeffs.push_back(2.0315);
        }
    }
    if (cfg && cfg->momentum_mode != MUON_MOMENTUM_SGD_NESTEROV && cfg->momentum_mode != MUON_MOMENTUM_EMA)
        return MUON_ERR_INVALID_ARG;
    if (cfg && !(std::isfinite(cfg->eps) && std::isfinite(cfg->wait_timeout_s))) return MUON_ERR_INVALID_ARG;

    muon_destroy();
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MUON_ERR_UNSUPPORTED_DEVICE;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return MUON_ERR_UNSUPPORTED_DEVICE;
    }
    if (!(prop.major == 10 && prop.minor == 3)) return MUON_ERR_UNSUPPORTED_DEVICE;

    Context* ctx = new Context();
    ctx->device = dev;
    ctx->sm_count = prop.multiProcessorCount;
    ctx->coeffs = coeffs;
    ctx->n_rows = static_cast<int>(coeffs.size() / 3);
    if (cfg) {
        if (cfg->eps > 0) ctx->eps = cfg->eps;
        ctx->momentum_mode = cfg->momentum_mode;
        ctx->debug = cfg->debug_flags;
        if (cfg->wait_timeout_s > 0)
            ctx->timeout_ns = static_cast<unsigned long long>(cfg->wait_timeout_s * 1e9);
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        delete ctx;
        return MUON_ERR_CUDA;
    }
    ctx->encode = reinterpret_cast<EncodeTiledFn>(fn);
    if (ns_pair_prepare(&ctx->max_clusters) != cudaSuccess ||
        ctx->max_clusters < 1 ||
        cudaMalloc(&ctx->status, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemset(ctx->status, 0, sizeof(unsigned int)) != cudaSuccess) {
        cudaGetLastError();
        if (ctx->status) cudaFree(ctx->status);
        delete ctx;
        return MUON_ERR_CUDA;
    }
    g_ctx = ctx;
    return MUON_OK;
}

static muon_status step_impl(float* const params[], const float* const grads[], float* const momentum_bufs[],
                             const muon_shape shapes[], int n_mats, float lr, float beta, int nesterov,
                             int ns_steps, muon_stream_t stream_, const NormuonCall* nm) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (n_mats < 0) return MUON_ERR_INVALID_ARG;
    if (n_mats == 0) {
        ctx->info = muon_step_info{};
        return MUON_OK;
    }
    if (!params || !grads || !momentum_bufs || !shapes) return MUON_ERR_INVALID_ARG;
    if (ns_steps < 0 || ns_steps > ctx->n_rows) return MUON_ERR_INVALID_ARG;
    if (!std::isfinite(lr) || !std::isfinite(beta)) return MUON_ERR_INVALID_ARG;
    if (check_shapes(shapes, n_mats) != MUON_OK) return MUON_ERR_UNSUPPORTED_SHAPE;
    for (int i = 0; i < n_mats; ++i) {
        if (!params[i] || !grads[i] || !momentum_bufs[i]) return MUON_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(params[i]) | reinterpret_cast<uintptr_t>(grads[i]) |
             reinterpret_cast<uintptr_t>(momentum_bufs[i])) & 15u)
            return MUON_ERR_MISALIGNED;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    NvtxScope step_range(nm ? "muon_step_normuon" : "muon_step");

    // the plan of this shape list: reused when cached (moved to the front), else built, dropping
    // the least recently used one when kMaxPlans are held
    Plan* P = nullptr;
    for (size_t k = 0; k < ctx->plans.size(); ++k) {
        if (same_shapes(ctx->plans[k], shapes, n_mats)) {
            P = ctx->plans[k];
            ctx->plans.erase(ctx->plans.begin() + static_cast<long>(k));
            break;
        }
    }
    if (!P) {
        if (static_cast<int>(ctx->plans.size()) >= kMaxPlans) {
            // work of earlier steps, on any stream, may still use the dropped workspace
            if (cudaDeviceSynchronize() != cudaSuccess) return MUON_ERR_CUDA;
            if (ctx->last == ctx->plans.back()) ctx->last = nullptr;
            free_plan(ctx->plans.back());
            ctx->plans.pop_back();
        }
        const muon_status st = build_plan(ctx, shapes, n_mats, &P);
        if (st != MUON_OK) return st;
    }
    ctx->plans.insert(ctx->plans.begin(), P);
    ctx->last = P;
    if (nm) {
        const muon_status st = ensure_normuon(ctx, P);
        if (st != MUON_OK) return st;
    }
    ctx->info = muon_step_info{};
    ctx->info.n_classes = static_cast<int>(P->classes.size());
    ctx->info.workspace_bytes = static_cast<long long>(P->arena_bytes);
    ctx->info.ns_alg_flops = P->ns_flops_per_iter * ns_steps;
    ctx->info.elementwise_alg_bytes = P->elem_bytes;

    if (ctx->debug & MUON_DEBUG_POISON_WORKSPACE) {
        if (cudaMemsetAsync(P->workspace_bf16, 0xFF, P->workspace_bf16_bytes, stream) != cudaSuccess)
            return MUON_ERR_CUDA;
    }

    // ---- momentum + norm (chunks of kMomentumMaxMats matrices, class order)
    static MomentumParams mp;  // ~12 KiB: kept off the stack
    nvtxRangePushA("muon momentum+norm");
    for (int base = 0; base < n_mats; base += kMomentumMaxMats) {
        const int cnt = std::min(kMomentumMaxMats, n_mats - base);
        std::memset(&mp, 0, sizeof(mp));
        int tiles = 0;
        for (int k = 0; k < cnt; ++k) {
            fill_momentum_mat(P, base + k, params, grads, momentum_bufs, tiles, &mp.mats[k]);
            tiles += mp.mats[k].ntiles;
        }
        mp.nmats = cnt;
        mp.total_tiles = tiles;
        mp.beta = beta;
        mp.nesterov = nesterov ? 1 : 0;
        mp.mode = ctx->momentum_mode;
        mp.eps = static_cast<float>(ctx->eps);
        mp.partials = P->partials;
        mp.counters = P->counters;
        mp.inv_norm = P->inv_norm;
        mp.norms = P->norms;
        const muon_status st = timed_launch(ctx, 0, stream, [&] { return launch_momentum_norm(mp, stream); });
        if (st != MUON_OK) {
            nvtxRangePop();
            return st;
        }
    }
    nvtxRangePop();

    const bool keep_o = (ctx->debug & MUON_DEBUG_KEEP_O) != 0;
    if (ns_steps == 0) {
        static UpdateParams up;
        for (int base = 0; base < n_mats; base += kMomentumMaxMats) {
            const int cnt = std::min(kMomentumMaxMats, n_mats - base);
            std::memset(&up, 0, sizeof(up));
            int tiles = 0;
            for (int k = 0; k < cnt; ++k) {
                fill_momentum_mat(P, base + k, params, grads, momentum_bufs, tiles, &up.mats[k]);
                tiles += up.mats[k].ntiles;
            }
            up.nmats = cnt;
            up.total_tiles = tiles;
            up.inv_norm = P->inv_norm;
            up.aspect = P->aspect;
            up.lr = lr;
            up.dbg_O = keep_o ? P->dbg_table : nullptr;
            const muon_status st = timed_launch(ctx, 5, stream, [&] { return launch_update(up, stream); });
            if (st != MUON_OK) return st;
        }
        return MUON_OK;
    }

    // ---- Newton-Schulz iterations: per group of <= kMaxClasses classes
    const int nclass = static_cast<int>(P->classes.size());
    // fp32 weight maps of the fused update: re-encoded only when the params change
    // (the NorMuon pass updates the weights in its own kernel)
    bool changed = false;
    for (int i = 0; i < n_mats && !changed && !nm; ++i) changed = P->mapped_p[i] != params[i];
    if (changed) {
        std::vector<CUtensorMap> pm(n_mats);
        for (int k = 0; k < n_mats; ++k) {
            const int i = P->order[k];
            if (encode_f32_map(ctx->encode, &pm[k], params[i], shapes[i].rows, shapes[i].cols) != MUON_OK)
                return MUON_ERR_CUDA;
        }
        // launches already enqueued, on any stream, may still read the previous maps
        if (cudaDeviceSynchronize() != cudaSuccess) return MUON_ERR_CUDA;
        if (cudaMemcpy(P->p_maps, pm.data(), n_mats * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess)
            return MUON_ERR_CUDA;
        P->mapped_p.assign(params, params + n_mats);
    }
    static PairParams pp;  // ~5 KiB: kept off the stack
    // step position of every class's first matrix (positions are class-ordered)
    std::vector<int> class_base(nclass, 0);
    for (int c = 1; c < nclass; ++c)
        class_base[c] = class_base[c - 1] + static_cast<int>(P->classes[c - 1].mats.size());
    for (int it = 0; it < ns_steps; ++it) {
        NvtxScope iter_range(kIterRange[it]);
        const double* row = &ctx->coeffs[3 * it];
        const int pin = it & 1, pout = pin ^ 1;
        const bool last = (it == ns_steps - 1);
        for (int g0 = 0; g0 < nclass; g0 += kMaxClasses) {
            const int gc = std::min(kMaxClasses, nclass - g0);
            for (int mode = MODE_GRAM; mode <= MODE_AXPY; ++mode) {
                std::memset(&pp, 0, sizeof(pp));
                const int eff_mode =
                    (mode == MODE_AXPY && last) ? (nm ? MODE_AXPY_O : MODE_AXPY_FINAL) : mode;
                pp.mode = eff_mode;
                pp.nclasses = gc;
                pp.first_iter = (it == 0 && mode != MODE_POLY) ? 1 : 0;
                pp.ca = static_cast<float>(row[0]);
                pp.cb = static_cast<float>(row[1]);
                pp.cc = static_cast<float>(row[2]);
                pp.inv_norm = P->inv_norm;
                pp.aspect = P->aspect;
                pp.lr = lr;
                pp.p_maps = P->p_maps;
                pp.dbg_maps = keep_o ? P->dbg_maps : nullptr;
                pp.o_maps = P->o_maps;
                pp.status = ctx->status;
                pp.timeout_ns = ctx->timeout_ns;
                pp.inject_lost_load = ((ctx->debug & MUON_DEBUG_INJECT_LOST_LOAD) && !ctx->injected &&
                                       it == 0 && mode == MODE_GRAM && g0 == 0)
                                          ? 1
                                          : 0;
                if (pp.inject_lost_load) ctx->injected = true;
                const bool bad_tiles = (ctx->debug & MUON_DEBUG_INJECT_BAD_TILES) && !ctx->injected_bad && it == 0 &&
                                       mode == MODE_GRAM && g0 == 0;
                if (bad_tiles) ctx->injected_bad = true;
                // The clusters take tiles round-robin in launch order, so the classes whose tiles
                // run longest (deepest K) go first and the last wave is made of the shortest
                // tiles; within a class the tiles of one matrix stay adjacent (their operands
                // share L2).
                int ord[kMaxClasses];
                for (int k = 0; k < gc; ++k) ord[k] = g0 + k;
                auto depth = [&](int c) { return mode == MODE_GRAM ? P->classes[c].n : P->classes[c].m; };
                std::stable_sort(ord, ord + gc, [&](int x, int y) { return depth(x) > depth(y); });
                int tiles = 0;
                for (int k = 0; k < gc; ++k) {
                    const ClassPlan& cp = P->classes[ord[k]];
                    PairClass& C = pp.cls[k];
                    const int G = static_cast<int>(cp.mats.size());
                    C.m = cp.m;
                    C.n = cp.n;
                    C.nmats = G;
                    C.tile_begin = tiles;
                    C.row_blocks = cp.row_blocks;
                    C.transposed = cp.transposed;
                    C.mat_base = class_base[ord[k]];
                    if (mode == MODE_GRAM) {
                        C.tiles_per_mat = cp.sym_pair_tiles;
                        C.col_groups = cp.col_pairs;
                        C.k_blocks = (cp.n + kPairBK - 1) / kPairBK;
                        pp.tmA[k] = cp.tmXk[pin];
                        pp.tmB[k] = cp.tmXk64[pin];
                        pp.tmA64[k] = cp.tmXk64[pin];
                        pp.tmOut[k] = cp.epiA64;
                    } else if (mode == MODE_POLY) {
                        C.tiles_per_mat = cp.sym_pair_tiles;
                        C.col_groups = cp.col_pairs;
                        C.k_blocks = (cp.m + kPairBK - 1) / kPairBK;
                        pp.tmA[k] = cp.tmAk;
                        pp.tmB[k] = cp.tmAk64;
                        pp.tmA64[k] = cp.tmAk64;
                        pp.tmIn[k] = cp.epiA64;
                        pp.tmOut[k] = cp.epiB64;
                    } else {
                        C.tiles_per_mat = cp.axpy_pair_tiles;
                        C.col_groups = cp.col_tiles;
                        C.k_blocks = (cp.m + kPairBK - 1) / kPairBK;
                        pp.tmA[k] = cp.tmBk;
                        pp.tmB[k] = cp.tmXmn128[pin];
                        pp.tmA64[k] = cp.tmBk64;
                        pp.tmOut[k] = cp.epiX64[pout];
                    }
                    tiles += C.tiles_per_mat * G;
                }
                pp.total_tiles = bad_tiles ? tiles + 1 : tiles;
                const int clusters = std::min(tiles, ctx->max_clusters);
                const int kind = eff_mode == MODE_GRAM ? 1 : eff_mode == MODE_POLY ? 2 : eff_mode == MODE_AXPY ? 3
                                 : eff_mode == MODE_AXPY_O ? 6 : 4;
                const muon_status st =
                    timed_launch(ctx, kind, stream, [&] { return launch_ns_pair(pp, clusters, stream); });
                if (st != MUON_OK) return st;
            }
        }
    }
    if (nm) {
        // ---- NorMuon: per-row statistics and ratio, then the weight update
        NvtxScope nm_range("muon NorMuon rows+update");
        static NormuonParams np;  // ~12 KiB: kept off the stack
        for (int base = 0; base < n_mats; base += kMomentumMaxMats) {
            const int cnt = std::min(kMomentumMaxMats, n_mats - base);
            std::memset(&np, 0, sizeof(np));
            int ctas = 0, tiles = 0;
            for (int k = 0; k < cnt; ++k) {
                const int pos = base + k;
                const int i = P->order[pos];
                NormuonMat& M = np.mats[k];
                M.O = P->o_bufs[i];
                M.V = nm->second_moments[i];
                M.p = params[i];
                M.dbg = keep_o ? P->dbg_O[i] : nullptr;
                M.rows = shapes[i].rows;
                M.cols = shapes[i].cols;
                M.cta_begin = ctas;
                M.nctas = (M.rows + kNormRowsPerCta - 1) / kNormRowsPerCta;
                M.tile_begin = tiles;
                M.tiles_x = (M.cols + 63) / 64;
                M.pos = pos;
                ctas += M.nctas;
                tiles += M.tiles_x * ((M.rows + 63) / 64);
            }
            np.nmats = cnt;
            np.beta2 = nm->beta2;
            np.eps = nm->eps;
            np.lr = lr;
            np.aspect = P->aspect;
            np.step = P->nm_step;
            np.row_base = P->nm_row_base;
            np.partials = P->nm_partials;
            np.counters = P->nm_counters;
            np.ratio = P->nm_ratio;
            np.total = ctas;
            muon_status st = timed_launch(ctx, 7, stream, [&] { return launch_normuon_rows(np, stream); });
            if (st != MUON_OK) return st;
            np.total = tiles;
            st = timed_launch(ctx, 7, stream, [&] { return launch_normuon_update(np, stream); });
            if (st != MUON_OK) return st;
        }
    }
    return MUON_OK;
}

muon_status muon_step(float* const params[], const float* const grads[], float* const momentum_bufs[],
                      const muon_shape shapes[], int n_mats, float lr, float beta, int nesterov,
                      int ns_steps, muon_stream_t stream) {
    return step_impl(params, grads, momentum_bufs, shapes, n_mats, lr, beta, nesterov, ns_steps, stream, nullptr);
}

muon_status muon_step_normuon(float* const params[], const float* const grads[], float* const momentum_bufs[],
                              float* const second_moments[], const muon_shape shapes[], int n_mats, float lr,
                              float beta, int nesterov, int ns_steps, float beta2, float eps2,
                              muon_stream_t stream) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (n_mats < 0) return MUON_ERR_INVALID_ARG;
    if (n_mats == 0) return step_impl(params, grads, momentum_bufs, shapes, 0, lr, beta, nesterov, ns_steps, stream,
                                      nullptr);
    if (!second_moments || ns_steps < 1) return MUON_ERR_INVALID_ARG;
    if (!(beta2 >= 0.0f && beta2 < 1.0f) || !(eps2 >= 0.0f) || !std::isfinite(eps2)) return MUON_ERR_INVALID_ARG;
    for (int i = 0; i < n_mats; ++i) {
        if (!second_moments[i]) return MUON_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(second_moments[i]) & 3u) return MUON_ERR_MISALIGNED;
    }
    const NormuonCall nm{second_moments, beta2, eps2};
    return step_impl(params, grads, momentum_bufs, shapes, n_mats, lr, beta, nesterov, ns_steps, stream, &nm);
}

muon_status muon_partition(const muon_shape shapes[], int n_mats, int world, int owner_out[]) {
    if (world < 1 || n_mats < 0 || (n_mats > 0 && (!shapes || !owner_out))) return MUON_ERR_INVALID_ARG;
    if (check_shapes(shapes, n_mats) != MUON_OK) return MUON_ERR_UNSUPPORTED_SHAPE;
    std::vector<double> cost(n_mats);
    std::vector<int> idx(n_mats);
    for (int i = 0; i < n_mats; ++i) {
        const double m = std::min(shapes[i].rows, shapes[i].cols), n = std::max(shapes[i].rows, shapes[i].cols);
        cost[i] = 3.0 * m * m * n + m * m * m;
        idx[i] = i;
    }
    // largest first; equal costs keep their index order
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) { return cost[x] > cost[y]; });
    std::vector<double> load(world, 0.0);
    for (int i : idx) {
        int best = 0;
        for (int r = 1; r < world; ++r)
            if (load[r] < load[best]) best = r;
        owner_out[i] = best;
        load[best] += cost[i];
    }
    return MUON_OK;
}

muon_status muon_plan_query(const muon_shape shapes[], int n_mats, int ns_steps, muon_plan_info* out) {
    if (!out || n_mats < 0 || (n_mats > 0 && !shapes)) return MUON_ERR_INVALID_ARG;
    const int max_rows = g_ctx ? g_ctx->n_rows : kMaxCoeffRows;
    if (ns_steps < 0 || ns_steps > max_rows) return MUON_ERR_INVALID_ARG;
    if (check_shapes(shapes, n_mats) != MUON_OK) return MUON_ERR_UNSUPPORTED_SHAPE;
    std::memset(out, 0, sizeof(*out));
    if (n_mats == 0) return MUON_OK;
    Plan P;
    Layout L;
    compute_layout(&P, shapes, n_mats, g_ctx && (g_ctx->debug & MUON_DEBUG_KEEP_O), &L);
    out->n_classes = static_cast<int>(P.classes.size());
    out->launches = launches_for(&P, ns_steps);
    out->workspace_bytes = static_cast<long long>(L.total);
    out->ns_alg_flops = P.ns_flops_per_iter * ns_steps;
    out->ns_executed_flops = L.ns_exec_flops_per_iter * ns_steps;
    out->elementwise_alg_bytes = P.elem_bytes;
    out->momentum_ctas = L.momentum_ctas;
    out->sym_tiles = L.sym_tiles;
    out->axpy_tiles = L.axpy_tiles;
    return MUON_OK;
}

muon_status muon_get_status(muon_stream_t stream) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
    unsigned int st = 0;
    if (cudaMemcpy(&st, ctx->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
    if (st != 0 && cudaMemset(ctx->status, 0, sizeof(unsigned int)) != cudaSuccess) return MUON_ERR_CUDA;
    if (st & STATUS_TIMEOUT) return MUON_ERR_DEVICE_TIMEOUT;
    if (st & STATUS_BOUNDS) return MUON_ERR_DEVICE_BOUNDS;
    return MUON_OK;
}

muon_status muon_get_step_info(muon_step_info* out) {
    if (!g_ctx) return MUON_ERR_NOT_INITIALIZED;
    if (!out) return MUON_ERR_INVALID_ARG;
    *out = g_ctx->info;
    return MUON_OK;
}

muon_status muon_kernel_times(double* ms_out, int* launches_out, int n_kinds) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (n_kinds < 0 || n_kinds > kKinds || (n_kinds > 0 && (!ms_out || !launches_out)))
        return MUON_ERR_INVALID_ARG;
    muon_status result = MUON_OK;
    for (auto& pt : ctx->pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(pt.b) != cudaSuccess || cudaEventElapsedTime(&ms, pt.a, pt.b) != cudaSuccess) {
            cudaGetLastError();
            result = MUON_ERR_CUDA;
        }
        ctx->kind_ms[pt.kind] += ms;
        ctx->kind_launches[pt.kind] += 1;
        ctx->event_pool.push_back(pt.a);
        ctx->event_pool.push_back(pt.b);
    }
    ctx->pending.clear();
    for (int k = 0; k < n_kinds; ++k) {
        ms_out[k] = ctx->kind_ms[k];
        launches_out[k] = ctx->kind_launches[k];
    }
    for (int k = 0; k < kKinds; ++k) {
        ctx->kind_ms[k] = 0;
        ctx->kind_launches[k] = 0;
    }
    return result;
}

muon_status muon_debug_copy_ns_output(int mat, float* dst_device, muon_stream_t stream) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (!(ctx->debug & MUON_DEBUG_KEEP_O) || !ctx->last || !dst_device) return MUON_ERR_INVALID_ARG;
    Plan* P = ctx->last;
    if (mat < 0 || mat >= static_cast<int>(P->shapes.size())) return MUON_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(P->shapes[mat].rows) * P->shapes[mat].cols * sizeof(float);
    return cudaMemcpyAsync(dst_device, P->dbg_O[mat], bytes, cudaMemcpyDeviceToDevice,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MUON_OK
               : MUON_ERR_CUDA;
}

muon_status muon_debug_copy_norms(float* dst_host, int n) {
    Context* ctx = g_ctx;
    if (!ctx) return MUON_ERR_NOT_INITIALIZED;
    if (!ctx->last || !dst_host || n < 0 || n > static_cast<int>(ctx->last->shapes.size()))
        return MUON_ERR_INVALID_ARG;
    Plan* P = ctx->last;
    std::vector<float> tmp(P->shapes.size());
    if (cudaDeviceSynchronize() != cudaSuccess) return MUON_ERR_CUDA;
    if (cudaMemcpy(tmp.data(), P->norms, tmp.size() * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MUON_ERR_CUDA;
    for (int i = 0; i < n; ++i) dst_host[i] = tmp[P->position[i]];
    return MUON_OK;
}

}  // extern "C"
