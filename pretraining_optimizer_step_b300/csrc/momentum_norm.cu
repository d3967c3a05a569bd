// momentum_norm.cu -- the HBM-bound passes of the Muon step.
//
// momentum_norm_kernel: one fused pass over every matrix of the step
//   m' = beta m + g (stored back), u = nesterov ? g + beta m' : m'
//   (EMA mode: m' = beta m + (1-beta) g, u = nesterov ? (1-beta) g + beta m' : m'),
//   X0 = bf16(u) written in the oriented layout (transposed through shared
//   memory when rows > cols), and ||u||_F reduced deterministically: each CTA
//   writes the fp32 sum of its 64 x 64 tile, and the last CTA of a matrix (an
//   atomic ticket) adds the partials in index order in fp64 and publishes
//   1/(||u|| + eps).  The momentum form is the reading stated in muon.h; the
//   pages ("Cara Melatih ChatGPT Sendiri dengan Budget 50 Dolar", section
//   "2. Pengoptimal Muon") only name momentum as the first part of the method.
// update_kernel: the weight update p -= lr sqrt(max(1, r/c)) O for ns_steps = 0,
//   where O = X0 / (||u|| + eps).
#include "kernels.cuh"
#include "ptx.cuh"

namespace muon {

namespace {

__device__ __forceinline__ int find_mat(const MomentumMat* mats, int nmats, int tile) {
    int lo = 0, hi = nmats - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mats[mid].tile_begin <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
    uint2 r;
    r.x = *reinterpret_cast<uint32_t*>(&lo);
    r.y = *reinterpret_cast<uint32_t*>(&hi);
    return r;
}

}  // namespace

__global__ void __launch_bounds__(kMomThreads)
    momentum_norm_kernel(const __grid_constant__ MomentumParams P) {
    __shared__ float tile[kMomTile][kMomTile + 1];
    __shared__ float warp_sums[kMomThreads / 32];
    __shared__ double warp_sums_d[kMomThreads / 32];
    __shared__ int is_last;
    // the first Gram launch (launched for programmatic serialization) may start launching once
    // every CTA of this grid has started; it waits in its own prologue for this grid to finish
    griddep_launch();

    const int t = blockIdx.x;
    const int mi = find_mat(P.mats, P.nmats, t);
    const MomentumMat& M = P.mats[mi];
    const int local = t - M.tile_begin;
    const int ty = local / M.tiles_x, tx = local - ty * M.tiles_x;
    const int r0 = ty * kMomTile, c0 = tx * kMomTile;
    const int tid = threadIdx.x;
    const int cq = tid & 15;   // column quad within the tile
    const int rr = tid >> 4;   // 0..15
    const float beta = P.beta;
    const float omb = 1.0f - beta;

    float ss = 0.0f;
    // all four rows' loads are issued before the first store (the compiler cannot prove that g and
    // the momentum buffer do not alias, so it would not move a load above an earlier store)
    float4 gv[4], mv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = r0 + rr + 16 * k;
        const int col = c0 + 4 * cq;
        gv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        mv[k] = gv[k];
        if (row < M.rows && col < M.cols) {
            const size_t off = static_cast<size_t>(row) * M.cols + col;
            gv[k] = __ldcs(reinterpret_cast<const float4*>(M.g + off));
            mv[k] = __ldcs(reinterpret_cast<const float4*>(M.mom + off));
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = r0 + rr + 16 * k;
        const int col = c0 + 4 * cq;
        float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < M.rows && col < M.cols) {
            const size_t off = static_cast<size_t>(row) * M.cols + col;
            const float4 g4 = gv[k];
            const float4 m4 = mv[k];
            float4 n4;
            if (P.mode == 1) {
                n4.x = fmaf(beta, m4.x, omb * g4.x);
                n4.y = fmaf(beta, m4.y, omb * g4.y);
                n4.z = fmaf(beta, m4.z, omb * g4.z);
                n4.w = fmaf(beta, m4.w, omb * g4.w);
                if (P.nesterov) {
                    u4.x = fmaf(beta, n4.x, omb * g4.x);
                    u4.y = fmaf(beta, n4.y, omb * g4.y);
                    u4.z = fmaf(beta, n4.z, omb * g4.z);
                    u4.w = fmaf(beta, n4.w, omb * g4.w);
                } else {
                    u4 = n4;
                }
            } else {
                n4.x = fmaf(beta, m4.x, g4.x);
                n4.y = fmaf(beta, m4.y, g4.y);
                n4.z = fmaf(beta, m4.z, g4.z);
                n4.w = fmaf(beta, m4.w, g4.w);
                if (P.nesterov) {
                    u4.x = fmaf(beta, n4.x, g4.x);
                    u4.y = fmaf(beta, n4.y, g4.y);
                    u4.z = fmaf(beta, n4.z, g4.z);
                    u4.w = fmaf(beta, n4.w, g4.w);
                } else {
                    u4 = n4;
                }
            }
            __stcs(reinterpret_cast<float4*>(M.mom + off), n4);
            ss = fmaf(u4.x, u4.x, ss);
            ss = fmaf(u4.y, u4.y, ss);
            ss = fmaf(u4.z, u4.z, ss);
            ss = fmaf(u4.w, u4.w, ss);
            if (!M.transposed) {
                *reinterpret_cast<uint2*>(M.x0 + off) = pack_bf16x4(u4.x, u4.y, u4.z, u4.w);
            }
        }
        if (M.transposed) {
            tile[rr + 16 * k][4 * cq + 0] = u4.x;
            tile[rr + 16 * k][4 * cq + 1] = u4.y;
            tile[rr + 16 * k][4 * cq + 2] = u4.z;
            tile[rr + 16 * k][4 * cq + 3] = u4.w;
        }
    }

    if (M.transposed) {
        // X0 is cols x rows: X0[c][r] = u[r][c]; write rows of X0 (stored columns).
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int oc = c0 + rr + 16 * k;   // X0 row = stored column
            const int orow = r0 + 4 * cq;      // X0 column = stored row
            if (oc < M.cols && orow < M.rows) {
                const int tc = rr + 16 * k, tr = 4 * cq;
                const size_t off = static_cast<size_t>(oc) * M.rows + orow;
                *reinterpret_cast<uint2*>(M.x0 + off) =
                    pack_bf16x4(tile[tr][tc], tile[tr + 1][tc], tile[tr + 2][tc], tile[tr + 3][tc]);
            }
        }
    }

    // Tile sum of squares: warp shuffle, then one value per warp in a fixed order.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) warp_sums[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kMomThreads / 32; ++w) s += warp_sums[w];
        P.partials[t] = s;
        __threadfence();
        const unsigned int ticket = atomicAdd(P.counters + M.gidx, 1u);
        is_last = (ticket == static_cast<unsigned int>(M.ntiles - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!is_last) return;

    // Last CTA of this matrix: fixed-order fp64 sum of its partials.
    __threadfence();
    double acc = 0.0;
    for (int i = tid; i < M.ntiles; i += kMomThreads)
        acc += static_cast<double>(__ldcg(P.partials + M.tile_begin + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((tid & 31) == 0) warp_sums_d[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kMomThreads / 32; ++w) s += warp_sums_d[w];
        const double nrm = sqrt(s);
        P.norms[M.gidx] = static_cast<float>(nrm);
        P.inv_norm[M.gidx] = static_cast<float>(1.0 / (nrm + static_cast<double>(P.eps)));
        P.counters[M.gidx] = 0u;
    }
}

__global__ void __launch_bounds__(kMomThreads) update_kernel(const __grid_constant__ UpdateParams P) {
    const int t = blockIdx.x;
    const int mi = find_mat(P.mats, P.nmats, t);
    const MomentumMat& M = P.mats[mi];
    const int local = t - M.tile_begin;
    const int ty = local / M.tiles_x, tx = local - ty * M.tiles_x;
    const int tid = threadIdx.x;
    const float s = P.inv_norm[M.gidx];
    const float sc = P.lr * P.aspect[M.gidx];
    float* dbg = P.dbg_O ? P.dbg_O[M.gidx] : nullptr;
    for (int e = tid; e < kMomTile * kMomTile; e += kMomThreads) {
        const int row = ty * kMomTile + e / kMomTile;
        const int col = tx * kMomTile + e % kMomTile;
        if (row >= M.rows || col >= M.cols) continue;
        const size_t xo = M.transposed ? static_cast<size_t>(col) * M.rows + row
                                       : static_cast<size_t>(row) * M.cols + col;
        const float O = s * __bfloat162float(M.x0[xo]);
        const size_t po = static_cast<size_t>(row) * M.cols + col;
        M.p[po] = fmaf(-sc, O, M.p[po]);
        if (dbg) dbg[po] = O;
    }
}

cudaError_t launch_momentum_norm(const MomentumParams& p, cudaStream_t s) {
    if (p.total_tiles <= 0) return cudaSuccess;
    momentum_norm_kernel<<<p.total_tiles, kMomThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_update(const UpdateParams& p, cudaStream_t s) {
    if (p.total_tiles <= 0) return cudaSuccess;
    update_kernel<<<p.total_tiles, kMomThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace muon
