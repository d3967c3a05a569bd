// normuon.cu -- the NorMuon scaling of the Muon update and the weight update
// that applies it.
//
// The apidog.com page, section "2. Pengoptimal Muon" (paragraph "Reduksi
// Varians NorMuon"), and the dev.to page ("NorMuon variance scaling") sketch a
// per-neuron rescale of the orthogonalised update O.  Reading (the sketch
// leaves red_dim, the second-moment state, step_size and v_norm_new open): a
// neuron is a stored row;
//   v_mean_i = mean_j O_ij^2 ;  V_i <- beta2 V_i + (1 - beta2) v_mean_i ;
//   step_i = 1 / sqrt(V_i + eps) ;
//   ratio = sqrt(sum_i v_mean_i) / max(sqrt(sum_i v_mean_i step_i^2), 1e-10)
//   p_ij <- p_ij - lr sqrt(max(1, r/c)) step_i ratio O_ij       (keeps ||O||_F)
//
// normuon_rows_kernel: one warp per stored row (8 rows per CTA) reads the row
//   of O (fp32, 16-byte loads), reduces its squares in a fixed order, updates V
//   and writes step_i; the last CTA of a matrix (atomic ticket) adds the CTAs'
//   double partial sums in index order and publishes ratio.  Deterministic.
// normuon_update_kernel: one CTA per 64 x 64 stored tile applies the update
//   (and writes O' = step ratio O when the debug copy is kept).
#include "kernels.cuh"

namespace muon {

namespace {

__device__ __forceinline__ int find_normuon_mat(const NormuonParams& P, int x, bool rows) {
    int lo = 0, hi = P.nmats - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int begin = rows ? P.mats[mid].cta_begin : P.mats[mid].tile_begin;
        if (begin <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

}  // namespace

__global__ void __launch_bounds__(256) normuon_rows_kernel(const __grid_constant__ NormuonParams P) {
    __shared__ double warp_old[kNormRowsPerCta], warp_new[kNormRowsPerCta];
    __shared__ int is_last;
    const int cta = blockIdx.x;
    const NormuonMat& M = P.mats[find_normuon_mat(P, cta, true)];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = (cta - M.cta_begin) * kNormRowsPerCta + warp;
    double s_old = 0.0, s_new = 0.0;
    if (row < M.rows) {
        const float4* o4 = reinterpret_cast<const float4*>(M.O + static_cast<size_t>(row) * M.cols);
        float acc = 0.f;
        for (int q = lane; q < (M.cols >> 2); q += 32) {
            const float4 o = __ldcg(o4 + q);
            acc = fmaf(o.x, o.x, acc);
            acc = fmaf(o.y, o.y, acc);
            acc = fmaf(o.z, o.z, acc);
            acc = fmaf(o.w, o.w, acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const double v_mean = static_cast<double>(acc) / M.cols;
        const double Vn = static_cast<double>(P.beta2) * M.V[row] + (1.0 - static_cast<double>(P.beta2)) * v_mean;
        const double step = 1.0 / sqrt(Vn + static_cast<double>(P.eps));
        if (lane == 0) {
            M.V[row] = static_cast<float>(Vn);
            P.step[P.row_base[M.pos] + row] = static_cast<float>(step);
        }
        s_old = v_mean;
        s_new = v_mean * step * step;
    }
    if (lane == 0) {
        warp_old[warp] = s_old;
        warp_new[warp] = s_new;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kNormRowsPerCta; ++w) {
            a += warp_old[w];
            b += warp_new[w];
        }
        P.partials[2 * cta] = a;
        P.partials[2 * cta + 1] = b;
        __threadfence();
        const unsigned int ticket = atomicAdd(P.counters + M.pos, 1u);
        is_last = ticket == static_cast<unsigned int>(M.nctas - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!is_last || threadIdx.x != 0) return;
    __threadfence();
    double a = 0.0, b = 0.0;
    for (int k = 0; k < M.nctas; ++k) {
        a += __ldcg(P.partials + 2 * (M.cta_begin + k));
        b += __ldcg(P.partials + 2 * (M.cta_begin + k) + 1);
    }
    const double nb = sqrt(b);
    P.ratio[M.pos] = static_cast<float>(sqrt(a) / (nb > 1e-10 ? nb : 1e-10));
    P.counters[M.pos] = 0u;
}

__global__ void __launch_bounds__(256) normuon_update_kernel(const __grid_constant__ NormuonParams P) {
    const int t = blockIdx.x;
    const NormuonMat& M = P.mats[find_normuon_mat(P, t, false)];
    const int local = t - M.tile_begin;
    const int ty = local / M.tiles_x, tx = local - ty * M.tiles_x;
    const int r0 = ty * 64, c0 = tx * 64;
    const int cq = threadIdx.x & 15, rr = threadIdx.x >> 4;
    const float ratio = P.ratio[M.pos];
    const float lr_aspect = P.lr * P.aspect[M.pos];
    const float* step = P.step + P.row_base[M.pos];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = r0 + rr + 16 * k;
        const int col = c0 + 4 * cq;
        if (row >= M.rows || col >= M.cols) continue;
        const size_t off = static_cast<size_t>(row) * M.cols + col;
        const float sr = step[row] * ratio;
        const float4 o = __ldcs(reinterpret_cast<const float4*>(M.O + off));
        float4 w = *reinterpret_cast<float4*>(M.p + off);
        const float sc = lr_aspect * sr;
        w.x = fmaf(-sc, o.x, w.x);
        w.y = fmaf(-sc, o.y, w.y);
        w.z = fmaf(-sc, o.z, w.z);
        w.w = fmaf(-sc, o.w, w.w);
        *reinterpret_cast<float4*>(M.p + off) = w;
        if (M.dbg) *reinterpret_cast<float4*>(M.dbg + off) = make_float4(sr * o.x, sr * o.y, sr * o.z, sr * o.w);
    }
}

cudaError_t launch_normuon_rows(const NormuonParams& p, cudaStream_t s) {
    if (p.total <= 0) return cudaSuccess;
    normuon_rows_kernel<<<p.total, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_normuon_update(const NormuonParams& p, cudaStream_t s) {
    if (p.total <= 0) return cudaSuccess;
    normuon_update_kernel<<<p.total, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace muon
