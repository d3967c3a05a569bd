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
// O arrives in bf16 (stored layout), written by the last Newton-Schulz launch.
// normuon_rows_kernel: one warp per stored row (4 rows per warp, 32 per CTA) reads the row
//   of O (16-byte loads of 8 bf16), reduces its squares in fp32 in a fixed order, updates V
//   and writes step_i; the last CTA of a matrix (atomic ticket) adds the CTAs'
//   double partial sums, spread over its threads in a fixed order, and
//   publishes ratio.  Deterministic.
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

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// sum of squares of the 8 bf16 values of a 16-byte word, added to acc
__device__ __forceinline__ float sq8(uint4 w, float acc) {
    acc = fmaf(bf_lo(w.x), bf_lo(w.x), acc);
    acc = fmaf(bf_hi(w.x), bf_hi(w.x), acc);
    acc = fmaf(bf_lo(w.y), bf_lo(w.y), acc);
    acc = fmaf(bf_hi(w.y), bf_hi(w.y), acc);
    acc = fmaf(bf_lo(w.z), bf_lo(w.z), acc);
    acc = fmaf(bf_hi(w.z), bf_hi(w.z), acc);
    acc = fmaf(bf_lo(w.w), bf_lo(w.w), acc);
    return fmaf(bf_hi(w.w), bf_hi(w.w), acc);
}

}  // namespace

__global__ void __launch_bounds__(256) normuon_rows_kernel(const __grid_constant__ NormuonParams P) {
    __shared__ double warp_old[kNormWarps], warp_new[kNormWarps];
    __shared__ int is_last;
    const int cta = blockIdx.x;
    const NormuonMat& M = P.mats[find_normuon_mat(P, cta, true)];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float s_old = 0.f, s_new = 0.f;  // lane 0: this warp's rows, added in row order
    for (int rw = 0; rw < kNormRowsPerWarp; ++rw) {
        const int row = (cta - M.cta_begin) * kNormRowsPerCta + rw * kNormWarps + warp;
        if (row >= M.rows) break;
        const uint4* o8 = reinterpret_cast<const uint4*>(M.O + static_cast<size_t>(row) * M.cols);
        // four independent sums, so four loads per lane are in flight
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const int nq = M.cols >> 3;
        int q = lane;
        for (; q + 96 < nq; q += 128) {
            const uint4 o0 = __ldcg(o8 + q), o1 = __ldcg(o8 + q + 32);
            const uint4 o2 = __ldcg(o8 + q + 64), o3 = __ldcg(o8 + q + 96);
            a0 = sq8(o0, a0);
            a1 = sq8(o1, a1);
            a2 = sq8(o2, a2);
            a3 = sq8(o3, a3);
        }
        for (; q < nq; q += 32) a0 = sq8(__ldcg(o8 + q), a0);
        float acc = (a0 + a1) + (a2 + a3);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        // fp32 (IEEE division and square root): the fp64 pipe of this part costs a full warp
        // instruction slot per operation even for one lane, and the row path would be bound by it
        if (lane == 0) {
            const float v_mean = acc / static_cast<float>(M.cols);
            const float Vn = fmaf(P.beta2, M.V[row], (1.0f - P.beta2) * v_mean);
            const float step = 1.0f / sqrtf(Vn + P.eps);
            M.V[row] = Vn;
            P.step[P.row_base[M.pos] + row] = step;
            s_old += v_mean;
            s_new += v_mean * step * step;
        }
    }
    if (lane == 0) {
        warp_old[warp] = static_cast<double>(s_old);
        warp_new[warp] = static_cast<double>(s_new);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kNormWarps; ++w) {
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
    if (!is_last) return;
    // Last CTA of the matrix: every thread adds a fixed strided subset of the CTAs' partials,
    // then a fixed xor tree per warp and the warp sums in index order (deterministic)
    __threadfence();
    double a = 0.0, b = 0.0;
    for (int k = threadIdx.x; k < M.nctas; k += blockDim.x) {
        a += __ldcg(P.partials + 2 * (M.cta_begin + k));
        b += __ldcg(P.partials + 2 * (M.cta_begin + k) + 1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    if (lane == 0) {
        warp_old[warp] = a;  // thread 0 finished reading these before the barrier above
        warp_new[warp] = b;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    double sa = 0.0, sb = 0.0;
    for (int w = 0; w < kNormWarps; ++w) {
        sa += warp_old[w];
        sb += warp_new[w];
    }
    const double nb = sqrt(sb);
    P.ratio[M.pos] = static_cast<float>(sqrt(sa) / (nb > 1e-10 ? nb : 1e-10));
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
        const uint2 ob = __ldcs(reinterpret_cast<const uint2*>(M.O + off));
        const float4 o = make_float4(bf_lo(ob.x), bf_hi(ob.x), bf_lo(ob.y), bf_hi(ob.y));
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
