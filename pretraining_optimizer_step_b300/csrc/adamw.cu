// adamw.cu -- muon_adamw_step: the AdamW step for the parameters the optimizer
// split keeps away from Muon (embeddings, lm_head, scalars; the dev.to page
// "Train your own ChatGPT", section "2. ตัวปรับปรุง Muon", optimizer table).
//
// Decoupled weight decay with bias-corrected moments, step t >= 1:
//   p <- p (1 - lr wd); m <- b1 m + (1 - b1) g; v <- b2 v + (1 - b2) g^2
//   p <- p - (lr / (1 - b1^t)) m / (sqrt(v / (1 - b2^t)) + eps)
// in fp32 (the bias corrections are formed on the host in fp64).
//
// One launch covers every tensor of the call: the tensors are cut into chunks
// of kChunk elements and each CTA (256 threads) updates one chunk with 16-byte
// loads and stores (a ragged tail of fewer than 4 elements goes scalar).
// 28 algorithmic bytes per element (p, g, m, v read; p, m, v written): HBM-bound.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/muon.h"

namespace {

constexpr int kAdamThreads = 256;
constexpr long long kChunk = 16384;          // elements per CTA (16 float4 per thread)
constexpr int kAdamMaxTensors = 128;         // tensors per launch (kernel parameter space)
constexpr int kAdamMaxDevices = 64;

struct AdamTensor {
    float* p;
    const float* g;
    float* m;
    float* v;
    long long n;
    long long chunk_begin;  // first CTA of this tensor in the launch
};

struct AdamParams {
    AdamTensor t[kAdamMaxTensors];
    int ntensors;
    long long total_chunks;
    float decay;      // 1 - lr wd
    float b1, omb1;   // beta1, 1 - beta1
    float b2, omb2;
    float step_size;  // lr / (1 - beta1^t)
    float inv_bc2;    // 1 / (1 - beta2^t)
    float eps;
};

__device__ __forceinline__ float adam_one(float p, float g, float& m, float& v, const AdamParams& P) {
    m = fmaf(P.b1, m, P.omb1 * g);
    v = fmaf(P.b2, v, P.omb2 * g * g);
    const float denom = sqrtf(v * P.inv_bc2) + P.eps;
    return fmaf(-P.step_size, m / denom, p * P.decay);
}

__global__ void __launch_bounds__(kAdamThreads) adamw_kernel(const __grid_constant__ AdamParams P) {
    const long long c = blockIdx.x;
    int lo = 0, hi = P.ntensors - 1;
    while (lo < hi) {  // last tensor whose first chunk is <= c
        const int mid = (lo + hi + 1) >> 1;
        if (P.t[mid].chunk_begin <= c) lo = mid;
        else hi = mid - 1;
    }
    const AdamTensor& T = P.t[lo];
    const long long e0 = (c - T.chunk_begin) * kChunk;
    const long long len = T.n - e0 < kChunk ? T.n - e0 : kChunk;
    const long long nvec = len >> 2;
    float4* p4 = reinterpret_cast<float4*>(T.p + e0);
    const float4* g4 = reinterpret_cast<const float4*>(T.g + e0);
    float4* m4 = reinterpret_cast<float4*>(T.m + e0);
    float4* v4 = reinterpret_cast<float4*>(T.v + e0);
    for (long long i = threadIdx.x; i < nvec; i += kAdamThreads) {
        const float4 g = __ldcs(g4 + i);
        float4 p = __ldcs(p4 + i), m = __ldcs(m4 + i), v = __ldcs(v4 + i);
        p.x = adam_one(p.x, g.x, m.x, v.x, P);
        p.y = adam_one(p.y, g.y, m.y, v.y, P);
        p.z = adam_one(p.z, g.z, m.z, v.z, P);
        p.w = adam_one(p.w, g.w, m.w, v.w, P);
        __stcs(p4 + i, p);
        __stcs(m4 + i, m);
        __stcs(v4 + i, v);
    }
    for (long long e = (nvec << 2) + threadIdx.x; e < len; e += kAdamThreads) {
        float m = T.m[e0 + e], v = T.v[e0 + e];
        T.p[e0 + e] = adam_one(T.p[e0 + e], T.g[e0 + e], m, v, P);
        T.m[e0 + e] = m;
        T.v[e0 + e] = v;
    }
}

int g_dev_ok[kAdamMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other

muon_status check_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kAdamMaxDevices) {
        cudaGetLastError();
        return MUON_ERR_UNSUPPORTED_DEVICE;
    }
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return MUON_ERR_UNSUPPORTED_DEVICE;
        }
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_dev_ok[dev] == 1 ? MUON_OK : MUON_ERR_UNSUPPORTED_DEVICE;
}

}  // namespace

extern "C" muon_status muon_adamw_step(float* const params[], const float* const grads[],
                                       float* const exp_avg[], float* const exp_avg_sq[],
                                       const long long numels[], int n_tensors, float lr, float beta1,
                                       float beta2, float eps, float weight_decay, int step,
                                       muon_stream_t stream_) {
    if (n_tensors < 0) return MUON_ERR_INVALID_ARG;
    if (n_tensors == 0) return MUON_OK;
    if (!params || !grads || !exp_avg || !exp_avg_sq || !numels) return MUON_ERR_INVALID_ARG;
    if (step < 1 || !std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(weight_decay) ||
        !(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || eps < 0.0f)
        return MUON_ERR_INVALID_ARG;
    for (int i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0) return MUON_ERR_INVALID_ARG;
        if (numels[i] == 0) continue;
        if (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i]) return MUON_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(params[i]) | reinterpret_cast<uintptr_t>(grads[i]) |
             reinterpret_cast<uintptr_t>(exp_avg[i]) | reinterpret_cast<uintptr_t>(exp_avg_sq[i])) & 15u)
            return MUON_ERR_MISALIGNED;
    }
    const muon_status dst = check_device();
    if (dst != MUON_OK) return dst;

    AdamParams P;  // ~5 KiB, by value
    std::memset(&P, 0, sizeof(P));
    const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), step);
    const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), step);
    P.decay = static_cast<float>(1.0 - static_cast<double>(lr) * weight_decay);
    P.b1 = beta1;
    P.omb1 = static_cast<float>(1.0 - static_cast<double>(beta1));
    P.b2 = beta2;
    P.omb2 = static_cast<float>(1.0 - static_cast<double>(beta2));
    P.step_size = static_cast<float>(lr / bc1);
    P.inv_bc2 = static_cast<float>(1.0 / bc2);
    P.eps = eps;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int k = 0;
    long long chunks = 0;
    auto flush = [&]() -> muon_status {
        if (k == 0) return MUON_OK;
        P.ntensors = k;
        P.total_chunks = chunks;
        // a grid dimension holds 2^31 - 1 CTAs: 3.5e13 elements per launch
        adamw_kernel<<<static_cast<unsigned int>(chunks), kAdamThreads, 0, stream>>>(P);
        k = 0;
        chunks = 0;
        return cudaGetLastError() == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    };
    for (int i = 0; i < n_tensors; ++i) {
        if (numels[i] == 0) continue;
        if (k == kAdamMaxTensors) {
            const muon_status st = flush();
            if (st != MUON_OK) return st;
        }
        AdamTensor& T = P.t[k++];
        T.p = params[i];
        T.g = grads[i];
        T.m = exp_avg[i];
        T.v = exp_avg_sq[i];
        T.n = numels[i];
        T.chunk_begin = chunks;
        chunks += (numels[i] + kChunk - 1) / kChunk;
    }
    return flush();
}
