// noalloc.cu -- muon_momentum_norm_noalloc: the momentum + norm pass of the
// Muon step for callers that cannot allocate device memory.  The kernel is the
// one muon_step runs (momentum_norm_kernel); only its scratch moves, from the
// step's cudaMalloc arena into a fixed array that lives in this file.
//
// Scratch layout (one array, shared by every call on a device):
//   partials  kNoAllocMaxTiles floats   one fp32 sum of squares per CTA (64 x 64 tile)
//   tickets   kNoAllocMaxMats  uint32   per-matrix arrival counters (must start at 0)
//   inv_norm  kNoAllocMaxMats  floats   1/(||u|| + eps), written by the kernel
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/muon.h"
#include "kernels.cuh"

using namespace muon;

namespace {

constexpr int kNoAllocMaxMats = 1024;
constexpr int kNoAllocMaxTiles = 262144;
constexpr int kNoAllocMaxDevices = 64;

constexpr size_t kOffPartials = 0;
constexpr size_t kOffTickets = kOffPartials + sizeof(float) * kNoAllocMaxTiles;
constexpr size_t kOffInvNorm = kOffTickets + sizeof(unsigned int) * kNoAllocMaxMats;
constexpr size_t kScratchBytes = kOffInvNorm + sizeof(float) * kNoAllocMaxMats;
static_assert(kOffTickets % 256 == 0 && kOffInvNorm % 256 == 0, "scratch sections stay 256-byte aligned");

// The fixed scratch.  In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device ordinal, looked up by the
// first call on that device, together with the ID of the context it belongs
// to.  A call whose current context has another ID (cudaDeviceReset ends a
// context; the next one may load the module elsewhere) looks it up again.
// The mutex makes concurrent first calls from several host threads safe.
struct ScratchSlot {
    unsigned char* addr = nullptr;
    unsigned long long ctx_id = 0;
};
ScratchSlot g_scratch[kNoAllocMaxDevices];
std::mutex g_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// ID of the calling thread's current context (0 when none is current or the
// driver does not offer the query).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
        resolved = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

muon_status scratch_for_current_device(unsigned char** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return MUON_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev >= kNoAllocMaxDevices) return MUON_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot& slot = g_scratch[dev];
    if (slot.addr != nullptr && slot.ctx_id != 0 && slot.ctx_id == current_context_id()) {
        *out = slot.addr;
        return MUON_OK;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MUON_ERR_UNSUPPORTED_DEVICE;
    }
    if (!(major == 10 && minor == 3)) return MUON_ERR_UNSUPPORTED_DEVICE;
    // with this device current: the symbol's address in its (primary) context
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return MUON_ERR_CUDA;
    }
    slot.addr = static_cast<unsigned char*>(ptr);
    slot.ctx_id = current_context_id();  // 0 (unknown) makes the next call look it up again
    *out = slot.addr;
    return MUON_OK;
}

int tiles_of(const muon_shape& s) {
    return ((s.rows + kMomTile - 1) / kMomTile) * ((s.cols + kMomTile - 1) / kMomTile);
}

}  // namespace

extern "C" muon_status muon_momentum_norm_noalloc(const float* const grads[], float* const momentum_bufs[],
                                                  void* const x0_out[], float* norms_out,
                                                  const muon_shape shapes[], int n_mats, float beta,
                                                  int nesterov, int momentum_mode, double eps,
                                                  muon_stream_t stream_) {
    // ---- every argument and limit is checked before the device is touched
    if (n_mats < 0) return MUON_ERR_INVALID_ARG;
    if (n_mats == 0) return MUON_OK;
    if (!grads || !momentum_bufs || !x0_out || !norms_out || !shapes) return MUON_ERR_INVALID_ARG;
    if (momentum_mode != MUON_MOMENTUM_SGD_NESTEROV && momentum_mode != MUON_MOMENTUM_EMA)
        return MUON_ERR_INVALID_ARG;
    if (!std::isfinite(beta) || !std::isfinite(eps)) return MUON_ERR_INVALID_ARG;
    for (int i = 0; i < n_mats; ++i) {
        const int r = shapes[i].rows, c = shapes[i].cols;
        if (r < 8 || c < 8 || (r % 8) != 0 || (c % 8) != 0 || r > 65536 || c > 65536)
            return MUON_ERR_UNSUPPORTED_SHAPE;
    }
    for (int i = 0; i < n_mats; ++i) {
        if (!grads[i] || !momentum_bufs[i] || !x0_out[i]) return MUON_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(grads[i]) | reinterpret_cast<uintptr_t>(momentum_bufs[i]) |
             reinterpret_cast<uintptr_t>(x0_out[i])) & 15u)
            return MUON_ERR_MISALIGNED;
    }
    if (reinterpret_cast<uintptr_t>(norms_out) & 3u) return MUON_ERR_MISALIGNED;
    if (n_mats > kNoAllocMaxMats) return MUON_ERR_SCRATCH_LIMIT;
    for (int base = 0; base < n_mats; base += kMomentumMaxMats) {
        const int cnt = n_mats - base < kMomentumMaxMats ? n_mats - base : kMomentumMaxMats;
        long long tiles = 0;
        for (int k = 0; k < cnt; ++k) tiles += tiles_of(shapes[base + k]);
        if (tiles > kNoAllocMaxTiles) return MUON_ERR_SCRATCH_LIMIT;
    }

    unsigned char* scratch = nullptr;
    const muon_status st = scratch_for_current_device(&scratch);
    if (st != MUON_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch + kOffTickets);

    // the kernel leaves every ticket it used at 0, but a previous call that
    // never finished (an error) could not; start from 0 on every call
    if (cudaMemsetAsync(tickets, 0, sizeof(unsigned int) * static_cast<size_t>(n_mats), stream) !=
        cudaSuccess)
        return MUON_ERR_CUDA;

    MomentumParams mp;  // kernel parameters, by value; ~12 KiB on the host stack
    for (int base = 0; base < n_mats; base += kMomentumMaxMats) {
        const int cnt = n_mats - base < kMomentumMaxMats ? n_mats - base : kMomentumMaxMats;
        std::memset(&mp, 0, sizeof(mp));
        int tiles = 0;
        for (int k = 0; k < cnt; ++k) {
            const int i = base + k;
            MomentumMat& M = mp.mats[k];
            M.g = grads[i];
            M.mom = momentum_bufs[i];
            M.p = nullptr;
            M.x0 = static_cast<__nv_bfloat16*>(x0_out[i]);
            M.rows = shapes[i].rows;
            M.cols = shapes[i].cols;
            M.transposed = M.rows > M.cols ? 1 : 0;
            M.tiles_x = (M.cols + kMomTile - 1) / kMomTile;
            M.ntiles = tiles_of(shapes[i]);
            M.tile_begin = tiles;
            M.gidx = i;
            tiles += M.ntiles;
        }
        mp.nmats = cnt;
        mp.total_tiles = tiles;
        mp.beta = beta;
        mp.nesterov = nesterov ? 1 : 0;
        mp.mode = momentum_mode;
        mp.eps = static_cast<float>(eps > 0 ? eps : 1e-7);
        mp.partials = reinterpret_cast<float*>(scratch + kOffPartials);
        mp.counters = tickets;
        mp.inv_norm = reinterpret_cast<float*>(scratch + kOffInvNorm);
        mp.norms = norms_out;
        if (launch_momentum_norm(mp, stream) != cudaSuccess) return MUON_ERR_CUDA;
    }
    return MUON_OK;
}
