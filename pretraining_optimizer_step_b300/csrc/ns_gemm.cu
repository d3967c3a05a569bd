// ns_gemm.cu -- the Newton-Schulz GEMMs of the Muon step on the sm_103a tensor cores.
//
// One iteration of the quintic loop ("Cara Melatih ChatGPT Sendiri dengan
// Budget 50 Dolar", section "2. Pengoptimal Muon", orthogonalization loop) is
// three launches of this persistent, warp-specialised kernel over every matrix
// of the step at once (grouped by oriented shape class):
//   MODE_GRAM  A = s^2 X X^T           only tiles on/above the diagonal; the
//                                      epilogue mirrors off-diagonal tiles so A
//                                      is stored whole (bf16)
//   MODE_POLY  B = b A + c A A         A is symmetric, so A A = A A^T: the same
//                                      K-major operand feeds both sides; the
//                                      epilogue reads the A tile and forms the
//                                      polynomial in fp32; mirrored like GRAM
//   MODE_AXPY  X' = s (a X + B X)      B (K-major) times X (MN-major operand);
//                                      the epilogue reads the X tile
//   MODE_AXPY_FINAL                    same product; O = s (a X + B X) stays in
//                                      fp32 and the epilogue applies
//                                      p -= lr sqrt(max(1, r/c)) O to the fp32
//                                      weights in their stored layout
// s = 1/(||u|| + eps) on the first iteration (X0 is stored unscaled), else 1.
//
// CTA layout (192 threads, one CTA per SM, grid-stride over tiles):
//   warp 0      TMA producer: 4-stage ring of {A 128x64, B 256x64} bf16 slices,
//               128-byte swizzled, completion by mbarrier transaction bytes
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma 128x256x16,
//               accumulators double-buffered in TMEM (2 x 256 fp32 columns)
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns per warp, one output
//               row per thread
// Every wait is bounded; on expiry the CTA latches STATUS_TIMEOUT, stops all
// roles, drains its own TMA loads and MMAs, frees TMEM and returns.
#include "kernels.cuh"
#include "ptx.cuh"

namespace muon {

namespace {

struct TileCoord {
    int ci;    // shape class
    int mat;   // matrix within the class
    int rb;    // 128-row block
    int cb;    // gram/poly: first 128-column block (tile spans 2); axpy: 256-column block
};

__device__ __forceinline__ TileCoord decode_tile(const GemmParams& P, int t) {
    TileCoord tc;
    int ci = 0;
    while (ci + 1 < P.nclasses && t >= P.cls[ci + 1].tile_begin) ++ci;
    const GemmClass& C = P.cls[ci];
    const int local = t - C.tile_begin;
    tc.ci = ci;
    tc.mat = local / C.tiles_per_mat;
    int lt = local - tc.mat * C.tiles_per_mat;
    if (P.mode == MODE_GRAM || P.mode == MODE_POLY) {
        // row block bi owns ceil((row_blocks - bi) / 2) tiles starting at column block bi
        int bi = 0;
        for (;;) {
            const int cnt = (C.row_blocks - bi + 1) >> 1;
            if (lt < cnt || bi + 1 >= C.row_blocks) break;
            lt -= cnt;
            ++bi;
        }
        tc.rb = bi;
        tc.cb = bi + 2 * lt;
    } else {
        tc.rb = lt / C.col_tiles;
        tc.cb = lt - tc.rb * C.col_tiles;
    }
    return tc;
}

__device__ __forceinline__ void latch_status(unsigned int* status, unsigned int bits) {
    atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Writes 32 fp32 values (one thread's slice of a tile row) as bf16 to row `r`,
// columns [c0, c0+32) of a row-major matrix with `ld` columns, in 16-byte
// groups; columns >= limit are skipped (limit is a multiple of 8).
__device__ __forceinline__ void store_row32(__nv_bfloat16* base, size_t ld, int r, int c0, int limit,
                                            const float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int c = c0 + 8 * g;
        if (c < limit) {
            uint4 w;
            w.x = pack2(v[8 * g + 0], v[8 * g + 1]);
            w.y = pack2(v[8 * g + 2], v[8 * g + 3]);
            w.z = pack2(v[8 * g + 4], v[8 * g + 5]);
            w.w = pack2(v[8 * g + 6], v[8 * g + 7]);
            *reinterpret_cast<uint4*>(base + static_cast<size_t>(r) * ld + c) = w;
        }
    }
}

// Reads 32 bf16 of row r, columns [c0, c0+32), as fp32 (zeros past limit).
__device__ __forceinline__ void load_row32(const __nv_bfloat16* base, size_t ld, int r, int c0,
                                           int limit, float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int c = c0 + 8 * g;
        if (c < limit) {
            const uint4 w = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(r) * ld + c);
            v[8 * g + 0] = bf16_lo(w.x); v[8 * g + 1] = bf16_hi(w.x);
            v[8 * g + 2] = bf16_lo(w.y); v[8 * g + 3] = bf16_hi(w.y);
            v[8 * g + 4] = bf16_lo(w.z); v[8 * g + 5] = bf16_hi(w.z);
            v[8 * g + 6] = bf16_lo(w.w); v[8 * g + 7] = bf16_hi(w.w);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[8 * g + j] = 0.f;
        }
    }
}

}  // namespace

__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ volatile int abort_flag;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t tiles_base = (raw + 1023u) & ~1023u;   // 128B-swizzle atoms need 1 KiB alignment
    uint8_t* tiles_ptr = smem_raw + (tiles_base - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool sym = (P.mode == MODE_GRAM || P.mode == MODE_POLY);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull_bar[a], 1);
            mbar_init(&tempty_bar[a], 4 * 32);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        for (int c = 0; c < P.nclasses; ++c) {
            tma_prefetch_desc(&P.tmA[c]);
            tma_prefetch_desc(&P.tmB[c]);
        }
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued[kStages] = {0, 0, 0, 0};
        bool aborted = false;
        bool injected = false;
        for (int t = blockIdx.x; t < P.total_tiles && !aborted; t += gridDim.x) {
            const TileCoord tc = decode_tile(P, t);
            const GemmClass& C = P.cls[tc.ci];
            const CUtensorMap* mA = &P.tmA[tc.ci];
            const CUtensorMap* mB = &P.tmB[tc.ci];
            const int bound = sym ? C.m : C.n;   // extent of the N-side rows / columns
            for (int kb = 0; kb < C.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_flag, P.timeout_ns)) {
                    latch_status(P.status, STATUS_TIMEOUT);
                    abort_flag = 1;
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles_ptr + stage * kStageBytes;
                uint8_t* sb = sa + kAStageBytes;
                const int k0 = kb * kBK;
                uint32_t bytes = kAStageBytes;
                if (sym) {
                    const int n0 = tc.cb * kBM;
                    bytes += (n0 + kBM < bound) ? 2 * kAStageBytes : kAStageBytes;
                } else {
                    const int n0 = tc.cb * kBN;
                    for (int q = 0; q < 4; ++q)
                        if (n0 + 64 * q < bound) bytes += kBK * 128;
                }
                if (P.inject_lost_load && !injected && blockIdx.x == 0) {
                    // test hook: this slice is never loaded, so its consumer's wait must expire
                    injected = true;
                } else {
                    mbar_arrive_expect_tx(&full_bar[stage], bytes);
                    tma_load_3d(sa, mA, &full_bar[stage], k0, tc.rb * kBM, tc.mat);
                    if (sym) {
                        const int n0 = tc.cb * kBM;
                        tma_load_3d(sb, mB, &full_bar[stage], k0, n0, tc.mat);
                        if (n0 + kBM < bound)
                            tma_load_3d(sb + kAStageBytes, mB, &full_bar[stage], k0, n0 + kBM, tc.mat);
                    } else {
                        const int n0 = tc.cb * kBN;
                        for (int q = 0; q < 4; ++q)
                            if (n0 + 64 * q < bound)
                                tma_load_3d(sb + q * (kBK * 128), mB, &full_bar[stage], n0 + 64 * q, k0,
                                            tc.mat);
                    }
                    issued[stage] += 1;
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (aborted) {
            // let every load this thread issued land before the CTA can exit
            for (int s = 0; s < kStages; ++s)
                if (issued[s] > 0)
                    mbar_wait_bounded(&full_bar[s], (issued[s] - 1u) & 1u, nullptr, P.timeout_ns);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_bf16_f32(kBM, kBN, sym ? 0 : 1);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool aborted = false;
        for (int t = blockIdx.x; t < P.total_tiles && !aborted; t += gridDim.x) {
            const TileCoord tc = decode_tile(P, t);
            const GemmClass& C = P.cls[tc.ci];
            if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, &abort_flag, P.timeout_ns)) {
                latch_status(P.status, STATUS_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
            for (int kb = 0; kb < C.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&full_bar[stage], phase, &abort_flag, P.timeout_ns)) {
                    latch_status(P.status, STATUS_TIMEOUT);
                    abort_flag = 1;
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = tiles_base + stage * kStageBytes;
                const uint32_t sb = sa + kAStageBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                    const uint64_t bdesc = sym ? smem_desc_sw128(sb + kk * 32, 16, 1024)
                                               : smem_desc_sw128(sb + kk * 2048, kBK * 128, 1024);
                    tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                tc_commit(&empty_bar[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            tc_commit(&tfull_bar[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // every MMA this thread issued must finish before TMEM is released
        tc_commit(&drain_bar);
        mbar_wait_bounded(&drain_bar, 0, nullptr, P.timeout_ns);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        const int lg = warp & 3;               // TMEM lane group this warp may access
        const int row_in_tile = lg * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < P.total_tiles; t += gridDim.x) {
            const TileCoord tc = decode_tile(P, t);
            const GemmClass& C = P.cls[tc.ci];
            // every lane waits; the outcome is made warp-uniform so that the
            // warp-collective TMEM loads below are reached by all lanes or none
            const bool ready = __all_sync(0xffffffffu,
                                          mbar_wait_bounded(&tfull_bar[acc], acc_phase, &abort_flag, P.timeout_ns));
            if (!ready) {
                if (lane == 0) latch_status(P.status, STATUS_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int gm = C.mat_base + tc.mat;
            const int r = tc.rb * kBM + row_in_tile;
            const bool row_ok = r < C.m;
            const float s = P.first_iter ? P.inv_norm[gm] : 1.0f;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) +
                                   static_cast<uint32_t>(acc * kBN);
            const size_t mm = static_cast<size_t>(C.m) * C.m;
            const size_t mn = static_cast<size_t>(C.m) * C.n;
            for (int ch = 0; ch < kBN / 32; ++ch) {
                uint32_t raw_v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + ch * 32, raw_v);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw_v[j]);
                if (!row_ok) continue;
                if (sym) {
                    const int c0 = tc.cb * kBM + ch * 32;
                    if (c0 >= C.m) continue;
                    __nv_bfloat16* out = C.out + static_cast<size_t>(tc.mat) * mm;
                    if (P.mode == MODE_GRAM) {
                        const float s2 = s * s;
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= s2;
                    } else {
                        float a[32];
                        load_row32(C.aux + static_cast<size_t>(tc.mat) * mm, C.m, r, c0, C.m, a);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = fmaf(P.cc, v[j], P.cb * a[j]);
                    }
                    store_row32(out, C.m, r, c0, C.m, v);
                    if (c0 >= (tc.rb + 1) * kBM) {
                        // strictly above the diagonal block: also write the mirrored element
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < C.m)
                                out[static_cast<size_t>(c0 + j) * C.m + r] = __float2bfloat16_rn(v[j]);
                    }
                } else {
                    const int c0 = tc.cb * kBN + ch * 32;
                    if (c0 >= C.n) continue;
                    float x[32];
                    load_row32(C.aux + static_cast<size_t>(tc.mat) * mn, C.n, r, c0, C.n, x);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = s * fmaf(P.ca, x[j], v[j]);
                    if (P.mode == MODE_AXPY) {
                        store_row32(C.out + static_cast<size_t>(tc.mat) * mn, C.n, r, c0, C.n, v);
                    } else {
                        float* p = P.p_table[gm];
                        float* dbg = P.dbg_O ? P.dbg_O[gm] : nullptr;
                        const float sc = P.lr * P.aspect[gm];
                        if (!C.transposed) {
                            // stored layout = oriented layout (m x n)
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const int c = c0 + 4 * g;
                                if (c < C.n) {
                                    float4* pp = reinterpret_cast<float4*>(p + static_cast<size_t>(r) * C.n + c);
                                    float4 w = *pp;
                                    w.x = fmaf(-sc, v[4 * g + 0], w.x);
                                    w.y = fmaf(-sc, v[4 * g + 1], w.y);
                                    w.z = fmaf(-sc, v[4 * g + 2], w.z);
                                    w.w = fmaf(-sc, v[4 * g + 3], w.w);
                                    *pp = w;
                                    if (dbg)
                                        *reinterpret_cast<float4*>(dbg + static_cast<size_t>(r) * C.n + c) =
                                            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                                }
                            }
                        } else {
                            // stored matrix is n x m: O_stored[c][r] = O[r][c]; consecutive
                            // lanes hold consecutive r, so each column c is a coalesced row segment
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int c = c0 + j;
                                if (c < C.n) {
                                    const size_t po = static_cast<size_t>(c) * C.m + r;
                                    p[po] = fmaf(-sc, v[j], p[po]);
                                    if (dbg) dbg[po] = v[j];
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty_bar[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

cudaError_t ns_gemm_prepare() {
    return cudaFuncSetAttribute(ns_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kGemmSmemBytes);
}

cudaError_t launch_ns_gemm(const GemmParams& p, int grid, cudaStream_t s) {
    if (p.total_tiles <= 0) return cudaSuccess;
    ns_gemm_kernel<<<grid, kGemmThreads, kGemmSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace muon
