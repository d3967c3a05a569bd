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
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns per warp into
//               registers, staged through a per-warp 32 x 33 fp32 shared block so
//               that global loads and stores run along rows (mirrored tiles and
//               n x m weights read the block transposed)
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

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Four consecutive bf16 <-> fp32 at element offset `off` (a multiple of 4, so
// the access is one aligned 8-byte word).
__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* base, size_t off, const float (&v)[4]) {
    uint2 w;
    w.x = pack2(v[0], v[1]);
    w.y = pack2(v[2], v[3]);
    *reinterpret_cast<uint2*>(base + off) = w;
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
    __shared__ float stage_all[4][32][33];   // epilogue: one 32 x 32 fp32 block per warp (padded)

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
        float (*stage)[33] = stage_all[lg];
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < P.total_tiles; t += gridDim.x) {
            const TileCoord tc = decode_tile(P, t);
            const GemmClass& C = P.cls[tc.ci];
            const int gm = C.mat_base + tc.mat;
            const size_t mm = static_cast<size_t>(C.m) * C.m;
            const size_t mn = static_cast<size_t>(C.m) * C.n;
            const int r0 = tc.rb * kBM + lg * 32;        // first oriented row of this warp
            const int ctile = sym ? tc.cb * kBM : tc.cb * kBN;
            const int climit = sym ? C.m : C.n;
            // While this tile's MMAs run, pull the global data its epilogue will read
            // (the A or X tile, and the fp32 weights of the final launch) into L2,
            // so that the epilogue's loads do not wait on DRAM.
            if (P.mode != MODE_GRAM && r0 < C.m) {
                const __nv_bfloat16* aux = C.aux + (sym ? static_cast<size_t>(tc.mat) * mm
                                                        : static_cast<size_t>(tc.mat) * mn);
                const int ld = sym ? C.m : C.n;
                const int ncols = min(kBN, climit - ctile);          // multiple of 8
                const int lines = (ncols * 2 + 127) / 128;           // 128-byte lines per row
#pragma unroll 1
                for (int q = lane; q < 32 * lines; q += 32) {
                    const int rr = r0 + q / lines;
                    if (rr < C.m)
                        prefetch_l2(aux + static_cast<size_t>(rr) * ld + ctile + (q % lines) * 64);
                }
                if (P.mode == MODE_AXPY_FINAL) {
                    const float* p = P.p_table[gm];
                    if (!C.transposed) {
                        const int plines = (ncols * 4 + 127) / 128;
#pragma unroll 1
                        for (int q = lane; q < 32 * plines; q += 32) {
                            const int rr = r0 + q / plines;
                            if (rr < C.m)
                                prefetch_l2(p + static_cast<size_t>(rr) * C.n + ctile + (q % plines) * 32);
                        }
                    } else {
                        // stored rows ctile .. ctile + ncols, columns r0 .. r0 + 31 (one line each)
#pragma unroll 1
                        for (int q = lane; q < ncols; q += 32)
                            prefetch_l2(p + static_cast<size_t>(ctile + q) * C.m + r0);
                    }
                }
            }
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
            const float s = P.first_iter ? P.inv_norm[gm] : 1.0f;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) +
                                   static_cast<uint32_t>(acc * kBN);
            // Each chunk is a 32 x 32 fp32 block: TMEM rows are lanes, so the block is
            // staged in shared memory and then read back by row segments (8 lanes x 4
            // columns per row, 4 rows per instruction), so every global access of the
            // epilogue is a run of >= 64 contiguous bytes.  A second pass over the
            // stage reads it transposed for the mirrored tile and for weights stored
            // n x m.  Each pass issues all of its global loads before using any.
            const int seg_row = lane >> 3;               // 0..3
            const int seg_col = (lane & 7) * 4;          // 0..28
            float* p = nullptr;
            float* dbg = nullptr;
            float sc = 0.f;
            if (P.mode == MODE_AXPY_FINAL) {
                p = P.p_table[gm];
                dbg = P.dbg_O ? P.dbg_O[gm] : nullptr;
                sc = P.lr * P.aspect[gm];
            }
            const __nv_bfloat16* aux = nullptr;
            __nv_bfloat16* out = nullptr;
            if (sym) {
                aux = P.mode == MODE_POLY ? C.aux + static_cast<size_t>(tc.mat) * mm : nullptr;
                out = C.out + static_cast<size_t>(tc.mat) * mm;
            } else {
                aux = C.aux + static_cast<size_t>(tc.mat) * mn;
                out = P.mode == MODE_AXPY ? C.out + static_cast<size_t>(tc.mat) * mn : nullptr;
            }
            const int ld = sym ? C.m : C.n;
            const bool final_t = (P.mode == MODE_AXPY_FINAL) && C.transposed;
            const bool final_n = (P.mode == MODE_AXPY_FINAL) && !C.transposed;
            for (int ch = 0; ch < kBN / 32; ++ch) {
                uint32_t raw_v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + ch * 32, raw_v);
                const int c0 = ctile + ch * 32;
                const bool live = c0 < climit;  // warp-uniform
                // issue this chunk's global loads while the TMEM load is in flight
                uint2 araw[8];
                float4 praw[8];
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int grow = r0 + it * 4 + seg_row;
                    const int gcol = c0 + seg_col;
                    araw[it] = make_uint2(0u, 0u);
                    praw[it] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (live && grow < C.m && gcol < climit) {
                        const size_t off = static_cast<size_t>(grow) * ld + gcol;
                        if (aux) araw[it] = *reinterpret_cast<const uint2*>(aux + off);
                        if (final_n) praw[it] = *reinterpret_cast<const float4*>(p + off);
                    }
                    if (final_t) {
                        // weights stored n x m: the pass-2 layout (stored row c0 + jj, columns r0 + rq ..)
                        const int jj = it * 4 + seg_row;
                        if (live && c0 + jj < climit && r0 + seg_col < C.m)
                            praw[it] = *reinterpret_cast<const float4*>(p + static_cast<size_t>(c0 + jj) * C.m + r0 +
                                                                        seg_col);
                    }
                }
                tmem_ld_wait();
                if (!live) continue;
#pragma unroll
                for (int j = 0; j < 32; ++j) stage[lane][j] = __uint_as_float(raw_v[j]);
                __syncwarp();
                const bool mirror = sym && c0 >= (tc.rb + 1) * kBM;
                // ---- pass 1: row segments of the oriented tile
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int i = it * 4 + seg_row;
                    const int grow = r0 + i;
                    const int gcol = c0 + seg_col;
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = stage[i][seg_col + e];
                    if (grow >= C.m || gcol >= climit) continue;
                    const size_t off = static_cast<size_t>(grow) * ld + gcol;
                    const float a[4] = {bf16_lo(araw[it].x), bf16_hi(araw[it].x), bf16_lo(araw[it].y),
                                        bf16_hi(araw[it].y)};
                    if (P.mode == MODE_GRAM) {
                        const float s2 = s * s;
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] *= s2;
                        store_bf16x4(out, off, o);
                    } else if (P.mode == MODE_POLY) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] = fmaf(P.cc, o[e], P.cb * a[e]);
                        store_bf16x4(out, off, o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] = s * fmaf(P.ca, a[e], o[e]);
                        if (P.mode == MODE_AXPY) {
                            store_bf16x4(out, off, o);
                        } else if (final_n) {
                            float4 w = praw[it];
                            w.x = fmaf(-sc, o[0], w.x);
                            w.y = fmaf(-sc, o[1], w.y);
                            w.z = fmaf(-sc, o[2], w.z);
                            w.w = fmaf(-sc, o[3], w.w);
                            *reinterpret_cast<float4*>(p + off) = w;
                            if (dbg) *reinterpret_cast<float4*>(dbg + off) = make_float4(o[0], o[1], o[2], o[3]);
                        }
                    }
                    if (mirror || final_t) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) stage[i][seg_col + e] = o[e];
                    }
                }
                if (!(mirror || final_t)) continue;  // warp-uniform
                __syncwarp();
                // ---- pass 2: the transposed block (stored row c0 + jj, columns r0 + rq ..)
                const int rq = seg_col;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int jj = it * 4 + seg_row;
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = stage[rq + e][jj];
                    if (c0 + jj >= climit || r0 + rq >= C.m) continue;
                    const size_t off = static_cast<size_t>(c0 + jj) * C.m + r0 + rq;
                    if (mirror) {
                        store_bf16x4(out, off, o);
                    } else {
                        // weights stored n x m: O_stored[c][r] = O[r][c]
                        float4 w = praw[it];
                        w.x = fmaf(-sc, o[0], w.x);
                        w.y = fmaf(-sc, o[1], w.y);
                        w.z = fmaf(-sc, o[2], w.z);
                        w.w = fmaf(-sc, o[3], w.w);
                        *reinterpret_cast<float4*>(p + off) = w;
                        if (dbg) *reinterpret_cast<float4*>(dbg + off) = make_float4(o[0], o[1], o[2], o[3]);
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
