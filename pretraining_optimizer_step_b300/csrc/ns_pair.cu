// ns_pair.cu -- the Newton-Schulz GEMMs of the Muon step on CTA pairs.
//
// One iteration of the quintic loop ("Cara Melatih ChatGPT Sendiri dengan
// Budget 50 Dolar", section "2. Pengoptimal Muon", orthogonalization loop) is
// three launches of this kernel over every matrix of the step (grouped by
// oriented shape class), one per mode:
//   MODE_GRAM        A = s^2 X X^T               tiles on/above the diagonal, upper blocks stored
//   MODE_POLY        B' = b A + c A A + a I      A symmetric: A A = A A^T, same operand both sides
//   MODE_AXPY        X' = s B' X                 X read MN-major as the B operand
//   MODE_AXPY_FINAL  O = s B' X in fp32, p += -lr sqrt(max(1, r/c)) O (TMA reduce-add)
//   MODE_AXPY_O      O = s B' X, stored in bf16 (stored layout) for the NorMuon pass
// Folding a I into the polynomial makes a X + B X = (B + a I) X a plain product, so the
// axpy epilogues read nothing but the accumulator; the only numerical change is one bf16
// rounding of B's diagonal entries plus a.  The final launch never reads the weights: it
// writes the fp32 weight change -lr s O to shared memory and a TMA reduce-add folds it into
// p in L2 (p' = p + fp32(-lr s O)).
//
// A cluster of two CTAs (one per SM) computes a 256 x N tile with
// tcgen05.mma.cta_group::2: CTA rank r holds rows [128 r, 128 r + 128) of the A
// operand and half of the N rows of the B operand in its shared memory, and
// receives its 128 accumulator rows in its own TMEM.  Per SM this halves the B
// operand traffic against a 128 x 256 single-CTA tile.
//   Gram/poly: with an even number of 128-row blocks, tile = row blocks (2 rp, 2 rp + 1)
//              x column blocks (2 q, 2 q + 1), rp <= q; the lower block of a diagonal
//              tile is computed but not stored.  With an odd number, tile = row blocks
//              (2 rp, 2 rp + 1) x column blocks (2 q - 1, 2 q) for rp < q, and for rp = q
//              the diagonal block 2 rp alone as an M = 128, N = 128 tile: every block
//              on or above the diagonal is computed once and nothing below it.
// Symmetric storage: A and B' are stored as their 128 x 128 blocks on and above
// the diagonal (diagonal blocks in full); nothing below is written.  A GEMM that
// reads A or B' as an operand takes a K panel that lies below the diagonal from
// the stored block across it, transposed: the same 64 x 128 TMA box with the
// coordinates swapped, consumed as an MN-major operand.  The two CTAs of a pair
// share one instruction descriptor, so a stage is read transposed on both
// halves when its K block is at or left of the pair's first row block (the
// diagonal block there is symmetric and stored whole, so either orientation of
// it is correct).
//   axpy:      tile = row blocks (2 rp, 2 rp + 1) x columns [256 ct, 256 ct + N).
// Half tiles: when a matrix has an odd number of 128-row blocks, its last row pair has
// one real block.  Those tiles run as M = 128 pair MMAs: each CTA loads 64 rows of that
// block, and each CTA's 64 x N accumulator is folded into TMEM as lanes 0..63 = columns
// [0, N/2), lanes 64..127 = columns [N/2, N), TMEM columns 0..N/2 - 1.  So every epilogue
// warp takes 32 rows x N/2 columns.
//
// CTA layout (192 threads, persistent over the pair tiles):
//   warp 0      TMA producer (both CTAs): ring of 3 stages (2 in the final launch when it
//               also stores the debug copy of O) of
//               {A 128 x 128, B-half <= 128 x 128} bf16 as 64-wide K panels; the loads
//               of both CTAs complete on the even CTA's mbarrier
//   warp 1      TMEM allocation (both CTAs); lane 0 of the even CTA issues 8 MMAs
//               (M 256, N 256/128, K 16) per stage and commits to both CTAs' barriers
//   warps 2..5  epilogue (both CTAs): per warp 32 rows, in chunks of 64 columns (Gram,
//               polynomial, axpy: bf16) or 32 columns (the final launch's fp32 weight
//               change, the bf16 O of the NorMuon step).  The polynomial's input (the A
//               subtile) arrives by TMA one chunk ahead into a swizzled shared slot that
//               then holds the chunk's output; outputs leave by TMA store (reduce-add
//               for the weights) from swizzled slots, and a slot is rewritten only once
//               the store that last read it has read it (one bulk group per chunk).
//               Threads touch shared memory only with conflict-free 16-byte vectors
//               (row access) or 4-byte/2-byte column access (transposes).
// Every wait is bounded; on expiry the CTA latches STATUS_TIMEOUT, raises its
// abort flag, lets its own copies land, and joins the final cluster barrier.
// Launches use programmatic dependent launch: a launch's CTAs take the SMs the previous
// launch releases, run the prologue (barriers, TMEM, descriptor prefetch), and wait
// (griddepcontrol.wait) for the previous grid before touching global memory.
#include "kernels.cuh"
#include "ptx.cuh"

namespace muon {

namespace {

struct PairTile {
    int ci;      // class
    int mat;     // matrix within the class
    int rb0;     // the pair's first row block
    int rb;      // this CTA's row block (128 rows; a half tile's single block for both CTAs)
    int row0;    // this CTA's first oriented row: rb * 128, or in a half tile rb0 * 128 + 64 rank
    int half_m;  // M = 128 tile (the pair's second row block does not exist)
    int c0;      // first output column of the tile
    int ncols;   // N: 256 or 128
};

__device__ __forceinline__ PairTile decode_pair_tile(const PairParams& P, int t, int rank, bool sym) {
    PairTile pt;
    int ci = 0;
    while (ci + 1 < P.nclasses && t >= P.cls[ci + 1].tile_begin) ++ci;
    const PairClass& C = P.cls[ci];
    const int local = t - C.tile_begin;
    pt.ci = ci;
    pt.mat = local / C.tiles_per_mat;
    const int lt = local - pt.mat * C.tiles_per_mat;
    if (sym) {
        // column step q has q + 1 tiles (row pairs rp = 0..q)
        int q = 0, base = 0;
        while (base + q + 1 <= lt) {
            base += q + 1;
            ++q;
        }
        const int rp = lt - base;
        pt.rb0 = 2 * rp;
        if ((C.row_blocks & 1) == 0) {
            // even block count: row blocks (2rp, 2rp+1) x column blocks (2q, 2q+1); the diagonal tile
            // (rp = q) computes its lower block too
            pt.c0 = 256 * q;
            pt.ncols = 256;
            pt.half_m = 0;
        } else if (rp < q) {
            // odd block count: row blocks (2rp, 2rp+1) x column blocks (2q-1, 2q), all on or above the
            // diagonal
            pt.c0 = 128 * (2 * q - 1);
            pt.ncols = 256;
            pt.half_m = 0;
        } else {
            // odd block count, rp = q: the diagonal block 2rp alone (M = 128, N = 128)
            pt.c0 = 256 * rp;
            pt.ncols = 128;
            pt.half_m = 1;
        }
    } else {
        const int rp = lt / C.col_groups;
        const int ct = lt - rp * C.col_groups;
        pt.rb0 = 2 * rp;
        pt.c0 = 256 * ct;
        pt.ncols = (C.n - pt.c0 > 128) ? 256 : 128;
        pt.half_m = pt.rb0 + 1 >= C.row_blocks ? 1 : 0;
    }
    pt.rb = pt.half_m ? pt.rb0 : pt.rb0 + rank;
    pt.row0 = pt.half_m ? pt.rb0 * 128 + 64 * rank : pt.rb * 128;
    return pt;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offsets inside the swizzled 32 x 32 subtiles the epilogue TMA maps use.
// bf16, 64-byte rows, 64B swizzle: 16-byte unit u of row r lives at unit u ^ ((r >> 1) & 3).
__device__ __forceinline__ uint32_t sw64_unit(int r, int u) { return r * 64 + ((u ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ uint32_t sw64_elem(int r, int c) { return sw64_unit(r, c >> 3) + ((c & 7) << 1); }
// fp32, 128-byte rows, 128B swizzle: 16-byte unit u of row r lives at unit u ^ (r & 7).
__device__ __forceinline__ uint32_t sw128_unit(int r, int u) { return r * 128 + ((u ^ (r & 7)) << 4); }
__device__ __forceinline__ uint32_t sw128_elem(int r, int c) { return sw128_unit(r, c >> 2) + ((c & 3) << 2); }

__device__ __forceinline__ void latch_status(unsigned int* status, unsigned int bits) { atomicOr(status, bits); }

// Bounded spin on the global timer (lets copies still in flight land before
// an aborting CTA leaves).
__device__ __forceinline__ void settle_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    ns_pair_kernel(const __grid_constant__ PairParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kPairMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kPairMaxStages];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ __align__(8) uint64_t in_bar[4][4];
    __shared__ uint32_t tmem_base_slot;
    __shared__ volatile int abort_flag;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t tiles_base = (raw + 1023u) & ~1023u;
    uint8_t* tiles_ptr = smem_raw + (tiles_base - raw);
    const bool final_mode = P.mode == MODE_AXPY_FINAL;
    const bool dbg_o = final_mode && P.dbg_maps != nullptr;   // debug copy of O in the final launch
    const int nstages = dbg_o ? 2 : 3;
    const int epi_warp_bytes = dbg_o ? 24576 : 8192;
    uint8_t* epi_ptr = tiles_ptr + nstages * kPairStageBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;
    const int cluster = static_cast<int>(cluster_id_x());
    const int nclusters = static_cast<int>(cluster_count_x());
    const bool sym = (P.mode == MODE_GRAM || P.mode == MODE_POLY);
    // The launch's tile list must be the one its classes describe (consecutive, non-empty
    // classes whose tile counts add up to total_tiles).  Every CTA checks the same parameters
    // and reaches the same verdict; on a mismatch the status word gets STATUS_BOUNDS and
    // every role's tile loop is empty, so no tile is decoded out of range and every role
    // still reaches the exit barrier.
    int expect_tiles = 0;
    bool params_ok = P.nclasses >= 1 && P.nclasses <= kMaxClasses && P.total_tiles >= 0;
    for (int c = 0; params_ok && c < P.nclasses; ++c) {
        const PairClass& C = P.cls[c];
        params_ok = C.tile_begin == expect_tiles && C.nmats >= 1 && C.tiles_per_mat >= 1 && C.k_blocks >= 1 &&
                    C.row_blocks >= 1 && C.m >= 8 && C.n >= C.m;
        expect_tiles += C.tiles_per_mat * C.nmats;
    }
    params_ok = params_ok && expect_tiles == P.total_tiles;
    const int total_tiles = params_ok ? P.total_tiles : 0;
    // The next launch on the stream (the next Newton-Schulz GEMM) may start launching now: its CTAs
    // take SMs only as this grid's CTAs exit, and run their prologue while the last tiles finish.
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairMaxStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull_bar[a], 1);
            mbar_init(&tempty_bar[a], 8);  // one arrive per epilogue warp of both CTAs
        }
        mbar_init(&drain_bar, 1);
        for (int w = 0; w < 4; ++w)
            for (int sl = 0; sl < 4; ++sl) mbar_init(&in_bar[w][sl], 1);
        abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc_pair(&tmem_base_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;
    // everything above touched only shared memory, TMEM and the launch parameters; the previous
    // kernel's outputs (this launch's operands) and the buffers it read are safe from here on
    griddep_wait();
    if (!params_ok && threadIdx.x == 0 && rank == 0 && cluster == 0) atomicOr(P.status, STATUS_BOUNDS);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        for (int c = 0; c < P.nclasses; ++c) {
            tma_prefetch_desc(&P.tmA[c]);
            tma_prefetch_desc(&P.tmB[c]);
        }
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        bool injected = false;
        for (int t = cluster; t < total_tiles && !aborted; t += nclusters) {
            const PairTile pt = decode_pair_tile(P, t, rank, sym);
            const PairClass& C = P.cls[pt.ci];
            const CUtensorMap* mA = &P.tmA[pt.ci];
            const CUtensorMap* mB = &P.tmB[pt.ci];
            const int half = pt.ncols >> 1;             // this CTA's B-side rows/columns: 64 or 128
            const int b0 = pt.c0 + rank * half;         // first of them
            // symmetric operands read from upper-block storage: first row / column block of the pair
            const bool a_symm = P.mode != MODE_GRAM;    // poly: A; axpy: B'
            const int a_first = pt.rb0;                 // the pair's first row block
            const int b_first = pt.c0 >> 7;             // the pair's first column block (poly)
            const uint32_t a_bytes = pt.half_m ? 16384u : 32768u;  // this CTA's A rows x 128 K
            // a diagonal tile of a symmetric product (N = 256, or the M = 128 diagonal block): each CTA's
            // half of the B operand is its own A panel (same rows, K block and orientation), so only the
            // A panels are loaded
            const bool diag = sym && b_first == a_first;
            const uint32_t total_bytes =
                diag ? 2u * a_bytes : 2u * (a_bytes + static_cast<uint32_t>(half) * kPairBK * 2u);
            for (int kb = 0; kb < C.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_flag, P.timeout_ns)) {
                    latch_status(P.status, STATUS_TIMEOUT);
                    abort_flag = 1;
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles_ptr + stage * kPairStageBytes;  // A: K panels at +0, +16 KiB
                uint8_t* sb = sa + 2 * kPairPanelBytes;               // B half: panels at +32, +48 KiB
                const int k0 = kb * kPairBK;
                const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);
                if (leader) mbar_arrive_expect_tx(&full_bar[stage], total_bytes);
                const bool a_tr = a_symm && kb <= a_first;   // this K block is below the stored triangle
                for (int h = 0; h < 2; ++h) {
                    if (a_tr && pt.half_m && h == 1) break;  // a half tile's 64 rows are one MN-major panel
                    if (P.inject_lost_load && leader && !injected && cluster == 0) {
                        injected = true;  // test hook: this A panel never arrives
                    } else if (a_tr) {
                        // MN-major: 64 of this CTA's rows (as columns of the stored block) x 128 K rows
                        tma_load_3d_pair(sa + h * kPairPanelBytes, mA, bar, pt.row0 + 64 * h, k0, pt.mat);
                    } else if (pt.half_m) {
                        // K-major, 64 rows: box 64 (K) x 64 rows
                        tma_load_3d_pair(sa + h * kPairPanelBytes, &P.tmA64[pt.ci], bar, k0 + 64 * h, pt.row0, pt.mat);
                    } else {
                        tma_load_3d_pair(sa + h * kPairPanelBytes, mA, bar, k0 + 64 * h, pt.row0, pt.mat);
                    }
                }
                if (diag) {
                    // the B halves are the A panels just loaded
                } else if (sym) {
                    const bool b_tr = P.mode == MODE_POLY && kb <= b_first;
                    if (b_tr) {
                        // MN-major B half: one 64 x 128 panel per 64 of this CTA's N rows
                        for (int j = 0; j < half / 64; ++j)
                            tma_load_3d_pair(sb + j * kPairPanelBytes, mA, bar, b0 + 64 * j, k0, pt.mat);
                    } else {
                        // K-major B half: 128 rows (box of tmA) or 64 rows (box of tmB) per K panel
                        const CUtensorMap* mBs = half == 128 ? mA : mB;
                        for (int h = 0; h < 2; ++h)
                            tma_load_3d_pair(sb + h * kPairPanelBytes, mBs, bar, k0 + 64 * h, b0, pt.mat);
                    }
                } else {
                    // MN-major X: one 64-column x 128-K panel per 64 columns of the B half
                    for (int j = 0; j < half / 64; ++j)
                        tma_load_3d_pair(sb + j * kPairPanelBytes, mB, bar, b0 + 64 * j, k0, pt.mat);
                }
                if (++stage == nstages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (aborted) settle_ns(100000);
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool aborted = false;
        bool issued = false;  // any MMA issued (only then is there anything to drain)
        for (int t = cluster; t < total_tiles && !aborted; t += nclusters) {
            const PairTile pt = decode_pair_tile(P, t, 0, sym);
            const PairClass& C = P.cls[pt.ci];
            const bool a_symm = P.mode != MODE_GRAM;
            const int a_first = pt.rb0;           // the pair's first row block
            const int b_first = pt.c0 >> 7;
            const bool diag = sym && b_first == a_first;  // B halves = A panels
            if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, &abort_flag, P.timeout_ns)) {
                latch_status(P.status, STATUS_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
            for (int kb = 0; kb < C.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&full_bar[stage], phase, &abort_flag, P.timeout_ns)) {
                    latch_status(P.status, STATUS_TIMEOUT);
                    abort_flag = 1;
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = tiles_base + stage * kPairStageBytes;
                const uint32_t sb = diag ? sa : sa + 2 * kPairPanelBytes;
                const int a_mn = (a_symm && kb <= a_first) ? 1 : 0;
                const int b_mn = sym ? ((P.mode == MODE_POLY && kb <= b_first) ? 1 : 0) : 1;
                const uint32_t idesc = idesc_bf16_f32_ab(pt.half_m ? 128 : 256, pt.ncols, a_mn, b_mn);
#pragma unroll
                for (int kk = 0; kk < kPairBK / 16; ++kk) {
                    // K-major: K panel kk / 4, 32 B per 16 of K; MN-major: 64-wide atoms 16 KiB apart,
                    // 2 KiB per 16 of K
                    const uint32_t kpan = (kk >> 2) * kPairPanelBytes + (kk & 3) * 32;
                    const uint64_t adesc = a_mn ? smem_desc_sw128(sa + kk * 2048, kPairPanelBytes, 1024)
                                                : smem_desc_sw128(sa + kpan, 16, 1024);
                    const uint64_t bdesc = b_mn ? smem_desc_sw128(sb + kk * 2048, kPairPanelBytes, 1024)
                                                : smem_desc_sw128(sb + kpan, 16, 1024);
                    tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                issued = true;
                tc_commit_pair_multicast(&empty_bar[stage], 0x3);
                if (++stage == nstages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            tc_commit_pair_multicast(&tfull_bar[acc], 0x3);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // every MMA issued must finish before TMEM is released
        if (issued) {
            tc_commit_pair_multicast(&drain_bar, 0x1);
            mbar_wait_bounded(&drain_bar, 0, nullptr, P.timeout_ns);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int lg = warp & 3;                       // TMEM lane group of this warp
        uint8_t* wbase = epi_ptr + lg * epi_warp_bytes;
        const bool has_in = P.mode == MODE_POLY;
        // The warp's epilogue slots, by mode (output slots alternate per committed store group, and
        // a slot is rewritten once the group that last read it -- n_out groups back -- has):
        //   gram, axpy (8 KiB): 2 output slots of a bf16 32 x 64 subtile
        //   poly (8 KiB):    2 slots of a bf16 32 x 64 subtile, each first the input (the A subtile,
        //                    loaded by TMA) and then, overwritten in place, the output B'; chunk c uses
        //                    slot c % 2, and its slot is refilled with chunk c + 2 once chunk c's store
        //                    has read it
        //   final (8 KiB):   2 output slots of the fp32 32 x 32 weight change -lr s O
        //   final, debug copy of O (24 KiB): 2 output slot pairs {weight change, O} of 8 KiB
        //   axpy_o (8 KiB):  4 output slots of bf16 32 x 32 (O in the stored layout)
        // Gram, polynomial and axpy take 64 columns per chunk: one slot wait, fence and TMA store per
        // 32 x 64 subtile halves that fixed cost per element, which bounds tiles with short K.
        const bool f32_out = final_mode;
        const bool wide = P.mode == MODE_GRAM || P.mode == MODE_AXPY || P.mode == MODE_POLY;
        const int cw = wide ? 64 : 32;  // columns per chunk
        const int n_in = has_in ? 2 : 0;
        const int in_stride = 4096;
        const int n_out = (f32_out || wide) ? 2 : 4;
        const int out_stride = dbg_o ? 8192 : ((f32_out || wide) ? 4096 : 2048);
        uint8_t* out_base = wbase + n_in * in_stride;
        auto in_b16 = [&](int sl) { return wbase + sl * in_stride; };
        uint64_t* ibar = in_bar[lg];
        uint32_t in_phase_bits = 0u, in_pending_bits = 0u;
        uint32_t groups = 0;  // bulk store groups committed by lane 0 (output slot = groups % n_out)
        const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty_bar[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty_bar[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool stores_issued = false;
        for (int t = cluster; t < total_tiles; t += nclusters) {
            const PairTile pt = decode_pair_tile(P, t, rank, sym);
            const PairClass& C = P.cls[pt.ci];
            const int gm = C.mat_base + pt.mat;
            // this warp's 32 rows and first column: a half tile folds each CTA's 64 rows x N columns
            // into lanes 0..63 (columns [0, N/2)) and 64..127 (columns [N/2, N))
            const int grow0 = pt.row0 + (pt.half_m ? (lg & 1) * 32 : lg * 32);  // first oriented row
            const int cb = pt.half_m ? (lg >> 1) * (pt.ncols >> 1) : 0;          // column offset in the tile
            const bool warp_rows = pt.rb < C.row_blocks && grow0 < C.m;
            const int climit = sym ? C.m : C.n;
            const int nch = (pt.half_m ? pt.ncols >> 1 : pt.ncols) / cw;
            const bool transposed = C.transposed != 0;
            const CUtensorMap* pmap = final_mode ? &P.p_maps[gm] : nullptr;
            // a chunk is live when this warp has rows, its columns exist, and (Gram/poly) its
            // 128-column block is not below the diagonal for this row block
            auto live = [&](int ch) {
                const int cc0 = pt.c0 + cb + ch * cw;
                if (!warp_rows || cc0 >= climit) return false;
                if (sym && (cc0 >> 7) < pt.rb) return false;
                return true;
            };
            auto issue_in = [&](int ch) {  // lane 0 only; only when n_in > 0 (polynomial: the A subtile)
                const int slot = ch % n_in;
                const int cc0 = pt.c0 + cb + ch * cw;
                mbar_arrive_expect_tx(&ibar[slot], 4096u);
                tma_load_3d(in_b16(slot), &P.tmIn[pt.ci], &ibar[slot], cc0, grow0, pt.mat);
                in_pending_bits |= 1u << slot;
            };
            // polynomial: load chunk c + 2 into chunk c's slot, once every store has read its slot
            auto refill = [&](int ch) {
                if (has_in && lane == 0 && ch + n_in < nch && live(ch + n_in)) {
                    bulk_wait_group_read0();
                    issue_in(ch + n_in);
                }
            };
            if (has_in && lane == 0) {
                bulk_wait_group_read0();  // the previous tile's last stores have read both slots
                for (int ch = 0; ch < n_in && ch < nch; ++ch)
                    if (live(ch)) issue_in(ch);
            }
            const bool ready = __all_sync(0xffffffffu, mbar_wait_bounded(&tfull_bar[acc], acc_phase, &abort_flag,
                                                                         P.timeout_ns));
            if (!ready) {
                if (lane == 0) latch_status(P.status, STATUS_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const float s = P.first_iter ? P.inv_norm[gm] : 1.0f;
            const float sc = final_mode ? P.lr * P.aspect[gm] : 0.f;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + static_cast<uint32_t>(acc * 256);
            bool failed = false;
            for (int ch = 0; ch < nch; ++ch) {
                if (wide) {
                    // Gram (A = s^2 acc), axpy (X' = s acc) and polynomial (B' = c acc + b A + a I):
                    // a 32 x 64 bf16 subtile per chunk
                    uint32_t r0[32], r1[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(t_row + ch * 64, r0);
                    tmem_ld_32x32b_x32(t_row + ch * 64 + 32, r1);
                    tmem_ld_wait();
                    if (ch == nch - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                    }
                    if (!live(ch)) {
                        refill(ch);
                        continue;
                    }
                    const int cc0 = pt.c0 + cb + ch * 64;
                    float v[64];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        v[j] = __uint_as_float(r0[j]);
                        v[32 + j] = __uint_as_float(r1[j]);
                    }
                    uint8_t* out_slot;
                    if (has_in) {
                        const int slot = ch & 1;
                        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ibar[slot], (in_phase_bits >> slot) & 1u,
                                                                                  &abort_flag, P.timeout_ns));
                        if (!ok) {
                            if (lane == 0) latch_status(P.status, STATUS_TIMEOUT);
                            abort_flag = 1;
                            failed = true;
                            break;
                        }
                        in_phase_bits ^= 1u << slot;
                        in_pending_bits &= ~(1u << slot);
                        out_slot = in_b16(slot);
                        // diagonal entries of this 32 x 64 subtile: column j = grow0 - cc0 + lane
                        const int doff = grow0 - cc0;
                        const int djl = (doff == 0 || doff == 32) ? doff + lane : -1;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 w = *reinterpret_cast<const uint4*>(out_slot + sw128_unit(lane, u));
                            const float a[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = 8 * u + e;
                                v[j] = fmaf(P.cc, v[j], P.cb * a[e]) + (j == djl ? P.ca : 0.0f);
                            }
                        }
                        __syncwarp();  // every lane has read the A subtile before B' overwrites it
                    } else {
                        const float f = P.mode == MODE_GRAM ? s * s : s;
#pragma unroll
                        for (int j = 0; j < 64; ++j) v[j] *= f;
                        if (lane == 0) bulk_wait_group_read1();  // the slot's previous store has read it
                        __syncwarp();
                        out_slot = out_base + (groups & 1u) * out_stride;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        uint4 w;
                        w.x = pack2(v[8 * u + 0], v[8 * u + 1]);
                        w.y = pack2(v[8 * u + 2], v[8 * u + 3]);
                        w.z = pack2(v[8 * u + 4], v[8 * u + 5]);
                        w.w = pack2(v[8 * u + 6], v[8 * u + 7]);
                        *reinterpret_cast<uint4*>(out_slot + sw128_unit(lane, u)) = w;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&P.tmOut[pt.ci], out_slot, cc0, grow0, pt.mat);
                        bulk_commit_group();
                        stores_issued = true;
                    }
                    ++groups;
                    refill(ch);
                    continue;
                }
                uint32_t raw_v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + ch * 32, raw_v);
                tmem_ld_wait();
                if (ch == nch - 1) {
                    // the accumulator is no longer read: hand it back to the MMA issuer
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                }
                // final and axpy_o: 32 x 32 subtiles (fp32 weight change, or bf16 O in the stored layout)
                if (live(ch)) {
                    const int cc0 = pt.c0 + cb + ch * 32;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw_v[j]) * s;
                    // the output slot about to be written must no longer be read by the store group
                    // that last used it, n_out groups back (the most recent n_out - 1 may still read)
                    if (lane == 0) {
                        if (n_out == 2) bulk_wait_group_read1();
                        else bulk_wait_group_read3();
                    }
                    __syncwarp();
                    uint8_t* out_slot = out_base + (groups % static_cast<uint32_t>(n_out)) * out_stride;
                    if (final_mode) {
                        // the fp32 weight change -sc O in the stored layout (rows = stored rows);
                        // a transposed subtile has stored rows = oriented columns j, columns = lanes
                        if (!transposed) {
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                *reinterpret_cast<float4*>(out_slot + sw128_unit(lane, u)) =
                                    make_float4(-sc * v[4 * u], -sc * v[4 * u + 1], -sc * v[4 * u + 2],
                                                -sc * v[4 * u + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                *reinterpret_cast<float*>(out_slot + sw128_elem(j, lane)) = -sc * v[j];
                        }
                        if (dbg_o) {
                            uint8_t* o_slot = out_slot + 4096;
                            if (!transposed) {
#pragma unroll
                                for (int u = 0; u < 8; ++u)
                                    *reinterpret_cast<float4*>(o_slot + sw128_unit(lane, u)) =
                                        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    *reinterpret_cast<float*>(o_slot + sw128_elem(j, lane)) = v[j];
                            }
                        }
                    } else if (transposed) {
                        // bf16 O subtile in the stored layout: stored rows are oriented columns j,
                        // stored columns are lanes (one 64-byte row per j, 2 bytes per lane)
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            *reinterpret_cast<__nv_bfloat16*>(out_slot + sw64_elem(j, lane)) = __float2bfloat16_rn(v[j]);
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint4 w;
                            w.x = pack2(v[8 * u + 0], v[8 * u + 1]);
                            w.y = pack2(v[8 * u + 2], v[8 * u + 3]);
                            w.z = pack2(v[8 * u + 4], v[8 * u + 5]);
                            w.w = pack2(v[8 * u + 6], v[8 * u + 7]);
                            *reinterpret_cast<uint4*>(out_slot + sw64_unit(lane, u)) = w;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (final_mode) {
                            if (transposed) tma_reduce_add_2d(pmap, out_slot, grow0, cc0);
                            else tma_reduce_add_2d(pmap, out_slot, cc0, grow0);
                            if (dbg_o) {
                                if (transposed) tma_store_2d(&P.dbg_maps[gm], out_slot + 4096, grow0, cc0);
                                else tma_store_2d(&P.dbg_maps[gm], out_slot + 4096, cc0, grow0);
                            }
                        } else {  // axpy_o
                            if (transposed) tma_store_2d(&P.o_maps[gm], out_slot, grow0, cc0);
                            else tma_store_2d(&P.o_maps[gm], out_slot, cc0, grow0);
                        }
                        bulk_commit_group();
                        stores_issued = true;
                    }
                    ++groups;  // every lane keeps the count (warp-uniform)
                }
            }
            if (failed) break;
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) {
            // loads still in flight (after an abort) must land before shared memory goes away
            for (int sl = 0; sl < n_in; ++sl)
                if ((in_pending_bits >> sl) & 1u) mbar_wait_bounded(&ibar[sl], (in_phase_bits >> sl) & 1u, nullptr, P.timeout_ns);
            if (stores_issued) bulk_wait_group0();
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // no CTA of the pair touches the other's shared memory or TMEM after this
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

cudaError_t ns_pair_prepare(int* max_clusters) {
    cudaError_t e = cudaFuncSetAttribute(ns_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, ns_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    *max_clusters = n;
    return cudaSuccess;
}

// Launched with programmatic stream serialization: the CTAs of a launch that follows another
// Newton-Schulz launch (or the momentum pass) start their prologue on SMs the previous grid has
// released, and wait in the kernel for its completion.
cudaError_t launch_ns_pair(const PairParams& p, int clusters, cudaStream_t s) {
    if (p.total_tiles <= 0 || clusters <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ns_pair_kernel, p);
}

}  // namespace muon
