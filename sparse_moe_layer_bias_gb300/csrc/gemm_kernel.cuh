// gemm_kernel.cuh -- persistent GEMM on the sm_103a tensor cores (tcgen05; bf16 x bf16,
// or e4m3 x e4m3 for the FP8 expert variant), used for every contraction of
// the Stable LatentMoE layer:
//   a1  h   = x W_down^T                       (A dense, B plain, bf16 out)
//   a2  s   = sigmoid(h W_router^T)            (A dense, B plain, fp32 out)
//   a5  act = SiTU(h W1^T) * softcap(h W2^T)   (A = h rows of the expert's
//            tokens, gathered with cp.async, 256 rows per tile as two 128-row
//            sub-tiles sharing each weight stage; B = the expert's W1|W2 rows)
//   a6  o   = gate * act W3^T                  (A = permuted act rows, B = the
//            expert's W3, rows scattered back to assignment order)
//   a8  y   = r W_up^T + shared_act Ws3^T       (K split over two A/B sources)
//   a8' shared_act = SiTU(x Ws1^T) * softcap(x Ws2^T)
// (SiTU-GLU: "Kimi-K3-Architecture-Deep-Dive" section 1; the layer's chain of
// projections: same page, section 2.)  In the FP8 variant a5 and a6 take e4m3
// operands (kind::f8f6f4, a K block of 128 elements = the same 128-byte rows)
// and their epilogues apply the power-of-two row scales: a5 writes e4m3(4 act),
// a6 undoes the 4 with the W3 row scale and the gate.
// For training (gemm_bwd.cu): EPI_SITU_GLU_SAVE (a5 / a8' that also keep the
// pre-activations p1 | p2 for the backward), EPI_F32 (fp32 weight gradients)
// and per-expert K segments (KSEG: each tile names its own K range, for the
// routed experts' weight gradients, whose output goes out by TMA store).
//
// Structure (one CTA per SM, 192 threads; 320 with the A gather):
//   warp 0      TMA producer: per 64-wide K block, one box of A and one or two
//               boxes of B into a STAGES-deep ring
//               of 128B-swizzled shared-memory tiles;
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (M=128, N=BN, K=16) x4 per stage (x2 for the two sub-tiles
//               of a pair tile) into TMEM and commits stage release / tile
//               completion.  Single tiles use two TMEM accumulators (the
//               epilogue of one overlaps the MMAs of the next); pair tiles
//               use the 512 columns for their two sub-tiles;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               the fused activation, and the global stores; releases the
//               accumulator so the next tile's MMAs overlap this epilogue;
//   warps 6..9  (gather mode only) copy the A rows named by a row list into
//               the stage with cp.async.
// All threads pass griddepcontrol.wait after the prologue (barrier init, TMEM
// allocation), so the kernel can be a programmatic dependent launch.
//
// CTA pairs (CG2, dense GEMMs fed by TMA; gemm_pair.cu): a cluster of two CTAs
// on two SMs computes a 256 x BN tile.  Each CTA's producer loads its own 128
// rows of A and half of the B rows; both CTAs' copies complete on CTA 0's
// stage barrier.  CTA 0's MMA thread issues tcgen05.mma.cta_group::2 (M = 256),
// which reads the operands from both CTAs' shared memory and leaves each
// CTA's 128 accumulator rows in that CTA's TMEM (allocated for the pair with
// cta_group::2), and its commits arrive on the barriers of both CTAs
// (multicast).  Each CTA's epilogue handles its own rows and releases the
// accumulator on CTA 0's barrier (one arrival per warp).  Before leaving, each
// CTA waits until every release aimed at it has arrived, and the pair meets at
// a cluster barrier before freeing TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "kernels.h"
#include "ptx.cuh"

namespace lmoe {

namespace {

constexpr int kThreads = 192;
constexpr int kTmemCols = 512;  // two accumulators of up to 256 fp32 columns
constexpr int kAccStride = 256;

// CG2: the tile is 256 x BN on a CTA pair; each CTA holds 128 rows of A and
// BN / 2 rows of B per stage.
template <int BN, bool PAIR, bool KSEG = false, bool CG2 = false, int EW = 4>
struct Cfg {
    static constexpr int kSub = PAIR ? 2 : 1;           // 128-row sub-tiles per tile
    static constexpr int kABytes = kSub * kBM * kBK * 2; // 16 or 32 KB
    static constexpr int kBRows = CG2 ? BN / 2 : BN;    // B rows per CTA and stage
    static constexpr int kBBytes = kBRows * kBK * 2;    // 14 to 32 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    // (eight epilogue warps, with their staging buffers, leave room for five
    // 32 KB or three 48 KB stages)
    static constexpr int kStages = EW == 8 ? ((kStageBytes <= 32768) ? 5 : 3)
                                           : (kStageBytes <= 32768) ? 6 : (kStageBytes <= 49152) ? 4 : 3;
    static constexpr int kEpiWarps = EW;
    static constexpr int kBarBytes = 256;
    // per epilogue warp: 32 rows x 64 bf16, row pitch 144 B (16 B of padding
    // keeps the 16-byte row writes and the 128-byte row reads conflict-free)
    static constexpr int kStgPitch = 144;
    static constexpr int kStgWarpBytes = 32 * kStgPitch;
    // per epilogue warp: the current tile's per-column scale factors (e4m3
    // epilogues; up to 256 fp32)
    static constexpr int kColWarpBytes = 1024;
    // K segments (fp32 weight gradients): per epilogue warp two 4 KB buffers
    // of a 32 x 32 fp32 block in the 128B-swizzled layout of a TMA store (one
    // for the TMA stores, one for the threads' stores),
    // 1024-byte aligned, in place of the staging and scale-factor areas the
    // other epilogues use (which leaves room for the full stage ring)
    static constexpr size_t kTmaStgOffset = (size_t(kStages) * kStageBytes + kBarBytes + 1023) / 1024 * 1024;
    static constexpr int kTmaStgWarpBytes = 2 * 4096;
    static constexpr size_t kSmem =
        KSEG ? 1024 + kTmaStgOffset + 4 * kTmaStgWarpBytes
             : 1024 + size_t(kStages) * kStageBytes + kBarBytes + EW * kStgWarpBytes + EW * kColWarpBytes;
    static_assert(kSmem <= 232448, "more dynamic shared memory than a CTA may have (227 KB)");
};

struct Tile {
    int row0;    // first output row (dense) / first permuted row (grouped) /
                 // first row of the expert's output block (K segments)
    int nrows;   // valid rows in this tile (<= 128, or <= 256 for pair tiles)
    int nt;      // N tile index
    int expert;  // grouped: expert id
    int k0, nk;  // first K block and number of K blocks
    int ks;      // dense split-K: the K range this tile sums (0 otherwise)
};

// CG2 (dense only): M tiles are 256 rows; CTA `rank` of the pair owns rows
// 128 * rank .. of the tile (nrows may then be <= 0: no valid rows).
template <bool GROUPED, bool KSEG = false, bool CG2 = false>
__device__ __forceinline__ Tile tile_at(const GemmArgs &a, int t, int n_m, uint32_t rank = 0) {
    Tile ti;
    ti.k0 = 0;
    ti.nk = a.k_blocks;
    ti.ks = 0;
    if (KSEG) {
        // per-expert K segments (weight gradients): {expert, first K block,
        // K blocks, first row of the expert's output block}
        const int mt = t / a.n_tiles;
        ti.nt = t % a.n_tiles;
        const int4 d = a.tiles[mt];
        ti.expert = d.x;
        ti.k0 = d.y;
        ti.nk = d.z;
        ti.row0 = d.w;
        ti.nrows = min(kBM, a.m_rows - d.w);
        if (kDebugChecks && !(idx_ok(mt, a.lim_tiles) && idx_ok(d.x, a.lim_experts) && d.y >= 0 && d.z >= 0 &&
                              d.w >= 0)) {
            ti.expert = 0;   // a bad entry becomes an empty tile
            ti.k0 = ti.nk = ti.row0 = ti.nrows = 0;
        }
    } else if (GROUPED) {
        // M-tile major: the N tiles of one M tile run side by side on
        // neighbouring SMs and share its activation rows through L2; the M
        // tiles of one expert follow each other, so its weights are read from
        // HBM about once and re-served from L2.
        const int mt = t / a.n_tiles;
        ti.nt = t % a.n_tiles;
        const int4 d = a.tiles[mt];
        ti.expert = d.x;
        ti.row0 = d.y;
        ti.nrows = d.z;
        if (kDebugChecks && !(idx_ok(mt, a.lim_tiles) && idx_ok(d.x, a.lim_experts) && d.z >= 1 &&
                              d.z <= 2 * kBM && idx_ok(d.y, a.lim_rows) && idx_ok(d.y + d.z - 1, a.lim_rows))) {
            ti.expert = 0;   // a bad entry becomes an empty tile
            ti.row0 = ti.nrows = 0;
        }
    } else {
        // Split-K: the K ranges are the slowest index of the tile list.
        if (a.k_splits > 1) {
            const int base = a.m_tiles * a.n_tiles;
            ti.ks = t / base;
            t -= ti.ks * base;
            ti.k0 = ti.ks * a.k_per_split;
            ti.nk = min(a.k_per_split, a.k_blocks - ti.k0);
        }
        // Rasterise in groups of 16 M tiles so the A rows of a group stay in L2
        // while every N tile visits them.
        constexpr int G = 16;
        const int group = G * a.n_tiles;
        const int g = t / group, r = t % group;
        const int m_first = g * G;
        const int gm = min(G, a.m_tiles - m_first);
        ti.nt = r / gm;
        const int mt = m_first + r % gm;
        ti.row0 = CG2 ? mt * (2 * kBM) + static_cast<int>(rank) * kBM : mt * kBM;
        ti.nrows = min(kBM, a.m_rows - ti.row0);
        ti.expert = 0;
    }
    return ti;
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// Hardware tanh (max relative error about 2^-11, far below the bf16 output's
// 2^-8).  The sigmoid is 1 / (1 + e^-x) from the fast exponential and
// division, which keeps its relative error small for very negative x, where
// (1 + tanh(x/2)) / 2 would cancel (relative error growing like e^-x * 2^-11).
// SiTU(x; b1) * softcap(y; b2) costs two tanh, one exp2 and one reciprocal;
// for b1 = 4 one tanh, one exp2 and one reciprocal.
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float situ_glu(float p1, float p2, float b1, float ib1, float b2, float ib2) {
    float situ;
    if (b1 == 4.0f) {
        // beta1 = 4 (K3): with u = e^(-x/2), tanh(x/4) = (1 - u) / (1 + u) and
        // sigma(x) = 1 / (1 + u^2), so SiTU(x) = 4 (1 - u) / ((1 + u)(1 + u^2)):
        // one exp2 and one reciprocal.  x is floored at -50, where
        // |SiTU| < 1e-21 (and (1 + u)(1 + u^2) stays finite).
        const float u = __expf(-0.5f * fmaxf(p1, -50.0f));
        situ = 4.0f * __fdividef(1.0f - u, (1.0f + u) * fmaf(u, u, 1.0f));
    } else {
        const float sig = __fdividef(1.0f, 1.0f + __expf(-p1));
        situ = b1 * tanh_fast(p1 * ib1) * sig;
    }
    return situ * (b2 * tanh_fast(p2 * ib2));
}

// 2^k as an fp32 built from the exponent bits, k clamped to the normal range
// [-126, 127] (an e4m3 scale exponent outside it belongs to a row whose
// largest magnitude is below 448 * 2^-127 or above 448 * 2^127).  Multiplying
// by it is exact while the product stays normal.
__device__ __forceinline__ float pow2f(int k) {
    k = max(-126, min(127, k));
    return __int_as_float((k + 127) << 23);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void store_f32_32(float *dst, const float (&v)[32], int ncols) {
    if (ncols >= 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
        for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < ncols) dst[j] = v[j];
    }
}

// Epilogue warps: eight for the e4m3 experts' W3 (its scaled bf16 epilogue,
// not its loads, sets its pace; warps 6..9 are free in a TMA-fed GEMM), four
// otherwise.
__host__ __device__ constexpr int epi_warps(int epi) { return epi == EPI_SCATTER_F8 ? 8 : 4; }
// A_GATHER adds four warps (6..9) that gather A rows with cp.async; eight
// epilogue warps take warps 6..9 instead.
__host__ __device__ constexpr int threads_for(int am, int epi = EPI_BF16) {
    return (am == A_GATHER || epi_warps(epi) == 8) ? kThreads + 128 : kThreads;
}

template <int BN, int AM, int BMD, int EPI, bool GROUPED, bool PAIR, bool KSEG = false, bool CG2 = false>
__global__ void __launch_bounds__(threads_for(AM, EPI), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const GemmArgs args) {
    using C = Cfg<BN, PAIR, KSEG, CG2, epi_warps(EPI)>;
    constexpr int S = C::kStages;
    constexpr int H = BN / 2;  // GLU: features per tile
    constexpr int NSUB = C::kSub;
    constexpr int NACC = PAIR ? 1 : 2;  // TMEM accumulator buffers (each NSUB x 256 columns)
    static_assert(!PAIR || (AM == A_GATHER && GROUPED), "pair tiles are built for the gathered expert GEMM");
    static_assert(C::kEpiWarps == 4 || (AM != A_GATHER && !KSEG && !CG2 && !PAIR),
                  "eight epilogue warps need warps 6..9 free");
    static_assert(!KSEG || (GROUPED && AM == A_DENSE && BMD == B_PLAIN && EPI == EPI_F32),
                  "K segments are built for the experts' weight gradients");
    static_assert(!CG2 || (!GROUPED && !PAIR && !KSEG && AM != A_GATHER && EPI != EPI_SITU_GLU_F8 &&
                           EPI != EPI_SCATTER_F8 && BN % 32 == 0),
                  "CTA pairs are built for the dense bf16 GEMMs fed by TMA");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *smA = smem;
    uint8_t *smB = smem + S * C::kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * C::kStageBytes);
    uint64_t *full = bars;             // [S]  TMA -> MMA
    uint64_t *empty = bars + S;        // [S]  MMA -> TMA
    uint64_t *tfull = bars + 2 * S;    // [2]  MMA -> epilogue
    uint64_t *tempty = bars + 2 * S + 2;  // [2]  epilogue -> MMA
    uint64_t *drain = bars + 2 * S + 4;   // [1]  final MMA completion
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pairs: this CTA's rank in the pair, and the pair's place in the
    // persistent tile loop (both CTAs walk the same tiles)
    const uint32_t rank = CG2 ? cluster_ctarank() : 0u;
    const int t_first = CG2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int t_step = CG2 ? static_cast<int>(n_clusters_x()) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // gather mode: one expect_tx arrival (B) + one per gathering thread
            mbar_init(smem_u32(&full[s]), AM == A_GATHER ? 1 + 128 : 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            // pairs: one arrival per epilogue warp of both CTAs (on CTA 0's barrier)
            mbar_init(smem_u32(&tempty[b]), CG2 ? 8 : 32 * C::kEpiWarps);
        }
        mbar_init(smem_u32(&drain[0]), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        if (CG2) {
            tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    // pairs: the other CTA's barriers must be initialised before anything
    // arrives on them or signals them
    if (CG2)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    grid_dependency_wait();   // inputs of this GEMM come from earlier kernels
    int n_m = GROUPED ? *args.n_mtiles : args.m_tiles;
    if (kDebugChecks && GROUPED && args.lim_tiles > 0 && !idx_ok(n_m, args.lim_tiles + 1)) n_m = 0;   // n_m <= capacity
    const int total = n_m * args.n_tiles * ((!GROUPED && args.k_splits > 1) ? args.k_splits : 1);
    const uint64_t lim = args.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        bool ok = true;
        for (int t = t_first; t < total && ok; t += t_step) {
            const Tile ti = tile_at<GROUPED, KSEG, CG2>(args, t, n_m, rank);
            constexpr uint32_t a_bytes = (AM == A_GATHER) ? 0u : C::kABytes;
            constexpr int TRB = (BMD == B_GLU) ? H : BN;     // rows per B box
            const int brow = args.b_packed ? (ti.expert * args.b_row_tiles + ti.nt) * args.k_blocks * TRB
                                           : ti.expert * args.b_expert_rows + ti.nt * TRB;
            for (int kb = 0; kb < ti.nk; ++kb) {
                // every lane waits; the warp proceeds only if all lanes saw the slot free
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                                       args.err, lim, true, CG2))) {
                    ok = false;
                    break;
                }
                // pairs: both CTAs' copies complete on CTA 0's barrier, which
                // CTA 0 arms with the bytes of both
                const uint32_t fb = CG2 ? mapa_shared(smem_u32(&full[stage]), 0) : smem_u32(&full[stage]);
                if (lane == 0 && rank == 0) mbar_arrive_expect_tx(smem_u32(&full[stage]), (CG2 ? 2u : 1u) * (a_bytes + C::kBBytes));
                __syncwarp();
                const uint32_t sa = smem_u32(smA + stage * C::kABytes);
                const uint32_t sb = smem_u32(smB + stage * C::kBBytes);
                const int kabs = ti.k0 + kb;   // K block in the operands' column space
                const bool second = (AM == A_SPLIT || BMD == B_SPLIT) && kabs >= args.k_split;
                const int kx = (second ? kabs - args.k_split : kabs) * kBK;
                // packed B: the K block is a row offset, the column is always 0
                // (K segments: both operands are packed by K block)
                const int bx = (KSEG || args.b_packed) ? 0 : kx;
                const int by = KSEG ? kabs * args.kseg_b_rows + ti.nt * TRB : args.b_packed ? brow + kabs * TRB : brow;
                const int ax = KSEG ? 0 : kx;
                const int ay = KSEG ? kabs * args.kseg_a_rows + ti.row0 : ti.row0;
                if (CG2 && lane == 0) {
                    // this CTA's 128 rows of A and its half of the B tile (GLU:
                    // CTA 0 the W1 rows, CTA 1 the W2 rows of the tile's features)
                    tma_load_2d_pair(sa, (AM == A_SPLIT && second) ? &tmA1 : &tmA0, ax, ay, fb);
                    if (BMD == B_GLU)
                        tma_load_2d_pair(sb, rank ? &tmB1 : &tmB0, bx, by, fb);
                    else
                        tma_load_2d_pair(sb, (BMD == B_SPLIT && second) ? &tmB1 : &tmB0, bx,
                                         by + static_cast<int>(rank) * C::kBRows, fb);
                } else if (lane == 0) {
                    if (AM != A_GATHER)
                        tma_load_2d(sa, (AM == A_SPLIT && second) ? &tmA1 : &tmA0, ax, ay, fb);
                    if (BMD == B_GLU) {
                        tma_load_2d(sb, &tmB0, bx, by, fb);
                        tma_load_2d(sb + H * (kBK * 2), &tmB1, bx, by, fb);
                    } else {
                        tma_load_2d(sb, (BMD == B_SPLIT && second) ? &tmB1 : &tmB0, bx, by, fb);
                    }
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Never leave while a copy into this CTA's shared memory is in flight.
        // (Pairs: CTA 0's barriers count both CTAs' copies.)
        if (lane == 0 && rank == 0) {
            for (int s = 0; s < S; ++s)
                if (issued_mask & (1u << s))
                    mbar_wait(smem_u32(&full[s]), (issued_parity >> s) & 1u, abort_flag, args.err,
                              lim, /*watch_abort=*/false);
        }
        // Pairs: every stage's last release, which the MMA thread of CTA 0
        // signals into both CTAs, must have arrived before this CTA may exit.
        if (CG2 && lane == 0) {
            for (int i = 0; i < S; ++i) {
                mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err, lim, true, true);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (AM == A_GATHER && warp >= 6) {
        // ------------------------------------------------------------ A gather
        // 128 threads copy the tile's 128 (pair: 256) rows x 128 bytes per
        // stage with 16-byte cp.async straight into the 128B-swizzled layout
        // the tensor core reads: thread i owns chunk c = i % 8 of rows i/8 + 16 j.
        // Each thread's arrival on the stage's full barrier fires when its
        // copies have landed (cp.async.mbarrier.arrive.noinc), so the threads
        // never wait on their own copies and run up to STAGES ahead; the MMA
        // thread issues the generic->async proxy fence after its wait.
        const int i = threadIdx.x - kThreads;
        const int c = i & 7;
        const int rb = i >> 3;
        const uint32_t sw = static_cast<uint32_t>((c ^ (rb & 7)) * 16);  // (rb + 16 j) & 7 == rb & 7
        bool ok = true;
        int g = 0;
        for (int t = t_first; t < total && ok; t += t_step) {
            const Tile ti = tile_at<GROUPED, KSEG, CG2>(args, t, n_m, rank);
            const uint16_t *src[8 * NSUB];
#pragma unroll
            for (int j = 0; j < 8 * NSUB; ++j) {
                const int r = rb + 16 * j;
                src[j] = nullptr;
                if (r < ti.nrows) {
                    const int32_t sr = args.gather_rows[ti.row0 + r];
                    if (idx_ok(sr, args.lim_src_rows)) src[j] = args.gather_src + int64_t(sr) * args.gather_ld + c * 8;
                }
            }
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                const int slot = g % S;
                const uint32_t par = static_cast<uint32_t>(g / S) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[slot]), par ^ 1u, abort_flag,
                                                       args.err, lim))) {
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_u32(smA + slot * C::kABytes);
#pragma unroll
                for (int j = 0; j < 8 * NSUB; ++j)
                    if (src[j]) cp_async_16(sa + (rb + 16 * j) * (kBK * 2) + sw, src[j] + kb * kBK);
                cp_async_arrive_noinc(smem_u32(&full[slot]));
                ++g;
            }
        }
        // finish (also after an abort): no copy may still be in flight
        cp_async_wait<0>();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // pairs: only CTA 0 issues; the accumulator rows of CTA 1 land in its own TMEM
        if (lane == 0 && rank == 0) {
            constexpr bool F8 = (EPI == EPI_SITU_GLU_F8 || EPI == EPI_SCATTER_F8);
            constexpr uint32_t idesc = F8 ? idesc_e4m3_m128(BN) : idesc_bf16(CG2 ? 2 * kBM : kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = t_first; t < total && ok; t += t_step) {
                if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, args.err, lim, true, CG2)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccStride);
                // a pair tile whose second sub-tile is empty skips its MMAs
                int nsub = 1;
                if (PAIR) nsub = (tile_at<GROUPED, KSEG>(args, t, n_m).nrows > kBM) ? 2 : 1;
                const int nkb = (KSEG || (!GROUPED && args.k_splits > 1)) ? tile_at<GROUPED, KSEG, CG2>(args, t, n_m, rank).nk
                                                                          : args.k_blocks;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err, lim)) {
                        ok = false;
                        break;
                    }
                    if (AM == A_GATHER) fence_proxy_async_smem();  // A was written by cp.async
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smA + stage * C::kABytes);
                    const uint32_t sb = smem_u32(smB + stage * C::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t bdesc = sdesc_sw128(sb + k * 32);
#pragma unroll
                        for (int sub = 0; sub < NSUB; ++sub)
                            if (sub < nsub) {
                                const uint64_t adesc = sdesc_sw128(sa + sub * (kBM * kBK * 2) + k * 32);
                                if (F8)
                                    tc_mma_e4m3(d + sub * kAccStride, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
                                else if (CG2)
                                    tc_mma_bf16_pair(d, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
                                else
                                    tc_mma_bf16(d + sub * kAccStride, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
                            }
                    }
                    if (CG2)
                        tc_commit_pair_mc(smem_u32(&empty[stage]), 0x3);   // both CTAs' producers
                    else
                        tc_commit(smem_u32(&empty[stage]));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (CG2)
                    tc_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);   // both CTAs' epilogues
                else
                    tc_commit(smem_u32(&tfull[acc]));
                if (++acc == NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // All MMAs this thread issued must finish before TMEM is freed.
            if (CG2)
                tc_commit_pair_mc(smem_u32(&drain[0]), 0x1);
            else
                tc_commit(smem_u32(&drain[0]));
            mbar_wait(smem_u32(&drain[0]), 0, abort_flag, args.err, lim, /*watch_abort=*/false);
            // Pairs: every accumulator's last release (four of the arrivals
            // come from the other CTA) must have arrived before this CTA exits.
            if (CG2) {
                for (int b = 0; b < NACC; ++b) {
                    mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, args.err, lim, true, true);
                    if (++acc == NACC) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < 2 + C::kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        // (eight warps: warps 2..5 take the first half of each tile's output
        // columns, warps 6..9 the second; both sets cover all lane quarters)
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;       // row of the tile held by this thread
        uint8_t *stg = smem + S * C::kStageBytes + C::kBarBytes + (warp - 2) * C::kStgWarpBytes;
        float *cscale = reinterpret_cast<float *>(smem + S * C::kStageBytes + C::kBarBytes +
                                                  C::kEpiWarps * C::kStgWarpBytes + (warp - 2) * C::kColWarpBytes);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t n_tma_stores = 0;   // K segments without split stores: TMA stores issued by this warp
        for (int t = t_first; t < total; t += t_step) {
            const Tile ti = tile_at<GROUPED, KSEG, CG2>(args, t, n_m, rank);
            // Per-row metadata of this thread's rows (destination row, gate,
            // token exponent), fetched before waiting for the accumulator so
            // their latency hides behind the MMAs.
            int64_t pre_drow[NSUB];
            float pre_scale[NSUB];
            int pre_he[NSUB];
            bool pre_ok[NSUB];   // false: a debug build's index check failed; the row is not written
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
                const int trow = sub * kBM + row;
                pre_drow[sub] = ti.row0 + trow;
                pre_scale[sub] = 1.0f;
                pre_he[sub] = 0;
                pre_ok[sub] = true;
                if (trow < ti.nrows) {
                    if (EPI == EPI_SCATTER_BF16 || EPI == EPI_SCATTER_F8) {
                        pre_drow[sub] = args.scatter_rows[ti.row0 + trow];
                        pre_ok[sub] = idx_ok(pre_drow[sub], args.lim_out_rows) && idx_ok(pre_drow[sub], args.lim_scale);
                        if (pre_ok[sub]) pre_scale[sub] = args.row_scale[pre_drow[sub]];
                    } else if (EPI == EPI_SITU_GLU_F8) {
                        const int32_t sr = args.gather_rows[ti.row0 + trow];
                        pre_ok[sub] = idx_ok(sr, args.lim_src_rows);
                        if (pre_ok[sub]) pre_he[sub] = args.row_exp[sr];
                    }
                }
            }
            // e4m3 epilogues: this tile's per-column power-of-two factors, into
            // the warp's own buffer (the warp finished reading the previous
            // tile's factors before it got here)
            if (EPI == EPI_SCATTER_F8) {        // 2^(W3 row exponent - 2) for the BN output columns
                const int8_t *ce = args.col_exp0 + ti.expert * args.col_exp_rows + ti.nt * BN;
                for (int i = lane; i < BN; i += 32) cscale[i] = pow2f(__ldg(ce + i) - 2);
                __syncwarp();
            } else if (EPI == EPI_SITU_GLU_F8) {   // 2^(W1 row exponent), then 2^(W2 row exponent)
                const int8_t *c1 = args.col_exp0 + ti.expert * args.col_exp_rows + ti.nt * H;
                const int8_t *c2 = args.col_exp1 + ti.expert * args.col_exp_rows + ti.nt * H;
                for (int i = lane; i < H; i += 32) {
                    cscale[i] = pow2f(__ldg(c1 + i));
                    cscale[H + i] = pow2f(__ldg(c2 + i));
                }
                __syncwarp();
            }
            // the whole warp must agree before the warp-collective tcgen05.ld
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, args.err, lim, true, CG2)))
                break;
            tc_fence_after();
#pragma unroll 1
            for (int sub = 0; sub < NSUB; ++sub) {
            if (sub * kBM >= ti.nrows) break;  // uniform across the CTA
            // this warp's 32 rows all lie past the tile's valid rows: nothing
            // to read or write (uniform across the warp)
            if (sub * kBM + q * 32 >= ti.nrows) continue;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>((acc + sub) * kAccStride);
            const int trow = sub * kBM + row;    // row of the tile (pair tiles: 0..255)
            const bool rv = trow < ti.nrows && ((NSUB > 1 && sub) ? pre_ok[NSUB - 1] : pre_ok[0]);
            if (EPI == EPI_SIGMOID_F32) {
                // fp32 scores: 32 columns (128 B) per row and group, staged like
                // the bf16 outputs below; the last partial group of a ragged N is
                // stored element by element.
                const int64_t orow = ti.row0 + trow;
                float *outf = reinterpret_cast<float *>(args.out);
                const bool vec_ok = (args.ld_out % 4) == 0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    const int64_t col = int64_t(ti.nt) * BN + c;
                    if (args.lout && rv)   // the logits themselves, for a backward pass
                        store_f32_32(args.lout + orow * args.ld_out + col, v, static_cast<int>(args.out_cols - col));
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = sigmoid_f(v[j]);
                    if (col + 32 <= args.out_cols && vec_ok) {
                        float4 *mine = reinterpret_cast<float4 *>(stg + lane * C::kStgPitch);
#pragma unroll
                        for (int j = 0; j < 8; ++j) mine[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        __syncwarp();
                        const int ch = lane & 7;
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int r = it * 4 + (lane >> 3);
                            const int64_t orr = __shfl_sync(0xffffffffu, orow, r);
                            const int ok = __shfl_sync(0xffffffffu, rv ? 1 : 0, r);
                            const float4 val = *reinterpret_cast<const float4 *>(stg + r * C::kStgPitch + ch * 16);
                            if (ok) *reinterpret_cast<float4 *>(outf + orr * args.ld_out + col + ch * 4) = val;
                        }
                        __syncwarp();
                    } else if (rv) {
                        store_f32_32(outf + orow * args.ld_out + col, v, static_cast<int>(args.out_cols - col));
                    }
                }
            } else if (EPI == EPI_F32 && KSEG) {
                // K segments (the experts' fp32 weight gradients): each warp
                // writes (accumulate: adds) its 32 rows in 32 x 32 blocks by
                // TMA store (reduction) through two swizzled 4 KB buffers, or,
                // with split_stores, half of them that way from one buffer and
                // the other half by the threads' own coalesced stores (atomic
                // adds) through the second: the two paths together carry more
                // than the TMA store path alone.
                // Rows of the expert's block below m_split go to the map in
                // tmA1 (out), the others to tmB1 (out2); m_split and the block
                // heights are multiples of 32, so a warp's rows are all valid
                // or all absent, and all in one output.
                uint8_t *tbuf = smem + C::kTmaStgOffset + (warp - 2) * C::kTmaStgWarpBytes;
                const int rblk = ti.row0 + q * 32;
                const bool rows_ok = q * 32 < ti.nrows;
                const bool first = rblk < args.m_split;
                const CUtensorMap *om = first ? &tmA1 : &tmB1;
                const int32_t y = first ? ti.expert * args.m_split + rblk
                                        : ti.expert * (args.m_rows - args.m_split) + (rblk - args.m_split);
                float *orow0 = reinterpret_cast<float *>(first ? args.out : args.out2) + int64_t(y) * args.ld_out;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);       // warp-collective: all lanes
                    const int col = ti.nt * BN + c;
                    if (rows_ok && col < args.out_cols) {   // warp-uniform
                        // split_stores: even 32-column groups leave by TMA store
                        // (buffer 0), odd ones by coalesced 16-byte stores from the
                        // threads (buffer 1), so both store paths of the SM carry
                        // output; else every group by TMA store, alternating buffers
                        const bool split = args.split_stores != 0;
                        const bool by_tma = !split || ((c >> 5) & 1) == 0;
                        uint8_t *buf = tbuf + (split ? (by_tma ? 0 : 4096) : (n_tma_stores & 1) * 4096);
                        if (by_tma) {
                            // the buffer's previous TMA store has read it
                            if (lane == 0) {
                                if (split)
                                    bulk_wait_read<0>();
                                else
                                    bulk_wait_read<1>();
                            }
                            __syncwarp();
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4 *>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        if (by_tma) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (args.accumulate)
                                    tma_reduce_add_2d(om, smem_u32(buf), col, y);
                                else
                                    tma_store_2d(om, smem_u32(buf), col, y);
                                bulk_commit();
                            }
                            ++n_tma_stores;
                        } else {
                            __syncwarp();
                            const int ch = lane & 7;
#pragma unroll
                            for (int it = 0; it < 8; ++it) {
                                const int r = it * 4 + (lane >> 3);   // 8 lanes per 128-byte row
                                const float4 val =
                                    *reinterpret_cast<const float4 *>(buf + r * 128 + ((ch ^ (r & 7)) << 4));
                                float4 *to = reinterpret_cast<float4 *>(orow0 + int64_t(r) * args.ld_out + col + ch * 4);
                                if (args.accumulate)
                                    atomicAdd(to, val);   // the only writer of these 4 floats
                                else
                                    *to = val;
                            }
                            __syncwarp();   // buffer 1 is read before the next odd group rewrites it
                        }
                    }
                }
            } else if (EPI == EPI_F32) {
                // fp32 rows (dense weight gradients, the router's share of the
                // latent gradient): staged like the scores above; accumulate
                // adds instead of storing (each element has one writer)
                // with out2, rows from m_split on go to out2 (two weights' gradients
                // of one GEMM, e.g. the shared experts' dWs1 | dWs2)
                // (split-K: this tile's K range has its own slab of partial sums)
                const int64_t r = ti.row0 + trow;
                float *dst = (args.out2 && r >= args.m_split)
                                 ? reinterpret_cast<float *>(args.out2) + (r - args.m_split) * args.ld_out
                                 : reinterpret_cast<float *>(args.out) + ti.ks * args.split_stride + r * args.ld_out;
                const bool vec_ok = (args.ld_out % 4) == 0;
                const unsigned long long dbits = reinterpret_cast<unsigned long long>(dst);
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    const int64_t col = int64_t(ti.nt) * BN + c;
                    if (col + 32 <= args.out_cols && vec_ok) {
                        float4 *mine = reinterpret_cast<float4 *>(stg + lane * C::kStgPitch);
#pragma unroll
                        for (int j = 0; j < 8; ++j) mine[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        __syncwarp();
                        const int ch = lane & 7;
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int rr = it * 4 + (lane >> 3);
                            const unsigned long long db = __shfl_sync(0xffffffffu, dbits, rr);
                            const int ok = __shfl_sync(0xffffffffu, rv ? 1 : 0, rr);
                            const float4 val = *reinterpret_cast<const float4 *>(stg + rr * C::kStgPitch + ch * 16);
                            float4 *to = reinterpret_cast<float4 *>(reinterpret_cast<float *>(db) + col + ch * 4);
                            if (ok) {
                                if (args.accumulate)
                                    atomicAdd(to, val);   // the only writer of these 4 floats
                                else
                                    *to = val;
                            }
                        }
                        __syncwarp();
                    } else if (rv) {
                        const int nc = static_cast<int>(args.out_cols - col);
                        if (args.accumulate) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nc) atomicAdd(dst + col + j, v[j]);
                        } else {
                            store_f32_32(dst + col, v, nc);
                        }
                    }
                }
            } else if (EPI == EPI_SITU_GLU_F8) {
                // e4m3 experts, W1|W2: p = acc * 2^(token exponent + weight-row
                // exponent) (exact), SiTU-GLU, then the fixed activation scale:
                // code = e4m3(4 * act), round to nearest even, saturating.  Each
                // thread writes its row's 32 codes per group (one 32-byte sector).
                const float rowf = pow2f((NSUB > 1 && sub) ? pre_he[NSUB - 1] : pre_he[0]);
                uint8_t *orow = reinterpret_cast<uint8_t *>(args.out) + (ti.row0 + trow) * args.ld_out;
                const float b1 = args.beta1, b2 = args.beta2;
                const float ib1 = 1.0f / b1, ib2 = 1.0f / b2;
#pragma unroll 1
                for (int c = 0; c < H; c += 32) {
                    float p1[32], p2[32];
                    tmem_ld32x2(taddr + c, taddr + H + c, p1, p2);
                    const int f0 = ti.nt * H + c;     // first feature of the group
                    uint32_t w[8];
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 s1 = *reinterpret_cast<const float4 *>(cscale + c + 4 * q4);
                        const float4 s2 = *reinterpret_cast<const float4 *>(cscale + H + c + 4 * q4);
                        const float f1[4] = {s1.x, s1.y, s1.z, s1.w}, f2[4] = {s2.x, s2.y, s2.z, s2.w};
                        uint32_t word = 0;
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int j = q4 * 4 + b;
                            const float x1 = p1[j] * rowf * f1[b];   // exact power-of-two scalings
                            const float x2 = p2[j] * rowf * f2[b];
                            const float a4 = 4.0f * situ_glu(x1, x2, b1, ib1, b2, ib2);
                            const uint32_t code = __nv_cvt_float_to_fp8(a4, __NV_SATFINITE, __NV_E4M3);
                            word |= code << (8 * b);
                        }
                        w[q4] = word;
                    }
                    if (rv) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + f0);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else {
                // bf16 outputs: each group of 64 columns goes through the warp's
                // staging buffer so the global stores are whole 128-byte lines
                // (4 rows x 128 B per warp instruction) instead of 16 bytes of
                // 32 different rows.
                const int64_t drow = (NSUB > 1 && sub) ? pre_drow[NSUB - 1] : pre_drow[0];
                const float scale = (NSUB > 1 && sub) ? pre_scale[NSUB - 1] : pre_scale[0];
                constexpr bool GLU = (EPI == EPI_SITU_GLU || EPI == EPI_SITU_GLU_SAVE);
                constexpr int NOUT = GLU ? H : BN;   // output columns per tile
                const int64_t col0 = int64_t(ti.nt) * NOUT;
                const float b1 = args.beta1, b2 = args.beta2;
                const float ib1 = 1.0f / b1, ib2 = 1.0f / b2;
                constexpr int CW = NOUT / (C::kEpiWarps / 4);   // columns per warp set
                const int c_begin = ((warp - 2) >> 2) * CW;
#pragma unroll 1
                for (int c = c_begin; c < c_begin + CW; c += 64) {
                    uint32_t packed[32];
                    float va[32], vb[32];
                    if (!GLU) tmem_ld32x2(taddr + c, taddr + c + 32, va, vb);   // both halves
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        float v[32];
                        if (GLU) {
                            float p2[32];
                            tmem_ld32x2(taddr + c + h2 * 32, taddr + H + c + h2 * 32, v, p2);
                            if (EPI == EPI_SITU_GLU_SAVE && rv) {
                                // keep the pre-activations for the backward: p1 | p2 in bf16
                                uint16_t *ps = args.pout + drow * args.pout_ld + col0 + c + h2 * 32;
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4) {
                                    reinterpret_cast<uint4 *>(ps)[q4] =
                                        make_uint4(pack_bf16x2(v[8 * q4], v[8 * q4 + 1]), pack_bf16x2(v[8 * q4 + 2], v[8 * q4 + 3]),
                                                   pack_bf16x2(v[8 * q4 + 4], v[8 * q4 + 5]), pack_bf16x2(v[8 * q4 + 6], v[8 * q4 + 7]));
                                    reinterpret_cast<uint4 *>(ps + args.pout_half)[q4] =
                                        make_uint4(pack_bf16x2(p2[8 * q4], p2[8 * q4 + 1]), pack_bf16x2(p2[8 * q4 + 2], p2[8 * q4 + 3]),
                                                   pack_bf16x2(p2[8 * q4 + 4], p2[8 * q4 + 5]), pack_bf16x2(p2[8 * q4 + 6], p2[8 * q4 + 7]));
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = situ_glu(v[j], p2[j], b1, ib1, b2, ib2);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = h2 ? vb[j] : va[j];
                        }
                        if (EPI == EPI_SCATTER_BF16) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] *= scale;
                        } else if (EPI == EPI_SCATTER_F8) {
                            // e4m3 experts' W3: gate * 2^(weight-row exponent - 2); the
                            // -2 undoes the activation's fixed scale of 4 (exact)
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4) {
                                const float4 f = *reinterpret_cast<const float4 *>(cscale + c + h2 * 32 + 4 * q4);
                                v[q4 * 4 + 0] = v[q4 * 4 + 0] * scale * f.x;
                                v[q4 * 4 + 1] = v[q4 * 4 + 1] * scale * f.y;
                                v[q4 * 4 + 2] = v[q4 * 4 + 2] * scale * f.z;
                                v[q4 * 4 + 3] = v[q4 * 4 + 3] * scale * f.w;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) packed[h2 * 16 + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                    }
                    uint4 *mine = reinterpret_cast<uint4 *>(stg + lane * C::kStgPitch);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        mine[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                    __syncwarp();
                    const int ch = lane & 7;                 // 16-byte chunk of a 128-byte row
                    const int64_t gcol = col0 + c + ch * 8;  // first output column of the chunk
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int r = it * 4 + (lane >> 3);
                        const int64_t dr = __shfl_sync(0xffffffffu, drow, r);
                        const int ok = __shfl_sync(0xffffffffu, rv ? 1 : 0, r);
                        const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * C::kStgPitch + ch * 16);
                        if (ok && gcol + 8 <= args.out_cols)
                            *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(args.out) + dr * args.ld_out +
                                                       gcol) = val;
                    }
                    __syncwarp();
                }
            }
            }  // sub-tiles
            tc_fence_before();
            if (CG2) {
                // one arrival per warp, on CTA 0's barrier
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            } else {
                mbar_arrive(smem_u32(&tempty[acc]));
            }
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // TMA stores read this CTA's shared memory: finish them before exit
        if (KSEG) {
            if (lane == 0) bulk_wait<0>();
            __syncwarp();
        }
    }

    tc_fence_before();
    // pairs: neither CTA frees its TMEM or leaves (its shared memory still
    // receiving the other's arrivals) before both are done
    if (CG2)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (CG2)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int BN, int AM, int BMD, int EPI, bool GROUPED, bool PAIR = false, bool KSEG = false>
cudaError_t launch_one(const GemmMaps &m, const GemmArgs &a, int grid, cudaStream_t st, bool dependent) {
    auto kern = gemm_kernel<BN, AM, BMD, EPI, GROUPED, PAIR, KSEG>;
    const size_t smem = Cfg<BN, PAIR, KSEG, false, epi_warps(EPI)>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(threads_for(AM, EPI)), smem, st, dependent, m.a0, m.a1, m.b0, m.b1, a);
}

// CTA pairs: clusters of two CTAs, as many pairs as fit on the GPU at once
// (at most `tiles`); the count is asked of the runtime once per device.
template <int BN, int AM, int BMD, int EPI>
cudaError_t launch_pair(const GemmMaps &m, const GemmArgs &a, int64_t tiles, cudaStream_t st, bool dependent) {
    auto kern = gemm_kernel<BN, AM, BMD, EPI, false, false, false, true>;
    const size_t smem = Cfg<BN, false, false, true>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(threads_for(AM, EPI));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
    constexpr int kMaxDev = 64;
    static std::atomic<int> pairs_on[kMaxDev];
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    int pairs = pairs_on[dev].load(std::memory_order_relaxed);
    if (pairs <= 0) {
        if ((e = cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg)) != cudaSuccess) return e;
        if (pairs <= 0) return cudaErrorInvalidConfiguration;
        pairs_on[dev].store(pairs, std::memory_order_relaxed);
    }
    if (tiles <= 0) return cudaSuccess;
    cfg.gridDim = dim3(2 * static_cast<unsigned>(tiles < pairs ? tiles : pairs));
    cfg.numAttrs = dependent ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, m.a0, m.a1, m.b0, m.b1, a);
}

}  // namespace

}  // namespace lmoe
