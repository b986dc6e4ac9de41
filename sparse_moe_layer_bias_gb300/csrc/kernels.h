// kernels.h -- internal interface between the C-ABI host code and the CUDA
// kernels of liblmoe.so (not installed, not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

// ------------------------------------------------------------------ launch
// Launch a kernel; with `dependent`, as a programmatic dependent launch: its
// CTAs may start while the previous kernel in the stream finishes, run their
// prologue, and wait in grid_dependency_wait() until that kernel has completed
// and its writes are visible.  Every kernel launched this way calls
// grid_dependency_wait() in all threads before touching memory that earlier
// work in the stream wrote, and before it can complete, so the chain of
// completions stays transitive.  (A kernel whose predecessor is not a kernel,
// e.g. a memset, is simply ordered after it.)
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          bool dependent, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Device status bits written by kernels (see lmoe_device_status).
constexpr unsigned kDevErrTimeout = 1u;

// ------------------------------------------------------------------ debug index checks
// A build with -DLMOE_DEBUG checks every index a kernel reads from a device
// list before using it: gathered and scattered rows, the permutation maps and
// the grouped GEMMs' tile lists.  A failed check sets this translation unit's
// debug word and the access is skipped (no trap); lmoe_device_status reports
// it as LMOE_ERR_INDEX.  In a release build idx_ok() is constant true and the
// checks compile away.
#ifdef LMOE_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

#if defined(__CUDACC__) && defined(LMOE_DEBUG)
static __device__ unsigned g_dbg_index_word;
#endif

#ifdef __CUDACC__
// 0 <= i < n (n <= 0: no known limit).  Debug builds record a violation.
__device__ __forceinline__ bool idx_ok(int64_t i, int64_t n) {
#ifdef LMOE_DEBUG
    if (n <= 0 || (i >= 0 && i < n)) return true;
    atomicOr(&g_dbg_index_word, 1u);
    return false;
#else
    (void)i;
    (void)n;
    return true;
#endif
}
#endif

// The debug word of each translation unit that checks indices (0 in a release
// build); `clear` resets it.  Synchronous.
unsigned debug_word_gemm(bool clear);
unsigned debug_word_pair(bool clear);
unsigned debug_word_split(bool clear);
unsigned debug_word_gemm_bwd(bool clear);
unsigned debug_word_route(bool clear);
unsigned debug_word_backward(bool clear);
unsigned debug_word_selftest(bool clear);
#ifdef LMOE_DEBUG
#define LMOE_DEBUG_WORD_READER(fn)                                                         \
    unsigned fn(bool clear) {                                                              \
        unsigned v = 0;                                                                    \
        if (cudaMemcpyFromSymbol(&v, g_dbg_index_word, sizeof v) != cudaSuccess) return ~0u; \
        if (clear && v) {                                                                  \
            const unsigned z = 0;                                                          \
            if (cudaMemcpyToSymbol(g_dbg_index_word, &z, sizeof z) != cudaSuccess) return ~0u; \
        }                                                                                  \
        return v;                                                                          \
    }
#else
#define LMOE_DEBUG_WORD_READER(fn) \
    unsigned fn(bool) { return 0; }
#endif
// One thread fails one index check (debug builds; nothing in a release build).
cudaError_t launch_index_check_selftest(cudaStream_t stream);

// ------------------------------------------------------------------ GEMM
// A operand source.
// A_GATHER: rows of A are gathered by a row-index list (cp.async by four
// extra producer warps); used for the routed experts' W1|W2 GEMM.
enum AMode { A_DENSE = 0, A_GATHER = 1, A_SPLIT = 2 };
// B operand source.
enum BMode { B_PLAIN = 0, B_GLU = 1, B_SPLIT = 2 };
// Epilogue.
// EPI_SITU_GLU_F8: e4m3 experts' W1|W2 -- rescale by the token's and the
// weight rows' power-of-two scales, SiTU-GLU, write e4m3(4 * act) bytes.
// EPI_SCATTER_F8: e4m3 experts' W3 -- rescale by 2^(row exponent - 2), gate,
// scatter bf16 rows (as EPI_SCATTER_BF16).
// Backward pass:
// EPI_F32: plain fp32 output rows (weight gradients; the router's share of the
// latent gradient).  With per-expert K segments (launch_gemm_bwd, kseg), the
// rows of expert e's output block go to out (rows < m_split) or out2.
// EPI_SITU_GLU_SAVE: EPI_SITU_GLU that also writes the pre-activations p1 | p2
// (bf16) to pout (p1 at the feature's column, p2 pout_half columns later), for
// a backward pass that does not recompute them.
enum Epi { EPI_BF16 = 0, EPI_SITU_GLU = 1, EPI_SIGMOID_F32 = 2, EPI_SCATTER_BF16 = 3, EPI_SITU_GLU_F8 = 4,
           EPI_SCATTER_F8 = 5, EPI_F32 = 6, EPI_SITU_GLU_SAVE = 7 };

constexpr int kBM = 128;  // rows per tile (one tcgen05 M=128 tile)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzled row of bf16 (128 e4m3)

struct GemmMaps {
    CUtensorMap a0, a1, b0, b1;
};

struct GemmArgs {
    int32_t m_rows;          // dense: rows of A / output
    int32_t m_tiles;         // dense: ceil(m_rows / 128)
    int32_t n_tiles;         // tiles along N
    int32_t k_blocks;        // ceil(K / 64)
    int32_t k_split;         // A_SPLIT/B_SPLIT: k-blocks served by map 0
    int32_t b_expert_rows;   // grouped: B-map rows per expert
    // grouped, tile-packed B (see launch_pack_tiles): B box (e, N tile nt, K
    // block kb) sits at row ((e * b_row_tiles + nt) * k_blocks + kb) * box rows
    int32_t b_packed;
    int32_t b_row_tiles;     // N tiles per expert in the packed layout
    const int4 *tiles;       // grouped: {expert, first permuted row, rows, 0} (pair tiles for A_GATHER)
    const int32_t *n_mtiles; // grouped: number of entries in `tiles` (device)
    const uint16_t *gather_src;   // A_GATHER: base of the row-major [*, K] bf16 source
    const int32_t *gather_rows;   // A_GATHER: source row for each grouped row
    int64_t gather_ld;            // A_GATHER: source row stride (elements)
    void *out;               // output base
    int64_t ld_out;          // output row stride (elements)
    int32_t out_cols;        // output columns that exist (masking of ragged N)
    const int32_t *scatter_rows;  // EPI_SCATTER_*: destination row per permuted row
    const float *row_scale;       // EPI_SCATTER_*: scale per destination row
    float beta1, beta2;
    // e4m3 experts: power-of-two scale exponents
    const int8_t *row_exp;        // EPI_SITU_GLU_F8: per source token row (indexed via gather_rows)
    const int8_t *col_exp0;       // per weight row of expert e: [e * col_exp_rows + col] (W1 or W3)
    const int8_t *col_exp1;       // EPI_SITU_GLU_F8: the W2 rows
    int32_t col_exp_rows;
    // training epilogues
    void *out2;                   // EPI_F32 with K segments: rows >= m_split of an expert's block
    int32_t m_split;
    // K segments: operand heights of the K-block packed A and B ([K blocks][rows][64]);
    // the box of K block kb, rows r.. sits at map row kb * rows + r
    int32_t kseg_a_rows, kseg_b_rows;
    int32_t accumulate;           // EPI_F32: add to the output instead of overwriting it
    int32_t split_stores;         // EPI_F32 with K segments: half the output by the threads' stores
    float *lout;                  // EPI_SIGMOID_F32: also the raw fp32 logits, ld_out apart (nullable)
    uint16_t *pout;               // EPI_SITU_GLU_SAVE: pre-activation rows (bf16)
    int64_t pout_ld;
    int32_t pout_half;
    unsigned *err;           // device status word
    uint64_t wait_limit_ns;  // bound on every mbarrier wait
    // limits for the debug build's index checks (0: no check): experts,
    // entries of the tile list, rows of the grouped row lists, rows of the
    // gathered source, rows of the scattered output, entries of row_scale
    int64_t lim_experts, lim_tiles, lim_rows, lim_src_rows, lim_out_rows, lim_scale;
    // dense split-K (EPI_F32): k_splits > 1 divides K into ranges of
    // k_per_split blocks; the tile list is m_tiles x n_tiles x k_splits and
    // range ks writes its fp32 partial sums at out + ks * split_stride
    int32_t k_splits, k_per_split;
    int64_t split_stride;
};

// Launch one persistent GEMM.  `bn` in {128, 256} (224 for the router).  With `pair`, A_GATHER runs
// pair tiles (two 128-row sub-tiles sharing each weight stage); without, 128-row
// tiles with a deeper stage ring.  Returns cudaErrorInvalidValue for a
// combination that is not compiled.
// The e4m3 epilogues select the kind::f8f6f4 MMA (A and B e4m3; a k-block is
// then 128 elements); every other epilogue multiplies bf16.
cudaError_t launch_gemm(int bn, AMode am, BMode bm, Epi epi, bool grouped, const GemmMaps &maps,
                        const GemmArgs &args, int grid, cudaStream_t stream, bool pair = false,
                        bool dependent = true);

// Dense GEMMs (A by TMA, not grouped) on CTA pairs (gemm_pair.cu): a
// 256 x bn tile per cluster of two CTAs, `args.m_tiles` = ceil(m_rows / 256)
// and `tiles` = m_tiles x n_tiles; the B maps' boxes are bn / 2 rows (each CTA
// loads its half of the tile's B rows).  The grid is chosen here (two CTAs
// per tile, at most as many pairs as fit on the GPU at once).  Compiled for
// bn = 256 with A_DENSE/B_PLAIN/EPI_BF16 (down-projection, backward dr),
// A_SPLIT/B_SPLIT/EPI_BF16 (up-projection, backward dx), A_DENSE/B_PLAIN/EPI_F32
// (backward dense weight gradients; the down-projection's split-K partials)
// and A_SPLIT/B_SPLIT/EPI_F32 (the up-projection's split-K partials);
// cudaErrorInvalidValue otherwise.
cudaError_t launch_gemm_pair(int bn, AMode am, BMode bm, Epi epi, const GemmMaps &maps, const GemmArgs &args,
                             int64_t tiles, cudaStream_t stream, bool dependent = true);

// Split-K of the dense GEMMs for small batches (splitk.cu): the single-CTA
// GEMM with the fp32 epilogue (args.k_splits, k_per_split, split_stride set;
// accumulate 0), bn / modes: 128, 224, 256 with A_DENSE/B_PLAIN; 128, 256 with
// A_DENSE/B_GLU; 128 with A_SPLIT/B_SPLIT.  (The 256-wide down- and
// up-projection split on CTA pairs: launch_gemm_pair with EPI_F32.)
cudaError_t launch_gemm_split(int bn, AMode am, BMode bm, const GemmMaps &maps, const GemmArgs &args, int grid,
                              cudaStream_t stream, bool dependent = true);
// The sum of the K ranges' partial slabs (fixed order) and the GEMM's epilogue.
enum SplitFinMode { FIN_BF16 = 0, FIN_SIGMOID = 1, FIN_GLU = 2 };
struct SplitFinArgs {
    const float *part;     // slab 0 of the partial sums: [rows][ld_part] fp32
    int64_t stride;        // elements from one slab to the next
    int32_t ks;            // number of slabs
    int32_t mode;          // SplitFinMode
    int64_t rows, cols;    // output rows and columns (FIN_GLU: features)
    int64_t ld_part;       // partial row stride (FIN_GLU: 2 x features, tile-interleaved)
    int32_t H;             // FIN_GLU: features per GEMM tile (W1 columns, then as many W2)
    float beta1, beta2;    // FIN_GLU
    uint16_t *out;         // FIN_BF16 / FIN_GLU: bf16 [rows][ld_out]
    float *outf;           // FIN_SIGMOID: sigmoid of the sums [rows][ld_out]
    float *lout;           // FIN_SIGMOID: the sums themselves (nullable)
    int64_t ld_out;
    uint16_t *pout;        // FIN_GLU: p1 | p2 in bf16 (nullable)
    int64_t pout_ld, pout_half;
};
cudaError_t launch_split_finalize(const SplitFinArgs &a, int num_sms, cudaStream_t stream);

// Backward-pass GEMMs (gemm_bwd.cu); same operand conventions.  With `kseg`
// (grouped, A and B dense): `tiles` holds {expert, first K block, K blocks,
// first row of the expert's output block} per 128-row tile, both operands are
// K-major over one shared column space in which each expert owns a segment,
// m_rows is the height of an expert's output block, and the fp32 output goes
// out by TMA store through maps.a1 (rows of the block below m_split; the map
// covers [E * m_split][out_cols]) and maps.b1 (the other rows): fp32 maps with
// 32 x 32 boxes and 128-byte swizzle (m_split and m_rows multiples of 32).
cudaError_t launch_gemm_bwd(int bn, AMode am, BMode bm, Epi epi, bool grouped, bool kseg, const GemmMaps &maps,
                            const GemmArgs &args, int grid, cudaStream_t stream);
// The forward's SiTU-GLU GEMMs that also keep their pre-activations
// (EPI_SITU_GLU_SAVE): the routed experts' (A_GATHER, grouped, 128-row or
// pair tiles) and the shared experts' (A_DENSE).
cudaError_t launch_gemm_save(int bn, AMode am, bool grouped, bool pair, const GemmMaps &maps, const GemmArgs &args,
                             int grid, cudaStream_t stream, bool dependent = true);

// Repack per-expert weights [E][R][K] (row-major bf16) into tile-contiguous
// order [E][R/TR][K/64][TR][64] so that one TMA box of TR rows x 64 columns is
// one contiguous TR*128-byte block of HBM.  R % TR == 0, K % 64 == 0.
cudaError_t launch_pack_tiles(const uint16_t *src, int64_t E, int R, int K, int TR, uint16_t *dst,
                              cudaStream_t stream);

// ------------------------------------------------------------------ routing
cudaError_t launch_topk(const float *scores, const float *bias, int64_t T, int E, int k,
                        int32_t *idx, float *gate, uint32_t *bitmap, int words_per_expert,
                        cudaStream_t stream);
cudaError_t launch_expert_scan(const uint32_t *bitmap, int E, int words_per_expert,
                               uint32_t *word_prefix, int32_t *counts, cudaStream_t stream);
// tiles: up to 128 rows each (ceil(count/128) per expert).  With tiles3 ==
// nullptr, tiles2 holds pair tiles of up to 256 rows for every expert
// (ceil(count/256) each); otherwise tiles2 holds them only for experts with
// more than 128 rows and tiles3 one tile for each expert with 1..128 rows.
cudaError_t launch_offsets_tiles(const int32_t *counts, int E, int32_t *offsets, int4 *tiles,
                                 int32_t *n_mtiles, int4 *tiles2, int32_t *n_mtiles2, int4 *tiles3,
                                 int32_t *n_mtiles3, cudaStream_t stream);
cudaError_t launch_scatter(const int32_t *idx, int64_t T, int k, int E, const uint32_t *bitmap,
                           const uint32_t *word_prefix, int words_per_expert,
                           const int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *tokrow,
                           cudaStream_t stream);

// ------------------------------------------------------------------ combine
// e4m3 quantisation of R rows of K bf16 values: exps[r] = smallest e with
// max|row| <= 448 * 2^e (0 for a zero row), codes = e4m3_rn_satfinite(v * 2^-e).
// K % 8 == 0.
cudaError_t launch_fp8_quantize_rows(const uint16_t *src, int64_t R, int K, uint8_t *codes, int8_t *exps,
                                     cudaStream_t stream);
// Row RMSNorm of bf16 rows (fp64 arithmetic, one rounding to bf16); L % 8 == 0.
cudaError_t launch_rms_rows(const uint16_t *h, int64_t T, int L, double eps, uint16_t *out, cudaStream_t stream);
cudaError_t launch_combine_rmsnorm(const uint16_t *o, int64_t T, int k, int L, float eps,
                                   uint16_t *r, unsigned *err, uint64_t wait_limit_ns, cudaStream_t stream);

// ------------------------------------------------------------------ QB
cudaError_t launch_qb_histogram(const float *scores, int64_t T, int E, int64_t ld, int B,
                                uint32_t *hist, int accumulate, int num_sms, cudaStream_t stream);
// One CTA waits (bounded) on an mbarrier nothing arrives on; sets the timeout
// bit in *err after limit_ns and *gave_up = 1 (nullable).
cudaError_t launch_bounded_wait_selftest(unsigned *err, uint64_t limit_ns, int *gave_up, cudaStream_t stream);
cudaError_t launch_sign_update(const int32_t *counts, int E, float gamma, float *bias, cudaStream_t stream);
cudaError_t launch_qb_quantile(const uint32_t *hist, int E, int B, double level, float *q,
                               float *bias, cudaStream_t stream);

// ------------------------------------------------------------------ backward
// out[b][c][q] = scale(q) * in[b][src(q)][c] (c < C, q < Q); src(q) = qsrc[q],
// or q when q < R without qsrc; a negative src gives 0.  Tiles starting at or
// past *q_limit (when given) are skipped.  packed_rows = C (batch 1, Q % 64
// == 0): K-block packed output, (c, q) at ((q / 64) * C + c) * 64 + q % 64.
cudaError_t launch_transpose(const uint16_t *in, int64_t ldi, int64_t in_batch_stride, int64_t R, int C,
                             uint16_t *out, int64_t ldo, int64_t out_batch_stride, int64_t Q, int batch,
                             const int32_t *qsrc, const float *qscale, const int32_t *q_limit, cudaStream_t stream,
                             int64_t packed_rows = 0);
// Per-expert column segments (assignments padded to 64), their column maps and
// the segment GEMMs' tile lists; n_tiles3 = {tiles in a, tiles in b, columns}.
// Counts come from the forward's offsets ([E+1] exclusive scan).
cudaError_t launch_segments(const int32_t *offsets, const int32_t *perm,
                            const int32_t *tokrow, const float *gates, int E, int32_t *segoff, int32_t *qperm,
                            int32_t *qtok, float *qgate, int4 *tiles_a, int m_tiles_a, int4 *tiles_b,
                            int m_tiles_b, int32_t *n_tiles3, cudaStream_t stream);
cudaError_t launch_zero_unused(const int32_t *offsets, int E, int64_t per_expert, float *g1, float *g2, float *g3,
                               cudaStream_t stream);
cudaError_t launch_rms_bwd(const uint16_t *o, int64_t T, int k, int L, float eps, const uint16_t *dr, int64_t ld_dr,
                           uint16_t *dz, cudaStream_t stream);
cudaError_t launch_router_bwd(const float *dg, const int32_t *inv, const int32_t *idx, const float *logits, int E,
                              int64_t T, int k, int ldl, uint16_t *dl, cudaStream_t stream);
cudaError_t launch_dh_sum(const uint16_t *dhp, const float *dhr, int64_t T, int k, int L, uint16_t *dh,
                          int num_sms, cudaStream_t stream);
cudaError_t launch_fill(float *p, int64_t n, float v, cudaStream_t stream);
// SiTU-GLU backward over rows at the pre-activations P (p1 | p2, p2 p_half
// columns after p1): dP (dp1 | dp2) from the activation gradient
// g_r * U[r][u_col0 ...], and dg[r] = sum of U * act when dg is not null.
cudaError_t launch_glu_bwd_rows(const uint16_t *P, int64_t p_ld, int p_half, const uint16_t *U, int64_t u_ld,
                                int u_col0, const int32_t *scale_rows, const float *scale, int64_t rows, int C,
                                float b1, float b2, uint16_t *dP, int64_t dp_ld, int dp_half, float *dg,
                                int num_sms, cudaStream_t stream);

}  // namespace lmoe
