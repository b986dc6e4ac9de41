// gemm.cu -- the forward pass's GEMM variants (the kernel template and its
// structure are described in gemm_kernel.cuh).
#include "gemm_kernel.cuh"

namespace lmoe {

#define LMOE_GEMM_CASE(BN_, AM_, BM_, EPI_, G_)                                   \
    if (bn == BN_ && am == AM_ && bm == BM_ && epi == EPI_ && grouped == G_)       \
        return launch_one<BN_, AM_, BM_, EPI_, G_>(maps, args, grid, stream, dependent);

cudaError_t launch_gemm(int bn, AMode am, BMode bm, Epi epi, bool grouped, const GemmMaps &maps,
                        const GemmArgs &args, int grid, cudaStream_t stream, bool pair, bool dependent) {
    // a1 down-projection, a8 up-projection + shared W3
    LMOE_GEMM_CASE(256, A_DENSE, B_PLAIN, EPI_BF16, false)
    LMOE_GEMM_CASE(128, A_DENSE, B_PLAIN, EPI_BF16, false)
    LMOE_GEMM_CASE(256, A_SPLIT, B_SPLIT, EPI_BF16, false)
    LMOE_GEMM_CASE(128, A_SPLIT, B_SPLIT, EPI_BF16, false)
    // a8' shared experts W1|W2 with the SiTU-GLU epilogue
    LMOE_GEMM_CASE(256, A_DENSE, B_GLU, EPI_SITU_GLU, false)
    LMOE_GEMM_CASE(128, A_DENSE, B_GLU, EPI_SITU_GLU, false)
    // a2 router scores
    LMOE_GEMM_CASE(256, A_DENSE, B_PLAIN, EPI_SIGMOID_F32, false)
    LMOE_GEMM_CASE(224, A_DENSE, B_PLAIN, EPI_SIGMOID_F32, false)   // E = 896 = 4 x 224: no padded columns
    LMOE_GEMM_CASE(128, A_DENSE, B_PLAIN, EPI_SIGMOID_F32, false)
    // a5 routed experts W1|W2 (token rows gathered per expert) with the
    // SiTU-GLU epilogue: pair tiles of 256 rows for experts with many tokens,
    // 128-row tiles (smaller stages, one more of them in flight) for the others
    if (am == A_GATHER && bm == B_GLU && epi == EPI_SITU_GLU && grouped) {
        if (pair) {
            if (bn == 256) return launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU, true, true>(maps, args, grid, stream, dependent);
            if (bn == 128) return launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU, true, true>(maps, args, grid, stream, dependent);
        } else {
            if (bn == 256) return launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU, true, false>(maps, args, grid, stream, dependent);
            if (bn == 128) return launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU, true, false>(maps, args, grid, stream, dependent);
        }
    }
    // a6 routed experts W3 with the gate-weighted scatter (also the backward's
    // experts' share of dh, rows scattered back to assignment order)
    LMOE_GEMM_CASE(256, A_DENSE, B_PLAIN, EPI_SCATTER_BF16, true)
    LMOE_GEMM_CASE(128, A_DENSE, B_PLAIN, EPI_SCATTER_BF16, true)
    // FP8 variant: e4m3 experts (kind::f8f6f4)
    if (am == A_GATHER && bm == B_GLU && epi == EPI_SITU_GLU_F8 && grouped) {
        if (pair) {
            if (bn == 256) return launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU_F8, true, true>(maps, args, grid, stream, dependent);
            if (bn == 128) return launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU_F8, true, true>(maps, args, grid, stream, dependent);
        } else {
            if (bn == 256) return launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU_F8, true, false>(maps, args, grid, stream, dependent);
            if (bn == 128) return launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU_F8, true, false>(maps, args, grid, stream, dependent);
        }
    }
    LMOE_GEMM_CASE(256, A_DENSE, B_PLAIN, EPI_SCATTER_F8, true)
    LMOE_GEMM_CASE(128, A_DENSE, B_PLAIN, EPI_SCATTER_F8, true)
    return cudaErrorInvalidValue;
}

#undef LMOE_GEMM_CASE

LMOE_DEBUG_WORD_READER(debug_word_gemm)

}  // namespace lmoe
