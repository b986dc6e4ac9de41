// gemm_pair.cu -- the dense GEMMs on CTA pairs (the forward's down- and
// up-projection; the backward's dr, dx and dense weight gradients): a
// 256 x 256 tile per cluster of two SMs, tcgen05.mma.cta_group::2 (M = 256)
// issued by the first CTA over both CTAs' shared memory, each CTA loading its
// own 128 rows of A and half of the B tile.  Per SM that is 32 KB of operands
// per 128 x 256 x 64 block of MMAs instead of 48 KB on one SM, so six stages
// fit.  The kernel template and its structure are described in
// gemm_kernel.cuh.
#include "gemm_kernel.cuh"

namespace lmoe {

#define LMOE_PAIR_CASE(BN_, AM_, BM_, EPI_)                        \
    if (bn == BN_ && am == AM_ && bm == BM_ && epi == EPI_)         \
        return launch_pair<BN_, AM_, BM_, EPI_>(maps, args, tiles, stream, dependent);

cudaError_t launch_gemm_pair(int bn, AMode am, BMode bm, Epi epi, const GemmMaps &maps, const GemmArgs &args,
                             int64_t tiles, cudaStream_t stream, bool dependent) {
    // a1 down-projection
    LMOE_PAIR_CASE(256, A_DENSE, B_PLAIN, EPI_BF16)
    // a8 up-projection + shared W3 (K split over the two sources); backward dx
    LMOE_PAIR_CASE(256, A_SPLIT, B_SPLIT, EPI_BF16)
    // backward: the dense weights' fp32 gradients (K = tokens); forward:
    // split-K partial sums of the down-projection (small batches)
    LMOE_PAIR_CASE(256, A_DENSE, B_PLAIN, EPI_F32)
    // split-K partial sums of the up-projection (small batches)
    LMOE_PAIR_CASE(256, A_SPLIT, B_SPLIT, EPI_F32)
    return cudaErrorInvalidValue;
}

#undef LMOE_PAIR_CASE

LMOE_DEBUG_WORD_READER(debug_word_pair)

}  // namespace lmoe
