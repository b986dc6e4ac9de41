// splitk.cu -- split-K for the dense GEMMs of small batches.  At decode sizes
// (tens of tokens) the down-projection, the router, the shared experts' W1|W2
// and the up-projection have only a few output tiles (one M tile): on one SM
// each, their weights stream at a few per cent of HBM.  Split-K spreads each
// tile's K blocks over enough CTAs to fill the GPU: every K range writes fp32
// partial sums (the persistent GEMM's fp32 epilogue) into its own slab, and
// split_finalize_kernel adds the slabs in a fixed order (the result does not
// depend on timing) and applies the GEMM's own epilogue: bf16 rounding, the
// router's sigmoid (and raw logits), or the SiTU-GLU of the shared experts
// ("Kimi-K3-Architecture-Deep-Dive" section 1) with its kept pre-activations.
#include "gemm_kernel.cuh"

namespace lmoe {

namespace {

__global__ void __launch_bounds__(256) split_finalize_kernel(const SplitFinArgs a) {
    grid_dependency_wait();   // the partial sums come from the GEMM before
    const int64_t total = a.rows * a.cols;
    const float ib1 = 1.0f / a.beta1, ib2 = 1.0f / a.beta2;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / a.cols, c = i % a.cols;
        const float *row = a.part + r * a.ld_part;
        if (a.mode == FIN_GLU) {
            // the GEMM's tile nt holds the W1 features nt*H.. in its first H
            // columns and the same W2 features in the next H
            const int64_t nt = c / a.H, j = c % a.H;
            const int64_t c1 = nt * 2 * a.H + j, c2 = c1 + a.H;
            float p1 = 0.0f, p2 = 0.0f;
            for (int ks = 0; ks < a.ks; ++ks) {
                p1 += row[ks * a.stride + c1];
                p2 += row[ks * a.stride + c2];
            }
            a.out[r * a.ld_out + c] = __bfloat16_as_ushort(__float2bfloat16_rn(situ_glu(p1, p2, a.beta1, ib1, a.beta2, ib2)));
            if (a.pout) {
                a.pout[r * a.pout_ld + c] = __bfloat16_as_ushort(__float2bfloat16_rn(p1));
                a.pout[r * a.pout_ld + a.pout_half + c] = __bfloat16_as_ushort(__float2bfloat16_rn(p2));
            }
        } else {
            float s = 0.0f;
            for (int ks = 0; ks < a.ks; ++ks) s += row[ks * a.stride + c];
            if (a.mode == FIN_SIGMOID) {
                if (a.lout) a.lout[r * a.ld_out + c] = s;
                a.outf[r * a.ld_out + c] = sigmoid_f(s);
            } else {
                a.out[r * a.ld_out + c] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
            }
        }
    }
}

}  // namespace

#define LMOE_SPLIT_CASE(BN_, AM_, BM_)                                  \
    if (bn == BN_ && am == AM_ && bm == BM_)                            \
        return launch_one<BN_, AM_, BM_, EPI_F32, false>(maps, args, grid, stream, dependent);

cudaError_t launch_gemm_split(int bn, AMode am, BMode bm, const GemmMaps &maps, const GemmArgs &args, int grid,
                              cudaStream_t stream, bool dependent) {
    // single CTAs, fp32 partial sums (the 256-wide down- and up-projection
    // split on CTA pairs instead: launch_gemm_pair with EPI_F32)
    LMOE_SPLIT_CASE(128, A_DENSE, B_PLAIN)    // down-projection (latent not a multiple of 256), router
    LMOE_SPLIT_CASE(224, A_DENSE, B_PLAIN)    // router, E a multiple of 224
    LMOE_SPLIT_CASE(256, A_DENSE, B_PLAIN)    // router
    LMOE_SPLIT_CASE(256, A_DENSE, B_GLU)      // shared experts W1|W2
    LMOE_SPLIT_CASE(128, A_DENSE, B_GLU)
    LMOE_SPLIT_CASE(128, A_SPLIT, B_SPLIT)    // up-projection (d not a multiple of 256)
    return cudaErrorInvalidValue;
}

#undef LMOE_SPLIT_CASE

cudaError_t launch_split_finalize(const SplitFinArgs &a, int num_sms, cudaStream_t stream) {
    const int64_t total = a.rows * a.cols;
    if (total <= 0) return cudaSuccess;
    const int64_t want = (total + 255) / 256;
    const int grid = static_cast<int>(want < 4 * num_sms ? want : 4 * num_sms);
    return launch_kernel(split_finalize_kernel, dim3(grid), dim3(256), 0, stream, true, a);
}

LMOE_DEBUG_WORD_READER(debug_word_split)

}  // namespace lmoe
