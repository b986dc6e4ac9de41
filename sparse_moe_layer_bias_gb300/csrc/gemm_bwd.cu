// gemm_bwd.cu -- the training GEMM variants of the persistent tcgen05 GEMM
// (gemm_kernel.cuh):
//   u     = dz W3[e]               (A = dz rows gathered by token, B = W3[e]^T)
//   dW    = G^T A for the dense weights (fp32; both operands transposed to
//           K-major over tokens)
//   dW[e] = G_e^T A_e for the routed experts (fp32; K = the expert's own
//           tokens: one K segment per expert in a shared column space)
// and the forward's SiTU-GLU GEMMs that keep their pre-activations p1 | p2
// for the backward's element-wise SiTU-GLU derivative.
#include "gemm_kernel.cuh"

namespace lmoe {

cudaError_t launch_gemm_bwd(int bn, AMode am, BMode bm, Epi epi, bool grouped, bool kseg, const GemmMaps &maps,
                            const GemmArgs &args, int grid, cudaStream_t stream) {
    const bool dep = true;
    if (bn != 256 && bn != 128) return cudaErrorInvalidValue;
    const bool b256 = (bn == 256);
    if (am == A_DENSE && bm == B_PLAIN && epi == EPI_F32) {
        if (kseg && grouped)
            return b256 ? launch_one<256, A_DENSE, B_PLAIN, EPI_F32, true, false, true>(maps, args, grid, stream, dep)
                        : launch_one<128, A_DENSE, B_PLAIN, EPI_F32, true, false, true>(maps, args, grid, stream, dep);
        if (!kseg && !grouped)
            return b256 ? launch_one<256, A_DENSE, B_PLAIN, EPI_F32, false>(maps, args, grid, stream, dep)
                        : launch_one<128, A_DENSE, B_PLAIN, EPI_F32, false>(maps, args, grid, stream, dep);
    }
    if (kseg) return cudaErrorInvalidValue;
    if (am == A_GATHER && bm == B_PLAIN && epi == EPI_BF16 && grouped)
        return b256 ? launch_one<256, A_GATHER, B_PLAIN, EPI_BF16, true>(maps, args, grid, stream, dep)
                    : launch_one<128, A_GATHER, B_PLAIN, EPI_BF16, true>(maps, args, grid, stream, dep);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_save(int bn, AMode am, bool grouped, bool pair, const GemmMaps &maps, const GemmArgs &args,
                             int grid, cudaStream_t stream, bool dependent) {
    if (bn != 256 && bn != 128) return cudaErrorInvalidValue;
    const bool b256 = (bn == 256);
    if (am == A_GATHER && grouped) {
        if (pair)
            return b256 ? launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU_SAVE, true, true>(maps, args, grid, stream, dependent)
                        : launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU_SAVE, true, true>(maps, args, grid, stream, dependent);
        return b256 ? launch_one<256, A_GATHER, B_GLU, EPI_SITU_GLU_SAVE, true>(maps, args, grid, stream, dependent)
                    : launch_one<128, A_GATHER, B_GLU, EPI_SITU_GLU_SAVE, true>(maps, args, grid, stream, dependent);
    }
    if (am == A_DENSE && !grouped && !pair)
        return b256 ? launch_one<256, A_DENSE, B_GLU, EPI_SITU_GLU_SAVE, false>(maps, args, grid, stream, dependent)
                    : launch_one<128, A_DENSE, B_GLU, EPI_SITU_GLU_SAVE, false>(maps, args, grid, stream, dependent);
    return cudaErrorInvalidValue;
}

LMOE_DEBUG_WORD_READER(debug_word_gemm_bwd)

}  // namespace lmoe
