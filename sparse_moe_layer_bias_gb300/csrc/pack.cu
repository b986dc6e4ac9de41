// pack.cu -- one-time weight layout change at handle creation.
//
// The routed experts' GEMMs stream each expert's weights from HBM in boxes of
// TR rows x 64 columns (128 bytes per row, one K block).  In the caller's
// row-major [R][K] layout those 128-byte pieces sit K*2 bytes apart; stored
// tile-contiguously ([R/TR][K/64][TR][64]) every box is one contiguous
// TR*128-byte block, so the weight stream is a sequence of large sequential
// HBM reads.
#include "kernels.h"

namespace lmoe {

namespace {

__global__ void pack_tiles_kernel(const uint4 *__restrict__ src, int64_t E, int R, int K, int TR,
                                  uint4 *__restrict__ dst) {
    // one thread per 16-byte chunk (8 bf16), in destination order
    const int64_t nchunk = E * R * int64_t(K / 8);
    const int KB = K / 64;
    const int NTR = R / TR;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nchunk;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % 8);           // chunk within the 64-column slice
        int64_t rest = i / 8;
        const int r = static_cast<int>(rest % TR);       // row within the tile
        rest /= TR;
        const int kb = static_cast<int>(rest % KB);
        rest /= KB;
        const int rt = static_cast<int>(rest % NTR);
        const int64_t e = rest / NTR;
        const int64_t srow = e * R + int64_t(rt) * TR + r;
        dst[i] = src[srow * (K / 8) + kb * 8 + c];
    }
}

}  // namespace

cudaError_t launch_pack_tiles(const uint16_t *src, int64_t E, int R, int K, int TR, uint16_t *dst,
                              cudaStream_t st) {
    if (R % TR != 0 || K % 64 != 0) return cudaErrorInvalidValue;
    pack_tiles_kernel<<<4096, 256, 0, st>>>(reinterpret_cast<const uint4 *>(src), E, R, K, TR,
                                           reinterpret_cast<uint4 *>(dst));
    return cudaGetLastError();
}

}  // namespace lmoe
