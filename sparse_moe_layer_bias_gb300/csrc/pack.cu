// pack.cu -- one-time weight layout change at handle creation.
//
// The routed experts' GEMMs stream each expert's weights from HBM in boxes of
// TR rows x 64 columns (128 bytes per row, one K block).  In the caller's
// row-major [R][K] layout those 128-byte pieces sit K*2 bytes apart; stored
// tile-contiguously ([R/TR][K/64][TR][64]) every box is one contiguous
// TR*128-byte block, so the weight stream is a sequence of large sequential
// HBM reads.
#include <cuda_fp8.h>

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

// e4m3 quantisation of one row per CTA (FP8 expert variant):
//   e     = smallest integer with max|row| <= 448 * 2^e  (0 for a zero row);
//           with max|row| = f * 2^x, f in [0.5, 1) and 448 = 0.875 * 2^9,
//           e = x - 9 if f <= 0.875 else x - 8
//   codes = e4m3(v * 2^-e), round to nearest even, saturating at 448
// The scaling by 2^-e is exact, so the code is the single e4m3 rounding of
// the bf16 value's scaled copy.
constexpr int kQuantThreads = 128;

__global__ void __launch_bounds__(kQuantThreads)
    fp8_quantize_rows_kernel(const uint4 *__restrict__ src, int K, uint2 *__restrict__ codes,
                             int8_t *__restrict__ exps) {
    grid_dependency_wait();
    const int64_t r = blockIdx.x;
    const int nvec = K / 8;
    const uint4 *row = src + r * nvec;
    float amax = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += kQuantThreads) {
        const uint4 w = __ldg(row + v);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[i] << 16)), fabsf(__uint_as_float(u[i] & 0xffff0000u))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __shared__ float part[kQuantThreads / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = part[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, part[w]);
    int e = 0;
    if (amax > 0.0f) {
        int x;
        const float f = frexpf(amax, &x);
        e = (f <= 0.875f) ? x - 9 : x - 8;
    }
    if (threadIdx.x == 0) exps[r] = static_cast<int8_t>(e);
    uint2 *crow = codes + r * nvec;
    for (int v = threadIdx.x; v < nvec; v += kQuantThreads) {
        const uint4 w = __ldg(row + v);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = ldexpf(__uint_as_float(u[i] << 16), -e);
            const float hi = ldexpf(__uint_as_float(u[i] & 0xffff0000u), -e);
            const uint32_t pair = uint32_t(__nv_cvt_float_to_fp8(lo, __NV_SATFINITE, __NV_E4M3)) |
                                  (uint32_t(__nv_cvt_float_to_fp8(hi, __NV_SATFINITE, __NV_E4M3)) << 8);
            out[i >> 1] |= pair << (16 * (i & 1));
        }
        crow[v] = make_uint2(out[0], out[1]);
    }
}

}  // namespace

cudaError_t launch_fp8_quantize_rows(const uint16_t *src, int64_t R, int K, uint8_t *codes, int8_t *exps,
                                     cudaStream_t st) {
    if (K % 8 != 0 || R < 0) return cudaErrorInvalidValue;
    if (R == 0) return cudaSuccess;
    if (R > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_kernel(fp8_quantize_rows_kernel, dim3(static_cast<unsigned>(R)), dim3(kQuantThreads), 0, st, true,
                         reinterpret_cast<const uint4 *>(src), K, reinterpret_cast<uint2 *>(codes), exps);
}

cudaError_t launch_pack_tiles(const uint16_t *src, int64_t E, int R, int K, int TR, uint16_t *dst,
                              cudaStream_t st) {
    if (R % TR != 0 || K % 64 != 0) return cudaErrorInvalidValue;
    pack_tiles_kernel<<<4096, 256, 0, st>>>(reinterpret_cast<const uint4 *>(src), E, R, K, TR,
                                           reinterpret_cast<uint4 *>(dst));
    return cudaGetLastError();
}

}  // namespace lmoe
