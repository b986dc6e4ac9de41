// combine.cu -- a7: gate-weighted aggregation of the routed experts and the
// single un-weighted RMSNorm ahead of the up-projection.
// ("Kimi-K3-Architecture-Deep-Dive" section 2: one RMS Norm before the
// up-projection; "Inside K3" section "RMSNorm insertion"; news write-up
// "Keeping the numbers in range": the norm sits after aggregation.)
//   z_t = sum_j o[t*k + j]          (o rows are already gate-weighted, bf16)
//   r_t = z_t / sqrt(mean(z_t^2) + eps)   -> bf16
// One CTA per token; each thread keeps VPT vectors of 8 latent channels in
// fp32 registers, so z is read once from the k expert rows and never stored.
#include <cuda_bf16.h>

#include "kernels.h"

namespace lmoe {

namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(u[i] << 16);
        acc[2 * i + 1] += __uint_as_float(u[i] & 0xffff0000u);
    }
}

template <int VPT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_rmsnorm_kernel(const uint16_t *__restrict__ o, int k, int L, float eps,
                           uint16_t *__restrict__ r) {
    grid_dependency_wait();
    const int64_t t = blockIdx.x;
    const int nvec = L / 8;
    float acc[VPT][8];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[v][i] = 0.0f;

    const uint4 *base = reinterpret_cast<const uint4 *>(o + t * k * int64_t(L));
    int j = 0;
    for (; j + 4 <= k; j += 4) {  // four expert rows in flight per step
        uint4 w[4][VPT];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int vi = threadIdx.x + v * kCombineThreads;
                w[jj][v] = (vi < nvec) ? __ldg(base + (int64_t)(j + jj) * nvec + vi) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int v = 0; v < VPT; ++v) add_bf16x8(acc[v], w[jj][v]);
    }
    for (; j < k; ++j)
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = threadIdx.x + v * kCombineThreads;
            if (vi < nvec) add_bf16x8(acc[v], __ldg(base + (int64_t)j * nvec + vi));
        }

    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += acc[v][i] * acc[v][i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ float part[kCombineThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) tot += part[w];
    const float inv_rms = 1.0f / sqrtf(tot / static_cast<float>(L) + eps);

    uint4 *out = reinterpret_cast<uint4 *>(r + t * int64_t(L));
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = threadIdx.x + v * kCombineThreads;
        if (vi >= nvec) continue;
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(acc[v][2 * i] * inv_rms, acc[v][2 * i + 1] * inv_rms);
            p[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        out[vi] = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

// Ablation variant's norm after the down-projection ("Kimi-K3-Architecture-
// Deep-Dive" section 2 and "Inside K3" section "RMSNorm insertion": the norm
// after the reduction that the ablation dropped): hn_t = h_t / sqrt(mean(h_t^2)
// + eps) on the bf16 row h_t.  The row's sum of squares, the scale and the
// products are fp64 (bf16 squares are exact in fp64), and each product is
// rounded once to bf16: first to fp32 with round-to-odd (truncate, then set
// the last bit if anything was cut off), then to bf16 with round-to-nearest-
// even.  Rounding to odd at a precision with at least two extra bits makes
// the second rounding equal to a direct one (Boldo and Melquiond, "Emulation
// of FMA and correctly rounded sums: proved algorithms using rounding to
// odd", IEEE Trans. Computers 57(4), 2008).  So the result is the correctly
// rounded bf16 of the fp64 quotient, as the routing decisions downstream need.
__device__ __forceinline__ float f64_to_f32_round_odd(double d) {
    float f = __double2float_rz(d);
    if (static_cast<double>(f) != d) f = __uint_as_float(__float_as_uint(f) | 1u);
    return f;
}

__global__ void __launch_bounds__(kCombineThreads)
    rms_rows_kernel(const uint16_t *__restrict__ h, int L, double eps, uint16_t *__restrict__ out) {
    grid_dependency_wait();
    const int64_t t = blockIdx.x;
    const int nvec = L / 8;
    const uint4 *row = reinterpret_cast<const uint4 *>(h + t * int64_t(L));
    double ss = 0.0;
    for (int vi = threadIdx.x; vi < nvec; vi += kCombineThreads) {
        const uint4 w = __ldg(row + vi);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const double lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xffff0000u);
            ss = fma(lo, lo, ss);
            ss = fma(hi, hi, ss);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ double part[kCombineThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) tot += part[w];
    const double rms = sqrt(tot / static_cast<double>(L) + eps);
    const double inv = rms > 0.0 ? 1.0 / rms : 0.0;
    uint4 *dst = reinterpret_cast<uint4 *>(out + t * int64_t(L));
    for (int vi = threadIdx.x; vi < nvec; vi += kCombineThreads) {
        const uint4 w = __ldg(row + vi);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const double lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xffff0000u);
            __nv_bfloat162 b = __floats2bfloat162_rn(f64_to_f32_round_odd(lo * inv), f64_to_f32_round_odd(hi * inv));
            p[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        dst[vi] = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

}  // namespace

cudaError_t launch_rms_rows(const uint16_t *h, int64_t T, int L, double eps, uint16_t *out, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    return launch_kernel(rms_rows_kernel, dim3(static_cast<unsigned>(T)), dim3(kCombineThreads), 0, st, true, h, L, eps,
                         out);
}

cudaError_t launch_combine_rmsnorm(const uint16_t *o, int64_t T, int k, int L, float eps,
                                   uint16_t *r, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int nvec = L / 8;
    const int vpt = (nvec + kCombineThreads - 1) / kCombineThreads;
    const dim3 grid(static_cast<unsigned>(T));
    const dim3 block(kCombineThreads);
    if (vpt <= 1) return launch_kernel(combine_rmsnorm_kernel<1>, grid, block, 0, st, true, o, k, L, eps, r);
    if (vpt <= 2) return launch_kernel(combine_rmsnorm_kernel<2>, grid, block, 0, st, true, o, k, L, eps, r);
    if (vpt <= 4) return launch_kernel(combine_rmsnorm_kernel<4>, grid, block, 0, st, true, o, k, L, eps, r);
    return cudaErrorInvalidValue;
}

}  // namespace lmoe
