// combine.cu -- a7: gate-weighted aggregation of the routed experts and the
// single un-weighted RMSNorm ahead of the up-projection.
// ("Kimi-K3-Architecture-Deep-Dive" section 2: one RMS Norm before the
// up-projection; "Inside K3" section "RMSNorm insertion"; news write-up
// "Keeping the numbers in range": the norm sits after aggregation.)
//   z_t = sum_j o[t*k + j]          (o rows are already gate-weighted, bf16)
//   r_t = z_t / sqrt(mean(z_t^2) + eps)   -> bf16
// One CTA per token; each thread keeps VPT vectors of 8 latent channels in
// fp32 registers, so z is read once from the k expert rows and never stored.
// A token's k rows are contiguous (assignment order), and the kernel is bound
// by the bytes it keeps in flight: where they fit in shared memory they
// arrive there by bulk copies (one per row, all in flight at once: 112 KB
// per token at K3 widths, two tokens per SM), else each thread loads four
// rows at a time into registers.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

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

// z (this thread's VPT vectors of 8 channels, fp32) -> r = z / sqrt(mean z^2
// + eps) in bf16: the sum of squares over the row by warp shuffles and one
// shared-memory step (the whole CTA takes part).
template <int VPT>
__device__ __forceinline__ void store_rms_row(const float (&acc)[VPT][8], int L, float eps, uint16_t *row) {
    const int nvec = L / 8;
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

    uint4 *out = reinterpret_cast<uint4 *>(row);
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

constexpr size_t kBulkRowsOffset = 64;          // the mbarrier and the abort flag come first
constexpr size_t kBulkSmemMax = 227 * 1024;

// The same with the token's k rows in shared memory: warp 0's lanes issue one
// bulk copy per row onto one mbarrier (armed first with all the bytes), every
// thread waits for it (bounded), then sums its channels over the rows in the
// same order as the kernel above (so both give the same bits).
template <int VPT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_rmsnorm_bulk_kernel(const uint16_t *__restrict__ o, int k, int L, float eps,
                                uint16_t *__restrict__ r, unsigned *err, uint64_t wait_limit_ns) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + 8);
    const uint4 *rows = reinterpret_cast<const uint4 *>(smem + kBulkRowsOffset);
    const int64_t t = blockIdx.x;
    const int nvec = L / 8;
    const uint32_t row_bytes = static_cast<uint32_t>(L) * 2u;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependency_wait();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) mbar_arrive_expect_tx(smem_u32(bar), row_bytes * static_cast<uint32_t>(k));
        __syncwarp();
        for (int j = threadIdx.x; j < k; j += 32)
            bulk_load(smem_u32(smem + kBulkRowsOffset + size_t(j) * row_bytes), o + (t * k + j) * int64_t(L),
                      row_bytes, smem_u32(bar));
    }
    const bool landed = mbar_wait(smem_u32(bar), 0u, abort_flag, err, wait_limit_ns, /*watch_abort=*/false);
    if (!__syncthreads_and(landed ? 1 : 0)) {
        // the copies did not land in time (the status bit is set): leave no
        // copy in flight into this CTA's shared memory, then give up the token
        if (threadIdx.x == 0) mbar_wait(smem_u32(bar), 0u, abort_flag, err, wait_limit_ns, false);
        __syncthreads();
        return;
    }
    float acc[VPT][8];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[v][i] = 0.0f;
    for (int j = 0; j < k; ++j)
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = threadIdx.x + v * kCombineThreads;
            if (vi < nvec) add_bf16x8(acc[v], rows[int64_t(j) * nvec + vi]);
        }
    store_rms_row<VPT>(acc, L, eps, r + t * int64_t(L));
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

    store_rms_row<VPT>(acc, L, eps, r + t * int64_t(L));
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
                                   uint16_t *r, unsigned *err, uint64_t wait_limit_ns, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int nvec = L / 8;
    const int vpt = (nvec + kCombineThreads - 1) / kCombineThreads;
    const dim3 grid(static_cast<unsigned>(T));
    const dim3 block(kCombineThreads);
    const size_t smem = kBulkRowsOffset + size_t(k) * size_t(L) * 2;
    if (L % 8 == 0 && (reinterpret_cast<uintptr_t>(o) % 16) == 0 && smem <= kBulkSmemMax) {
        auto bulk = [&](auto kern) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return launch_kernel(kern, grid, block, smem, st, true, o, k, L, eps, r, err, wait_limit_ns);
        };
        if (vpt <= 1) return bulk(combine_rmsnorm_bulk_kernel<1>);
        if (vpt <= 2) return bulk(combine_rmsnorm_bulk_kernel<2>);
        if (vpt <= 4) return bulk(combine_rmsnorm_bulk_kernel<4>);
    }
    if (vpt <= 1) return launch_kernel(combine_rmsnorm_kernel<1>, grid, block, 0, st, true, o, k, L, eps, r);
    if (vpt <= 2) return launch_kernel(combine_rmsnorm_kernel<2>, grid, block, 0, st, true, o, k, L, eps, r);
    if (vpt <= 4) return launch_kernel(combine_rmsnorm_kernel<4>, grid, block, 0, st, true, o, k, L, eps, r);
    return cudaErrorInvalidValue;
}

}  // namespace lmoe
