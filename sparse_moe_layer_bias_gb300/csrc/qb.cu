// qb.cu -- Quantile Balancing: per-expert B-bin histogram of router scores
// and the quantile read that sets each expert's selection bias.
// ("Kimi-K3-Architecture-Deep-Dive" section 3: map scores into [0,1], keep a
// local B-bin histogram, histograms are additive so one all-reduce of the
// counts rebuilds the global distribution, 1000 bins suffice; "Inside K3"
// section "Quantile Balancing (QB)": read the quantile from that histogram;
// news write-up "Keeping the numbers in range": solve for each expert's
// threshold directly.)
//
// Histogram layout on the GPU: CTA (expert group g, token chunk c) owns the
// counters of EPC consecutive experts in shared memory, streams its chunk of
// rows with 16-byte loads (EPC = 32 -> each row segment is one 128-byte line),
// counts with shared-memory atomics, and adds its non-zero counters into the
// global histogram at the end.  The global adds are the on-chip analogue of
// the cross-node all-reduce.  For large B (where 32-bit counters would leave
// fewer than 32 experts per CTA) the counters are 16-bit, two bins per 32-bit
// word, spilled to the global histogram before they could carry into their
// neighbour: twice the experts per CTA, so each row segment a CTA reads is a
// whole 32-byte sector or more.
#include <algorithm>

#include "kernels.h"

namespace lmoe {

namespace {

constexpr int kHistThreads = 1024;
constexpr size_t kHistSmemBudget = 200 * 1024;

__device__ __forceinline__ int bin_of(float s, float fB, int B) {
    const float f = floorf(__fmul_rn(s, fB));  // one fp32 rounding, then floor
    // s < 1/B (and NaN) -> bin 0; large values clamp to B-1
    return (f >= 1.0f) ? min(static_cast<int>(fminf(f, 2147483520.0f)), B - 1) : 0;
}

// Vector path: E % 4 == 0, ld % 4 == 0, 16-byte aligned rows; EPC in {4..32}.
// PACK16: counters of bins 2w and 2w+1 share word w (low / high 16 bits).  A
// 16-bit counter must never reach 65536 (it would carry into its neighbour),
// so the rows are counted in spans of kSpan16 = 32768: after each span every
// counter that has reached 32768 is added to the global histogram and
// cleared; any other counter can take at most 32768 more counts before the
// next check.  The global adds are so far fewer than a flush per 65535 rows
// (a counter of a 10000-bin histogram rarely gets near 32768).
constexpr int64_t kSpan16 = 32768;

// U: row sweeps whose loads are in flight per thread.  (With 16-bit counters
// for 10000 bins one CTA fills an SM's shared memory; 8 or 16 sweeps in flight
// measured slower than 4 there: that kernel is bound by its shared-memory
// atomics, not by loads in flight.)
template <int EPC, bool PACK16, int U>
__global__ void __launch_bounds__(kHistThreads)
    qb_hist_vec_kernel(const float *__restrict__ s, int64_t T, int E, int64_t ld, int B,
                       uint32_t *__restrict__ hist, int n_groups, int64_t rows_per_chunk) {
    extern __shared__ uint32_t cnt[];  // [EPC][WB] words
    const int WB = PACK16 ? (B + 1) / 2 : B;   // counter words per expert
    constexpr int NQ = EPC / 4;                 // float4 per row segment
    constexpr int ROWS = kHistThreads / NQ;     // rows per sweep
    const int g = blockIdx.x % n_groups;
    const int64_t chunk = blockIdx.x / n_groups;
    const int e0 = g * EPC;
    const int ne = min(EPC, E - e0);
    const int64_t r_begin = chunk * rows_per_chunk;
    const int64_t r_end = min(T, r_begin + rows_per_chunk);
    for (int i = threadIdx.x; i < ne * WB; i += kHistThreads) cnt[i] = 0u;
    __syncthreads();

    const float fB = static_cast<float>(B);
    auto count = [&](int c, float v) {
        const int b = bin_of(v, fB, B);
        if (PACK16)
            atomicAdd(&cnt[c * WB + (b >> 1)], 1u << ((b & 1) << 4));
        else
            atomicAdd(&cnt[c * WB + b], 1u);
    };
    uint32_t *dst = hist + int64_t(e0) * B;
    // 16-bit counters: add the halves at or above `min_count` to the global
    // histogram and clear them (the caller synchronised the block before)
    auto spill16 = [&](uint32_t min_count) {
        for (int i = threadIdx.x; i < ne * WB; i += kHistThreads) {
            const uint32_t c = cnt[i];
            if (!c) continue;
            const uint32_t lo = c & 0xffffu, hi = c >> 16;
            const bool tlo = lo && lo >= min_count, thi = hi && hi >= min_count;
            if (!(tlo || thi)) continue;
            const int e = i / WB, b = 2 * (i % WB);
            if (tlo) atomicAdd(&dst[int64_t(e) * B + b], lo);
            if (thi) atomicAdd(&dst[int64_t(e) * B + b + 1], hi);   // b + 1 < B when non-zero
            cnt[i] = (tlo ? 0u : lo) | (thi ? 0u : (hi << 16));
        }
    };
    const int q = threadIdx.x % NQ;
    const int rl = threadIdx.x / NQ;
    const bool qv = 4 * q < ne;
    const float *col = s + e0 + 4 * q;
    const int64_t span = PACK16 ? kSpan16 : (r_end - r_begin);
    for (int64_t s0 = r_begin; s0 < r_end; s0 += span) {
        const int64_t s1 = min(r_end, s0 + span);
        for (int64_t r0 = s0; r0 < s1; r0 += int64_t(ROWS) * U) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = r0 + int64_t(u) * ROWS + rl;
                v[u] = (qv && row < s1) ? __ldcs(reinterpret_cast<const float4 *>(col + row * ld))
                                        : make_float4(-1.f, -1.f, -1.f, -1.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = r0 + int64_t(u) * ROWS + rl;
                if (!(qv && row < s1)) continue;
                const int c = 4 * q;
                count(c + 0, v[u].x);
                count(c + 1, v[u].y);
                count(c + 2, v[u].z);
                count(c + 3, v[u].w);
            }
        }
        if (PACK16 && s1 < r_end) {   // more rows follow: spill the counters that could overflow
            __syncthreads();
            spill16(static_cast<uint32_t>(kSpan16));
            __syncthreads();
        }
    }
    __syncthreads();
    if (PACK16) {
        spill16(1u);
    } else {
        for (int i = threadIdx.x; i < ne * WB; i += kHistThreads) {
            const uint32_t c = cnt[i];
            if (c) atomicAdd(&dst[i], c);
        }
    }
}

// Scalar path for any E / ld / alignment.
__global__ void __launch_bounds__(kHistThreads)
    qb_hist_scalar_kernel(const float *__restrict__ s, int64_t T, int E, int64_t ld, int B,
                          uint32_t *__restrict__ hist, int epc, int n_groups,
                          int64_t rows_per_chunk) {
    extern __shared__ uint32_t cnt[];
    const int g = blockIdx.x % n_groups;
    const int64_t chunk = blockIdx.x / n_groups;
    const int e0 = g * epc;
    const int ne = min(epc, E - e0);
    const int64_t r_begin = chunk * rows_per_chunk;
    const int64_t r_end = min(T, r_begin + rows_per_chunk);
    for (int i = threadIdx.x; i < ne * B; i += kHistThreads) cnt[i] = 0u;
    __syncthreads();
    const float fB = static_cast<float>(B);
    const int64_t n = (r_end - r_begin) * ne;
    for (int64_t i = threadIdx.x; i < n; i += kHistThreads) {
        const int64_t row = r_begin + i / ne;
        const int c = static_cast<int>(i % ne);
        atomicAdd(&cnt[c * B + bin_of(s[row * ld + e0 + c], fB, B)], 1u);
    }
    __syncthreads();
    uint32_t *dst = hist + int64_t(e0) * B;
    for (int i = threadIdx.x; i < ne * B; i += kHistThreads) {
        const uint32_t c = cnt[i];
        if (c) atomicAdd(&dst[i], c);
    }
}

// Bins too many for shared memory: count straight into the global histogram.
__global__ void qb_hist_global_kernel(const float *__restrict__ s, int64_t T, int E, int64_t ld,
                                      int B, uint32_t *__restrict__ hist) {
    const float fB = static_cast<float>(B);
    const int64_t n = T * E;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = i / E;
        const int c = static_cast<int>(i % E);
        atomicAdd(&hist[int64_t(c) * B + bin_of(s[row * ld + c], fB, B)], 1u);
    }
}

// One warp per expert: N, the rank r, the first bin whose cumulative count
// reaches r (found in two levels: the lanes' spans of bins, then the bins of
// one span), and the in-bin linear interpolation, all in fp64.
__global__ void qb_quantile_kernel(const uint32_t *__restrict__ hist, int E, int B, double level,
                                   float *__restrict__ q_out, float *__restrict__ b_out) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (e >= E) return;
    const uint32_t *row = hist + int64_t(e) * B;
    // Two levels: lane l sums the bins of its span [l*span, (l+1)*span); one
    // scan over the lanes gives n and the span holding the r-th count; the
    // warp then scans that span alone for the first bin whose cumulative
    // count reaches r.
    const int span = (B + 31) / 32;
    const int s0 = min(B, lane * span), s1 = min(B, s0 + span);
    unsigned long long part = 0;
    for (int j = s0; j < s1; ++j) part += row[j];
    unsigned long long incl = part;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const unsigned long long n = __shfl_sync(0xffffffffu, incl, 31);
    double q = 0.0;
    if (n > 0) {
        double rr = ceil(level * static_cast<double>(n));
        if (rr < 1.0) rr = 1.0;
        if (rr > static_cast<double>(n)) rr = static_cast<double>(n);
        const unsigned long long r = static_cast<unsigned long long>(rr);
        // the first span whose cumulative count reaches r (lane 31's is n >= r)
        const int fs = __ffs(__ballot_sync(0xffffffffu, incl >= r)) - 1;
        unsigned long long below = __shfl_sync(0xffffffffu, incl - part, fs);   // counts before that span
        const int j_begin = __shfl_sync(0xffffffffu, s0, fs), j_end = __shfl_sync(0xffffffffu, s1, fs);
        for (int j0 = j_begin; j0 < j_end; j0 += 32) {
            const int j = j0 + lane;
            const unsigned long long c = (j < j_end) ? row[j] : 0ull;
            unsigned long long inc = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += o;
            }
            const unsigned ballot = __ballot_sync(0xffffffffu, j < j_end && below + inc >= r);
            if (ballot) {
                const int f = __ffs(ballot) - 1;
                const unsigned long long cf = __shfl_sync(0xffffffffu, c, f);
                const unsigned long long inf = __shfl_sync(0xffffffffu, inc, f);
                const unsigned long long before = below + inf - cf;  // C_{j*-1}
                q = (static_cast<double>(j0 + f) +
                     static_cast<double>(r - before) / static_cast<double>(cf)) /
                    static_cast<double>(B);
                break;
            }
            below += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    if (lane == 0) {
        if (q_out) q_out[e] = static_cast<float>(q);
        b_out[e] = static_cast<float>(-q);
    }
}

}  // namespace

cudaError_t launch_qb_histogram(const float *scores, int64_t T, int E, int64_t ld, int B,
                                uint32_t *hist, int accumulate, int num_sms, cudaStream_t st) {
    cudaError_t err;
    if (!accumulate) {
        err = cudaMemsetAsync(hist, 0, size_t(E) * size_t(B) * sizeof(uint32_t), st);
        if (err != cudaSuccess) return err;
    }
    if (T == 0) return cudaSuccess;
    const size_t per_expert = size_t(B) * sizeof(uint32_t);
    if (per_expert > kHistSmemBudget) {
        qb_hist_global_kernel<<<num_sms * 4, 512, 0, st>>>(scores, T, E, ld, B, hist);
        return cudaGetLastError();
    }
    // at most 16 experts per CTA: a 64-byte piece of each row already streams
    // well, and the smaller counter block leaves room for two CTAs per SM
    int epc = 16;
    while (epc > 1 && size_t(epc) * per_expert > kHistSmemBudget) epc >>= 1;
    const bool vec = epc >= 4 && (E % 4 == 0) && (ld % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(scores) % 16 == 0);
    // 16-bit counters where they let a CTA hold more experts (vector path)
    const size_t per_expert16 = size_t((B + 1) / 2) * sizeof(uint32_t);
    int epc16 = 16;
    while (epc16 > 1 && size_t(epc16) * per_expert16 > kHistSmemBudget) epc16 >>= 1;
    const bool pack16 = vec && epc16 > epc;
    if (pack16) epc = epc16;
    const int n_groups = (E + epc - 1) / epc;
    const size_t smem = size_t(epc) * (pack16 ? per_expert16 : per_expert);
    const int ctas_per_sm = max(1, min(2, static_cast<int>((227 * 1024) / (smem + 1024))));
    // Token chunks per expert group: the fewest (each chunk ends with one
    // global add per non-zero counter) that fill the GPU in whole waves --
    // the first count whose last wave is at least 90% full.
    const int slots = num_sms * ctas_per_sm;
    const int64_t min_rows = 512;
    const int64_t max_chunks = (T + min_rows - 1) / min_rows;
    // at least one wave's worth of CTAs (few expert groups: more chunks), no
    // chunk shorter than min_rows; then up to 16 more chunks if that fills
    // the last wave to 90%
    const int first = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(slots / n_groups, max_chunks)));
    int n_chunks = first;
    for (int c = first; c <= first + 16 && c <= max_chunks; ++c) {
        const int ctas = n_groups * c;
        const int waves = (ctas + slots - 1) / slots;
        if (ctas * 10 >= waves * slots * 9) {
            n_chunks = c;
            break;
        }
    }
    const int64_t rows_per_chunk = (T + n_chunks - 1) / n_chunks;
    const unsigned grid = static_cast<unsigned>(n_groups) * static_cast<unsigned>(n_chunks);

#define LMOE_QB_VEC(N_, P_, U_)                                                                     \
    case N_:                                                                                        \
        err = cudaFuncSetAttribute(qb_hist_vec_kernel<N_, P_, U_>,                                  \
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
        if (err != cudaSuccess) return err;                                                         \
        qb_hist_vec_kernel<N_, P_, U_><<<grid, kHistThreads, smem, st>>>(scores, T, E, ld, B, hist,  \
                                                                         n_groups, rows_per_chunk); \
        break;
    if (vec && pack16) {
        switch (epc) {
            LMOE_QB_VEC(8, true, 4)
            LMOE_QB_VEC(16, true, 4)
            default:
                return cudaErrorInvalidValue;
        }
    } else if (vec) {
        switch (epc) {
            LMOE_QB_VEC(4, false, 4)
            LMOE_QB_VEC(8, false, 4)
            LMOE_QB_VEC(16, false, 4)
            default:
                return cudaErrorInvalidValue;
        }
    } else {
        err = cudaFuncSetAttribute(qb_hist_scalar_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
        if (err != cudaSuccess) return err;
        qb_hist_scalar_kernel<<<grid, kHistThreads, smem, st>>>(scores, T, E, ld, B, hist, epc,
                                                               n_groups, rows_per_chunk);
    }
#undef LMOE_QB_VEC
    return cudaGetLastError();
}

// Fixed-step bias update (the rule QB replaces): one CTA sums the loads, then
// every expert's bias moves by +gamma (under-loaded), -gamma (over-loaded) or
// not at all; the comparison counts[e] * E <=> total is exact in integers.
__global__ void __launch_bounds__(1024) sign_update_kernel(const int32_t *__restrict__ counts, int E, float gamma,
                                                           float *__restrict__ bias) {
    __shared__ long long s_part[32];
    long long part = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) part += counts[e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = part;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < (int(blockDim.x) + 31) / 32; ++w) total += s_part[w];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const long long scaled = static_cast<long long>(counts[e]) * E;
        if (scaled < total)
            bias[e] = __fadd_rn(bias[e], gamma);
        else if (scaled > total)
            bias[e] = __fsub_rn(bias[e], gamma);
    }
}

cudaError_t launch_sign_update(const int32_t *counts, int E, float gamma, float *bias, cudaStream_t st) {
    sign_update_kernel<<<1, 1024, 0, st>>>(counts, E, gamma, bias);
    return cudaGetLastError();
}

cudaError_t launch_qb_quantile(const uint32_t *hist, int E, int B, double level, float *q,
                               float *bias, cudaStream_t st) {
    const int wpb = 8;
    qb_quantile_kernel<<<(E + wpb - 1) / wpb, wpb * 32, 0, st>>>(hist, E, B, level, q, bias);
    return cudaGetLastError();
}

}  // namespace lmoe
