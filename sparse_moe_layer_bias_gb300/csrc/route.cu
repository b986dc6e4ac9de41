// route.cu -- biased top-k expert selection and the token permutation.
//
// a3 ("Kimi-K3-Architecture-Deep-Dive" section 3; news write-up "Keeping the
// numbers in range"): the loss-free selection bias shifts which experts a
// token picks, not how their outputs are weighted.  Per token, one warp:
//   u_e = fp32(s_e + b_e); take the top_k largest u (ties: lower expert id),
//   gate_j = s at the chosen expert (unbiased).
// a4: the T*top_k assignments are grouped by expert with a deterministic,
// stable counting sort (and, for the forward, each assignment's latent row is
// copied into its grouped position).  A token picks an expert at most once, so "stable by
// assignment id" is "ordered by token": each expert keeps a bitmap over
// tokens, the rank of token t inside expert e is a popcount prefix of that
// bitmap, and no atomic ever decides an order.
#include "kernels.h"

namespace lmoe {

namespace {

constexpr int kTopkWarps = 8;

template <int V>  // experts per lane (E <= 32*V)
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float *__restrict__ scores, const float *__restrict__ bias, int64_t T, int E,
                int k, int32_t *__restrict__ idx, float *__restrict__ gate,
                uint32_t *__restrict__ bitmap, int words) {
    const int lane = threadIdx.x & 31;
    const int64_t t = int64_t(blockIdx.x) * kTopkWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *srow = scores + t * E;
    float s[V], u[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int e = i * 32 + lane;
        s[i] = (e < E) ? srow[e] : 0.0f;
        u[i] = (e < E) ? __fadd_rn(s[i], bias[e]) : 0.0f;
    }
    uint32_t taken = 0;
    int my_e = -1;
    float my_g = 0.0f;
    for (int j = 0; j < k; ++j) {
        // lane-local best: larger u, then lower id (ids grow with i)
        float bv = 0.0f;
        int be = 0x7fffffff;
        bool have = false;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = i * 32 + lane;
            if (e < E && !(taken & (1u << i)) && (!have || u[i] > bv)) {
                bv = u[i];
                be = e;
                have = true;
            }
        }
        // warp argmax over (u desc, id asc); lanes without a candidate lose
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            const bool ohave = __shfl_xor_sync(0xffffffffu, have ? 1 : 0, off) != 0;
            const bool better = ohave && (!have || ov > bv || (ov == bv && oe < be));
            if (better) {
                bv = ov;
                be = oe;
                have = true;
            }
        }
        // the owner lane marks it taken and hands the unbiased score over
        float gsc = 0.0f;
        if ((be & 31) == lane) {
            const int i = be >> 5;
#pragma unroll
            for (int ii = 0; ii < V; ++ii)
                if (ii == i) {
                    taken |= 1u << ii;
                    gsc = s[ii];
                }
        }
        gsc = __shfl_sync(0xffffffffu, gsc, be & 31);
        if (lane == j) {
            my_e = be;
            my_g = gsc;
        }
    }
    if (lane < k) {
        idx[t * k + lane] = my_e;
        gate[t * k + lane] = my_g;
        atomicOr(&bitmap[int64_t(my_e) * words + (t >> 5)], 1u << (t & 31));
    }
}

// word_prefix[e][w] = number of tokens < 32*w that picked e; counts[e] = total.
__global__ void expert_scan_kernel(const uint32_t *__restrict__ bitmap, int E, int words,
                                   uint32_t *__restrict__ word_prefix, int32_t *__restrict__ counts) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (e >= E) return;
    const uint32_t *row = bitmap + int64_t(e) * words;
    uint32_t *pre = word_prefix + int64_t(e) * words;
    uint32_t running = 0;
    for (int w0 = 0; w0 < words; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t c = (w < words) ? __popc(row[w]) : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (w < words) pre[w] = running + incl - c;
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = static_cast<int32_t>(running);
}

// One CTA: offsets = exclusive scan of counts; the grouped-GEMM tile list
// (expert, first permuted row, rows) with ceil(count/128) tiles per expert,
// experts in id order.
__global__ void __launch_bounds__(1024)
    offsets_tiles_kernel(const int32_t *__restrict__ counts, int E, int32_t *__restrict__ offsets,
                         int4 *__restrict__ tiles, int32_t *__restrict__ n_mtiles) {
    __shared__ int32_t s_cnt[1024];
    __shared__ int32_t s_til[1024];
    const int e = threadIdx.x;
    const int32_t c = (e < E) ? counts[e] : 0;
    const int32_t nt = (c + kBM - 1) / kBM;
    s_cnt[e] = c;
    s_til[e] = nt;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // Hillis-Steele inclusive scan
        int32_t a = 0, b = 0;
        if (e >= off) {
            a = s_cnt[e - off];
            b = s_til[e - off];
        }
        __syncthreads();
        s_cnt[e] += a;
        s_til[e] += b;
        __syncthreads();
    }
    if (e < E) {
        const int32_t row0 = s_cnt[e] - c;
        const int32_t tile0 = s_til[e] - nt;
        offsets[e] = row0;
        for (int32_t m = 0; m < nt; ++m)
            tiles[tile0 + m] = make_int4(e, row0 + m * kBM, min(kBM, c - m * kBM), 0);
    }
    if (e == E - 1) {
        offsets[E] = s_cnt[e];
        *n_mtiles = s_til[e];
    }
}

__global__ void scatter_kernel(const int32_t *__restrict__ idx, int64_t T, int k,
                               const uint32_t *__restrict__ bitmap,
                               const uint32_t *__restrict__ word_prefix, int words,
                               const int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                               int32_t *__restrict__ inv, int32_t *__restrict__ tokrow) {
    const int64_t a = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (a >= T * k) return;
    const int64_t t = a / k;
    const int e = idx[a];
    const int64_t w = int64_t(e) * words + (t >> 5);
    const uint32_t below = bitmap[w] & ((1u << (t & 31)) - 1u);
    const int32_t p = offsets[e] + static_cast<int32_t>(word_prefix[w] + __popc(below));
    perm[p] = static_cast<int32_t>(a);
    inv[a] = p;
    tokrow[p] = static_cast<int32_t>(t);
}

// Same maps as scatter_kernel, one warp per assignment, plus the copy of the
// assignment's latent row into its permuted slot: h_perm[p] = h[t].  The
// grouped expert GEMM then reads each expert's rows as dense TMA boxes.
constexpr int kCopyWarps = 8;
__global__ void __launch_bounds__(kCopyWarps * 32)
    scatter_copy_kernel(const int32_t *__restrict__ idx, int64_t T, int k,
                        const uint32_t *__restrict__ bitmap, const uint32_t *__restrict__ word_prefix,
                        int words, const int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                        int32_t *__restrict__ inv, int32_t *__restrict__ tokrow,
                        const uint16_t *__restrict__ h, int L, uint16_t *__restrict__ h_perm) {
    const int lane = threadIdx.x & 31;
    const int64_t a = int64_t(blockIdx.x) * kCopyWarps + (threadIdx.x >> 5);
    if (a >= T * k) return;
    const int64_t t = a / k;
    int32_t p = 0;
    if (lane == 0) {
        const int e = idx[a];
        const int64_t w = int64_t(e) * words + (t >> 5);
        const uint32_t below = bitmap[w] & ((1u << (t & 31)) - 1u);
        p = offsets[e] + static_cast<int32_t>(word_prefix[w] + __popc(below));
        perm[p] = static_cast<int32_t>(a);
        inv[a] = p;
        tokrow[p] = static_cast<int32_t>(t);
    }
    p = __shfl_sync(0xffffffffu, p, 0);
    const uint4 *src = reinterpret_cast<const uint4 *>(h + t * int64_t(L));
    uint4 *dst = reinterpret_cast<uint4 *>(h_perm + int64_t(p) * L);
    const int nvec = L / 8;
    for (int i0 = 0; i0 < nvec; i0 += 32 * 8) {   // 8 loads in flight per lane
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * 32 + lane;
            if (i < nvec) v[u] = __ldg(src + i);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * 32 + lane;
            if (i < nvec) dst[i] = v[u];
        }
    }
}

}  // namespace

cudaError_t launch_topk(const float *scores, const float *bias, int64_t T, int E, int k,
                        int32_t *idx, float *gate, uint32_t *bitmap, int words, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((T + kTopkWarps - 1) / kTopkWarps));
    const dim3 block(kTopkWarps * 32);
    const int v = (E + 31) / 32;
    if (v <= 1)
        topk_kernel<1><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 4)
        topk_kernel<4><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 8)
        topk_kernel<8><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 16)
        topk_kernel<16><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 28)
        topk_kernel<28><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    else
        topk_kernel<32><<<grid, block, 0, st>>>(scores, bias, T, E, k, idx, gate, bitmap, words);
    return cudaGetLastError();
}

cudaError_t launch_expert_scan(const uint32_t *bitmap, int E, int words, uint32_t *word_prefix,
                               int32_t *counts, cudaStream_t st) {
    const int wpb = 8;
    expert_scan_kernel<<<(E + wpb - 1) / wpb, wpb * 32, 0, st>>>(bitmap, E, words, word_prefix, counts);
    return cudaGetLastError();
}

cudaError_t launch_offsets_tiles(const int32_t *counts, int E, int32_t *offsets, int4 *tiles,
                                 int32_t *n_mtiles, cudaStream_t st) {
    offsets_tiles_kernel<<<1, 1024, 0, st>>>(counts, E, offsets, tiles, n_mtiles);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t *idx, int64_t T, int k, const uint32_t *bitmap,
                           const uint32_t *word_prefix, int words, const int32_t *offsets,
                           int32_t *perm, int32_t *inv, int32_t *tokrow, const uint16_t *h, int L,
                           uint16_t *h_perm, cudaStream_t st) {
    const int64_t n = T * k;
    if (n == 0) return cudaSuccess;
    if (h) {
        scatter_copy_kernel<<<static_cast<unsigned>((n + kCopyWarps - 1) / kCopyWarps), kCopyWarps * 32, 0,
                              st>>>(idx, T, k, bitmap, word_prefix, words, offsets, perm, inv, tokrow, h,
                                    L, h_perm);
    } else {
        scatter_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
            idx, T, k, bitmap, word_prefix, words, offsets, perm, inv, tokrow);
    }
    return cudaGetLastError();
}

}  // namespace lmoe
