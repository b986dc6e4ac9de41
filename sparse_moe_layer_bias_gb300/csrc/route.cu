// route.cu -- biased top-k expert selection and the token permutation.
//
// a3 ("Kimi-K3-Architecture-Deep-Dive" section 3; news write-up "Keeping the
// numbers in range"): the loss-free selection bias shifts which experts a
// token picks, not how their outputs are weighted.  Per token, one warp:
//   u_e = fp32(s_e + b_e); take the top_k largest u (ties: lower expert id),
//   gate_j = s at the chosen expert (unbiased).
// The k-th largest of the 32 lanes' largest keys is a lower bound tau on the
// token's k-th largest key (k lanes each hold a key at least that large), so
// every key of the top k is >= tau.  Typically only ~20 keys are; they are
// gathered into one per lane and put in order by one bitonic sort over the
// warp (key descending, expert id ascending).  A token with more than 32 such
// keys (e.g. a row of saturated scores) takes k rounds instead, each of two
// warp reductions (max of the lanes' best keys, then the lowest expert id
// among the lanes holding it).  Both give the same, exact result.
// a4: the T*top_k assignments are grouped by expert with a deterministic,
// stable counting sort.  A token picks an expert at most once, so "stable by
// assignment id" is "ordered by token": each expert keeps a bitmap over
// tokens, the rank of token t inside expert e is a popcount prefix of that
// bitmap, and no atomic ever decides an order.
#include "kernels.h"

namespace lmoe {

namespace {

constexpr int kTopkWarps = 8;

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0 is folded into +0 first so that the two compare equal, as floats do.
// Key 0 is the NaN pattern 0xffffffff and never occurs for finite scores; it
// marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float u) {
    const uint32_t b = __float_as_uint(__fadd_rn(u, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Bitonic sort of one value per lane, largest in lane 0.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
            // runs of `size` lanes alternate direction; the last run (all
            // 32 lanes) is descending, where the lower lane keeps the larger
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            v = (lower == desc) ? max(v, o) : min(v, o);
        }
    }
    return v;
}

// The same over (key, id) pairs, best first: larger key, then lower id (all
// ids distinct, so no two pairs compare equal).
__device__ __forceinline__ void warp_sort_pairs_desc(uint32_t &key, uint32_t &id, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, key, stride);
            const uint32_t oi = __shfl_xor_sync(0xffffffffu, id, stride);
            const bool other_better = ok > key || (ok == key && oi < id);
            const bool keep_better = ((lane & stride) == 0) == ((lane & size) == 0);
            if (keep_better == other_better) {
                key = ok;
                id = oi;
            }
        }
    }
}

template <int V>  // experts per lane (E <= 32*V)
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float *__restrict__ scores, const float *__restrict__ bias, int64_t T, int E,
                int k, int32_t *__restrict__ idx, float *__restrict__ gate,
                uint32_t *__restrict__ bitmap, int words) {
    grid_dependency_wait();
    __shared__ uint2 s_cand[kTopkWarps][32];   // a warp's candidates: (key, expert)
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t t = int64_t(blockIdx.x) * kTopkWarps + wib;
    if (t >= T) return;   // the whole warp; nothing below synchronises the block
    const float *srow = scores + t * E;
    uint32_t key[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int e = i * 32 + lane;
        key[i] = (e < E) ? order_key(__fadd_rn(srow[e], bias[e])) : 0u;
    }
    int my_e = -1;
    // tau: the k-th largest of the lanes' largest keys.  Lanes 0 .. min(E,32)-1
    // each hold an expert and k <= E, so tau is a real key (> 0), and the
    // experts past E (key 0) are never candidates.
    uint32_t lmax = 0u;
#pragma unroll
    for (int i = 0; i < V; ++i) lmax = max(lmax, key[i]);
    const uint32_t tau = __shfl_sync(0xffffffffu, warp_sort_desc(lmax, lane), k - 1);
    uint32_t cmask = 0u;   // bit i: key[i] is a candidate (V <= 32)
#pragma unroll
    for (int i = 0; i < V; ++i) cmask |= (key[i] >= tau ? 1u : 0u) << i;
    const int c = __popc(cmask);
    const int n_cand = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(c)));
    if (n_cand <= 32) {
        int incl = c;   // inclusive prefix of the lanes' candidate counts
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int pos0 = incl - c;   // the lane's candidates go to pos0, pos0 + 1, ...
#pragma unroll
        for (int i = 0; i < V; ++i)
            if ((cmask >> i) & 1u)
                s_cand[wib][pos0 + __popc(cmask & ((1u << i) - 1u))] =
                    make_uint2(key[i], static_cast<uint32_t>(i * 32 + lane));
        __syncwarp();
        // one candidate per lane; the empty lanes rank last (key 0, ids
        // above every expert's)
        uint32_t ck = 0u, ce = 0x10000u + static_cast<uint32_t>(lane);
        if (lane < n_cand) {
            const uint2 cv = s_cand[wib][lane];
            ck = cv.x;
            ce = cv.y;
        }
        warp_sort_pairs_desc(ck, ce, lane);
        my_e = static_cast<int>(ce);
    } else {
        uint32_t taken = 0u;   // bit i: key[i] was chosen in an earlier round
        for (int j = 0; j < k; ++j) {
            // lane-local best: largest key not yet taken, lowest expert id (=
            // lowest i) on ties
            uint32_t bk = 0u;
            int bi = 0;
#pragma unroll
            for (int i = V - 1; i >= 0; --i)
                if (!((taken >> i) & 1u) && key[i] >= bk) {
                    bk = key[i];
                    bi = i;
                }
            // warp: the largest key, then the lowest expert id holding it
            const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
            const int cand = (bk == wk && bk != 0u) ? bi * 32 + lane : 0x7fffffff;
            const int we = __reduce_min_sync(0xffffffffu, cand);
            if (we != 0x7fffffff && (we & 31) == lane) taken |= 1u << (we >> 5);
            if (lane == j) my_e = we;
        }
    }
    if (lane < k) {
        idx[t * k + lane] = my_e;
        gate[t * k + lane] = srow[my_e];          // the unbiased score
        atomicOr(&bitmap[int64_t(my_e) * words + (t >> 5)], 1u << (t & 31));
    }
}

// word_prefix[e][w] = number of tokens < 32*w that picked e; counts[e] = total.
__global__ void expert_scan_kernel(const uint32_t *__restrict__ bitmap, int E, int words,
                                   uint32_t *__restrict__ word_prefix, int32_t *__restrict__ counts) {
    grid_dependency_wait();
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

// One CTA: offsets = exclusive scan of counts, and two grouped-GEMM tile lists
// (expert, first permuted row, rows), experts in id order: ceil(count/128)
// tiles of up to 128 rows, and ceil(count/256) pair tiles of up to 256 rows.
__global__ void __launch_bounds__(1024)
    offsets_tiles_kernel(const int32_t *__restrict__ counts, int E, int32_t *__restrict__ offsets,
                         int4 *__restrict__ tiles, int32_t *__restrict__ n_mtiles,
                         int4 *__restrict__ tiles2, int32_t *__restrict__ n_mtiles2,
                         int4 *__restrict__ tiles3, int32_t *__restrict__ n_mtiles3) {
    grid_dependency_wait();
    __shared__ int32_t s_cnt[1024];
    __shared__ int32_t s_til[1024];
    __shared__ int32_t s_til2[1024];
    __shared__ int32_t s_til3[1024];
    const int e = threadIdx.x;
    const bool split = tiles3 != nullptr;
    const int32_t c = (e < E) ? counts[e] : 0;
    const int32_t nt = (c + kBM - 1) / kBM;
    const int32_t nt3 = (split && c > 0 && c <= kBM) ? 1 : 0;   // light: one 128-row tile
    const int32_t nt2 = nt3 ? 0 : (c + 2 * kBM - 1) / (2 * kBM);
    s_cnt[e] = c;
    s_til[e] = nt;
    s_til2[e] = nt2;
    s_til3[e] = nt3;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // Hillis-Steele inclusive scans
        int32_t a = 0, b = 0, b2 = 0, b3 = 0;
        if (e >= off) {
            a = s_cnt[e - off];
            b = s_til[e - off];
            b2 = s_til2[e - off];
            b3 = s_til3[e - off];
        }
        __syncthreads();
        s_cnt[e] += a;
        s_til[e] += b;
        s_til2[e] += b2;
        s_til3[e] += b3;
        __syncthreads();
    }
    if (e < E) {
        const int32_t row0 = s_cnt[e] - c;
        offsets[e] = row0;
        const int32_t tile0 = s_til[e] - nt;
        for (int32_t m = 0; m < nt; ++m)
            tiles[tile0 + m] = make_int4(e, row0 + m * kBM, min(kBM, c - m * kBM), 0);
        const int32_t pair0 = s_til2[e] - nt2;
        for (int32_t m = 0; m < nt2; ++m)
            tiles2[pair0 + m] = make_int4(e, row0 + m * 2 * kBM, min(2 * kBM, c - m * 2 * kBM), 0);
        if (nt3) tiles3[s_til3[e] - 1] = make_int4(e, row0, c, 0);
    }
    if (e == E - 1) {
        offsets[E] = s_cnt[e];
        *n_mtiles = s_til[e];
        *n_mtiles2 = s_til2[e];
        if (split) *n_mtiles3 = s_til3[e];
    }
}

__global__ void scatter_kernel(const int32_t *__restrict__ idx, int64_t T, int k, int E,
                               const uint32_t *__restrict__ bitmap,
                               const uint32_t *__restrict__ word_prefix, int words,
                               const int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                               int32_t *__restrict__ inv, int32_t *__restrict__ tokrow) {
    grid_dependency_wait();
    const int64_t a = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (a >= T * k) return;
    const int64_t t = a / k;
    const int e = idx[a];
    if (!idx_ok(e, E)) return;
    const int64_t w = int64_t(e) * words + (t >> 5);
    const uint32_t below = bitmap[w] & ((1u << (t & 31)) - 1u);
    const int32_t p = offsets[e] + static_cast<int32_t>(word_prefix[w] + __popc(below));
    if (!idx_ok(p, T * k)) return;
    perm[p] = static_cast<int32_t>(a);
    inv[a] = p;
    tokrow[p] = static_cast<int32_t>(t);
}

}  // namespace

cudaError_t launch_topk(const float *scores, const float *bias, int64_t T, int E, int k,
                        int32_t *idx, float *gate, uint32_t *bitmap, int words, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((T + kTopkWarps - 1) / kTopkWarps));
    const dim3 block(kTopkWarps * 32);
    const int v = (E + 31) / 32;
    if (v <= 1)
        return launch_kernel(topk_kernel<1>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 4)
        return launch_kernel(topk_kernel<4>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 8)
        return launch_kernel(topk_kernel<8>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 16)
        return launch_kernel(topk_kernel<16>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
    else if (v <= 28)
        return launch_kernel(topk_kernel<28>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
    return launch_kernel(topk_kernel<32>, grid, block, 0, st, true, scores, bias, T, E, k, idx, gate, bitmap, words);
}

cudaError_t launch_expert_scan(const uint32_t *bitmap, int E, int words, uint32_t *word_prefix,
                               int32_t *counts, cudaStream_t st) {
    const int wpb = 8;
    return launch_kernel(expert_scan_kernel, dim3((E + wpb - 1) / wpb), dim3(wpb * 32), 0, st, true, bitmap, E, words,
                         word_prefix, counts);
}

cudaError_t launch_offsets_tiles(const int32_t *counts, int E, int32_t *offsets, int4 *tiles,
                                 int32_t *n_mtiles, int4 *tiles2, int32_t *n_mtiles2, int4 *tiles3,
                                 int32_t *n_mtiles3, cudaStream_t st) {
    return launch_kernel(offsets_tiles_kernel, dim3(1), dim3(1024), 0, st, true, counts, E, offsets, tiles, n_mtiles,
                         tiles2, n_mtiles2, tiles3, n_mtiles3);
}

cudaError_t launch_scatter(const int32_t *idx, int64_t T, int k, int E, const uint32_t *bitmap,
                           const uint32_t *word_prefix, int words, const int32_t *offsets,
                           int32_t *perm, int32_t *inv, int32_t *tokrow, cudaStream_t st) {
    const int64_t n = T * k;
    if (n == 0) return cudaSuccess;
    return launch_kernel(scatter_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st, true, idx, T,
                         k, E, bitmap, word_prefix, words, offsets, perm, inv, tokrow);
}

LMOE_DEBUG_WORD_READER(debug_word_route)

}  // namespace lmoe
