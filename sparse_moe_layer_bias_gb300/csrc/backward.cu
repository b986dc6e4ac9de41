// backward.cu -- the memory-bound kernels of the layer's backward pass:
// transposes (plain, or gathering the rows of each expert's assignments into
// a padded per-expert column segment), the per-expert segment maps and
// weight-gradient tile lists, the RMSNorm backward, the router backward, the
// latent-gradient sum, the zeroing of unused experts' weight gradients and
// the SiTU-GLU backward at the pre-activations the forward kept.
//
// The gradient follows "Kimi-K3-Architecture-Deep-Dive" section 2 (the chain
// down-projection -> routed experts -> aggregate -> RMSNorm -> up-projection)
// and section 1 (SiTU-GLU; the tanh softcap is differentiable everywhere);
// the routing choice itself carries no gradient, the gates do.
#include <cuda_bf16.h>

#include "kernels.h"

namespace lmoe {

namespace {

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ uint16_t f_to_bf16(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

constexpr int kTT = 64;  // transpose tile: 64 x 64 elements

// out[b][c][q] = scale(q) * in[b][src(q)][c] for c < C, q < Q, where
// src(q) = qsrc[q] (or q when q < R without qsrc) and a negative src gives 0.
// Tiles whose first q is at or past *q_limit are skipped (never read later).
// 16-byte accesses on both sides: a thread loads 8 columns of one source row
// and stores 8 consecutive q of one output row (element-wise at a ragged C or
// Q).  With packed_rows > 0 the output is K-block packed: element (c, q) sits
// at ((q / 64) * packed_rows + c) * 64 + q % 64, so each 64-column block of q
// is one contiguous [packed_rows][64] slab and a TMA box of consecutive rows
// in it is one contiguous run of memory (ldo and obs are then unused).  The
// shared tile is stored with its 16-byte chunks XOR-swizzled by (q / 8) % 8 so
// that the column reads of the store phase spread over the banks.  Requires
// ldi, ldo, the batch strides and the pointers to be multiples of 8 elements
// (16 bytes).
__device__ __forceinline__ int swz(int q, int c) { return q * kTT + ((((c >> 3) ^ (q >> 3)) & 7) << 3) + (c & 7); }

__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t *__restrict__ in, int64_t ldi, int64_t ibs,
                                                        int64_t R, int C, uint16_t *__restrict__ out, int64_t ldo,
                                                        int64_t obs, int64_t Q, const int32_t *__restrict__ qsrc,
                                                        const float *__restrict__ qscale,
                                                        const int32_t *__restrict__ q_limit, int64_t packed_rows) {
    grid_dependency_wait();
    __shared__ __align__(16) uint16_t tile[kTT * kTT];
    const int64_t q0 = int64_t(blockIdx.x) * kTT;
    const int c0 = blockIdx.y * kTT;
    const int64_t b = blockIdx.z;
    if (q_limit && q0 >= *q_limit) return;
    const int chunk = threadIdx.x & 7, r8 = threadIdx.x >> 3;   // 8 chunks x 32 rows
    const uint16_t *inb = in + b * ibs;
    uint16_t *outb = out + b * obs;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int qq = r8 + 32 * i;
        const int64_t q = q0 + qq;
        int64_t src = -1;
        float sc = 1.0f;
        if (q < Q) {
            src = qsrc ? qsrc[q] : (q < R ? q : -1);
            if (src >= 0 && !idx_ok(src, R)) src = -1;   // debug builds: a row outside the input
            if (qscale && src >= 0) sc = qscale[q];
        }
        const int c = c0 + chunk * 8;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (src >= 0) {
            const uint16_t *p = inb + src * ldi + c;
            if (c + 8 <= C) {
                const uint4 v = *reinterpret_cast<const uint4 *>(p);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
                for (int e = 0; e < 8; ++e)
                    if (c + e < C) w[e >> 1] |= uint32_t(p[e]) << (16 * (e & 1));
            }
            if (qscale) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t lo = f_to_bf16(sc * bf16_to_f(uint16_t(w[e] & 0xffffu)));
                    const uint16_t hi = f_to_bf16(sc * bf16_to_f(uint16_t(w[e] >> 16)));
                    w[e] = uint32_t(lo) | (uint32_t(hi) << 16);
                }
            }
        }
        *reinterpret_cast<uint4 *>(&tile[swz(qq, chunk * 8)]) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int cc = r8 + 32 * i;
        const int c = c0 + cc;
        if (c >= C) continue;
        const int64_t q = q0 + chunk * 8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = uint32_t(tile[swz(chunk * 8 + 2 * e, cc)]) | (uint32_t(tile[swz(chunk * 8 + 2 * e + 1, cc)]) << 16);
        uint16_t *p = packed_rows > 0 ? out + ((q0 >> 6) * packed_rows + c) * kTT + chunk * 8
                                      : outb + int64_t(c) * ldo + q;
        if (q + 8 <= Q) {
            *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            for (int e = 0; e < 8; ++e)
                if (q + e < Q) p[e] = uint16_t(w[e >> 1] >> (16 * (e & 1)));
        }
    }
}

// One block: the per-expert column segments (each expert's assignments padded
// to a multiple of 64 columns), in expert order, and the weight-gradient tile
// lists {expert, first K block, K blocks, first output row} for the experts
// with at least one assignment: m_tiles_a (resp. b) 128-row tiles each.
constexpr int kSegThreads = 1024;
// Each expert's count is offsets[e + 1] - offsets[e] (the forward's scan).
__global__ void __launch_bounds__(kSegThreads) segments_kernel(const int32_t *__restrict__ offsets, int E,
                                                               int32_t *__restrict__ segoff, int4 *__restrict__ tiles_a,
                                                               int m_tiles_a, int4 *__restrict__ tiles_b, int m_tiles_b,
                                                               int32_t *__restrict__ n_tiles2) {
    grid_dependency_wait();
    __shared__ int32_t s_pad[kSegThreads], s_ne[kSegThreads];
    const int e = threadIdx.x;
    const int cnt = (e < E) ? offsets[e + 1] - offsets[e] : 0;
    const int pad = (cnt + 63) / 64 * 64;
    s_pad[e] = pad;
    s_ne[e] = cnt > 0 ? 1 : 0;
    __syncthreads();
    // inclusive scans (Hillis-Steele over the block)
    for (int off = 1; off < kSegThreads; off <<= 1) {
        const int a = (e >= off) ? s_pad[e - off] : 0;
        const int b = (e >= off) ? s_ne[e - off] : 0;
        __syncthreads();
        s_pad[e] += a;
        s_ne[e] += b;
        __syncthreads();
    }
    const int seg0 = s_pad[e] - pad;       // exclusive
    const int ne0 = s_ne[e] - (cnt > 0 ? 1 : 0);
    if (e < E) segoff[e] = seg0;
    if (e == E - 1) {
        segoff[E] = s_pad[e];
        n_tiles2[0] = s_ne[e] * m_tiles_a;
        n_tiles2[1] = s_ne[e] * m_tiles_b;
        n_tiles2[2] = s_pad[e];   // columns in use
    }
    if (e < E && cnt > 0) {
        for (int mt = 0; mt < m_tiles_a; ++mt)
            tiles_a[ne0 * m_tiles_a + mt] = make_int4(e, seg0 / 64, pad / 64, mt * 128);
        for (int mt = 0; mt < m_tiles_b; ++mt)
            tiles_b[ne0 * m_tiles_b + mt] = make_int4(e, seg0 / 64, pad / 64, mt * 128);
    }
}

// Column maps of the segments: for column q = segoff[e] + c (c < padded
// count), qperm = the permuted row offsets[e] + c (or -1 past the count),
// qtok = that row's token, qgate = its gate.  One block per expert.
__global__ void __launch_bounds__(256) segment_maps_kernel(const int32_t *__restrict__ offsets,
                                                           const int32_t *__restrict__ segoff,
                                                           const int32_t *__restrict__ perm,
                                                           const int32_t *__restrict__ tokrow,
                                                           const float *__restrict__ gates, int32_t *__restrict__ qperm,
                                                           int32_t *__restrict__ qtok, float *__restrict__ qgate) {
    grid_dependency_wait();
    const int e = blockIdx.x;
    const int cnt = offsets[e + 1] - offsets[e];
    const int pad = (cnt + 63) / 64 * 64;
    const int64_t s0 = segoff[e];
    for (int c = threadIdx.x; c < pad; c += blockDim.x) {
        int32_t p = -1, t = -1;
        float g = 0.0f;
        if (c < cnt) {
            p = offsets[e] + c;
            t = tokrow[p];
            const int32_t a = perm[p];
            g = idx_ok(a, offsets[gridDim.x]) ? gates[a] : 0.0f;   // offsets[E] = assignments
        }
        qperm[s0 + c] = p;
        qtok[s0 + c] = t;
        qgate[s0 + c] = g;
    }
}

// Zero the routed weight gradients of experts no token chose (the segment
// GEMMs have no tile for them).  grid (E, chunks).
__global__ void __launch_bounds__(256) zero_unused_kernel(const int32_t *__restrict__ offsets, int64_t per_expert,
                                                          float *__restrict__ g1, float *__restrict__ g2,
                                                          float *__restrict__ g3) {
    grid_dependency_wait();
    const int e = blockIdx.x;
    if (offsets[e + 1] != offsets[e]) return;
    const int64_t n4 = per_expert / 4;
    float4 *p1 = reinterpret_cast<float4 *>(g1 + int64_t(e) * per_expert);
    float4 *p2 = reinterpret_cast<float4 *>(g2 + int64_t(e) * per_expert);
    float4 *p3 = reinterpret_cast<float4 *>(g3 + int64_t(e) * per_expert);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = int64_t(blockIdx.y) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.y) * blockDim.x) {
        p1[i] = z;
        p2[i] = z;
        p3[i] = z;
    }
}

// RMSNorm backward, one block per token.  z = sum_j o[t*k + j] (the
// gate-weighted expert rows the forward stored, fp32 sum), ms = mean(z^2),
// r = z / sqrt(ms + eps);
// dz = dr / sqrt(ms + eps) - z (dr . z) / (L (ms + eps)^(3/2)), stored bf16.
constexpr int kRmsThreads = 256;
__global__ void __launch_bounds__(kRmsThreads) rms_bwd_kernel(const uint16_t *__restrict__ o, int k, int L, float eps,
                                                              const uint16_t *__restrict__ dr, int64_t ld_dr,
                                                              uint16_t *__restrict__ dz) {
    grid_dependency_wait();
    extern __shared__ float zs[];   // [L]
    __shared__ float red[2][kRmsThreads / 32];
    const int64_t t = blockIdx.x;
    float ss = 0.0f, drz = 0.0f;
    for (int c = threadIdx.x * 8; c < L; c += kRmsThreads * 8) {
        float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < k; ++j) {
            const uint4 v = *reinterpret_cast<const uint4 *>(o + (t * k + j) * L + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                z[2 * i] += __uint_as_float(w[i] << 16);
                z[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
            }
        }
        const uint4 dv = *reinterpret_cast<const uint4 *>(dr + t * ld_dr + c);
        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ss = fmaf(z[2 * i], z[2 * i], ss);
            ss = fmaf(z[2 * i + 1], z[2 * i + 1], ss);
            drz = fmaf(__uint_as_float(dw[i] << 16), z[2 * i], drz);
            drz = fmaf(__uint_as_float(dw[i] & 0xffff0000u), z[2 * i + 1], drz);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) zs[c + i] = z[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
        drz += __shfl_xor_sync(0xffffffffu, drz, off);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = ss;
        red[1][threadIdx.x >> 5] = drz;
    }
    __syncthreads();
    ss = 0.0f;
    drz = 0.0f;
#pragma unroll
    for (int w = 0; w < kRmsThreads / 32; ++w) {
        ss += red[0][w];
        drz += red[1][w];
    }
    const float den = ss / static_cast<float>(L) + eps;
    const float inv = 1.0f / sqrtf(den);
    const float coef = drz * inv / (static_cast<float>(L) * den);
    for (int c = threadIdx.x * 8; c < L; c += kRmsThreads * 8) {
        const uint4 dv = *reinterpret_cast<const uint4 *>(dr + t * ld_dr + c);
        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = __uint_as_float(dw[i] << 16) * inv - zs[c + 2 * i] * coef;
            const float b = __uint_as_float(dw[i] & 0xffff0000u) * inv - zs[c + 2 * i + 1] * coef;
            w[i] = uint32_t(f_to_bf16(a)) | (uint32_t(f_to_bf16(b)) << 16);
        }
        *reinterpret_cast<uint4 *>(dz + t * L + c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Router backward, one warp per token.  Lane j < k takes the token's j-th
// chosen expert e_j: the gate's gradient dg[p] (p = the assignment's permuted
// row) times sigma'(x) = sigma(x) sigma(-x) at the expert's fp32 logit x as
// the forward's router GEMM computed it (kept in logits [T][E]); this form
// stays accurate where the fp32 gate sigma(x) has rounded to 1 (g (1 - g)
// would give 0 there).  Written into a dense bf16 row dl[t][0..ldl) that is
// zero elsewhere.
__global__ void __launch_bounds__(256) router_bwd_kernel(const float *__restrict__ dg,
                                                         const int32_t *__restrict__ inv,
                                                         const int32_t *__restrict__ idx,
                                                         const float *__restrict__ logits, int E, int64_t T,
                                                         int k, int ldl, uint16_t *__restrict__ dl) {
    grid_dependency_wait();
    const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;   // whole warps
    int e = -1;
    float v = 0.0f;
    if (lane < k) {
        const int64_t a = t * k + lane;
        e = idx[a];
        if (e >= 0 && e < E) {   // else not a routing the forward produced: no gradient
            const float x = logits[t * E + e];
            const float sp = 1.0f / (1.0f + __expf(-x));
            const float sm = 1.0f / (1.0f + __expf(x));
            const int32_t p = inv[a];
            v = idx_ok(p, T * k) ? dg[p] * (sp * sm) : 0.0f;
        } else {
            e = -1;
        }
    }
    for (int c0 = 0; c0 < ldl; c0 += 64) {
        const int c = c0 + 2 * lane;
        float v0 = 0.0f, v1 = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int ej = __shfl_sync(0xffffffffu, e, j);
            const float vj = __shfl_sync(0xffffffffu, v, j);
            if (ej == c) v0 = vj;
            if (ej == c + 1) v1 = vj;
        }
        if (c < ldl)
            *reinterpret_cast<uint32_t *>(dl + t * ldl + c) = uint32_t(f_to_bf16(v0)) | (uint32_t(f_to_bf16(v1)) << 16);
    }
}

// dh[t] = dhr[t] (fp32, the router's share) + sum_j dhp[t*k + j] (bf16 rows
// of the experts' shares, assignment order), stored bf16.  8 columns per thread.
__global__ void __launch_bounds__(256) dh_sum_kernel(const uint16_t *__restrict__ dhp, const float *__restrict__ dhr,
                                                     int64_t T, int k, int L, uint16_t *__restrict__ dh) {
    grid_dependency_wait();
    const int64_t per_row = L / 8;
    const int64_t total = T * per_row;
    for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = v / per_row;
        const int c = static_cast<int>(v % per_row) * 8;
        const float4 r0 = *reinterpret_cast<const float4 *>(dhr + t * L + c);
        const float4 r1 = *reinterpret_cast<const float4 *>(dhr + t * L + c + 4);
        float acc[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        for (int j = 0; j < k; ++j) {
            const uint4 u = *reinterpret_cast<const uint4 *>(dhp + (t * k + j) * L + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += __uint_as_float(w[i] << 16);
                acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = uint32_t(f_to_bf16(acc[2 * i])) | (uint32_t(f_to_bf16(acc[2 * i + 1])) << 16);
        *reinterpret_cast<uint4 *>(dh + t * L + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// tanh(y) and its derivative 1 - tanh(y)^2 from one exponential: with
// u = e^(-2|y|), tanh(y) = sign(y) (1 - u) / (1 + u) and
// 1 - tanh(y)^2 = 4u / (1 + u)^2.  The derivative keeps its relative accuracy
// where tanh saturates (1 - t*t from an approximate t would not).
__device__ __forceinline__ void tanh_and_slope(float y, float &t, float &slope) {
    const float u = __expf(-2.0f * fabsf(y));
    const float inv = __fdividef(1.0f, 1.0f + u);   // 1 + u in [1, 2]
    t = copysignf((1.0f - u) * inv, y);
    slope = 4.0f * u * inv * inv;
}

// Backward of one SiTU-GLU element ("Kimi-K3-Architecture-Deep-Dive" section 1:
// the tanh softcap is differentiable everywhere).  With sigma = sigmoid(p1):
//   SiTU   = b1 tanh(p1/b1) sigma        SiTU'   = (1 - tanh^2) sigma + SiTU (1 - sigma)
//   softcap = b2 tanh(p2/b2)             softcap' = 1 - tanh^2(p2/b2)
// da is the activation's gradient; returns act = SiTU softcap as well.
__device__ __forceinline__ void situ_glu_bwd(float p1, float p2, float da, float b1, float ib1, float b2,
                                             float ib2, float &dp1, float &dp2, float &act) {
    float t2, s2;
    tanh_and_slope(p2 * ib2, t2, s2);
    float situ, dsitu;
    if (b1 == 4.0f) {
        // beta1 = 4 (K3): with u = e^(-x/2) and D = (1 + u)(1 + u^2),
        // tanh(x/4) = (1 - u)/(1 + u) and sigma(x) = 1/(1 + u^2), so
        //   SiTU  = 4 (1 - u) / D
        //   SiTU' = (1 - tanh^2) sigma + SiTU (1 - sigma)
        //         = 4 (u / D) ((1 + u + u^2 - u^3) / D)
        // from one exponential and one reciprocal; the two factors stay in
        // range where 1/D^2 alone would underflow.  x is floored at -50 as
        // in the forward (there |SiTU'| < 1e-21).
        const float u = __expf(-0.5f * fmaxf(p1, -50.0f));
        const float u2 = u * u;
        const float inv_d = __fdividef(1.0f, (1.0f + u) * (1.0f + u2));
        situ = 4.0f * (1.0f - u) * inv_d;
        dsitu = 4.0f * (u * inv_d) * (fmaf(u2, 1.0f - u, 1.0f + u) * inv_d);
    } else {
        float t1, s1;
        tanh_and_slope(p1 * ib1, t1, s1);
        const float sig = __fdividef(1.0f, 1.0f + __expf(-p1));   // 0 once e^(-p1) passes 2^126
        situ = b1 * t1 * sig;
        dsitu = s1 * sig + situ * (1.0f - sig);
    }
    const float cap = b2 * t2;
    dp1 = da * dsitu * cap;
    dp2 = da * situ * s2;
    act = situ * cap;
}

// SiTU-GLU backward of one row per warp, at the saved pre-activations:
//   p1 = P[r][f], p2 = P[r][p_half + f], da = g_r * U[r][u_col0 + f]
//   dP[r][f] = da SiTU'(p1) softcap(p2), dP[r][dp_half + f] = da SiTU(p1) softcap'(p2)
//   dg[r] = sum_f U[r][u_col0 + f] SiTU(p1) softcap(p2)    (when dg is given)
// with g_r = scale[scale_rows[r]] (1 without scale).  C features per row, a
// multiple of 8; each lane takes 8 consecutive features per step (16-byte
// accesses), two steps in flight.  Strides and offsets are multiples of 8
// elements.
constexpr int kGluWarps = 8;
__global__ void __launch_bounds__(kGluWarps * 32) glu_bwd_rows_kernel(
    const uint16_t *__restrict__ P, int64_t p_ld, int p_half, const uint16_t *__restrict__ U, int64_t u_ld,
    int u_col0, const int32_t *__restrict__ scale_rows, const float *__restrict__ scale, int64_t rows, int C,
    float b1, float b2, uint16_t *__restrict__ dP, int64_t dp_ld, int dp_half, float *__restrict__ dg) {
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = int64_t(blockIdx.x) * kGluWarps + (threadIdx.x >> 5);
    const int64_t nwarps = int64_t(gridDim.x) * kGluWarps;
    const float ib1 = 1.0f / b1, ib2 = 1.0f / b2;   // once per thread
    const int chunks = C >> 3;
    for (int64_t r = warp0; r < rows; r += nwarps) {
        const int64_t si = scale_rows ? scale_rows[r] : r;
        const float g = (scale && idx_ok(si, rows)) ? scale[si] : (scale ? 0.0f : 1.0f);
        const uint16_t *p1r = P + r * p_ld, *p2r = p1r + p_half, *ur = U + r * u_ld + u_col0;
        uint16_t *d1r = dP + r * dp_ld, *d2r = d1r + dp_half;
        float acc = 0.0f;
        for (int j0 = lane; j0 < chunks; j0 += 64) {
            uint4 a1[2], a2[2], au[2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int j = j0 + 32 * s;
                if (j < chunks) {
                    a1[s] = *reinterpret_cast<const uint4 *>(p1r + 8 * j);
                    a2[s] = *reinterpret_cast<const uint4 *>(p2r + 8 * j);
                    au[s] = *reinterpret_cast<const uint4 *>(ur + 8 * j);
                }
            }
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int j = j0 + 32 * s;
                if (j >= chunks) continue;
                const uint32_t w1[4] = {a1[s].x, a1[s].y, a1[s].z, a1[s].w};
                const uint32_t w2[4] = {a2[s].x, a2[s].y, a2[s].z, a2[s].w};
                const uint32_t wu[4] = {au[s].x, au[s].y, au[s].z, au[s].w};
                uint32_t o1[4], o2[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float d1[2], d2[2];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float p1 = __uint_as_float(hh ? (w1[b] & 0xffff0000u) : (w1[b] << 16));
                        const float p2 = __uint_as_float(hh ? (w2[b] & 0xffff0000u) : (w2[b] << 16));
                        const float uu = __uint_as_float(hh ? (wu[b] & 0xffff0000u) : (wu[b] << 16));
                        float a;
                        situ_glu_bwd(p1, p2, g * uu, b1, ib1, b2, ib2, d1[hh], d2[hh], a);
                        acc = fmaf(uu, a, acc);
                    }
                    o1[b] = uint32_t(f_to_bf16(d1[0])) | (uint32_t(f_to_bf16(d1[1])) << 16);
                    o2[b] = uint32_t(f_to_bf16(d2[0])) | (uint32_t(f_to_bf16(d2[1])) << 16);
                }
                *reinterpret_cast<uint4 *>(d1r + 8 * j) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                *reinterpret_cast<uint4 *>(d2r + 8 * j) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
            }
        }
        if (dg) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) dg[r] = acc;
        }
    }
}

__global__ void __launch_bounds__(256) fill_kernel(float *__restrict__ p, int64_t n, float v) {
    grid_dependency_wait();
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        p[i] = v;
}

int blocks_for(int64_t work, int per_block, int cap) {
    const int64_t b = (work + per_block - 1) / per_block;
    return static_cast<int>(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_transpose(const uint16_t *in, int64_t ldi, int64_t in_batch_stride, int64_t R, int C,
                             uint16_t *out, int64_t ldo, int64_t out_batch_stride, int64_t Q, int batch,
                             const int32_t *qsrc, const float *qscale, const int32_t *q_limit, cudaStream_t stream,
                             int64_t packed_rows) {
    if (Q <= 0 || C <= 0 || batch <= 0) return cudaSuccess;
    if (packed_rows > 0 && (batch != 1 || packed_rows != C || Q % kTT != 0)) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>((Q + kTT - 1) / kTT), static_cast<unsigned>((C + kTT - 1) / kTT),
                    static_cast<unsigned>(batch));
    return launch_kernel(transpose_kernel, grid, dim3(256), 0, stream, true, in, ldi, in_batch_stride, R, C, out, ldo,
                         out_batch_stride, Q, qsrc, qscale, q_limit, packed_rows);
}

cudaError_t launch_segments(const int32_t *offsets, const int32_t *perm,
                            const int32_t *tokrow, const float *gates, int E, int32_t *segoff, int32_t *qperm,
                            int32_t *qtok, float *qgate, int4 *tiles_a, int m_tiles_a, int4 *tiles_b,
                            int m_tiles_b, int32_t *n_tiles3, cudaStream_t stream) {
    if (E > kSegThreads) return cudaErrorInvalidValue;
    cudaError_t e = launch_kernel(segments_kernel, dim3(1), dim3(kSegThreads), 0, stream, true, offsets, E, segoff,
                                  tiles_a, m_tiles_a, tiles_b, m_tiles_b, n_tiles3);
    if (e != cudaSuccess) return e;
    return launch_kernel(segment_maps_kernel, dim3(E), dim3(256), 0, stream, true, offsets,
                         static_cast<const int32_t *>(segoff), perm, tokrow, gates, qperm, qtok, qgate);
}

cudaError_t launch_zero_unused(const int32_t *offsets, int E, int64_t per_expert, float *g1, float *g2, float *g3,
                               cudaStream_t stream) {
    return launch_kernel(zero_unused_kernel, dim3(E, 64), dim3(256), 0, stream, true, offsets, per_expert, g1, g2, g3);
}

cudaError_t launch_rms_bwd(const uint16_t *o, int64_t T, int k, int L, float eps, const uint16_t *dr, int64_t ld_dr,
                           uint16_t *dz, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const size_t smem = size_t(L) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(rms_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(rms_bwd_kernel, dim3(static_cast<unsigned>(T)), dim3(kRmsThreads), smem, stream, true, o, k,
                         L, eps, dr, ld_dr, dz);
}

cudaError_t launch_router_bwd(const float *dg, const int32_t *inv, const int32_t *idx, const float *logits, int E,
                              int64_t T, int k, int ldl, uint16_t *dl, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    if (k > 32) return cudaErrorInvalidValue;
    const unsigned blocks = static_cast<unsigned>((T * 32 + 255) / 256);
    return launch_kernel(router_bwd_kernel, dim3(blocks), dim3(256), 0, stream, true, dg, inv, idx, logits, E, T, k,
                         ldl, dl);
}

cudaError_t launch_dh_sum(const uint16_t *dhp, const float *dhr, int64_t T, int k, int L, uint16_t *dh,
                          int num_sms, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const int blocks = blocks_for(T * (L / 8), 256, num_sms * 8);
    return launch_kernel(dh_sum_kernel, dim3(blocks), dim3(256), 0, stream, true, dhp, dhr, T, k, L, dh);
}

cudaError_t launch_glu_bwd_rows(const uint16_t *P, int64_t p_ld, int p_half, const uint16_t *U, int64_t u_ld,
                                int u_col0, const int32_t *scale_rows, const float *scale, int64_t rows, int C,
                                float b1, float b2, uint16_t *dP, int64_t dp_ld, int dp_half, float *dg,
                                int num_sms, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    if (C <= 0 || (C & 7) || (p_ld & 7) || (p_half & 7) || (u_ld & 7) || (u_col0 & 7) || (dp_ld & 7) ||
        (dp_half & 7) || p_half < C || dp_half < C || u_col0 + C > u_ld || p_half + C > p_ld ||
        dp_half + C > dp_ld || num_sms <= 0)
        return cudaErrorInvalidValue;
    const int64_t want = (rows + kGluWarps - 1) / kGluWarps;
    const int64_t cap = int64_t(num_sms) * 8;   // 8 blocks of 8 warps per SM, grid-stride beyond
    return launch_kernel(glu_bwd_rows_kernel, dim3(static_cast<unsigned>(want < cap ? want : cap)),
                         dim3(kGluWarps * 32), 0, stream, true, P, p_ld, p_half, U, u_ld, u_col0, scale_rows, scale,
                         rows, C, b1, b2, dP, dp_ld, dp_half, dg);
}

cudaError_t launch_fill(float *p, int64_t n, float v, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int blocks = blocks_for(n, 256, 1024);
    return launch_kernel(fill_kernel, dim3(blocks), dim3(256), 0, stream, true, p, n, v);
}

LMOE_DEBUG_WORD_READER(debug_word_backward)

}  // namespace lmoe
