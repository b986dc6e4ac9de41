// lmoe_api.cu -- host side of the C ABI declared in include/lmoe.h: argument
// validation, workspace layout, TMA descriptors, and the launch sequences of
// one Stable LatentMoE forward pass and of its backward pass.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>

#include "lmoe.h"
#include "kernels.h"

using namespace lmoe;

struct lmoe_handle {
    lmoe_config cfg;
    lmoe_weights w;
    int device;
    int num_sms;
    unsigned *d_status;  // device status word (bounded-wait timeouts)
    // Weight-side TMA descriptors, built once.
    int bn_down, bn_shared, bn_exp1, bn_exp3, bn_up, bn_router;
    // down- / up-projection on CTA pairs (256-row tiles over two SMs; B boxes of bn / 2 rows)
    bool pair_down, pair_up;
    CUtensorMap m_wdown, m_wrouter, m_ws1, m_ws2, m_w1, m_w2, m_w3, m_wup, m_ws3;
    // routed experts' weights repacked tile-contiguously (handle-owned): bf16,
    // or e4m3 codes (expert_fp8) with one int8 scale exponent per weight row
    uint16_t *w1p, *w2p, *w3p;
    int8_t *w1e, *w2e, *w3e;
    cudaEvent_t *stage_events;  // optional timing hook (LMOE_NUM_STAGES + 1 events)
    cudaEvent_t *bwd_events;    // optional timing hook of the backward (LMOE_BWD_NUM_STAGES + 1)
    // lmoe_forward_host: input / output copy streams and, per staging slot, the
    // events "input landed", "forward done" and "output copied".
    cudaStream_t io_in, io_out;
    cudaEvent_t ev_in[2], ev_fwd[2], ev_out[2];
    unsigned io_calls;
    // The shared experts depend only on x: without the timing hook they run on
    // this side stream, concurrently with the routing kernels.
    cudaStream_t side;
    cudaEvent_t ev_fork, ev_join;
    // with_backward: transposed copies of the weights (handle-owned), K-major
    // for the backward's data-gradient GEMMs:
    //   t_ups3 [latent + S][d]        = [W_up^T ; Ws3^T]
    //   t_w3   [E][inter][latent]     = W3[e]^T
    //   t_w12  [E][latent][2 inter]   = [W1[e]^T | W2[e]^T]
    //   t_wr   [latent][E rounded up to 64] = W_router^T (zero columns past E)
    //   t_wd   [d][latent]            = W_down^T
    //   t_ws12 [d][2 S]               = [Ws1^T | Ws2^T]
    uint16_t *t_ups3, *t_w3, *t_w12, *t_wr, *t_wd, *t_ws12;
    CUtensorMap m_t_ups3, m_t_w3, m_t_w12, m_t_wr, m_t_wd, m_t_ws12;
    int bn_drs, bn_u, bn_s;
    bool pair_dr;   // dr on CTA pairs (dx follows pair_up, the dense weight gradients their own width)
    // backward: fork / join events of the side-stream copies
    cudaEvent_t bev[6];
};

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder_ready() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 2-D bf16 row-major [rows][cols] (row stride ld elements), box = 64 columns
// (128 bytes, 128B swizzle) x box_rows rows.
bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t ld,
              uint32_t box_rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D fp32 row-major [rows][cols] (row stride ld elements) as a TMA store
// target: 32 x 32 boxes (128-byte rows, 128B swizzle).
bool make_store_map_f32(CUtensorMap *m, void *ptr, uint64_t rows, uint64_t cols, uint64_t ld) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 4};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t h, scores, idx, gates, counts, offsets, bitmap, wprefix, tiles, tiles2, nmt, perm, inv, tokrow,
        tiles3, act, o, r, sact, hn, h8, h8e, pre, spre, logit, part, total;
};

// Split-K of a dense GEMM for small batches: when its output tiles (256-row
// tiles on CTA pairs, else 128-row) would fill less than half of the GPU,
// K is divided into ks ranges of `per` K blocks (at least 4 each) so that
// tiles x ks CTAs (or pairs) fill it once; ks == 1: no split.
struct DenseSplit {
    int ks, per;
};
DenseSplit plan_split(int num_sms, bool pair, int64_t T, int64_t n_tiles, int k_blocks) {
    DenseSplit sp{1, k_blocks};
    const int64_t base = ceil_div(T, pair ? 2 * kBM : kBM) * n_tiles;
    const int64_t units = pair ? num_sms / 2 : num_sms;
    if (base <= 0 || 2 * base > units) return sp;
    const int64_t ks = std::min<int64_t>(units / base, k_blocks / 4);
    if (ks < 2) return sp;
    const int per = static_cast<int>(ceil_div(k_blocks, ks));
    const int ks2 = static_cast<int>(ceil_div(k_blocks, per));
    if (ks2 >= 2) sp = DenseSplit{ks2, per};
    return sp;
}

// The forward's four dense GEMMs: {split, output columns of the partial sums}.
struct DenseSplits {
    DenseSplit down, router, shared, up;
    int64_t n_down, n_router, n_shared, n_up;
};
DenseSplits plan_dense_splits(const lmoe_handle *h, int64_t T) {
    const lmoe_config &c = h->cfg;
    const int64_t d = c.d, L = c.latent, E = c.n_experts;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    DenseSplits p;
    p.down = plan_split(h->num_sms, h->pair_down, T, ceil_div(L, h->bn_down), static_cast<int>(d / kBK));
    p.router = plan_split(h->num_sms, false, T, ceil_div(E, h->bn_router), static_cast<int>(L / kBK));
    p.shared = plan_split(h->num_sms, false, T, S / (h->bn_shared / 2), static_cast<int>(d / kBK));
    p.up = plan_split(h->num_sms, h->pair_up, T, ceil_div(d, h->bn_up), static_cast<int>((L + S) / kBK));
    p.n_down = L;
    p.n_router = E;
    p.n_shared = 2 * S;
    p.n_up = d;
    return p;
}

// fp32 elements of the split-K slot for a batch of T tokens: the largest
// need of any batch of at most T tokens, so that a workspace sized for T (for
// instance for max_tokens) also serves every smaller batch -- a smaller batch
// can split more ways (fewer tiles) and need more.  For a fixed number of
// row tiles the need grows with the batch, so T and the multiples of 128 below
// it cover every case.  A GEMM splits only while twice its row tiles fit in
// the SMs (pairs: in half of them), i.e. for at most 64 rows per SM.
int64_t split_slot_elems(const lmoe_handle *h, int64_t T) {
    int64_t pe = 0;
    auto at = [&](int64_t t) {
        const DenseSplits p = plan_dense_splits(h, t);
        for (auto [sp, nc] : {std::pair<DenseSplit, int64_t>{p.down, p.n_down}, {p.router, p.n_router},
                              {p.shared, p.n_shared}, {p.up, p.n_up}})
            if (sp.ks > 1) pe = std::max(pe, int64_t(sp.ks) * t * nc);
    };
    if (T > 0) at(T);
    const int64_t t_max = std::min<int64_t>(T - 1, int64_t(h->num_sms) * kBM);
    for (int64_t t = kBM; t <= t_max; t += kBM) at(t);
    return pe;
}

Layout compute_layout(const lmoe_handle *h, int64_t T, bool own_scores, bool own_idx,
                      bool own_gates, bool own_counts) {
    const lmoe_config &c = h->cfg;
    Layout l{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    const int64_t L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    const int64_t words = ceil_div(T, 32);
    const int64_t n = T * K;
    const size_t none = SIZE_MAX;
    l.h = take(size_t(T * L * 2));
    l.scores = own_scores ? take(size_t(T * E * 4)) : none;
    l.idx = own_idx ? take(size_t(n * 4)) : none;
    l.gates = own_gates ? take(size_t(n * 4)) : none;
    l.counts = own_counts ? take(size_t(E * 4)) : none;
    l.offsets = take(size_t((E + 1) * 4));
    l.bitmap = take(size_t(E * words * 4));
    l.wprefix = take(size_t(E * words * 4));
    l.tiles = take(size_t((ceil_div(n, kBM) + E) * 16));
    l.tiles2 = take(size_t((ceil_div(n, 2 * kBM) + E) * 16));
    l.tiles3 = take(size_t(E * 16));
    l.nmt = take(16);
    l.perm = take(size_t(n * 4));
    l.inv = take(size_t(n * 4));
    l.tokrow = take(size_t(n * 4));
    l.act = take(size_t(n * I * 2));
    l.o = take(size_t(n * L * 2));
    l.r = take(size_t(T * L * 2));
    l.sact = take(size_t(T * S * 2));
    l.hn = c.norm_after_down ? take(size_t(T * L * 2)) : none;
    l.h8 = c.expert_fp8 ? take(size_t(T * L)) : none;
    l.h8e = c.expert_fp8 ? take(size_t(T)) : none;
    // with_backward: the SiTU-GLU pre-activations p1 | p2 (bf16), kept for
    // the backward (routed rows in permuted order, shared rows by token)
    l.pre = c.with_backward ? take(size_t(n * 2 * I * 2)) : none;
    l.spre = c.with_backward ? take(size_t(T * 2 * S * 2)) : none;
    l.logit = c.with_backward ? take(size_t(T * E * 4)) : none;   // the router's fp32 logits
    // small batches: the dense GEMMs' split-K partial sums (one slab per K
    // range, fp32; the four GEMMs use the slot one after another)
    {
        const int64_t pe = split_slot_elems(h, T);
        l.part = pe ? take(size_t(pe * 4)) : none;
    }
    l.total = off;
    return l;
}

int validate_config(const lmoe_config *c) {
    if (!c) return LMOE_ERR_INVALID_ARG;
    if (c->d <= 0 || c->latent <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->inter <= 0 ||
        c->n_shared <= 0 || c->shared_inter <= 0 || c->max_tokens < 0)
        return LMOE_ERR_INVALID_ARG;
    if (!(c->beta1 > 0.0f) || !(c->beta2 > 0.0f) || !(c->rms_eps >= 0.0f)) return LMOE_ERR_INVALID_ARG;
    if (c->norm_after_down != 0 && c->norm_after_down != 1) return LMOE_ERR_INVALID_ARG;
    if (c->expert_fp8 != 0 && c->expert_fp8 != 1) return LMOE_ERR_INVALID_ARG;
    if (c->with_backward != 0 && c->with_backward != 1) return LMOE_ERR_INVALID_ARG;
    if (c->with_backward && c->expert_fp8) return LMOE_ERR_UNSUPPORTED_SHAPE;
    if (c->expert_fp8 && c->inter % 128) return LMOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t S = int64_t(c->n_shared) * c->shared_inter;
    if (c->d % 64 || c->latent % 128 || c->inter % 64 || S % 64) return LMOE_ERR_UNSUPPORTED_SHAPE;
    if (c->latent > 8192 || c->top_k > 32 || c->top_k > c->n_experts || c->n_experts > 1024)
        return LMOE_ERR_UNSUPPORTED_SHAPE;
    // 32-bit row coordinates of the TMA descriptors and permuted-row indices
    if (int64_t(c->n_experts) * c->latent * (c->inter / 64) >= (int64_t(1) << 31) ||
        int64_t(c->n_experts) * c->inter * (c->latent / 64) >= (int64_t(1) << 31) ||
        int64_t(c->n_experts) * c->latent >= (int64_t(1) << 31) ||
        int64_t(c->n_experts) * c->inter >= (int64_t(1) << 31) ||
        c->max_tokens * c->top_k >= (int64_t(1) << 31))
        return LMOE_ERR_UNSUPPORTED_SHAPE;
    return LMOE_OK;
}

int check_device(int *dev, int *sms) {
    if (cudaGetDevice(dev) != cudaSuccess) return LMOE_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
        return LMOE_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return LMOE_ERR_NO_DEVICE;
    return LMOE_OK;
}

GemmArgs base_args(const lmoe_handle *h) {
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.beta1 = h->cfg.beta1;
    a.beta2 = h->cfg.beta2;
    a.err = h->d_status;
    a.wait_limit_ns = kWaitLimitNs;
    return a;
}

int gemm_status(cudaError_t e) { return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA; }

// A dense GEMM of a small batch as split-K: the GEMM's fp32 epilogue writes
// each K range's partial sums into its slab of `part`, then the finalize adds
// the slabs in a fixed order and applies the GEMM's own epilogue (`fin`: its
// mode and outputs).  `a` carries the operands and the shape (n_tiles,
// k_blocks, k_split); `n_cols` is the partial sums' row length.
int run_split(const lmoe_handle *h, const GemmMaps &m, GemmArgs a, int bn, AMode am, BMode bm, bool pair,
              const DenseSplit &sp, int64_t T, int64_t n_cols, float *part, SplitFinArgs fin, cudaStream_t s,
              bool dependent) {
    a.m_rows = static_cast<int32_t>(T);
    a.m_tiles = static_cast<int32_t>(ceil_div(T, pair ? 2 * kBM : kBM));
    a.k_splits = sp.ks;
    a.k_per_split = sp.per;
    a.split_stride = T * n_cols;
    a.out = part;
    a.ld_out = n_cols;
    a.out_cols = static_cast<int32_t>(n_cols);
    a.lout = nullptr;
    a.pout = nullptr;
    a.accumulate = 0;
    const int64_t tiles = int64_t(a.m_tiles) * a.n_tiles * sp.ks;
    const cudaError_t e =
        pair ? launch_gemm_pair(bn, am, bm, EPI_F32, m, a, tiles, s, dependent)
             : launch_gemm_split(bn, am, bm, m, a, static_cast<int>(std::min<int64_t>(tiles, h->num_sms)), s, dependent);
    if (e != cudaSuccess) return LMOE_ERR_CUDA;
    fin.part = part;
    fin.stride = T * n_cols;
    fin.ks = sp.ks;
    fin.rows = T;
    fin.ld_part = n_cols;
    return gemm_status(launch_split_finalize(fin, h->num_sms, s));
}

// Staging slot of lmoe_forward_host: x [max_tokens][d] bf16, bias [E] fp32,
// y [max_tokens][d] bf16.
struct IoSlot {
    size_t x, bias, y, bytes;
};

IoSlot io_slot(const lmoe_config &c) {
    IoSlot s;
    const size_t xb = align256(size_t(c.max_tokens) * c.d * 2);
    s.x = 0;
    s.bias = xb;
    s.y = xb + align256(size_t(c.n_experts) * 4);
    s.bytes = s.y + xb;
    return s;
}

void release_streams(lmoe_handle *h);

// Free whatever a (possibly half-built) handle holds, then the handle.
void free_handle(lmoe_handle *h) {
    cudaFree(h->d_status);
    cudaFree(h->w1p);
    cudaFree(h->w2p);
    cudaFree(h->w3p);
    cudaFree(h->w1e);
    cudaFree(h->w2e);
    cudaFree(h->w3e);
    cudaFree(h->t_ups3);
    cudaFree(h->t_w3);
    cudaFree(h->t_w12);
    cudaFree(h->t_wr);
    cudaFree(h->t_wd);
    cudaFree(h->t_ws12);
    release_streams(h);
    delete h;
}

// e4m3 expert weights: quantise [E][R][K] bf16 rows (one scale exponent per
// row) through a temporary code buffer, then pack the codes tile-contiguously
// like the bf16 weights (a 128-byte box row holds 128 codes).
bool quantize_pack(const uint16_t *src, uint64_t E, uint64_t R, uint64_t K, int TR, uint16_t **packed,
                   int8_t **exps) {
    uint8_t *codes = nullptr;
    const size_t n = size_t(E) * R * K;
    if (cudaMalloc(packed, n) != cudaSuccess || cudaMalloc(exps, size_t(E) * R) != cudaSuccess ||
        cudaMalloc(&codes, n) != cudaSuccess)
        return false;
    const bool ok = launch_fp8_quantize_rows(src, int64_t(E * R), static_cast<int>(K), codes, *exps, 0) ==
                        cudaSuccess &&
                    launch_pack_tiles(reinterpret_cast<const uint16_t *>(codes), E, static_cast<int>(R),
                                      static_cast<int>(K / 2), TR, *packed, 0) == cudaSuccess &&
                    cudaDeviceSynchronize() == cudaSuccess;
    cudaFree(codes);
    return ok;
}

void release_streams(lmoe_handle *h) {
    for (int i = 0; i < 6; ++i)
        if (h->bev[i]) cudaEventDestroy(h->bev[i]);
    if (h->side) cudaStreamDestroy(h->side);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->io_in) cudaStreamDestroy(h->io_in);
    if (h->io_out) cudaStreamDestroy(h->io_out);
    for (int s = 0; s < 2; ++s) {
        if (h->ev_in[s]) cudaEventDestroy(h->ev_in[s]);
        if (h->ev_fwd[s]) cudaEventDestroy(h->ev_fwd[s]);
        if (h->ev_out[s]) cudaEventDestroy(h->ev_out[s]);
    }
}

int64_t round64(int64_t v) { return (v + 63) / 64 * 64; }

// Transposed weight copies for the backward pass (see lmoe_handle).
bool build_transposed(lmoe_handle *h) {
    const lmoe_config &c = h->cfg;
    const lmoe_weights &w = h->w;
    const int64_t d = c.d, L = c.latent, E = c.n_experts, I = c.inter;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    const int64_t Ep = round64(E);
    h->bn_drs = ((L + S) % 256 == 0) ? 256 : 128;
    h->bn_u = (I % 256 == 0) ? 256 : 128;
    h->bn_s = (S % 256 == 0) ? 256 : 128;
    if (cudaMalloc(&h->t_ups3, size_t((L + S) * d) * 2) != cudaSuccess ||
        cudaMalloc(&h->t_w3, size_t(E * I * L) * 2) != cudaSuccess ||
        cudaMalloc(&h->t_w12, size_t(E * L * 2 * I) * 2) != cudaSuccess ||
        cudaMalloc(&h->t_wr, size_t(L * Ep) * 2) != cudaSuccess ||
        cudaMalloc(&h->t_wd, size_t(d * L) * 2) != cudaSuccess ||
        cudaMalloc(&h->t_ws12, size_t(d * 2 * S) * 2) != cudaSuccess)
        return false;
    const int Li = static_cast<int>(L), Ii = static_cast<int>(I), di = static_cast<int>(d);
    const int Si = static_cast<int>(S), Ei = static_cast<int>(E);
    // launch_transpose(in, ldi, in_batch, R, C, out, ldo, out_batch, Q, batch, ...):
    // out[b][c][q] = in[b][q][c]
    bool ok = launch_transpose(w.w_up, L, 0, d, Li, h->t_ups3, d, 0, d, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.ws3, S, 0, d, Si, h->t_ups3 + L * d, d, 0, d, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.w3, I, L * I, L, Ii, h->t_w3, L, I * L, L, Ei, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.w1, L, I * L, I, Li, h->t_w12, 2 * I, L * 2 * I, I, Ei, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.w2, L, I * L, I, Li, h->t_w12 + I, 2 * I, L * 2 * I, I, Ei, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.w_router, L, 0, E, Li, h->t_wr, Ep, 0, Ep, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.w_down, d, 0, L, di, h->t_wd, L, 0, L, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.ws1, d, 0, S, di, h->t_ws12, 2 * S, 0, S, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              launch_transpose(w.ws2, d, 0, S, di, h->t_ws12 + S, 2 * S, 0, S, 1, nullptr, nullptr, nullptr, 0) == cudaSuccess &&
              cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) return false;
    h->pair_dr = h->bn_drs == 256;
    return make_map(&h->m_t_ups3, h->t_ups3, L + S, d, d, h->pair_dr ? h->bn_drs / 2 : h->bn_drs) &&
           make_map(&h->m_t_w3, h->t_w3, E * I, L, L, h->bn_u) &&
           make_map(&h->m_t_w12, h->t_w12, E * L, 2 * I, 2 * I, h->bn_exp3) &&
           make_map(&h->m_t_wr, h->t_wr, L, Ep, Ep, h->bn_down) &&
           make_map(&h->m_t_wd, h->t_wd, d, L, L, h->pair_up ? h->bn_up / 2 : h->bn_up) &&
           make_map(&h->m_t_ws12, h->t_ws12, d, 2 * S, 2 * S, h->pair_up ? h->bn_up / 2 : h->bn_up);
}

// Backward workspace: gradients of the intermediates, their K-major
// (transposed) copies for the weight-gradient GEMMs, and the per-expert
// column segments.  Tp = T and Qmax = T*top_k + 64 E rounded up to 64;
// Ep = E rounded up to 64.
struct BwdLayout {
    size_t ones, drs, dps, dz, u, dp, dgate, dl, dhp, dhr, dh, dhraw, dyT, xT, rT, sT, dpsT, dhT, hT, dlT, segoff, qperm,
        qtok, qgate, kt_a, kt_b, nkt, doT, aT, hgT, dpT, total;
    int64_t Tp, Ep, Qmax;
};

BwdLayout bwd_layout(const lmoe_handle *h, int64_t T) {
    const lmoe_config &c = h->cfg;
    BwdLayout l{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    const int64_t d = c.d, L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    const int64_t n = T * K;
    l.Tp = round64(T);
    l.Ep = round64(E);
    l.Qmax = round64(n) + 64 * E;
    l.ones = take(size_t(n) * 4);
    l.drs = take(size_t(T * (L + S)) * 2);
    l.dps = take(size_t(T * 2 * S) * 2);
    l.dz = take(size_t(T * L) * 2);
    l.u = take(size_t(n * I) * 2);
    l.dp = take(size_t(n * 2 * I) * 2);
    l.dgate = take(size_t(n) * 4);   // the gates' gradients, per permuted row
    l.dl = take(size_t(T * l.Ep) * 2);
    l.dhp = take(size_t(n * L) * 2);
    l.dhr = take(size_t(T * L) * 4);
    l.dh = take(size_t(T * L) * 2);
    l.dhraw = take(size_t(T * L) * 2);   // norm-after-down variant: gradient at the down-projection's output
    l.dyT = take(size_t(d * l.Tp) * 2);
    l.xT = take(size_t(d * l.Tp) * 2);
    l.rT = take(size_t(L * l.Tp) * 2);
    l.sT = take(size_t(S * l.Tp) * 2);
    l.dpsT = take(size_t(2 * S * l.Tp) * 2);
    l.dhT = take(size_t(L * l.Tp) * 2);
    l.hT = take(size_t(L * l.Tp) * 2);
    l.dlT = take(size_t(E * l.Tp) * 2);
    l.segoff = take(size_t(E + 1) * 4);
    l.qperm = take(size_t(l.Qmax) * 4);
    l.qtok = take(size_t(l.Qmax) * 4);
    l.qgate = take(size_t(l.Qmax) * 4);
    l.kt_a = take(size_t(E * (L / kBM)) * 16);
    l.kt_b = take(size_t(E * ceil_div(2 * I, kBM)) * 16);
    l.nkt = take(16);
    l.doT = take(size_t(L * l.Qmax) * 2);
    l.aT = take(size_t(I * l.Qmax) * 2);
    l.hgT = take(size_t(L * l.Qmax) * 2);
    l.dpT = take(size_t(2 * I * l.Qmax) * 2);
    l.total = off;
    return l;
}

}  // namespace

extern "C" {

const char *lmoe_status_string(int s) {
    switch (s) {
        case LMOE_OK: return "LMOE_OK";
        case LMOE_ERR_INVALID_ARG: return "LMOE_ERR_INVALID_ARG";
        case LMOE_ERR_UNSUPPORTED_SHAPE: return "LMOE_ERR_UNSUPPORTED_SHAPE";
        case LMOE_ERR_ALIGNMENT: return "LMOE_ERR_ALIGNMENT";
        case LMOE_ERR_WORKSPACE: return "LMOE_ERR_WORKSPACE";
        case LMOE_ERR_CUDA: return "LMOE_ERR_CUDA";
        case LMOE_ERR_TIMEOUT: return "LMOE_ERR_TIMEOUT";
        case LMOE_ERR_NO_DEVICE: return "LMOE_ERR_NO_DEVICE";
        case LMOE_ERR_INDEX: return "LMOE_ERR_INDEX";
        default: return "LMOE_ERR_UNKNOWN";
    }
}

int lmoe_create(const lmoe_config *cfg, const lmoe_weights *w, lmoe_handle **out) {
    if (!out) return LMOE_ERR_INVALID_ARG;
    *out = nullptr;
    int st = validate_config(cfg);
    if (st) return st;
    if (!w || !w->w_down || !w->w_router || !w->w1 || !w->w2 || !w->w3 || !w->ws1 || !w->ws2 ||
        !w->ws3 || !w->w_up)
        return LMOE_ERR_INVALID_ARG;
    const void *ptrs[] = {w->w_down, w->w_router, w->w1, w->w2, w->w3, w->ws1, w->ws2, w->ws3, w->w_up};
    for (const void *p : ptrs)
        if (!aligned16(p)) return LMOE_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    st = check_device(&dev, &sms);
    if (st) return st;
    if (!encoder_ready()) return LMOE_ERR_CUDA;

    lmoe_handle *h = new (std::nothrow) lmoe_handle;
    if (!h) return LMOE_ERR_CUDA;
    std::memset(h, 0, sizeof *h);
    h->cfg = *cfg;
    h->w = *w;
    h->device = dev;
    h->num_sms = sms;
    const lmoe_config &c = h->cfg;
    const uint64_t d = c.d, L = c.latent, E = c.n_experts, I = c.inter;
    const uint64_t S = uint64_t(c.n_shared) * c.shared_inter;
    h->bn_down = (L % 256 == 0) ? 256 : 128;
    h->bn_shared = (S % 128 == 0) ? 256 : 128;
    h->bn_exp1 = (I % 128 == 0) ? 256 : 128;
    h->bn_exp3 = (L % 256 == 0) ? 256 : 128;   // latent % 128 == 0: the boxes tile each expert's W3
    h->bn_up = (d % 256 == 0) ? 256 : 128;
    // router: 224-wide N tiles when they cover E exactly (K3: 896 = 4 x 224),
    // else 256-wide unless E fits one 128-wide tile
    h->bn_router = (E % 224 == 0) ? 224 : (E > 128) ? 256 : 128;
    // the 256-wide down- and up-projections run on CTA pairs: per SM, half the
    // B tile per stage, six stages instead of four.  The router (one and a half
    // waves of tiles) and the shared experts' W1|W2 measured slower on pairs
    // and stay on single CTAs.
    h->pair_down = h->bn_down == 256;
    h->pair_up = h->bn_up == 256;
    // Repack W1, W2 (boxes of bn_exp1/2 rows) and W3 (boxes of bn_exp3 rows)
    // so each box is one contiguous block of HBM; in the FP8 variant the
    // boxes hold e4m3 codes (128 per 128-byte row) instead of bf16.
    const int tr12 = h->bn_exp1 / 2, tr3 = h->bn_exp3;
    bool ok = true;
    uint64_t kb12 = L / 64, kb3 = I / 64;   // 128-byte K blocks per weight row
    if (c.expert_fp8) {
        kb12 = L / 128;
        kb3 = I / 128;
        ok = quantize_pack(w->w1, E, I, L, tr12, &h->w1p, &h->w1e) &&
             quantize_pack(w->w2, E, I, L, tr12, &h->w2p, &h->w2e) &&
             quantize_pack(w->w3, E, L, I, tr3, &h->w3p, &h->w3e);
    } else {
        const size_t bytes12 = size_t(E) * I * L * 2, bytes3 = size_t(E) * L * I * 2;
        ok = cudaMalloc(&h->w1p, bytes12) == cudaSuccess && cudaMalloc(&h->w2p, bytes12) == cudaSuccess &&
             cudaMalloc(&h->w3p, bytes3) == cudaSuccess &&
             launch_pack_tiles(w->w1, E, static_cast<int>(I), static_cast<int>(L), tr12, h->w1p, 0) == cudaSuccess &&
             launch_pack_tiles(w->w2, E, static_cast<int>(I), static_cast<int>(L), tr12, h->w2p, 0) == cudaSuccess &&
             launch_pack_tiles(w->w3, E, static_cast<int>(L), static_cast<int>(I), tr3, h->w3p, 0) == cudaSuccess &&
             cudaDeviceSynchronize() == cudaSuccess;
    }
    if (!ok) {
        free_handle(h);
        return LMOE_ERR_CUDA;
    }
    ok = make_map(&h->m_wdown, w->w_down, L, d, d, h->pair_down ? h->bn_down / 2 : h->bn_down) &&
         make_map(&h->m_wrouter, w->w_router, E, L, L, h->bn_router) &&
         make_map(&h->m_ws1, w->ws1, S, d, d, h->bn_shared / 2) &&
         make_map(&h->m_ws2, w->ws2, S, d, d, h->bn_shared / 2) &&
         make_map(&h->m_w1, h->w1p, E * I * kb12, 64, 64, tr12) &&
         make_map(&h->m_w2, h->w2p, E * I * kb12, 64, 64, tr12) &&
         make_map(&h->m_w3, h->w3p, E * L * kb3, 64, 64, tr3) &&
         make_map(&h->m_wup, w->w_up, d, L, L, h->pair_up ? h->bn_up / 2 : h->bn_up) &&
         make_map(&h->m_ws3, w->ws3, d, S, S, h->pair_up ? h->bn_up / 2 : h->bn_up);
    if (!ok) {
        free_handle(h);
        return LMOE_ERR_CUDA;
    }
    if (c.with_backward && !build_transposed(h)) {
        free_handle(h);
        return LMOE_ERR_CUDA;
    }
    bool io_ok = cudaStreamCreateWithFlags(&h->io_in, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&h->io_out, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 6 && io_ok && c.with_backward; ++i)
        io_ok = cudaEventCreateWithFlags(&h->bev[i], cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < 2 && io_ok; ++s)
        io_ok = cudaEventCreateWithFlags(&h->ev_in[s], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&h->ev_fwd[s], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&h->ev_out[s], cudaEventDisableTiming) == cudaSuccess;
    if (!io_ok || cudaMalloc(&h->d_status, 256) != cudaSuccess || cudaMemset(h->d_status, 0, 256) != cudaSuccess) {
        free_handle(h);
        return LMOE_ERR_CUDA;
    }
    *out = h;
    return LMOE_OK;
}

int lmoe_destroy(lmoe_handle *h) {
    if (!h) return LMOE_ERR_INVALID_ARG;
    const cudaError_t e = cudaDeviceSynchronize();
    free_handle(h);
    return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

int lmoe_workspace_size(const lmoe_handle *h, int64_t T, size_t *bytes) {
    if (!h || !bytes || T < 0) return LMOE_ERR_INVALID_ARG;
    if (T > h->cfg.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    *bytes = compute_layout(h, T, true, true, true, true).total;
    return LMOE_OK;
}

int lmoe_workspace_layout(const lmoe_handle *h, int64_t T, lmoe_ws_layout *out) {
    if (!h || !out || T < 0) return LMOE_ERR_INVALID_ARG;
    if (T > h->cfg.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    const Layout l = compute_layout(h, T, true, true, true, true);
    out->h = int64_t(l.h);
    out->scores = int64_t(l.scores);
    out->topk_idx = int64_t(l.idx);
    out->gates = int64_t(l.gates);
    out->counts = int64_t(l.counts);
    out->offsets = int64_t(l.offsets);
    out->perm = int64_t(l.perm);
    out->inv = int64_t(l.inv);
    out->act = int64_t(l.act);
    out->o = int64_t(l.o);
    out->r = int64_t(l.r);
    out->shared_act = int64_t(l.sact);
    out->h_norm = (l.hn == SIZE_MAX) ? -1 : int64_t(l.hn);
    out->h_fp8 = (l.h8 == SIZE_MAX) ? -1 : int64_t(l.h8);
    out->h_fp8_exp = (l.h8e == SIZE_MAX) ? -1 : int64_t(l.h8e);
    out->pre_act = (l.pre == SIZE_MAX) ? -1 : int64_t(l.pre);
    out->shared_pre_act = (l.spre == SIZE_MAX) ? -1 : int64_t(l.spre);
    out->logits = (l.logit == SIZE_MAX) ? -1 : int64_t(l.logit);
    return LMOE_OK;
}

int lmoe_forward(lmoe_handle *h, const uint16_t *x, int64_t T, const float *bias, uint16_t *y,
                 float *scores_out, int32_t *topk_idx_out, float *gates_out,
                 int32_t *expert_counts_out, void *workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
    if (!h || T < 0) return LMOE_ERR_INVALID_ARG;
    const lmoe_config &c = h->cfg;
    if (T > c.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return LMOE_OK;
    if (!x || !bias || !y || !workspace) return LMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(bias) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) || (scores_out && !aligned16(scores_out)) ||
        (topk_idx_out && !aligned16(topk_idx_out)) || (gates_out && !aligned16(gates_out)) ||
        (expert_counts_out && !aligned16(expert_counts_out)))
        return LMOE_ERR_ALIGNMENT;
    // The workspace is sized for every intermediate; caller-provided outputs
    // simply leave their slot unused, so the documented offsets never move.
    const Layout l = compute_layout(h, T, true, true, true, true);
    if (workspace_bytes < l.total) return LMOE_ERR_WORKSPACE;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t d = c.d, L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    const int64_t n = T * K;
    const int words = static_cast<int>(ceil_div(T, 32));
    uint16_t *hbuf = reinterpret_cast<uint16_t *>(ws + l.h);
    float *scores = scores_out ? scores_out : reinterpret_cast<float *>(ws + l.scores);
    int32_t *idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t *>(ws + l.idx);
    float *gates = gates_out ? gates_out : reinterpret_cast<float *>(ws + l.gates);
    int32_t *counts = expert_counts_out ? expert_counts_out : reinterpret_cast<int32_t *>(ws + l.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + l.offsets);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(ws + l.bitmap);
    uint32_t *wprefix = reinterpret_cast<uint32_t *>(ws + l.wprefix);
    int4 *tiles = reinterpret_cast<int4 *>(ws + l.tiles);
    int4 *tiles2 = reinterpret_cast<int4 *>(ws + l.tiles2);
    int4 *tiles3 = reinterpret_cast<int4 *>(ws + l.tiles3);
    // [0]: 128-row tiles, [1]: pair tiles (heavy experts), [2]: light-expert tiles
    int32_t *nmt = reinterpret_cast<int32_t *>(ws + l.nmt);
    int32_t *perm = reinterpret_cast<int32_t *>(ws + l.perm);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + l.inv);
    int32_t *tokrow = reinterpret_cast<int32_t *>(ws + l.tokrow);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + l.act);
    uint16_t *obuf = reinterpret_cast<uint16_t *>(ws + l.o);
    uint16_t *rbuf = reinterpret_cast<uint16_t *>(ws + l.r);
    uint16_t *sact = reinterpret_cast<uint16_t *>(ws + l.sact);
    // the latent the router and the experts read: h, or RMSNorm(h) in the
    // norm-after-down variant
    uint16_t *hlat = c.norm_after_down ? reinterpret_cast<uint16_t *>(ws + l.hn) : hbuf;
    uint8_t *h8 = c.expert_fp8 ? ws + l.h8 : nullptr;              // e4m3 codes of hlat
    int8_t *h8e = c.expert_fp8 ? reinterpret_cast<int8_t *>(ws + l.h8e) : nullptr;
    // with_backward: the SiTU-GLU GEMMs also keep their pre-activations
    const bool save = c.with_backward != 0;
    uint16_t *pre = save ? reinterpret_cast<uint16_t *>(ws + l.pre) : nullptr;
    uint16_t *spre = save ? reinterpret_cast<uint16_t *>(ws + l.spre) : nullptr;
    float *logit = save ? reinterpret_cast<float *>(ws + l.logit) : nullptr;
    // small batches: the dense GEMMs split over K (partial sums in the workspace)
    const DenseSplits dsp = plan_dense_splits(h, T);
    float *part = l.part != SIZE_MAX ? reinterpret_cast<float *>(ws + l.part) : nullptr;

    // Activation-side TMA descriptors for this T and workspace.
    CUtensorMap m_x, m_h, m_act, m_r, m_sact;
    if (!make_map(&m_x, x, T, d, d, kBM) || !make_map(&m_h, hlat, T, L, L, kBM) ||
        !(c.expert_fp8 ? make_map(&m_act, act, n, I / 2, I / 2, kBM)   // e4m3 codes as 2-byte pairs
                       : make_map(&m_act, act, n, I, I, kBM)) ||
        !make_map(&m_r, rbuf, T, L, L, kBM) || !make_map(&m_sact, sact, T, S, S, kBM))
        return LMOE_ERR_CUDA;

    const int m_tiles = static_cast<int>(ceil_div(T, kBM));
    const int m_tiles2 = static_cast<int>(ceil_div(T, 2 * kBM));   // CTA pairs: 256-row tiles
    auto mark = [&](int stage) {
        if (h->stage_events) cudaEventRecord(h->stage_events[stage], stream);
    };
    auto grid_for = [&](int64_t tiles_) {
        return static_cast<int>(tiles_ < h->num_sms ? tiles_ : h->num_sms);
    };
    int st;

    if (cudaMemsetAsync(bitmap, 0, size_t(E) * words * 4, stream) != cudaSuccess) return LMOE_ERR_CUDA;

    mark(LMOE_STAGE_DOWN);
    {   // a1: h = x W_down^T
        GemmMaps m{m_x, m_x, h->m_wdown, h->m_wdown};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = h->pair_down ? m_tiles2 : m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(L, h->bn_down));
        a.k_blocks = static_cast<int32_t>(d / kBK);
        a.out = hbuf;
        a.ld_out = L;
        a.out_cols = static_cast<int32_t>(L);
        // the first kernel of the forward follows a memset: ordinary stream order
        if (dsp.down.ks > 1) {
            SplitFinArgs f{};
            f.mode = FIN_BF16;
            f.cols = L;
            f.out = hbuf;
            f.ld_out = L;
            st = run_split(h, m, a, h->bn_down, A_DENSE, B_PLAIN, h->pair_down, dsp.down, T, dsp.n_down, part, f,
                           stream, /*dependent=*/false);
        } else {
            st = gemm_status(h->pair_down
                                 ? launch_gemm_pair(h->bn_down, A_DENSE, B_PLAIN, EPI_BF16, m, a,
                                                    a.m_tiles * a.n_tiles, stream, /*dependent=*/false)
                                 : launch_gemm(h->bn_down, A_DENSE, B_PLAIN, EPI_BF16, false, m, a,
                                               grid_for(int64_t(m_tiles) * a.n_tiles), stream, /*pair=*/false,
                                               /*dependent=*/false));
        }
        if (st) return st;
    }
    if (c.norm_after_down &&   // ablation variant: hn = h / sqrt(mean(h^2) + eps), per token
        launch_rms_rows(hbuf, T, static_cast<int>(L), static_cast<double>(c.rms_eps), hlat, stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    // a8': shared experts, act_s = SiTU(x Ws1^T) * softcap(x Ws2^T)
    auto run_shared = [&](cudaStream_t s_) {
        GemmMaps m{m_x, m_x, h->m_ws1, h->m_ws2};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = m_tiles;
        a.n_tiles = static_cast<int32_t>(S / (h->bn_shared / 2));
        a.k_blocks = static_cast<int32_t>(d / kBK);
        a.out = sact;
        a.ld_out = S;
        a.out_cols = static_cast<int32_t>(S);
        if (dsp.shared.ks > 1) {
            SplitFinArgs f{};
            f.mode = FIN_GLU;
            f.cols = S;
            f.H = h->bn_shared / 2;
            f.beta1 = c.beta1;
            f.beta2 = c.beta2;
            f.out = sact;
            f.ld_out = S;
            f.pout = save ? spre : nullptr;
            f.pout_ld = 2 * S;
            f.pout_half = S;
            return run_split(h, m, a, h->bn_shared, A_DENSE, B_GLU, false, dsp.shared, T, dsp.n_shared, part, f, s_,
                             true);
        }
        if (save) {
            a.pout = spre;
            a.pout_ld = 2 * S;
            a.pout_half = static_cast<int32_t>(S);
            return gemm_status(launch_gemm_save(h->bn_shared, A_DENSE, false, false, m, a,
                                                grid_for(int64_t(m_tiles) * a.n_tiles), s_));
        }
        return gemm_status(launch_gemm(h->bn_shared, A_DENSE, B_GLU, EPI_SITU_GLU, false, m, a,
                                       grid_for(int64_t(m_tiles) * a.n_tiles), s_));
    };
    // a2: s = sigmoid(h W_router^T), fp32
    auto run_router = [&]() {
        GemmMaps m{m_h, m_h, h->m_wrouter, h->m_wrouter};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(E, h->bn_router));
        a.k_blocks = static_cast<int32_t>(L / kBK);
        a.out = scores;
        a.lout = logit;                  // with_backward: the logits as well
        a.ld_out = E;
        a.out_cols = static_cast<int32_t>(E);
        if (dsp.router.ks > 1) {
            SplitFinArgs f{};
            f.mode = FIN_SIGMOID;
            f.cols = E;
            f.outf = scores;
            f.lout = logit;
            f.ld_out = E;
            return run_split(h, m, a, h->bn_router, A_DENSE, B_PLAIN, false, dsp.router, T, dsp.n_router, part, f,
                             stream, true);
        }
        return gemm_status(launch_gemm(h->bn_router, A_DENSE, B_PLAIN, EPI_SIGMOID_F32, false, m, a,
                                       grid_for(int64_t(m_tiles) * a.n_tiles), stream));
    };
    // Without the timing hook the shared experts run on the side stream once
    // the router is done, while the routing kernels (small and latency-bound)
    // run here on the same SMs; the join comes before the routed experts'
    // GEMMs, which need every SM: the HBM-bound expert launches reach the
    // memory roofline only with every SM's loads in flight, so giving some
    // SMs to the shared experts beside them measured slower (design notes).
    // With the hook, the stages run in stream order so that each stage's
    // events bracket it alone.
    const bool overlap = (h->stage_events == nullptr);
    if (overlap) {
        st = run_router();
        if (st) return st;
        if (cudaEventRecord(h->ev_fork, stream) != cudaSuccess ||
            cudaStreamWaitEvent(h->side, h->ev_fork, 0) != cudaSuccess)
            return LMOE_ERR_CUDA;
        st = run_shared(h->side);
        if (st) return st;
        if (cudaEventRecord(h->ev_join, h->side) != cudaSuccess) return LMOE_ERR_CUDA;
    } else {
        mark(LMOE_STAGE_SHARED);
        st = run_shared(stream);
        if (st) return st;
        mark(LMOE_STAGE_ROUTER);
        st = run_router();
        if (st) return st;
    }
    // a3 + a4: biased top-k, then the stable grouping of assignments by expert
    mark(LMOE_STAGE_TOPK);
    if (launch_topk(scores, bias, T, static_cast<int>(E), static_cast<int>(K), idx, gates, bitmap,
                    words, stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    mark(LMOE_STAGE_SCAN);
    if (launch_expert_scan(bitmap, static_cast<int>(E), words, wprefix, counts, stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    mark(LMOE_STAGE_OFFSETS);
    if (launch_offsets_tiles(counts, static_cast<int>(E), offsets, tiles, nmt, tiles2, nmt + 1, tiles3, nmt + 2,
                             stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    mark(LMOE_STAGE_SCATTER);
    if (launch_scatter(idx, T, static_cast<int>(K), static_cast<int>(E), bitmap, wprefix, words, offsets, perm, inv, tokrow,
                       stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    if (overlap && cudaStreamWaitEvent(stream, h->ev_join, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    mark(LMOE_STAGE_EXPERT_W12_LIGHT);
    {   // a5: act = SiTU(W1[e] h) * softcap(W2[e] h) over the rows of each expert's tokens.
        // Experts with more than 128 rows run pair tiles (two 128-row sub-tiles
        // share each weight stage); the others run 128-row tiles whose smaller
        // stages leave room for more weight stages in flight.
        // FP8 variant: the latent rows are quantised to e4m3 first (one
        // power-of-two scale per token) and the GEMM multiplies e4m3 codes;
        // its epilogue writes the activation as e4m3(4 * act).
        const bool f8 = c.expert_fp8 != 0;
        if (f8 && launch_fp8_quantize_rows(hlat, T, static_cast<int>(L), h8, h8e, stream) != cudaSuccess)
            return LMOE_ERR_CUDA;
        GemmMaps m{m_h, m_h, h->m_w1, h->m_w2};
        GemmArgs a = base_args(h);
        a.n_tiles = static_cast<int32_t>(I / (h->bn_exp1 / 2));
        a.k_blocks = static_cast<int32_t>(f8 ? L / 128 : L / kBK);   // 128-byte K blocks
        a.b_expert_rows = static_cast<int32_t>(I);
        a.b_packed = 1;
        a.b_row_tiles = static_cast<int32_t>(I / (h->bn_exp1 / 2));
        a.gather_src = f8 ? reinterpret_cast<const uint16_t *>(h8) : hlat;
        a.gather_rows = tokrow;
        a.gather_ld = f8 ? L / 2 : L;    // in 2-byte units
        a.out = act;
        a.ld_out = I;                    // elements: bf16, or bytes of e4m3 codes
        a.out_cols = static_cast<int32_t>(I);
        a.row_exp = h8e;
        a.col_exp0 = h->w1e;
        a.col_exp1 = h->w2e;
        a.col_exp_rows = static_cast<int32_t>(I);
        const Epi epi = f8 ? EPI_SITU_GLU_F8 : EPI_SITU_GLU;
        a.pout = pre;                    // with_backward: p1 | p2 per permuted row
        a.pout_ld = 2 * I;
        a.pout_half = static_cast<int32_t>(I);
        auto w12 = [&](bool pair, int grid) {
            return save ? launch_gemm_save(h->bn_exp1, A_GATHER, true, pair, m, a, grid, stream)
                        : launch_gemm(h->bn_exp1, A_GATHER, B_GLU, epi, true, m, a, grid, stream, pair);
        };
        a.lim_experts = E;               // limits of the debug build's index checks
        a.lim_rows = n;
        a.lim_src_rows = T;
        a.tiles = tiles3;
        a.n_mtiles = nmt + 2;
        a.lim_tiles = E;
        st = gemm_status(w12(/*pair=*/false, grid_for(E * a.n_tiles)));
        if (st) return st;
        mark(LMOE_STAGE_EXPERT_W12_HEAVY);
        // an expert holds at most one row per token, so with T <= 128 no
        // expert is heavy and the pair-tile list is empty: no launch
        if (T > kBM) {
            a.tiles = tiles2;
            a.n_mtiles = nmt + 1;
            a.lim_tiles = ceil_div(n, 2 * kBM) + E;
            const int64_t max_pairs = (ceil_div(n, 2 * kBM) + E) * a.n_tiles;
            st = gemm_status(w12(/*pair=*/true, grid_for(max_pairs)));
            if (st) return st;
        }
    }
    mark(LMOE_STAGE_EXPERT_W3);
    {   // a6: o[a] = gate[a] * W3[e] act, written back in assignment order
        const bool f8 = c.expert_fp8 != 0;
        GemmMaps m{m_act, m_act, h->m_w3, h->m_w3};
        GemmArgs a = base_args(h);
        a.n_tiles = static_cast<int32_t>(ceil_div(L, h->bn_exp3));
        a.k_blocks = static_cast<int32_t>(f8 ? I / 128 : I / kBK);
        a.col_exp0 = h->w3e;
        a.col_exp_rows = static_cast<int32_t>(L);
        a.b_expert_rows = static_cast<int32_t>(L);
        a.b_packed = 1;
        a.b_row_tiles = static_cast<int32_t>(L / h->bn_exp3);
        a.tiles = tiles;
        a.n_mtiles = nmt;
        a.lim_tiles = ceil_div(n, kBM) + E;
        a.lim_experts = E;
        a.lim_rows = n;
        a.lim_out_rows = n;
        a.lim_scale = n;
        a.out = obuf;
        a.ld_out = L;
        a.out_cols = static_cast<int32_t>(L);
        a.scatter_rows = perm;
        a.row_scale = gates;
        const int64_t max_tiles = (ceil_div(n, kBM) + E) * a.n_tiles;
        st = gemm_status(launch_gemm(h->bn_exp3, A_DENSE, B_PLAIN, f8 ? EPI_SCATTER_F8 : EPI_SCATTER_BF16, true,
                                     m, a, grid_for(max_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_STAGE_COMBINE);
    // a7: z = sum of the token's gate-weighted expert rows; r = RMSNorm(z)
    if (launch_combine_rmsnorm(obuf, T, static_cast<int>(K), static_cast<int>(L), c.rms_eps, rbuf, h->d_status,
                               kWaitLimitNs, stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    mark(LMOE_STAGE_UP);
    {   // a8: y = r W_up^T + act_s Ws3^T  (one GEMM, K split over the two sources)
        GemmMaps m{m_r, m_sact, h->m_wup, h->m_ws3};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = h->pair_up ? m_tiles2 : m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(d, h->bn_up));
        a.k_split = static_cast<int32_t>(L / kBK);
        a.k_blocks = static_cast<int32_t>((L + S) / kBK);
        a.out = y;
        a.ld_out = d;
        a.out_cols = static_cast<int32_t>(d);
        if (dsp.up.ks > 1) {
            SplitFinArgs f{};
            f.mode = FIN_BF16;
            f.cols = d;
            f.out = y;
            f.ld_out = d;
            st = run_split(h, m, a, h->bn_up, A_SPLIT, B_SPLIT, h->pair_up, dsp.up, T, dsp.n_up, part, f, stream, true);
        } else {
            st = gemm_status(h->pair_up ? launch_gemm_pair(h->bn_up, A_SPLIT, B_SPLIT, EPI_BF16, m, a,
                                                           a.m_tiles * a.n_tiles, stream)
                                        : launch_gemm(h->bn_up, A_SPLIT, B_SPLIT, EPI_BF16, false, m, a,
                                                      grid_for(int64_t(m_tiles) * a.n_tiles), stream));
        }
        if (st) return st;
    }
    mark(LMOE_NUM_STAGES);
    return LMOE_OK;
}

int lmoe_backward_workspace_size(const lmoe_handle *h, int64_t T, size_t *bytes) {
    if (!h || !bytes || T < 0) return LMOE_ERR_INVALID_ARG;
    if (!h->cfg.with_backward) return LMOE_ERR_INVALID_ARG;
    if (T > h->cfg.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    *bytes = bwd_layout(h, T).total;
    return LMOE_OK;
}

int lmoe_backward(lmoe_handle *h, const uint16_t *x, int64_t T, const uint16_t *dy, const int32_t *idx_in,
                  const float *gates_in, const void *fwd_workspace,
                  size_t fwd_workspace_bytes, uint16_t *dx, const lmoe_grads *g, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    if (!h || T < 0) return LMOE_ERR_INVALID_ARG;
    const lmoe_config &c = h->cfg;
    if (!c.with_backward) return LMOE_ERR_INVALID_ARG;
    if (T > c.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return LMOE_OK;
    if (!x || !dy || !fwd_workspace || !dx || !g || !workspace || !g->w_down || !g->w_router || !g->w1 ||
        !g->w2 || !g->w3 || !g->ws1 || !g->ws2 || !g->ws3 || !g->w_up || (g->accumulate != 0 && g->accumulate != 1))
        return LMOE_ERR_INVALID_ARG;
    const void *al[] = {x, dy, dx, g->w_down, g->w_router, g->w1, g->w2, g->w3, g->ws1, g->ws2, g->ws3, g->w_up};
    for (const void *p : al)
        if (!aligned16(p)) return LMOE_ERR_ALIGNMENT;
    if ((idx_in && !aligned16(idx_in)) || (gates_in && !aligned16(gates_in)) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        (reinterpret_cast<uintptr_t>(fwd_workspace) & 255u))
        return LMOE_ERR_ALIGNMENT;
    const Layout fl = compute_layout(h, T, true, true, true, true);
    const BwdLayout bl = bwd_layout(h, T);
    if (fwd_workspace_bytes < fl.total || workspace_bytes < bl.total) return LMOE_ERR_WORKSPACE;

    const int64_t d = c.d, L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int64_t S = int64_t(c.n_shared) * c.shared_inter;
    const int64_t n = T * K;
    const int64_t Tp = bl.Tp, Ep = bl.Ep, Qmax = bl.Qmax;
    const int Li = static_cast<int>(L), Ii = static_cast<int>(I), di = static_cast<int>(d);
    const int Si = static_cast<int>(S), Ei = static_cast<int>(E), Ki = static_cast<int>(K);
    // the forward's intermediates
    const uint8_t *fw = static_cast<const uint8_t *>(fwd_workspace);
    const uint16_t *hbuf = reinterpret_cast<const uint16_t *>(fw + fl.h);
    // the latent the router and the experts read: h, or RMSNorm(h) in the
    // norm-after-down variant (whose backward ends in that norm's backward)
    const uint16_t *hlat = c.norm_after_down ? reinterpret_cast<const uint16_t *>(fw + fl.hn) : hbuf;
    const int32_t *idx = idx_in ? idx_in : reinterpret_cast<const int32_t *>(fw + fl.idx);
    const float *gates = gates_in ? gates_in : reinterpret_cast<const float *>(fw + fl.gates);
    const int32_t *offsets = reinterpret_cast<const int32_t *>(fw + fl.offsets);
    const int4 *tiles = reinterpret_cast<const int4 *>(fw + fl.tiles);     // 128-row tiles, every expert
    const int32_t *nmt = reinterpret_cast<const int32_t *>(fw + fl.nmt);
    const int32_t *perm = reinterpret_cast<const int32_t *>(fw + fl.perm);
    const int32_t *inv = reinterpret_cast<const int32_t *>(fw + fl.inv);
    const int32_t *tokrow = reinterpret_cast<const int32_t *>(fw + fl.tokrow);
    const uint16_t *act = reinterpret_cast<const uint16_t *>(fw + fl.act);
    const uint16_t *obuf = reinterpret_cast<const uint16_t *>(fw + fl.o);
    const uint16_t *rbuf = reinterpret_cast<const uint16_t *>(fw + fl.r);
    const uint16_t *sact = reinterpret_cast<const uint16_t *>(fw + fl.sact);
    // the SiTU-GLU pre-activations the forward kept: p1 | p2 per row
    const uint16_t *pre = reinterpret_cast<const uint16_t *>(fw + fl.pre);
    const uint16_t *spre = reinterpret_cast<const uint16_t *>(fw + fl.spre);
    const float *logit = reinterpret_cast<const float *>(fw + fl.logit);   // the router's, [T][E]
    // the backward's own buffers
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto bf = [&](size_t off) { return reinterpret_cast<uint16_t *>(ws + off); };
    float *ones = reinterpret_cast<float *>(ws + bl.ones);
    uint16_t *drs = bf(bl.drs), *dps = bf(bl.dps), *dz = bf(bl.dz), *u = bf(bl.u), *dp = bf(bl.dp);
    float *dgate = reinterpret_cast<float *>(ws + bl.dgate);
    uint16_t *dl = bf(bl.dl), *dhp = bf(bl.dhp), *dh = bf(bl.dh), *dhraw = bf(bl.dhraw);
    // the gradient at the down-projection's output: dh, or in the variant dh
    // taken back through the norm after the down-projection
    uint16_t *dhx = c.norm_after_down ? dhraw : dh;
    float *dhr = reinterpret_cast<float *>(ws + bl.dhr);
    uint16_t *dyT = bf(bl.dyT), *xT = bf(bl.xT), *rT = bf(bl.rT), *sT = bf(bl.sT), *dpsT = bf(bl.dpsT);
    uint16_t *dhT = bf(bl.dhT), *hT = bf(bl.hT), *dlT = bf(bl.dlT);
    int32_t *segoff = reinterpret_cast<int32_t *>(ws + bl.segoff);
    int32_t *qperm = reinterpret_cast<int32_t *>(ws + bl.qperm);
    int32_t *qtok = reinterpret_cast<int32_t *>(ws + bl.qtok);
    float *qgate = reinterpret_cast<float *>(ws + bl.qgate);
    int4 *kt_a = reinterpret_cast<int4 *>(ws + bl.kt_a);
    int4 *kt_b = reinterpret_cast<int4 *>(ws + bl.kt_b);
    int32_t *nkt = reinterpret_cast<int32_t *>(ws + bl.nkt);
    uint16_t *doT = bf(bl.doT), *aT = bf(bl.aT), *hgT = bf(bl.hgT), *dpT = bf(bl.dpT);

    auto wbox = [](int bn) { return bn == 256 ? bn / 2 : bn; };
    CUtensorMap m_dy, m_x, m_dp, m_dl, m_dh, m_dps, m_dyT, m_xT, m_rT, m_sT, m_dpsT, m_dhT, m_hT, m_dlT,
        m_doT, m_aT, m_hgT, m_dpT;
    if (!make_map(&m_dy, dy, T, d, d, kBM) || !make_map(&m_x, x, T, d, d, kBM) ||
        !make_map(&m_dp, dp, n, 2 * I, 2 * I, kBM) || !make_map(&m_dl, dl, T, Ep, Ep, kBM) ||
        !make_map(&m_dh, dhx, T, L, L, kBM) || !make_map(&m_dps, dps, T, 2 * S, 2 * S, kBM) ||
        // (B of the dense weight-gradient GEMMs: 256-wide ones run on CTA pairs,
        // each CTA loading half of the tile's rows)
        !make_map(&m_dyT, dyT, d, Tp, Tp, kBM) || !make_map(&m_xT, xT, d, Tp, Tp, wbox(h->bn_up)) ||
        !make_map(&m_rT, rT, L, Tp, Tp, wbox(h->bn_down)) || !make_map(&m_sT, sT, S, Tp, Tp, wbox(h->bn_s)) ||
        !make_map(&m_dpsT, dpsT, 2 * S, Tp, Tp, kBM) ||
        !make_map(&m_dhT, dhT, L, Tp, Tp, kBM) || !make_map(&m_hT, hT, L, Tp, Tp, wbox(h->bn_down)) ||
        !make_map(&m_dlT, dlT, E, Tp, Tp, kBM) ||
        // K-block packed segment copies: [Qmax / 64 * rows][64]
        !make_map(&m_doT, doT, Qmax / 64 * L, 64, 64, kBM) || !make_map(&m_aT, aT, Qmax / 64 * I, 64, 64, h->bn_u) ||
        !make_map(&m_hgT, hgT, Qmax / 64 * L, 64, 64, h->bn_down) ||
        !make_map(&m_dpT, dpT, Qmax / 64 * 2 * I, 64, 64, kBM))
        return LMOE_ERR_CUDA;

    const int m_tiles = static_cast<int>(ceil_div(T, kBM));
    auto grid_for = [&](int64_t tiles_) { return static_cast<int>(tiles_ < h->num_sms ? tiles_ : h->num_sms); };
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    int st;
    const int64_t grouped_tiles = ceil_div(n, kBM) + E;   // bound on the forward's 128-row tile list

    auto mark = [&](int stage) {
        if (h->bwd_events) cudaEventRecord(h->bwd_events[stage], stream);
    };
    // The copies the weight-gradient GEMMs read (token-major transposes and the
    // per-expert segments) are memory-bound and only read earlier results.
    // Without the timing hook they run on the handle's side stream next to
    // the tensor-core GEMMs of the main chain (whose one CTA per SM leaves
    // shared memory and threads for the copies' blocks): the input copies
    // beside dr and the shared experts, the segments beside dx and the dense
    // weight gradients; each group is joined before the GEMMs that read it.
    // With the hook, everything runs in stream order so each stage's events
    // bracket it alone.
    const bool overlap = (h->bwd_events == nullptr);
    cudaStream_t s2 = overlap ? h->side : stream;
    auto fork = [&](int i) {
        return !overlap ||
               (cudaEventRecord(h->bev[i], stream) == cudaSuccess && cudaStreamWaitEvent(s2, h->bev[i], 0) == cudaSuccess);
    };
    const int64_t Tl = T;
    auto tr = [&](const uint16_t *in, int64_t ldi, int64_t R, int C, uint16_t *out, int64_t Q, const int32_t *qsrc,
                  const float *qscale, const int32_t *qlim, bool packed = false) {
        return ok(launch_transpose(in, ldi, 0, R, C, out, Q, 0, Q, 1, qsrc, qscale, qlim, s2, packed ? C : 0));
    };
    auto copies_inputs = [&]() {   // inputs of the backward: dy, x and the forward's r, act_s, h
        return tr(dy, d, Tl, di, dyT, Tp, nullptr, nullptr, nullptr) && tr(x, d, Tl, di, xT, Tp, nullptr, nullptr, nullptr) &&
               tr(rbuf, L, Tl, Li, rT, Tp, nullptr, nullptr, nullptr) &&
               tr(sact, S, Tl, Si, sT, Tp, nullptr, nullptr, nullptr) && tr(hlat, L, Tl, Li, hT, Tp, nullptr, nullptr, nullptr);
    };
    auto copies_dps = [&]() { return tr(dps, 2 * S, Tl, 2 * Si, dpsT, Tp, nullptr, nullptr, nullptr); };
    auto copies_dl = [&]() { return tr(dl, Ep, Tl, Ei, dlT, Tp, nullptr, nullptr, nullptr); };
    auto copies_dh = [&]() { return tr(dhx, L, Tl, Li, dhT, Tp, nullptr, nullptr, nullptr); };
    const int mt_a = static_cast<int>(L / kBM), mt_b = static_cast<int>(ceil_div(2 * I, kBM));
    auto copies_segments = [&]() {   // after dz and dp exist
        return ok(launch_segments(offsets, perm, tokrow, gates, Ei, segoff, qperm, qtok, qgate, kt_a, mt_a, kt_b,
                                  mt_b, nkt, s2)) &&
               (g->accumulate || ok(launch_zero_unused(offsets, Ei, I * L, g->w1, g->w2, g->w3, s2))) &&
               // do = gate * dz rows, act rows, h rows, dp rows, each in its expert's
               // column segment, K-block packed ([Qmax / 64][rows][64])
               tr(dz, L, Tl, Li, doT, Qmax, qtok, qgate, nkt + 2, true) &&
               tr(act, I, n, Ii, aT, Qmax, qperm, nullptr, nkt + 2, true) &&
               tr(hlat, L, Tl, Li, hgT, Qmax, qtok, nullptr, nkt + 2, true) &&
               tr(dp, 2 * I, n, 2 * Ii, dpT, Qmax, qperm, nullptr, nkt + 2, true);
    };
    if (overlap && !(fork(0) && copies_inputs())) return LMOE_ERR_CUDA;

    mark(LMOE_BWD_STAGE_DR);
    if (!ok(launch_fill(ones, n, 1.0f, stream))) return LMOE_ERR_CUDA;
    {   // dr | da_s = dy [W_up | Ws3]
        GemmMaps m{m_dy, m_dy, h->m_t_ups3, h->m_t_ups3};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = h->pair_dr ? static_cast<int32_t>(ceil_div(T, 2 * kBM)) : m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(L + S, h->bn_drs));
        a.k_blocks = static_cast<int32_t>(d / kBK);
        a.out = drs;
        a.ld_out = L + S;
        a.out_cols = static_cast<int32_t>(L + S);
        st = gemm_status(h->pair_dr ? launch_gemm_pair(h->bn_drs, A_DENSE, B_PLAIN, EPI_BF16, m, a,
                                                       int64_t(a.m_tiles) * a.n_tiles, stream)
                                    : launch_gemm(h->bn_drs, A_DENSE, B_PLAIN, EPI_BF16, false, m, a,
                                                  grid_for(int64_t(m_tiles) * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_STAGE_SHARED);
    // shared experts: dp_s = SiTU-GLU backward at the kept x Ws1^T | x Ws2^T with
    // da_s from dr | da_s
    if (!ok(launch_glu_bwd_rows(spre, 2 * S, Si, drs, L + S, Li, nullptr, nullptr, T, Si, c.beta1, c.beta2, dps,
                                2 * S, Si, nullptr, h->num_sms, stream)))
        return LMOE_ERR_CUDA;
    if (overlap && !(fork(1) && copies_dps())) return LMOE_ERR_CUDA;
    mark(LMOE_BWD_STAGE_RMSNORM);
    // RMSNorm backward: dz
    if (!ok(launch_rms_bwd(obuf, T, Ki, Li, c.rms_eps, drs, L + S, dz, stream))) return LMOE_ERR_CUDA;
    mark(LMOE_BWD_STAGE_EXPERT_U);
    {   // u = W3[e]^T dz for every assignment (dz rows gathered by token), permuted order
        GemmMaps m{h->m_t_w3, h->m_t_w3, h->m_t_w3, h->m_t_w3};
        GemmArgs a = base_args(h);
        a.n_tiles = static_cast<int32_t>(ceil_div(I, h->bn_u));
        a.k_blocks = static_cast<int32_t>(L / kBK);
        a.b_expert_rows = static_cast<int32_t>(I);
        a.gather_src = dz;
        a.gather_rows = tokrow;
        a.gather_ld = L;
        a.out = u;
        a.ld_out = I;
        a.out_cols = static_cast<int32_t>(I);
        // 128-row tiles for every expert (pair tiles, which hold the whole
        // TMEM, measured slower here, for every expert and for those with
        // more than 128 rows alike: their epilogue cannot overlap the MMAs)
        a.tiles = tiles;
        a.n_mtiles = nmt;
        a.lim_tiles = ceil_div(n, kBM) + E;
        a.lim_experts = E;
        a.lim_rows = n;
        a.lim_src_rows = T;
        st = gemm_status(launch_gemm_bwd(h->bn_u, A_GATHER, B_PLAIN, EPI_BF16, true, false, m, a,
                                         grid_for(grouped_tiles * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_STAGE_EXPERT_GLU);
    // routed experts: dp = SiTU-GLU backward at the kept W1[e] h | W2[e] h with
    // da = gate * u (permuted rows; the gate of the row's assignment), and
    // dgate = u . act per row
    if (!ok(launch_glu_bwd_rows(pre, 2 * I, Ii, u, I, 0, perm, gates, n, Ii, c.beta1, c.beta2, dp, 2 * I, Ii, dgate,
                                h->num_sms, stream)))
        return LMOE_ERR_CUDA;

    mark(LMOE_BWD_STAGE_ROUTER);
    // router: dl = dgate * sigma'(logit) at the chosen experts (the forward's
    // logits), dense [T][Ep]
    if (!ok(launch_router_bwd(dgate, inv, idx, logit, Ei, T, Ki, static_cast<int>(Ep), dl, stream)))
        return LMOE_ERR_CUDA;
    if (overlap && !(fork(2) && copies_dl())) return LMOE_ERR_CUDA;
    mark(LMOE_BWD_STAGE_DH_EXPERTS);
    {   // experts' share of dh: W1[e]^T dp1 + W2[e]^T dp2, rows back in assignment order
        GemmMaps m{m_dp, m_dp, h->m_t_w12, h->m_t_w12};
        GemmArgs a = base_args(h);
        a.n_tiles = static_cast<int32_t>(ceil_div(L, h->bn_exp3));
        a.k_blocks = static_cast<int32_t>(2 * I / kBK);
        a.b_expert_rows = static_cast<int32_t>(L);
        a.tiles = tiles;
        a.n_mtiles = nmt;
        a.out = dhp;
        a.ld_out = L;
        a.out_cols = static_cast<int32_t>(L);
        a.scatter_rows = perm;
        a.row_scale = ones;
        a.lim_tiles = ceil_div(n, kBM) + E;
        a.lim_experts = E;
        a.lim_rows = n;
        a.lim_out_rows = n;
        a.lim_scale = n;
        st = gemm_status(launch_gemm(h->bn_exp3, A_DENSE, B_PLAIN, EPI_SCATTER_BF16, true, m, a,
                                     grid_for(grouped_tiles * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_STAGE_DH_ROUTER);
    {   // router's share of dh: dl W_router (fp32)
        GemmMaps m{m_dl, m_dl, h->m_t_wr, h->m_t_wr};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(L, h->bn_down));
        a.k_blocks = static_cast<int32_t>(Ep / kBK);
        a.out = dhr;
        a.ld_out = L;
        a.out_cols = static_cast<int32_t>(L);
        st = gemm_status(launch_gemm_bwd(h->bn_down, A_DENSE, B_PLAIN, EPI_F32, false, false, m, a,
                                         grid_for(int64_t(m_tiles) * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_STAGE_DH_SUM);
    if (!ok(launch_dh_sum(dhp, dhr, T, Ki, Li, dh, h->num_sms, stream))) return LMOE_ERR_CUDA;
    // norm-after-down variant: dh is the gradient at RMSNorm(h); take it back
    // through that norm (the same kernel as the aggregate's norm, one row per
    // token: z = h) to the down-projection's output
    if (c.norm_after_down &&
        !ok(launch_rms_bwd(hbuf, T, 1, Li, c.rms_eps, dh, L, dhraw, stream)))
        return LMOE_ERR_CUDA;
    // side stream: the last token-major copy, then (join point 4 for the dense
    // weight gradients) the per-expert segments, which so run next to dx and
    // the dense weight-gradient GEMMs (join point 5 for the experts')
    if (overlap && !(fork(3) && copies_dh() && cudaEventRecord(h->bev[4], s2) == cudaSuccess && copies_segments() &&
                     cudaEventRecord(h->bev[5], s2) == cudaSuccess))
        return LMOE_ERR_CUDA;
    mark(LMOE_BWD_STAGE_DX);
    {   // dx = dh W_down + dp_s [Ws1 ; Ws2]  (K split over the two sources)
        GemmMaps m{m_dh, m_dps, h->m_t_wd, h->m_t_ws12};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(T);
        a.m_tiles = h->pair_up ? static_cast<int32_t>(ceil_div(T, 2 * kBM)) : m_tiles;
        a.n_tiles = static_cast<int32_t>(ceil_div(d, h->bn_up));
        a.k_split = static_cast<int32_t>(L / kBK);
        a.k_blocks = static_cast<int32_t>((L + 2 * S) / kBK);
        a.out = dx;
        a.ld_out = d;
        a.out_cols = static_cast<int32_t>(d);
        st = gemm_status(h->pair_up ? launch_gemm_pair(h->bn_up, A_SPLIT, B_SPLIT, EPI_BF16, m, a,
                                                       int64_t(a.m_tiles) * a.n_tiles, stream)
                                    : launch_gemm(h->bn_up, A_SPLIT, B_SPLIT, EPI_BF16, false, m, a,
                                                  grid_for(int64_t(m_tiles) * a.n_tiles), stream));
        if (st) return st;
    }
    // ---- weight gradients of the dense weights: K = tokens (transposed operands, zero past T)
    mark(LMOE_BWD_STAGE_TRANSPOSE);
    if (overlap) {   // the token-major copies are done
        if (cudaStreamWaitEvent(stream, h->bev[4], 0) != cudaSuccess) return LMOE_ERR_CUDA;
    } else if (!(copies_inputs() && copies_dps() && copies_dh() && copies_dl())) {
        return LMOE_ERR_CUDA;
    }
    auto wgrad = [&](const CUtensorMap &ma, const CUtensorMap &mb, int64_t M, int64_t N, int bn, float *out,
                     float *out2 = nullptr, int64_t m_split = 0) {
        GemmMaps m{ma, ma, mb, mb};
        GemmArgs a = base_args(h);
        const bool pair = bn == 256;   // (B maps made with wbox)
        a.m_rows = static_cast<int32_t>(M);
        a.m_tiles = static_cast<int32_t>(ceil_div(M, pair ? 2 * kBM : kBM));
        a.n_tiles = static_cast<int32_t>(ceil_div(N, bn));
        a.k_blocks = static_cast<int32_t>(Tp / kBK);
        a.out = out;
        a.out2 = out2;
        a.m_split = static_cast<int32_t>(m_split);
        a.ld_out = N;
        a.out_cols = static_cast<int32_t>(N);
        a.accumulate = g->accumulate;
        if (pair)
            return gemm_status(launch_gemm_pair(bn, A_DENSE, B_PLAIN, EPI_F32, m, a, int64_t(a.m_tiles) * a.n_tiles,
                                                stream));
        return gemm_status(launch_gemm_bwd(bn, A_DENSE, B_PLAIN, EPI_F32, false, false, m, a,
                                           grid_for(int64_t(a.m_tiles) * a.n_tiles), stream));
    };
    mark(LMOE_BWD_STAGE_WGRAD_DENSE);
    if ((st = wgrad(m_dyT, m_rT, d, L, h->bn_down, g->w_up)) || (st = wgrad(m_dyT, m_sT, d, S, h->bn_s, g->ws3)) ||
        // dWs1 | dWs2 in one GEMM over the 2S rows of dp_s^T (rows from S on go to dWs2)
        (st = wgrad(m_dpsT, m_xT, 2 * S, d, h->bn_up, g->ws1, g->ws2, S)) ||
        (st = wgrad(m_dhT, m_xT, L, d, h->bn_up, g->w_down)) || (st = wgrad(m_dlT, m_hT, E, L, h->bn_down, g->w_router)))
        return st;
    // ---- weight gradients of the routed experts: K = each expert's own assignments
    mark(LMOE_BWD_STAGE_SEGMENTS);
    if (overlap) {   // the segments are done: every side-stream copy has finished
        if (cudaStreamWaitEvent(stream, h->bev[5], 0) != cudaSuccess) return LMOE_ERR_CUDA;
    } else if (!copies_segments()) {
        return LMOE_ERR_CUDA;
    }
    mark(LMOE_BWD_STAGE_WGRAD_W3);
    CUtensorMap m_g3, m_g1, m_g2;
    if (!make_store_map_f32(&m_g3, g->w3, E * L, I, I) || !make_store_map_f32(&m_g1, g->w1, E * I, L, L) ||
        !make_store_map_f32(&m_g2, g->w2, E * I, L, L))
        return LMOE_ERR_CUDA;
    {   // dW3[e] = sum over e's assignments of (gate dz) act^T
        GemmMaps m{m_doT, m_g3, m_aT, m_g3};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(L);
        a.m_split = static_cast<int32_t>(L);
        a.kseg_a_rows = static_cast<int32_t>(L);
        a.kseg_b_rows = static_cast<int32_t>(I);
        a.accumulate = g->accumulate;
        a.n_tiles = static_cast<int32_t>(ceil_div(I, h->bn_u));
        a.tiles = kt_a;
        a.n_mtiles = nkt;
        a.lim_tiles = E * mt_a;
        a.lim_experts = E;
        a.out = g->w3;
        a.out2 = g->w3;
        a.ld_out = I;
        a.out_cols = static_cast<int32_t>(I);
        st = gemm_status(launch_gemm_bwd(h->bn_u, A_DENSE, B_PLAIN, EPI_F32, true, true, m, a,
                                         grid_for(E * mt_a * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_STAGE_WGRAD_W12);
    {   // dW1[e] | dW2[e] = sum over e's assignments of (dp1 | dp2) h^T
        GemmMaps m{m_dpT, m_g1, m_hgT, m_g2};
        GemmArgs a = base_args(h);
        a.m_rows = static_cast<int32_t>(2 * I);
        a.m_split = static_cast<int32_t>(I);
        a.kseg_a_rows = static_cast<int32_t>(2 * I);
        a.kseg_b_rows = static_cast<int32_t>(L);
        a.accumulate = g->accumulate;
        a.n_tiles = static_cast<int32_t>(ceil_div(L, h->bn_down));
        a.tiles = kt_b;
        a.n_mtiles = nkt + 1;
        a.lim_tiles = E * mt_b;
        a.lim_experts = E;
        a.out = g->w1;
        a.out2 = g->w2;
        // dW1 | dW2 tiles hold few K blocks and are nearly all output: both
        // store paths (measured faster; dW3 measured the same either way and
        // keeps TMA stores alone)
        a.split_stores = 1;
        a.ld_out = L;
        a.out_cols = static_cast<int32_t>(L);
        st = gemm_status(launch_gemm_bwd(h->bn_down, A_DENSE, B_PLAIN, EPI_F32, true, true, m, a,
                                         grid_for(E * mt_b * a.n_tiles), stream));
        if (st) return st;
    }
    mark(LMOE_BWD_NUM_STAGES);
    return LMOE_OK;
}

int lmoe_host_io_size(const lmoe_handle *h, size_t *bytes) {
    if (!h || !bytes) return LMOE_ERR_INVALID_ARG;
    *bytes = 2 * io_slot(h->cfg).bytes;
    return LMOE_OK;
}

int lmoe_forward_host(lmoe_handle *h, const uint16_t *x_host, int64_t T, const float *bias_host,
                      uint16_t *y_host, float *scores_out, int32_t *topk_idx_out, float *gates_out,
                      int32_t *expert_counts_out, void *io_dev, size_t io_bytes, void *workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
    if (!h || T < 0) return LMOE_ERR_INVALID_ARG;
    const lmoe_config &c = h->cfg;
    if (T > c.max_tokens) return LMOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return LMOE_OK;
    if (!x_host || !bias_host || !y_host || !io_dev || !workspace) return LMOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(io_dev) & 255u) return LMOE_ERR_ALIGNMENT;
    const IoSlot sl = io_slot(c);
    if (io_bytes < 2 * sl.bytes) return LMOE_ERR_WORKSPACE;
    if (workspace_bytes < compute_layout(h, T, true, true, true, true).total) return LMOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || (scores_out && !aligned16(scores_out)) ||
        (topk_idx_out && !aligned16(topk_idx_out)) || (gates_out && !aligned16(gates_out)) ||
        (expert_counts_out && !aligned16(expert_counts_out)))
        return LMOE_ERR_ALIGNMENT;

    const int s = static_cast<int>(h->io_calls & 1u);
    uint8_t *base = static_cast<uint8_t *>(io_dev) + s * sl.bytes;
    uint16_t *xs = reinterpret_cast<uint16_t *>(base + sl.x);
    float *bs = reinterpret_cast<float *>(base + sl.bias);
    uint16_t *ys = reinterpret_cast<uint16_t *>(base + sl.y);
    const size_t xbytes = size_t(T) * c.d * 2;
    // 1. input copy, after the forward that last read this slot
    if (cudaStreamWaitEvent(h->io_in, h->ev_fwd[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(xs, x_host, xbytes, cudaMemcpyHostToDevice, h->io_in) != cudaSuccess ||
        cudaMemcpyAsync(bs, bias_host, size_t(c.n_experts) * 4, cudaMemcpyHostToDevice, h->io_in) !=
            cudaSuccess ||
        cudaEventRecord(h->ev_in[s], h->io_in) != cudaSuccess)
        return LMOE_ERR_CUDA;
    // From here on the slot's input copy is queued.  If anything below fails,
    // the slot's "forward done" event is still recorded after whatever this
    // call queued on `stream`, and the call counter moves on, so that the
    // next call that copies into this slot waits for that work first.
    auto fail = [&](int status) {
        cudaEventRecord(h->ev_fwd[s], stream);
        ++h->io_calls;
        return status;
    };
    // 2. the forward, after its input landed and the slot's last output copy
    if (cudaStreamWaitEvent(stream, h->ev_in[s], 0) != cudaSuccess ||
        cudaStreamWaitEvent(stream, h->ev_out[s], 0) != cudaSuccess)
        return fail(LMOE_ERR_CUDA);
    const int st = lmoe_forward(h, xs, T, bs, ys, scores_out, topk_idx_out, gates_out, expert_counts_out,
                                workspace, workspace_bytes, stream);
    if (st) return fail(st);
    if (cudaEventRecord(h->ev_fwd[s], stream) != cudaSuccess) return fail(LMOE_ERR_CUDA);
    // 3. output copy
    if (cudaStreamWaitEvent(h->io_out, h->ev_fwd[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(y_host, ys, xbytes, cudaMemcpyDeviceToHost, h->io_out) != cudaSuccess ||
        cudaEventRecord(h->ev_out[s], h->io_out) != cudaSuccess) {
        ++h->io_calls;   // the forward's event is recorded; a queued part of the copy runs on io_out in order
        return LMOE_ERR_CUDA;
    }
    ++h->io_calls;
    return LMOE_OK;
}

int lmoe_host_wait(lmoe_handle *h, cudaStream_t stream) {
    if (!h) return LMOE_ERR_INVALID_ARG;
    for (int s = 0; s < 2; ++s)
        if (cudaStreamWaitEvent(stream, h->ev_out[s], 0) != cudaSuccess) return LMOE_ERR_CUDA;
    return LMOE_OK;
}

int lmoe_set_stage_events(lmoe_handle *h, cudaEvent_t *events, int n_events) {
    if (!h) return LMOE_ERR_INVALID_ARG;
    if (!events) {
        if (n_events != 0) return LMOE_ERR_INVALID_ARG;
        h->stage_events = nullptr;
        return LMOE_OK;
    }
    if (n_events != LMOE_NUM_STAGES + 1) return LMOE_ERR_INVALID_ARG;
    h->stage_events = events;
    return LMOE_OK;
}

int lmoe_set_backward_events(lmoe_handle *h, cudaEvent_t *events, int n_events) {
    if (!h) return LMOE_ERR_INVALID_ARG;
    if (events == nullptr && n_events == 0) {
        h->bwd_events = nullptr;
        return LMOE_OK;
    }
    if (!events || n_events != LMOE_BWD_NUM_STAGES + 1) return LMOE_ERR_INVALID_ARG;
    h->bwd_events = events;
    return LMOE_OK;
}

int lmoe_selftest_timeout(lmoe_handle *h, uint64_t limit_ns, cudaStream_t stream) {
    if (!h || limit_ns < 1000ull || limit_ns > 1000000000ull) return LMOE_ERR_INVALID_ARG;
    return launch_bounded_wait_selftest(h->d_status, limit_ns, nullptr, stream) == cudaSuccess ? LMOE_OK
                                                                                            : LMOE_ERR_CUDA;
}

int lmoe_device_status(lmoe_handle *h, cudaStream_t stream, int clear, int *device_status) {
    if (!h || !device_status) return LMOE_ERR_INVALID_ARG;
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, h->d_status, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return LMOE_ERR_CUDA;
    if (clear && v) {
        if (cudaMemsetAsync(h->d_status, 0, sizeof v, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return LMOE_ERR_CUDA;
    }
    // a debug build's failed index checks (every translation unit's word)
    const bool cl = clear != 0;
    const unsigned dbg = debug_word_gemm(cl) | debug_word_pair(cl) | debug_word_split(cl) | debug_word_gemm_bwd(cl) | debug_word_route(cl) |
                         debug_word_backward(cl) | debug_word_selftest(cl);
    if (dbg == ~0u) return LMOE_ERR_CUDA;
    *device_status = dbg ? LMOE_ERR_INDEX : (v & kDevErrTimeout) ? LMOE_ERR_TIMEOUT : LMOE_OK;
    return LMOE_OK;
}

int lmoe_debug_checks(void) { return kDebugChecks ? 1 : 0; }

int lmoe_selftest_index(cudaStream_t stream) {
    if (!kDebugChecks) return LMOE_ERR_INVALID_ARG;
    return launch_index_check_selftest(stream) == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

int qb_histogram(const float *scores, int64_t T, int32_t E, int64_t ld, int32_t B, uint32_t *hist,
                 int accumulate, cudaStream_t stream) {
    if (T < 0 || E < 1 || ld < E || B < 1 || B > 65536 || !hist || (T > 0 && !scores) ||
        (accumulate != 0 && accumulate != 1))
        return LMOE_ERR_INVALID_ARG;
    if (!aligned16(hist) || (scores && !aligned16(scores))) return LMOE_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    int st = check_device(&dev, &sms);
    if (st) return st;
    return launch_qb_histogram(scores, T, E, ld, B, hist, accumulate, sms, stream) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
}

int qb_quantile_bias(const uint32_t *hist, int32_t E, int32_t B, double level, float *quantile_out,
                     float *bias_out, cudaStream_t stream) {
    if (!hist || !bias_out || E < 1 || B < 1 || B > 65536 || !(level >= 0.0 && level <= 1.0))
        return LMOE_ERR_INVALID_ARG;
    if (!aligned16(hist) || !aligned16(bias_out) || (quantile_out && !aligned16(quantile_out)))
        return LMOE_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    int st = check_device(&dev, &sms);
    if (st) return st;
    return launch_qb_quantile(hist, E, B, level, quantile_out, bias_out, stream) == cudaSuccess
               ? LMOE_OK
               : LMOE_ERR_CUDA;
}

int qb_sign_update(const int32_t *counts, int32_t E, float gamma, float *bias, cudaStream_t stream) {
    if (!counts || !bias || E < 1 || E > 65536 || !(gamma == gamma)) return LMOE_ERR_INVALID_ARG;
    if (!aligned16(counts) || !aligned16(bias)) return LMOE_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    int st = check_device(&dev, &sms);
    if (st) return st;
    return launch_sign_update(counts, E, gamma, bias, stream) == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

}  // extern "C"
