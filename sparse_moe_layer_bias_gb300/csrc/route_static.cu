// route_static.cu -- lmoe_route_static: the biased top-k and the stable
// grouping of assignments by expert, with its scratch memory in a fixed
// device array inside this library instead of a caller workspace.
//
// Why it exists: some callers cannot call cudaMalloc or hand out device
// memory at run time -- e.g. an inference-engine plugin that is given no
// allocator, or a latency-critical serving loop that forbids allocation once it
// has started.  They still pass their inputs and outputs; the bitmaps, popcount
// prefixes and the other scratch of the permutation live in kScratch below.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library holds kScratchBytes of it until the process exits.  Host code cannot
// use its name as a device address: at set-up, once per device and with that
// device current, cudaGetSymbolAddress gives the address the kernels receive.
#include <mutex>

#include "lmoe.h"
#include "kernels.h"

namespace {

// 8 MiB: enough for 896 experts x 8192 tokens x top-16 (about 2.4 MiB) with
// room to spare; larger problems are rejected with LMOE_ERR_UNSUPPORTED_SHAPE.
constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char kScratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of kScratch on the current device (looked up once per device).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LMOE_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, kScratch) != cudaSuccess || !p) return LMOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LMOE_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int lmoe_route_static(const float *scores, int64_t T, int32_t E, int32_t top_k,
                                 const float *bias, int32_t *topk_idx, float *gates,
                                 int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                                 cudaStream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E) return LMOE_ERR_INVALID_ARG;
    if (T == 0) return LMOE_OK;
    if (!scores || !bias || !topk_idx || !gates || !counts || !offsets || !perm || !inv)
        return LMOE_ERR_INVALID_ARG;
    if (T * top_k >= (int64_t(1) << 31)) return LMOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t words = (T + 31) / 32;
    const int64_t n = T * top_k;
    // scratch layout: bitmap | word prefix | tile lists (128 and 256 rows) | tile counts |
    // token of each permuted row
    const size_t b_bitmap = align256(size_t(E) * words * 4);
    const size_t b_prefix = align256(size_t(E) * words * 4);
    const size_t b_tiles = align256(size_t((n + lmoe::kBM - 1) / lmoe::kBM + E) * 16);
    const size_t b_tiles2 = align256(size_t((n + 2 * lmoe::kBM - 1) / (2 * lmoe::kBM) + E) * 16);
    const size_t b_nmt = 256;
    const size_t b_tokrow = align256(size_t(n) * 4);
    if (b_bitmap + b_prefix + b_tiles + b_tiles2 + b_nmt + b_tokrow > kScratchBytes)
        return LMOE_ERR_UNSUPPORTED_SHAPE;

    void *base = nullptr;
    const int st = scratch_address(&base);
    if (st != LMOE_OK) return st;
    unsigned char *p = static_cast<unsigned char *>(base);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(p);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(p + b_bitmap);
    int4 *tiles = reinterpret_cast<int4 *>(p + b_bitmap + b_prefix);
    int4 *tiles2 = reinterpret_cast<int4 *>(p + b_bitmap + b_prefix + b_tiles);
    int32_t *nmt = reinterpret_cast<int32_t *>(p + b_bitmap + b_prefix + b_tiles + b_tiles2);
    int32_t *tokrow = reinterpret_cast<int32_t *>(p + b_bitmap + b_prefix + b_tiles + b_tiles2 + b_nmt);

    // The bitmap is the only scratch that must start at zero; the array keeps
    // the previous call's contents.
    if (cudaMemsetAsync(bitmap, 0, size_t(E) * words * 4, stream) != cudaSuccess) return LMOE_ERR_CUDA;
    const int w = static_cast<int>(words);
    if (lmoe::launch_topk(scores, bias, T, E, top_k, topk_idx, gates, bitmap, w, stream) != cudaSuccess ||
        lmoe::launch_expert_scan(bitmap, E, w, prefix, counts, stream) != cudaSuccess ||
        lmoe::launch_offsets_tiles(counts, E, offsets, tiles, nmt, tiles2, nmt + 1, nullptr, nullptr, stream) != cudaSuccess ||
        lmoe::launch_scatter(topk_idx, T, top_k, E, bitmap, prefix, w, offsets, perm, inv, tokrow, stream) !=
            cudaSuccess)
        return LMOE_ERR_CUDA;
    return LMOE_OK;
}
