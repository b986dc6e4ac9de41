/*
 * lmoe.h -- C ABI of the GB300 (sm_103a) Stable LatentMoE layer (forward and
 * backward) and Quantile Balancing (QB) library, liblmoe.so.
 *
 * The operations follow three public write-ups of Kimi K3's architecture:
 *   [DD] "Kimi-K3-Architecture-Deep-Dive": section 1 (SiTU-GLU), section 2
 *        (Stable LatentMoE), section 3 (Quantile Balancing).
 *   [IN] "Inside K3: How Stable Latent MoE and MLA Attention Are Designed":
 *        sections "SiTU-GLU", "RMSNorm insertion", "Quantile Balancing (QB)".
 *   [NW] "Notes on the MoE and Attention of K3" (news write-up): sections
 *        "LatentMoE: paying for a bigger pool", "Keeping the numbers in range".
 *
 * Conventions shared by every call:
 *   - Tensors are caller-owned DEVICE memory, dense row-major.  bf16 tensors are
 *     passed as uint16_t bit patterns.  Every tensor pointer must be 16-byte
 *     aligned (LMOE_ERR_ALIGNMENT otherwise).
 *   - Calls enqueue kernels on `stream` and return without synchronising.
 *     Errors found on the host (bad arguments, shapes, alignment, workspace
 *     size) are reported synchronously and then nothing is enqueued; errors the
 *     GPU raises surface at the caller's next synchronisation of the stream.
 *   - No call allocates device memory except lmoe_create (handle state).
 *   - Every call returns an lmoe_status (0 = success).
 */
#ifndef LMOE_H_
#define LMOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    LMOE_OK = 0,
    LMOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum          */
    LMOE_ERR_UNSUPPORTED_SHAPE = 2, /* a dimension outside what the kernels tile      */
    LMOE_ERR_ALIGNMENT = 3,         /* a pointer not 16-byte aligned                  */
    LMOE_ERR_WORKSPACE = 4,         /* workspace missing or smaller than required     */
    LMOE_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed           */
    LMOE_ERR_TIMEOUT = 6,           /* a kernel's bounded wait gave up (device error) */
    LMOE_ERR_NO_DEVICE = 7,         /* the current device is not sm_103 (GB300)       */
    LMOE_ERR_INDEX = 8              /* a debug build's index check failed (device error) */
} lmoe_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *lmoe_status_string(int status);

/* ------------------------------------------------------------------------ */
/* Layer configuration and weights                                          */
/* ------------------------------------------------------------------------ */

/* Shape of one Stable LatentMoE layer.  [DD] section 2: d -> d/2 latent,
 * 2n routed experts of which 2k are active per token; [NW] "LatentMoE": K3 has
 * d = 7168, latent 3584, 896 experts, 16 active, 2 shared experts.
 * Supported: d, inter, n_shared*shared_inter multiples of 64, latent a multiple of 128;
 * 1 <= top_k <= 32; top_k <= n_experts <= 1024; max_tokens >= 0. */
typedef struct {
    int32_t d;            /* hidden size                                      */
    int32_t latent;       /* routed latent width (d/2 in K3)                  */
    int32_t n_experts;    /* routed experts E                                 */
    int32_t top_k;        /* experts chosen per token                         */
    int32_t inter;        /* routed expert intermediate size I                */
    int32_t n_shared;     /* shared experts (always active)                   */
    int32_t shared_inter; /* intermediate size of each shared expert Is       */
    float beta1;          /* SiTU cap; 4 in K3 ([DD] section 1)               */
    float beta2;          /* linear-branch softcap; 25 in K3 ([DD] section 1) */
    float rms_eps;        /* epsilon inside the RMSNorm square root (1e-6)    */
    int64_t max_tokens;   /* largest T a forward call will be given           */
    int32_t norm_after_down; /* 0: K3's layer.  1: ablation variant with a
                           * second un-weighted RMSNorm right after the
                           * down-projection, h = RMSNorm(W_down x), which the
                           * router and the experts then see ([DD] section 2,
                           * [IN] "RMSNorm insertion": the variant the ablation
                           * dropped) */
    int32_t expert_fp8;   /* 0: bf16 routed experts (K3's layer).  1: FP8
                           * variant: lmoe_create quantises W1, W2, W3 to e4m3
                           * with one power-of-two scale per weight row, each
                           * forward quantises the routed latent per token the
                           * same way, and the expert GEMMs run e4m3 x e4m3 on
                           * the tensor cores (fp32 accumulation); the SiTU-GLU
                           * activation is stored as e4m3(4 * act), exact scale
                           * from its bound |act| < beta1*beta2 = 100 ([NW]
                           * "Keeping the numbers in range").  Requires inter %
                           * 128 == 0.  Codes round to nearest even and saturate
                           * at 448; a row's scale is the smallest 2^e with
                           * max|row| <= 448 * 2^e. */
    int32_t with_backward; /* 1: lmoe_create also keeps transposed copies of
                           * every weight (about as much device memory again as
                           * the weights) so that lmoe_backward can run, and
                           * lmoe_forward also keeps the SiTU-GLU pre-activations
                           * (pre_act, shared_pre_act: p1 | p2 in bf16, 4 bytes per
                           * activation element) and the router's fp32 logits in
                           * its workspace for it; 0: the
                           * handle serves forwards only.  The backward covers
                           * K3's layer and the norm_after_down variant;
                           * with_backward together with expert_fp8 returns
                           * LMOE_ERR_UNSUPPORTED_SHAPE. */
} lmoe_config;

/* Weight pointers (device, bf16, row-major, K-major rows as "out x in").
 * w1, w2 and w3 are COPIED at lmoe_create into a handle-owned, tile-contiguous
 * order (one more copy of the routed weights in device memory); the caller may
 * free or change them afterwards.  For the other six the handle keeps the
 * POINTERS: the caller must keep them alive and unchanged until lmoe_destroy.
 * S = n_shared * shared_inter. */
typedef struct {
    const uint16_t *w_down;   /* [latent][d]           down-projection            */
    const uint16_t *w_router; /* [n_experts][latent]   router rows                */
    const uint16_t *w1;       /* [n_experts][inter][latent]  SiTU branch          */
    const uint16_t *w2;       /* [n_experts][inter][latent]  softcapped branch    */
    const uint16_t *w3;       /* [n_experts][latent][inter]  expert output        */
    const uint16_t *ws1;      /* [S][d]  shared SiTU branch (expert s: rows s*Is..) */
    const uint16_t *ws2;      /* [S][d]  shared softcapped branch                */
    const uint16_t *ws3;      /* [d][S]  shared output (expert s: columns s*Is..) */
    const uint16_t *w_up;     /* [d][latent]           up-projection              */
} lmoe_weights;

typedef struct lmoe_handle lmoe_handle;

/* Validate `cfg`, check the device (sm_103), and build the handle: the
 * repacked routed weights, the TMA descriptors of all weights and a small
 * device status word (LMOE_ERR_CUDA if the copy does not fit).  On success
 * *out owns a handle to release with lmoe_destroy.  Synchronous. */
int lmoe_create(const lmoe_config *cfg, const lmoe_weights *weights, lmoe_handle **out);

/* Release the handle and its device state (synchronises the device first). */
int lmoe_destroy(lmoe_handle *handle);

/* Bytes of caller-provided device workspace lmoe_forward needs for T tokens
 * (0 <= T <= max_tokens).  The workspace holds the routing maps and the
 * intermediate activations (see lmoe_workspace_layout) and, for batches
 * small enough that the dense GEMMs are split over K, their fp32 partial
 * sums in an internal slot after the documented ones.  The size depends on
 * the handle's device (its number of SMs) and never decreases with T: a
 * workspace sized for T (e.g. for max_tokens) serves every smaller batch. */
int lmoe_workspace_size(const lmoe_handle *handle, int64_t T, size_t *bytes);

/* Byte offsets, inside the workspace, of the intermediates a forward of T
 * tokens leaves behind (for inspection and tests; valid after the stream has
 * reached the end of the forward).  Every slot is always reserved; when the
 * caller passes its own buffer for scores, topk_idx, gates or counts, the
 * values go there and that slot is left untouched. */
typedef struct {
    int64_t h;        /* [T][latent] bf16        latent after the down-projection */
    int64_t scores;   /* [T][n_experts] fp32     sigmoid router scores            */
    int64_t topk_idx; /* [T][top_k] int32        chosen experts                   */
    int64_t gates;    /* [T][top_k] fp32         unbiased scores of those experts */
    int64_t counts;   /* [n_experts] int32       assignments per expert           */
    int64_t offsets;  /* [n_experts+1] int32     exclusive scan of counts         */
    int64_t perm;     /* [T*top_k] int32         assignment at each permuted row  */
    int64_t inv;      /* [T*top_k] int32         permuted row of each assignment  */
    int64_t act;      /* [T*top_k][inter] bf16   expert SiTU-GLU activations, permuted order
                       * (expert_fp8: e4m3 codes of 4 * act, one byte each) */
    int64_t o;        /* [T*top_k][latent] bf16  gate-weighted expert outputs, assignment order */
    int64_t r;        /* [T][latent] bf16        RMS-normalised aggregate          */
    int64_t shared_act; /* [T][S] bf16           shared-expert activations        */
    int64_t h_norm;   /* [T][latent] bf16        RMSNorm(h) when norm_after_down, else -1 */
    int64_t h_fp8;    /* [T][latent] e4m3 codes of the routed latent (expert_fp8), else -1 */
    int64_t h_fp8_exp; /* [T] int8 scale exponents of those rows (expert_fp8), else -1 */
    int64_t pre_act;  /* [T*top_k][2*inter] bf16 SiTU-GLU pre-activations W1[e] h | W2[e] h of
                       * each permuted row (with_backward, read by lmoe_backward), else -1 */
    int64_t shared_pre_act; /* [T][2*S] bf16 the shared experts' Ws1 x | Ws2 x (with_backward), else -1 */
    int64_t logits;   /* [T][n_experts] fp32 router logits W_router h (with_backward), else -1 */
} lmoe_ws_layout;

int lmoe_workspace_layout(const lmoe_handle *handle, int64_t T, lmoe_ws_layout *layout);

/* One forward pass of the Stable LatentMoE layer on T tokens:
 *   h  = W_down x                              (a1; [DD] section 2)
 *        (norm_after_down: h = RMSNorm(W_down x), same eps, no weight)
 *   s  = sigmoid(W_router h)                   (a2; routing in the latent)
 *   u  = fp32(s + bias); pick the top_k experts by u (ties: lower id)
 *        gates = s at the chosen experts       (a3; [DD] section 3, [NW])
 *   group the T*top_k assignments by expert    (a4; stable)
 *   act = SiTU(W1[e] h; beta1) * softcap(W2[e] h; beta2)   (a5; [DD] section 1)
 *   o   = gate * W3[e] act                     (a6)
 *   z   = sum over the token's experts of o;  r = z / sqrt(mean(z^2) + eps)
 *                                              (a7; [DD] section 2, [IN] "RMSNorm insertion")
 *   y  = W_up r + sum_s Ws3_s (SiTU(Ws1_s x) * softcap(Ws2_s x))   (a8; [NW] shared experts)
 * x: [T][d] bf16 input.  bias: [n_experts] fp32 selection bias.  y: [T][d]
 * bf16 output.  Optional outputs (NULL = keep them in the workspace):
 * scores_out [T][n_experts] fp32, topk_idx_out [T][top_k] int32, gates_out
 * [T][top_k] fp32, expert_counts_out [n_experts] int32.  workspace: at least
 * lmoe_workspace_size(T) bytes, 256-byte aligned.  T = 0 enqueues nothing.
 * A handle may be used from one stream at a time per workspace.  Unless the
 * timing hook (lmoe_set_stage_events) is set, the shared experts' GEMM runs on
 * a side stream of the handle, ordered after the work already in `stream`
 * and joined back into `stream` before the routed experts, so everything the
 * call enqueues is ordered within `stream` as seen from outside.  The
 * result is bitwise reproducible: no sum depends on the order in which the
 * kernels' threads run. */
int lmoe_forward(lmoe_handle *handle, const uint16_t *x, int64_t T, const float *bias,
                 uint16_t *y, float *scores_out, int32_t *topk_idx_out, float *gates_out,
                 int32_t *expert_counts_out, void *workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* Bytes of device staging memory lmoe_forward_host needs: two slots, each
 * holding x [max_tokens][d] bf16, bias [n_experts] fp32 and y [max_tokens][d]
 * bf16 (256-byte aligned sub-buffers).  The size depends only on the handle. */
int lmoe_host_io_size(const lmoe_handle *handle, size_t *bytes);

/* lmoe_forward from and to HOST memory, pipelined across calls.  Enqueues,
 * without waiting for any of it:
 *   1. on the handle's input copy stream, once the forward that last read
 *      staging slot (call number % 2) is done: x_host [T][d] bf16 and
 *      bias_host [n_experts] fp32 into that slot of io_dev;
 *   2. on `stream`, once copy 1 has landed and the output copy that last read
 *      the slot's y is done: lmoe_forward (y into the slot; the optional
 *      device outputs and the workspace as in lmoe_forward);
 *   3. on the handle's output copy stream, once 2 is done: y into y_host.
 * So the input copy of one call overlaps the forward of the one before, and
 * its output copy the forward of the one after.  y_host holds the result once
 * `stream` has passed a later lmoe_host_wait (or after a device
 * synchronisation).  The caller keeps x_host and bias_host unchanged, and
 * y_host untouched, until then.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to run asynchronously.
 * io_dev: lmoe_host_io_size bytes, 256-byte aligned, used only through this
 * call.  Argument errors are reported before anything is enqueued, as in
 * lmoe_forward.  A CUDA error after the input copy was queued leaves the
 * staging slot ordered after the work the call did queue, so later calls stay
 * correct; the failed call's y_host is not written.
 * One host thread and one `stream` per handle at a time.  The pages describe
 * no host-memory interface; this is an addition of this library. */
int lmoe_forward_host(lmoe_handle *handle, const uint16_t *x_host, int64_t T, const float *bias_host,
                      uint16_t *y_host, float *scores_out, int32_t *topk_idx_out, float *gates_out,
                      int32_t *expert_counts_out, void *io_dev, size_t io_bytes, void *workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/* Make `stream` wait for every output copy lmoe_forward_host has enqueued so
 * far (enqueues a wait; does not block the host). */
int lmoe_host_wait(lmoe_handle *handle, cudaStream_t stream);

/* Stages of lmoe_forward, in launch order (for lmoe_set_stage_events). */
typedef enum {
    LMOE_STAGE_DOWN = 0,       /* a1 down-projection GEMM                          */
    LMOE_STAGE_SHARED = 1,     /* shared experts' W1|W2 GEMM + SiTU-GLU            */
    LMOE_STAGE_ROUTER = 2,     /* a2 router GEMM + sigmoid                         */
    LMOE_STAGE_TOPK = 3,       /* a3 biased top-k                                  */
    LMOE_STAGE_SCAN = 4,       /* a4 per-expert counts                             */
    LMOE_STAGE_OFFSETS = 5,    /* a4 offsets and grouped-GEMM tile list            */
    LMOE_STAGE_SCATTER = 6,    /* a4 permutation maps                              */
    LMOE_STAGE_EXPERT_W12_LIGHT = 7, /* a5 grouped expert W1|W2 GEMM + SiTU-GLU, experts
                                      * with at most 128 rows (FP8 variant: after the
                                      * latent's e4m3 quantisation, also in this stage) */
    LMOE_STAGE_EXPERT_W12_HEAVY = 8, /* a5 the same for experts with more rows (pair tiles) */
    LMOE_STAGE_EXPERT_W3 = 9,  /* a6 grouped expert W3 GEMM + gate scatter         */
    LMOE_STAGE_COMBINE = 10,   /* a7 aggregation + RMSNorm                         */
    LMOE_STAGE_UP = 11,        /* a8 up-projection + shared W3 GEMM                */
    LMOE_NUM_STAGES = 12
} lmoe_stage;

/* Timing hook: with n_events == LMOE_NUM_STAGES + 1 (cudaEvent_t handles
 * created by the caller), every later lmoe_forward records events[i] on its
 * stream just before stage i and events[LMOE_NUM_STAGES] after the last one.
 * events = NULL (n_events = 0) turns it off.  The handle keeps the array
 * pointer: it must stay valid while set. */
int lmoe_set_stage_events(lmoe_handle *handle, cudaEvent_t *events, int n_events);

/* ------------------------------------------------------------------------ */
/* Backward pass                                                             */
/* ------------------------------------------------------------------------ */

/* Weight gradients (device fp32, each laid out like its weight in
 * lmoe_weights; all required, 16-byte aligned).  accumulate = 0: lmoe_backward
 * overwrites them; 1: it adds this pass's gradients to their contents (one
 * fp32 addition per element, e.g. to sum micro-batches without an extra
 * pass over the gradients). */
typedef struct {
    float *w_down;   /* [latent][d]                  */
    float *w_router; /* [n_experts][latent]          */
    float *w1;       /* [n_experts][inter][latent]   */
    float *w2;       /* [n_experts][inter][latent]   */
    float *w3;       /* [n_experts][latent][inter]   */
    float *ws1;      /* [S][d]                       */
    float *ws2;      /* [S][d]                       */
    float *ws3;      /* [d][S]                       */
    float *w_up;     /* [d][latent]                  */
    int32_t accumulate; /* 0 or 1 (else LMOE_ERR_INVALID_ARG)            */
} lmoe_grads;

/* Bytes of device workspace lmoe_backward needs for T tokens (separate from
 * the forward's workspace, which it reads). */
int lmoe_backward_workspace_size(const lmoe_handle *handle, int64_t T, size_t *bytes);

/* Gradient of the layer ("Kimi-K3-Architecture-Deep-Dive" sections 1 and 2):
 * given dy = dL/dy [T][d] bf16 for the forward lmoe_forward ran on x [T][d]
 * with this handle, computes dx [T][d] bf16 and the fp32 weight gradients.
 * The forward's routing is held fixed: the top-k choice has no gradient; the
 * router's gradient flows through the gates (gate = sigmoid(w_router[e] . h)).
 * The selection bias gets none.  The bf16 roundings of the forward pass the
 * gradient through unchanged.  Per token:
 *   dr  = W_up^T dy,  da_s = Ws3^T dy  (shared experts: SiTU-GLU backward at
 *         the forward's kept Ws1 x, Ws2 x)
 *   dz  = RMSNorm backward of dr at z = sum of the forward's rows o
 *   per chosen expert: u = W3[e]^T dz; da = gate * u; dgate = u . act;
 *         dp1, dp2 = SiTU-GLU backward at the forward's kept W1[e] h, W2[e] h
 *         (bf16);
 *         dh += W1[e]^T dp1 + W2[e]^T dp2 + w_router[e] dgate sigma'(logit)
 *   dx  = W_down^T dh + Ws1^T dp_s1 + Ws2^T dp_s2
 * and the weight gradients are the sums over tokens of the matching outer
 * products (dW_up = sum dy r^T, ..., dW3[e] = sum over e's assignments of
 * gate dz act^T, dW1[e] = sum dp1 h^T).
 * The forward's intermediates are read from fwd_workspace (the workspace of
 * that forward, unchanged since; its layout for T): h, perm, inv, the
 * permuted activations and pre-activations, the router's logits, the rows
 * o, r, the shared activations and pre-activations and the tile
 * lists, and the offsets of the expert groups (always in the workspace; the
 * per-expert counts are their differences).  topk_idx, gates: the forward's
 * outputs when the caller had it write them to its own buffers (they are then
 * not in the workspace), or NULL for the workspace's copies; an expert id
 * outside [0, n_experts) contributes no gradient.  sigma'(logit) is taken
 * as sigma(logit) sigma(-logit) at the forward's kept fp32 logit, which stays
 * accurate where the fp32 gate has rounded to 1.  workspace: lmoe_backward_workspace_size(T) bytes,
 * 256-byte aligned.  The handle must have been created with with_backward =
 * 1 (else LMOE_ERR_INVALID_ARG).  Errors are reported before anything is
 * enqueued, as in lmoe_forward.  Unless lmoe_set_backward_events is set, the
 * memory-bound copies run on a side stream of the handle, forked from and
 * joined back into `stream`, so the call is ordered within `stream` as seen
 * from outside.  T = 0 enqueues nothing (the gradients are left untouched). */
int lmoe_backward(lmoe_handle *handle, const uint16_t *x, int64_t T, const uint16_t *dy,
                  const int32_t *topk_idx, const float *gates, const void *fwd_workspace,
                  size_t fwd_workspace_bytes, uint16_t *dx, const lmoe_grads *grads, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/* Stages of lmoe_backward, in launch order (for lmoe_set_backward_events). */
typedef enum {
    LMOE_BWD_STAGE_DR = 0,          /* dr | da_s = dy [W_up | Ws3]                        */
    LMOE_BWD_STAGE_SHARED = 1,      /* shared experts: SiTU-GLU backward (recomputed)    */
    LMOE_BWD_STAGE_RMSNORM = 2,     /* RMSNorm backward: dz                              */
    LMOE_BWD_STAGE_EXPERT_U = 3,    /* u = W3[e]^T dz per assignment (two launches)       */
    LMOE_BWD_STAGE_EXPERT_GLU = 4,  /* routed SiTU-GLU backward (recomputed; two launches) */
    LMOE_BWD_STAGE_ROUTER = 5,      /* gate and logit gradients                          */
    LMOE_BWD_STAGE_DH_EXPERTS = 6,  /* experts' share of dh                              */
    LMOE_BWD_STAGE_DH_ROUTER = 7,   /* router's share of dh                              */
    LMOE_BWD_STAGE_DH_SUM = 8,      /* dh                                                */
    LMOE_BWD_STAGE_DX = 9,          /* dx                                                */
    LMOE_BWD_STAGE_TRANSPOSE = 10,  /* token-major copies for the dense weight gradients */
    LMOE_BWD_STAGE_WGRAD_DENSE = 11, /* six dense weight gradients                       */
    LMOE_BWD_STAGE_SEGMENTS = 12,   /* per-expert segments, their copies, unused experts */
    LMOE_BWD_STAGE_WGRAD_W3 = 13,   /* routed experts' dW3                               */
    LMOE_BWD_STAGE_WGRAD_W12 = 14,  /* routed experts' dW1 | dW2                         */
    LMOE_BWD_NUM_STAGES = 15
} lmoe_bwd_stage;

/* Timing hook of lmoe_backward, as lmoe_set_stage_events for the forward:
 * n_events == LMOE_BWD_NUM_STAGES + 1 events recorded before each stage and
 * after the last; NULL / 0 turns it off. */
int lmoe_set_backward_events(lmoe_handle *handle, cudaEvent_t *events, int n_events);

/* Routing without caller scratch: the biased top-k (a3) and the stable
 * grouping of assignments by expert (a4) of lmoe_forward, for callers that
 * cannot allocate device memory -- e.g. an inference-engine plugin given no
 * allocator, or a serving loop that forbids allocation once running.  The
 * pages describe no such call; it is an interface addition of this library.
 * Inputs: scores [T][E] fp32 (sigmoid router scores), bias [E] fp32.
 * Outputs (caller memory, same meaning as in lmoe_forward): topk_idx [T][top_k]
 * int32, gates [T][top_k] fp32, counts [E] int32, offsets [E+1] int32,
 * perm [T*top_k] int32, inv [T*top_k] int32.
 * Scratch lives in one fixed 8 MiB array inside the library (every GPU that
 * loads the library holds it until exit); problems whose scratch exceeds it
 * return LMOE_ERR_UNSUPPORTED_SHAPE.  With n = T*top_k and each term rounded
 * up to a multiple of 256 bytes, the scratch is
 *   4*E*ceil(T/32)                (token bitmap of each expert)
 * + 4*E*ceil(T/32)                (popcount prefix of each bitmap word)
 * + 16*(ceil(n/128) + E)          (128-row tile list)
 * + 16*(ceil(n/256) + E)          (256-row tile list)
 * + 256                           (tile counts)
 * + 4*n                           (token of each permuted row) bytes.
 * It calls no cudaMalloc/cudaFree.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress).  All calls share the array:
 * calls whose work overlaps on the GPU (other streams, other threads) race and
 * must be serialised by the caller.  1 <= top_k <= 32, top_k <= E <= 1024. */
int lmoe_route_static(const float *scores, int64_t T, int32_t E, int32_t top_k, const float *bias,
                      int32_t *topk_idx, float *gates, int32_t *counts, int32_t *offsets,
                      int32_t *perm, int32_t *inv, cudaStream_t stream);

/* Self-test of the failure path (no fault, no hang): enqueues one CTA that
 * waits, with the same bounded mbarrier wait every GEMM role uses, on a
 * barrier nothing arrives on.  After limit_ns (1 us .. 1 s) the wait gives up
 * and sets the handle's device status, so a following lmoe_device_status
 * reports LMOE_ERR_TIMEOUT; the kernel returns normally and the context stays
 * usable.  The pages describe no such call; it is an addition of this library. */
int lmoe_selftest_timeout(lmoe_handle *handle, uint64_t limit_ns, cudaStream_t stream);

/* Device-side status of the handle's kernels (bounded waits that gave up;
 * in a debug build also failed index checks).  Synchronises `stream`, copies
 * the status word, and clears it when `clear` is non-zero.  *device_status is
 * LMOE_OK, LMOE_ERR_TIMEOUT or (debug builds) LMOE_ERR_INDEX, which takes
 * precedence.  The index-check words are per library, not per handle. */
int lmoe_device_status(lmoe_handle *handle, cudaStream_t stream, int clear, int *device_status);

/* 1 if this library was built with index checks (-DLMOE_DEBUG), else 0.
 * Such a build checks, before every use, each index that a kernel reads from
 * a device list -- the rows the expert GEMMs gather and scatter (and their
 * gates), the permutation maps, the grouped GEMMs' tile lists and their
 * counts, the backward's column maps.  A failed check skips the access (the
 * affected rows are left unwritten), records the failure, and
 * lmoe_device_status then returns LMOE_ERR_INDEX.  Nothing traps.  The
 * pages describe no such build; it is an addition of this library. */
int lmoe_debug_checks(void);

/* Self-test of that reporting path: in a debug build enqueues one thread that
 * fails one index check without touching memory, so a following
 * lmoe_device_status (any handle) reports LMOE_ERR_INDEX.  A release build
 * returns LMOE_ERR_INVALID_ARG and enqueues nothing. */
int lmoe_selftest_index(cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Quantile Balancing                                                        */
/* ------------------------------------------------------------------------ */

/* QB histogram ([DD] section 3, steps 1-3; [IN] "Quantile Balancing (QB)").
 * scores: [T][ld] fp32 (the first E columns are the experts), values in [0,1]
 * (sigmoid scores need no further map).  hist: [E][B] uint32.
 *   bin(s) = min(B-1, floor(fp32(s*B)))  (fp32 multiply; s < 0 -> bin 0)
 *   hist[e][bin(scores[t][e])] += 1 for all t < T.
 * accumulate = 0 replaces hist's contents (every bin is written); 1 adds to
 * it (histograms are additive).
 * Constraints: T >= 0, 1 <= E <= ld, 1 <= B <= 65536.  NaN scores are not
 * allowed (their bin is undefined). */
int qb_histogram(const float *scores, int64_t T, int32_t E, int64_t ld, int32_t B,
                 uint32_t *hist, int accumulate, cudaStream_t stream);

/* QB quantile read and bias ([DD] section 3; [IN] "Quantile Balancing (QB)";
 * [NW] "Keeping the numbers in range").  For each expert e with N = sum of its
 * row: r = clamp(ceil(level*N), 1, N); j* = first bin whose cumulative count
 * reaches r; q[e] = (j* + (r - C_{j*-1}) / hist[e][j*]) / B (linear inside
 * the bin, computed in fp64, stored fp32); bias[e] = -q[e].  An empty row
 * gives q = 0, bias = 0.  level is normally 1 - top_k/n_experts.
 * hist: [E][B] uint32; quantile_out: [E] fp32 (nullable); bias_out: [E] fp32. */
int qb_quantile_bias(const uint32_t *hist, int32_t E, int32_t B, double level,
                     float *quantile_out, float *bias_out, cudaStream_t stream);

/* The fixed-step selection-bias update that Quantile Balancing replaces, for
 * closed-loop comparisons ("Notes on the MoE and Attention of K3", paragraph
 * on Quantile Balancing: K2 changed each expert's bias by a constant amount
 * per update, which the page likens to SignSGD).  Reading:
 *   mean = sum(counts) / E;  bias[e] += gamma * sign(mean - counts[e]),
 * sign(0) = 0, the comparison exact in integers, the add one fp32 addition.
 * counts: [E] int32 assignments per expert (e.g. lmoe_forward's
 * expert_counts_out); bias: [E] fp32, updated in place.  1 <= E <= 65536;
 * device pointers, 16-byte aligned; argument errors enqueue nothing. */
int qb_sign_update(const int32_t *counts, int32_t E, float gamma, float *bias, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LMOE_H_ */
