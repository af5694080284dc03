/*
 * moe_gb300.h -- C ABI of the routed Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * One layer: T tokens of hidden size H are scored by a router against E experts,
 * each token is sent to its top-k experts, every expert is a SwiGLU MLP whose
 * three matrices are stored in NVFP4, and the k expert outputs of each token are
 * weighted and summed. Sources (web pages on serving Kimi-K3):
 *   - "Kimi-K3 NVFP4 station eight sparks", section "The number the project hangs
 *     on": a layer is attention, then a router, then 16 experts, then a sum;
 *     table "What we verified today": 16 of 896 experts per token, one expert is
 *     18,579,480 bytes in 12 tensors; section "What has to be built": NVFP4 is an
 *     FP8 scale per 16 values plus a per-expert global scale.
 *   - "Serving Kimi-K3 ... with 8xB300 GPUs", section "The model, as the serving
 *     system sees it": 3 matrices per expert, 4-bit E2M1 values two per byte.
 *   - "Computation and Data Movement for Inference" (Chinese translation of an essay
 *     on MoE serving), sections 4 and 15:
 *     route records are sorted by expert so one weight load serves a bucket, then
 *     expert outputs are restored to token order, weighted and merged.
 * The pages leave open the score function, tie rule, activation and global-scale
 * granularity; this library uses: fp32 router logits; top-k by (logit descending,
 * expert index ascending, -0 == +0); gate weights = softmax over the k selected
 * logits; SwiGLU silu(gate) * up with gate rows first; one fp32 scale per
 * projection tensor (gate, up, down) per expert.
 *
 * Conventions for every call:
 *   - Return value: MOE_OK (0) or a negative moe_status. Argument errors are
 *     detected on the host before any GPU work is enqueued; nothing is written.
 *   - "device" pointers are CUDA global memory on the context's device; "host"
 *     pointers are CPU memory. Streams are passed as void* and must be a
 *     cudaStream_t of the context's device (NULL = legacy default stream).
 *   - Kernels never trap. Device-side anomalies (an expert id out of range, a
 *     count overflow) set a sticky error word read by moe_get_error().
 *   - A context is used by one host thread and one stream at a time.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx; /* opaque; owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, T out of range, aliasing */
  MOE_ERR_UNSUPPORTED = -2,  /* shape outside the supported set, or device is not sm_103 */
  MOE_ERR_NOT_LOADED = -3,   /* forward before moe_load_layer */
  MOE_ERR_OOM = -4,          /* device allocation failed */
  MOE_ERR_CUDA = -5,         /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_FLAG = -6   /* a kernel raised the device error word */
} moe_status;

/* Layer shape and capacity.
 * Supported: hidden % 256 == 0, inter % 128 == 0, 1 <= top_k <= 32,
 * top_k <= n_experts <= 1024, 1 <= max_tokens, max_tokens * top_k < 2^31,
 * hidden <= 14336.
 * Expert range (expert-parallel serving; "Kimi-K3 NVFP4 station eight sparks", section
 * "What has to be built": the split is a mask on the router's chosen ids, and the routed
 * kernel takes a local expert offset): a context may hold only the experts
 * [expert_begin, expert_begin + expert_count) of the layer's n_experts. The router still
 * scores all n_experts and every token still picks its top_k among them; routes to
 * experts outside the range are masked, so the context's output is the part of the
 * layer's output that its experts contribute, and the outputs of contexts whose ranges
 * partition the experts add up to the layer. expert_count = 0 (with expert_begin = 0)
 * means all experts.
 * LatentMoE block ("Kimi K3 optimization on GB300, Part I", section "Routed-down
 * projection: column sharding and latent assembly": every MoE block projects the 7,168
 * hidden dimensions into a 3,584-wide routed latent with a [3584, 7168] BF16 weight, and
 * back after the experts; "Serving Kimi K3 End to End", section 3.3: 2 shared experts that
 * every token uses, unquantized in the NVFP4 checkpoint): with latent = d > 0 the routed
 * experts work in d dimensions,
 *   lat = bf16(x W_down^T)  (W_down bf16 [d][H]),  routed = the expert sum on lat (width d),
 *   out = bf16(routed W_up^T + shared(x))  (W_up bf16 [H][d]),
 * where shared(x) = W_sd (silu(W_sg x) * (W_su x)) with bf16 weights of intermediate size
 * shared_inter (all shared experts together: two experts of width f are one of width 2f),
 * present when shared_inter > 0 (only together with latent > 0). The router scores the
 * hidden state x. Supported: latent % 256 == 0, latent <= 14336, shared_inter % 64 == 0,
 * and no expert range (expert_count == 0): the projections and shared experts belong to
 * the whole layer, so the outputs of range contexts would each carry the shared experts
 * and would not add up to the layer (MOE_ERR_UNSUPPORTED). */
typedef struct {
  int32_t hidden;       /* H */
  int32_t inter;        /* I, the expert intermediate size */
  int32_t n_experts;    /* E, experts of the layer (the router's outputs) */
  int32_t top_k;        /* k */
  int32_t max_tokens;   /* the largest T a forward call may pass; sizes the workspace */
  uint32_t flags;       /* reserved, must be 0 */
  int32_t expert_begin; /* first expert this context holds (global id) */
  int32_t expert_count; /* experts this context holds, or 0 for all n_experts */
  int32_t latent;       /* d: the routed experts' width in a LatentMoE block, or 0 (they work in H) */
  int32_t shared_inter; /* intermediate size of the shared experts together, or 0 for none */
} moe_config;

/* One layer's weights in HOST memory, caller-owned, read only during moe_load_layer.
 * Per-expert pointers let a caller hand over experts wherever they sit (a loader
 * must map expert ids to tensors explicitly; checkpoints may store them out of order).
 * The expert arrays cover the context's experts only: entry l is global expert
 * expert_begin + l, for l < n_local (n_local = expert_count, or n_experts for all).
 *   router_w    fp32 [H][E], row-major: logit[t][e] = sum_h x[t][h] * router_w[h][e]
 *   router_bias fp32 [E] added to the logits, or NULL for none
 *   gu_codes[l] uint8 [2I][H/2]: rows 0..I-1 gate, I..2I-1 up; element k of a row is
 *               in byte k/2, low nibble = even k; a nibble is an E2M1 code
 *   gu_scales[l] uint8 [2I][H/16]: E4M3 ("fn") scale of elements 16b..16b+15 of a row
 *   gu_global   fp32 [n_local][2]: (gate, up) tensor scales
 *   dn_codes[l] uint8 [H][I/2], dn_scales[l] uint8 [H][I/16], dn_global fp32 [n_local]
 * Weight element = e2m1(code) * e4m3(block scale) * tensor scale. In a LatentMoE block
 * (latent = d > 0) the expert tensors are at width d in place of H ([2I][d/2], [d][I/2], ...)
 * and the block's dense weights are bf16 (NULL when not used):
 *   proj_down   bf16 [d][H]: lat[t][j] = sum_h x[t][h] * proj_down[j][h]
 *   proj_up     bf16 [H][d]: out[t][c] = sum_j routed[t][j] * proj_up[c][j] + shared
 *   shared_gu   bf16 [2 Is][H]: rows 0..Is-1 gate, Is..2Is-1 up (Is = shared_inter)
 *   shared_dn   bf16 [H][Is] */
typedef struct {
  const float* router_w;
  const float* router_bias;
  const uint8_t* const* gu_codes;
  const uint8_t* const* gu_scales;
  const float* gu_global;
  const uint8_t* const* dn_codes;
  const uint8_t* const* dn_scales;
  const float* dn_global;
  const uint16_t* proj_down;
  const uint16_t* proj_up;
  const uint16_t* shared_gu;
  const uint16_t* shared_dn;
} moe_layer_host;

/* Create a context on CUDA device `device`: checks the device is sm_103 and
 * allocates the device workspace for cfg->max_tokens. *out receives the context
 * (NULL on failure). */
MOE_API int moe_create(const moe_config* cfg, int device, moe_ctx** out);

/* Copy a layer's weights to the device and repack them into the kernels' layouts.
 * Synchronous. May be called again to replace the layer. */
MOE_API int moe_load_layer(moe_ctx* ctx, const moe_layer_host* layer);

/* The layer on T tokens: out[t][:] = sum_j w[t][j] * FFN_{idx[t][j]}(x[t][:]).
 *   x    device bf16 [T][H], row-major, 16-byte aligned
 *   out  device bf16 [T][H], 16-byte aligned, must not overlap x
 * Asynchronous on `stream`; allocates nothing; does not synchronise the host; may be
 * captured in a CUDA graph. T == 0 returns MOE_OK and enqueues nothing; T > max_tokens
 * is an error. At decode sizes (T*k/E < 8) the kernels are launched with programmatic
 * stream serialisation and the last one lets the next kernel on the stream launch
 * before it has finished: a following kernel that is itself launched with that
 * attribute must wait on its grid dependency (griddepcontrol.wait) before reading out;
 * kernels launched without it, copies and events wait for completion as usual. */
MOE_API int moe_forward(moe_ctx* ctx, void* stream, const void* x, void* out, int32_t T);

/* The expert stage on caller-given routing ("Kimi-K3 NVFP4 station eight sparks",
 * section "What has to be built": a worker takes each token's 16 global expert ids,
 * with -1 for a masked id, and returns rows plus the ids it actually served):
 *   out[t][:] = sum over j ascending, where idx[t][j] is one of this context's experts,
 *               of w[t][j] * FFN_{idx[t][j]}(x[t][:])   (zero if no route is served)
 *   x       device bf16 [T][H], 16-byte aligned
 *   idx     device int32 [T][k]: global expert ids; -1 = masked; ids of other contexts'
 *           experts are skipped. A token must not list one expert twice (error bit 16,
 *           that token's output is then undefined); an id outside [-1, E) raises error
 *           bit 1 and is skipped.
 *   w       device fp32 [T][k]: the weight of each route, applied as given
 *   out     device bf16 [T][H], 16-byte aligned, must not overlap x
 *   served  device int32 [T][k] or NULL: idx[t][j] where this context computed the route,
 *           else -1
 * Asynchronous on `stream`; allocates nothing; may be captured in a CUDA graph; the same
 * launch rules as moe_forward. */
MOE_API int moe_forward_routed(moe_ctx* ctx, void* stream, const void* x, const int32_t* idx, const float* w,
                               void* out, int32_t T, int32_t* served);

/* The same through HOST buffers: copies x (host bf16 [T][H]) to the device,
 * runs moe_forward, copies the result to out (host bf16 [T][H]) and waits for
 * the stream. Use page-locked host memory for asynchronous copies. */
MOE_API int moe_forward_host(moe_ctx* ctx, void* stream, const void* x_host, void* out_host, int32_t T);

/* Release everything the context owns. NULL is a no-op. */
MOE_API int moe_destroy(moe_ctx* ctx);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_str(int status);

/* Read and clear the device error word (synchronises the device). Returns
 * MOE_OK if no kernel raised it, MOE_ERR_DEVICE_FLAG otherwise; *bits (may be
 * NULL) receives the raw word: 1 = expert id out of range, 2 = row count overflow,
 * 4 = a bounded wait inside a GEMM gave up (the kernel stopped early), 8 = an f16
 * intermediate (SwiGLU or down-projection value, stored in normalised units) was
 * beyond the f16 range or not finite; it is stored as the conversion gives it (an
 * infinity or NaN, never clamped), so the output shows it too; 16 = a token of a
 * caller-given routing listed one expert twice. */
MOE_API int moe_get_error(moe_ctx* ctx, uint32_t* bits);

/* ---- inspection hooks (tests and benchmarking) ----------------------------- */

/* Routing of T tokens (router, select, permute). Every output is a device
 * pointer and may be NULL:
 *   logits fp32 [T][E]; idx int32 [T][k] (descending logit, global ids); w fp32 [T][k];
 *   offsets int32 [n_local+1] (routed rows of the context's experts; inv = -1 for a
 *   masked route); perm int32 [T*k] (token of routed row p);
 *   slot int32 [T*k] (j of routed row p); inv int32 [T*k] (row p of (t, j)). */
MOE_API int moe_debug_route(moe_ctx* ctx, void* stream, const void* x, int32_t T, float* logits, int32_t* idx, float* w,
                    int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv);

/* Select and permute from caller-given logits (device fp32 [T][E]); the
 * outputs are as for moe_debug_route. */
MOE_API int moe_debug_select(moe_ctx* ctx, void* stream, const float* logits, int32_t T, int32_t* idx, float* w,
                     int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv);

/* The expert stage on its own: runs the whole layer on x and copies the SwiGLU
 * activations h (device fp32 [T*k][I], rows in routed order p) and the
 * unweighted down projections y (device fp32 [T*k][D], D = latent or H) out. Either
 * may be NULL. In a LatentMoE block, lat (device bf16 [T][d], may be NULL) receives the
 * routed-down projection the experts read. */
MOE_API int moe_debug_experts(moe_ctx* ctx, void* stream, const void* x, int32_t T, float* h, float* y, void* lat);

/* A dependent consumer as moe_forward describes it: copies `bytes` (a multiple of 16)
 * from device src to device dst (both 16-byte aligned, not overlapping) with a kernel
 * launched on `stream` with programmatic stream serialisation that waits on its grid
 * dependency (griddepcontrol.wait) before its first read. Enqueued after moe_forward,
 * dst receives the finished output although the kernel may launch before the forward's
 * last kernel has completed. For tests of that contract; runs on the current device.
 * Errors: MOE_ERR_INVALID_ARG for NULL, misaligned, overlapping or odd-sized
 * arguments; MOE_ERR_CUDA if the launch fails. */
MOE_API int moe_debug_pdl_copy(void* stream, const void* src, void* dst, int64_t bytes);

/* Per-kernel timing with CUDA events recorded on the forward's stream.
 * moe_profile_begin arms the next `max_calls` forwards; moe_profile_end waits
 * for them and writes, for each of `n` stages (n <= moe_profile_stages()), the
 * summed milliseconds and the number of launches timed. Stage names come from
 * moe_profile_stage_name(i). Forwards armed inside a CUDA-graph capture are timed
 * by the graph's replays (the last replay counts); a captured forward whose graph
 * was never replayed is not counted. */
MOE_API int moe_profile_stages(void);
MOE_API const char* moe_profile_stage_name(int i);
MOE_API int moe_profile_begin(moe_ctx* ctx, int32_t max_calls);
MOE_API int moe_profile_end(moe_ctx* ctx, float* ms, int32_t* launches, int32_t n);

/* ---- routing without allocation ---------------------------------------------- */

/* Limits of moe_route_noalloc (its scratch is a fixed-size array inside the library). */
#define MOE_NOALLOC_MAX_TOKENS 256
#define MOE_NOALLOC_MAX_EXPERTS 1024
#define MOE_NOALLOC_MAX_PARTIALS (1024 * 1024) /* router partial sums, 4-byte words */

/* The routing step (router logits, top-k select, per-expert permutation) for
 * callers that may not allocate device memory: engines that reserve their whole
 * HBM budget at start-up and forbid cudaMalloc on the request path, plugin hosts
 * that only hand out pre-planned buffers, or decode loops that cannot take the
 * device-wide synchronisation an allocation may cause. The pages have no
 * counterpart to this call; it adds no new arithmetic, only a different owner for
 * the scratch memory.
 * It needs no context and allocates nothing: its scratch (about 5.3 MB) is one
 * static __device__ array that every GPU loading this library holds until the
 * process exits. Runs on the CURRENT device, on `stream`.
 *   x          device bf16 [T][H], 16-byte aligned
 *   router_w   device fp32 [H][E]; router_bias device fp32 [E] or NULL
 *   idx, w, offsets, perm, slot, inv: device outputs, caller-allocated, laid out
 *              as for moe_debug_route (all required)
 *   err        device uint32 or NULL: when given, the routing kernels OR the error
 *              bits of moe_get_error into it (1 = expert id out of range); the caller
 *              clears it and reads it after the stream has finished
 * Limits: H % 64 == 0, 1 <= k <= 32, k <= E <= MOE_NOALLOC_MAX_EXPERTS,
 * 1 <= T <= MOE_NOALLOC_MAX_TOKENS; larger sizes return MOE_ERR_UNSUPPORTED.
 * The first call on a device looks up the scratch's device address (make it
 * before any stream capture); the address belongs to the device's primary context,
 * so only that context (the one the CUDA runtime uses) is supported. All calls share
 * the one array: calls whose GPU work overlaps (unordered streams) race and corrupt
 * each other's results. The logits come from an fp32 SIMT router and may differ from
 * moe_forward's tensor-core logits in the last bits, so two experts whose logits are
 * that close may be ordered differently. */
MOE_API int moe_route_noalloc(void* stream, const void* x, const float* router_w, const float* router_bias,
                              int32_t H, int32_t E, int32_t k, int32_t T, int32_t* idx, float* w, int32_t* offsets,
                              int32_t* perm, int32_t* slot, int32_t* inv, uint32_t* err);

/* Number of kernels this context has enqueued so far (all calls that run kernels). */
MOE_API int64_t moe_launch_count(const moe_ctx* ctx);

/* The launch plan moe_forward uses for T tokens on a GPU with sm_count SMs, computed on
 * the host only (no GPU; for tests and capacity planning). plan (caller-owned, 11
 * entries):
 *   [0] 1 for the prefill GEMM variant, 0 for decode   [1] routed rows per work item
 *   [2] K splits of the gate/up GEMM                     [3] K splits of the down GEMM
 *   [4] CTAs of the expert GEMMs                         [5] K splits of the router GEMM
 *   [6] CTAs of the router GEMM                          [7] 1 if routing runs as one launch
 *   [8] row-chunk capacity of the workspace              [9] device workspace bytes
 *   [10] experts with at most this many rows run on the decode GEMM in a prefill-sized
 *        call (0: no split)
 * Errors: what moe_create returns for cfg; MOE_ERR_INVALID_ARG for a NULL plan,
 * sm_count < 1 or T outside 1..max_tokens. */
MOE_API int moe_plan(const moe_config* cfg, int32_t sm_count, int32_t T, int64_t* plan);

/* Device bytes held by the context (weights + workspace). */
MOE_API int64_t moe_device_bytes(const moe_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
