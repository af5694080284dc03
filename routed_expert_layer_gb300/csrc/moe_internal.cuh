// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/moe_gb300.h"

namespace moe {

// ---- programmatic dependent launch ----------------------------------------------------
// Every kernel of the forward is launched with programmatic stream serialisation. It
// waits for the kernel before it (griddepcontrol.wait: that grid has completed and its
// writes are visible) before it touches any memory, and only then lets the kernel after
// it launch (griddepcontrol.launch_dependents), so at most two kernels overlap: one
// running, the next one launched and in its prologue. Launch latency and prologues
// (barrier setup, tensor-memory allocation) are hidden; results cannot change. When a
// kernel is launched without the attribute both instructions do nothing.
__device__ __forceinline__ void pdl_entry() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Whether launch_pdl adds the attribute: set for the duration of a decode-sized forward
// by the host thread that enqueues it. At prefill sizes launch latency is noise, and a
// dependent grid that becomes resident early only holds SM slots, so there the kernels
// are launched plainly (griddepcontrol.wait is then a no-op).
extern thread_local bool g_launch_pdl;

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  return [&](std::remove_cv_t<KArgs>... a) {
    void* p[] = {(void*)&a...};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = g_launch_pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, (const void*)kernel, p);
  }(std::forward<Args>(args)...);
}

// Device error word bits (also documented in moe_get_error).
constexpr uint32_t kErrExpertRange = 1u;
constexpr uint32_t kErrCountOverflow = 2u;
// (bit 4 = a bounded wait in the tensor-core GEMM gave up; see tc_ptx.cuh)
constexpr uint32_t kErrF16Range = 8u;  // a stored f16 intermediate was out of range or not finite
constexpr uint32_t kErrDuplicate = 16u;  // a token listed the same expert twice (caller-given routing)

// Profiled stages of one forward.
enum Stage {
  kStageRouter = 0,
  kStageSelect,
  kStagePermute,
  kStagePrep,      // f16 activation rows + work list
  kStageGateUp,
  kStageFinalize,  // K-split reduction + SwiGLU (only when the gate/up GEMM splits K)
  kStageDown,
  kStageCombine,
  kStageBlockIn,   // LatentMoE block: routed-down projection + shared experts' gate/up
  kStageBlockOut,  // LatentMoE block: routed-up projection + shared experts' down, summed
  kNumStages
};

// Tile of the SIMT router (used by the allocation-free routing entry point).
constexpr int kRouterTT = 16;     // router tile: tokens
constexpr int kRouterTE = 128;    // router tile: experts (one per thread)

// Device copy of one layer. Expert weights are repacked into the tensor-core tile
// layout (see expert_tc.cu): [E][M tiles][K chunks of 128][9216 B].
struct DeviceLayer {
  const float* router_w = nullptr;      // [H][E] fp32
  const float* router_bias = nullptr;   // [E] (zeros when the caller gave none)
  const uint16_t* router_w3 = nullptr;  // [E_pad][3H] bf16: three-term split of W_r, transposed
  const uint8_t* gu_tc = nullptr;       // [E][2I/128][H/128][9216] gate/up tiles (rows interleaved)
  const uint8_t* dn_tc = nullptr;       // [E][H/128][I/128][9216] down tiles
  const float* gu_global = nullptr;     // [E][2] (gate, up) tensor scales
  const float* dn_global = nullptr;     // [E]
  const float* gu_norm = nullptr;       // [E][2] 2^-n_gate, 2^-n_up: accumulator normalisers (below)
  const float* dn_norm = nullptr;       // [E] 2^-n_down
  const int32_t* norm_exp = nullptr;    // [E][4] (n_gate, n_up, n_down, 0)
};

// ---- normalised f16 intermediates ----------------------------------------------------------
// The SwiGLU rows h and the down rows y are stored in f16 between kernels. So that their
// range does not depend on the size of x or of the tensor scales, they are stored in
// normalised units. With A = e2m1 * e4m3 (the dequantised weight without its tensor scale,
// |A| <= 6 * M where M is the projection's largest block scale) and B = the f16 activation
// row scaled by 2^sigma so its largest element lies in [2^13, 2^14):
//   gn = acc_gate * 2^-n_gate, un = acc_up * 2^-n_up with 2^n >= 6 * M * 2^14 (so |gn|, |un|
//        <= H, typically O(1)); exact, being powers of two;
//   gv = gn * gate_f[p] is the true gate pre-activation (gate_f = g_gate * 2^(n_gate - sigma));
//   h  = gn * un * sigmoid(gv) * 2^-6 is stored (the true SwiGLU value is h * 2^6 * g_gate *
//        g_up * 2^(n_gate + n_up - 2 sigma)); x and the tensor scales reach h only through the
//        bounded sigmoid;
//   y  = acc_down * 2^-n_down with 2^n_down >= 6 * M_down is stored;
//   the combine multiplies y by comb_f[p] = g_down * g_gate * g_up * 2^(n_gate + n_up + n_down
//        + 6 - 2 sigma) (computed in fp32 with ldexp, so it over- or underflows only where the
//        true output does) and by the gate weight.
// A stored value that is not finite or beyond the f16 range raises kErrF16Range.
constexpr float kHStore = 1.0f / 64.0f;
constexpr int kHStoreExp = 6;

// ---- tensor-core path ------------------------------------------------------------------
constexpr int kTcDecodeN = 16;        // rows per work item, decode variant
constexpr int kTcDecodeStages = 6;    // shared-memory pipeline stages, decode variant (two CTAs per SM;
                                      // measured: 6 and 8 alike within 0.5 %, odd counts 2-3 % slower)
constexpr int kTcDecodeAStages = 3;   // dequantised A stages in TMEM, decode variant
constexpr int kTcPrefillN = 192;      // rows per work item, prefill variant
constexpr int kTcPrefillStages = 6;   // pipeline stages, prefill variant (1 CTA per SM, 2 weight tiles)
constexpr int kTcPrefillAStages = 2;  // dequantised A stages in TMEM, prefill variant
constexpr int kTcPrefillKH = 1;       // 64-element K halves per stage, prefill variant
// Midfill (8 <= T*k/E < kTcMidMaxAvg routed rows per expert on average): the prefill kernel
// with 128-row items and 128-element K stages (two A stages of 128 K fit in TMEM).
constexpr int kTcMidN = 128;
constexpr int kTcMidStages = 4;
constexpr int kTcMidAStages = 2;
constexpr int kTcMidKH = 2;
constexpr int kTcMidMaxAvg = 96;
// Small midfill (8 <= T*k/E < kTcMid64MaxAvg): 64-row items, so each stage's activation
// tile is half as large and six stages fit in shared memory instead of four (deeper
// weight prefetch); with 40 rows per expert on average an expert rarely needs two items.
constexpr int kTcMid64N = 64;
constexpr int kTcMid64Stages = 6;
constexpr int kTcMid64MaxAvg = 40;
// A K split is taken when it shortens the decode GEMM's critical path (waves x chunks per
// item) by at least this many percent.
constexpr int kTcSplitMinGainPct = 10;
constexpr int kTcModePartial = 0;     // epilogue writes normalised fp32 partial sums
constexpr int kTcModeSwiglu = 1;      // epilogue applies SwiGLU and writes normalised f16 h
constexpr int kTcModeOutF16 = 2;      // epilogue writes normalised f16 values to out16

// A run of at most nmax routed rows of one expert; every (chunk, M tile, K split)
// is one work item of the grouped GEMM, decoded arithmetically from its index.
struct TcChunk {
  int e;   // expert
  int p0;  // first routed row
  int n;   // rows (<= nmax)
  int pad;
};

struct TcPlan {
  bool prefill = false;
  int nmax = kTcDecodeN;
  int ctas_per_sm = 2;
  int grid = 0;
  int S1 = 1, S2 = 1;  // K splits of the gate/up and down GEMMs
  // Prefill-sized calls on the general routing path: experts with at most cold_rows rows
  // (the cold tail of a skewed batch) run on the decode GEMM, the rest on the prefill GEMM.
  int cold_rows = 0;
};

struct TcGemmParams {
  const uint8_t* w = nullptr;        // tile-layout weights [E][M][KC][4608]
  int M = 0, KC = 0, S = 1;
  const TcChunk* chunks = nullptr;
  const int32_t* n_chunks = nullptr;
  const float* gscale = nullptr;     // accumulator normalisers 2^-n per expert
  int gstride = 1, gsel = 0;         // gscale[e*gstride + (gsel ? row&1 : 0)]
  const float* gate_f = nullptr;     // per routed row: normalised gate -> true gate pre-activation
  int mode = kTcModePartial;
  float* out = nullptr;              // partial output [S][rows][ldo]
  uint16_t* out16 = nullptr;         // f16 output [S][rows][ldo] (kTcModeOutF16)
  size_t out_slice = 0;
  int ldo = 0;
  uint16_t* h16 = nullptr;           // SwiGLU output [rows][I]
  int I = 0;
  uint32_t* err = nullptr;
};

struct RouterTcPlan {
  int nt = 16;        // tokens per N tile
  int n_tiles = 1, m_tiles = 1;
  int kc_total = 0;   // K stages of 64 over the 3H concatenated terms
  int S = 1;          // K splits
  int grid = 1;
  bool small = true;  // N tile <= 64 (deeper pipeline variant)
};

struct RouterTcParams {
  int T = 0, E = 0, H = 0;
  int nt = 16, n_tiles = 1, m_tiles = 1, kc_total = 0, S = 1;
  float* part = nullptr;  // [S][T][E]
  uint32_t* err = nullptr;
};

struct Workspace {
  float* router_part = nullptr;   // [S][T][E]
  float* logits = nullptr;        // [T][E]
  int32_t* idx = nullptr;         // [T][k]
  float* w = nullptr;             // [T][k]
  uint32_t* masks = nullptr;      // [ceil(T/32)][E]
  int32_t* chunk_base = nullptr;  // [ceil(T/32)][E]
  int32_t* counts = nullptr;      // [E]
  int32_t* offsets = nullptr;     // [E+1]
  int32_t* active = nullptr;      // [E] touched experts, ascending
  int32_t* meta = nullptr;        // [4]: [0] touched experts, [1] max rows per expert, [2] row chunks
  int32_t* perm = nullptr;        // [T*k]
  int32_t* slot = nullptr;        // [T*k]
  int32_t* inv = nullptr;         // [T*k]
  uint16_t* x_stage = nullptr;    // [T][H] for moe_forward_host
  uint16_t* out_stage = nullptr;  // [T][H]
  uint32_t* err = nullptr;        // device error word
  uint32_t* ticket = nullptr;     // CTAs finished in route_small_kernel (zero between calls)
  // tensor-core path
  uint16_t* xg = nullptr;         // [T*k][H] f16 activation rows in routed order (row p x 2^sigma_p)
  float* gate_f = nullptr;        // [T*k] g_gate * 2^(n_gate - sigma_p) of each routed row
  float* comb_f = nullptr;        // [T*k] factor from stored y to the true down projection
  float* wc = nullptr;            // [T][k] per route: gate weight * comb_f of its row
  uint16_t* h16 = nullptr;        // [T*k][I] f16 SwiGLU activations, normalised
  float* part1 = nullptr;         // [S1][T*k][2I] normalised gate/up partial sums (split K only)
  uint16_t* ytc = nullptr;        // [S2][T*k][H] f16 down-projection partial sums, normalised
  TcChunk* chunks = nullptr;     // row chunks of the touched experts (count in meta[2])
  int chunk_cap = 0;
  TcChunk* chunks_cold = nullptr;  // prefill-sized calls: experts of few rows, for the decode GEMM (meta[3])
  int chunk_cap_cold = 0;
  // LatentMoE block
  uint16_t* lat = nullptr;        // [T][d] bf16 routed latent (the experts' input)
  uint16_t* hcat = nullptr;       // [T][d + Is] bf16: routed latent output | shared SwiGLU rows
  float* blk_part = nullptr;      // [S][T][M] fp32 partial sums of the block GEMMs
};

// E is the layer's expert count (the router scores all of them); a context may hold
// only the experts [e0, e0 + El) (an expert range: expert-parallel serving), and every
// route to an expert outside it, or with id -1, is masked. Local expert l is global e0 + l.
// H is the width of the layer's input and output rows (the router reads rows of H); D the
// width the routed experts work in (the routed latent of a LatentMoE block, else H).
struct Shape {
  int H, I, E, k;
  int e0 = 0, El = 0;
  int D = 0;
};

// Global expert id -> local expert of the context, or -1 when the route is masked: id -1,
// an expert outside the context's range, or (raising kErrExpertRange through `bad`) an id
// outside [0, E).
__device__ __forceinline__ int local_expert(int id, int E, int e0, int El, bool& bad) {
  if (id < -1 || id >= E) {
    bad = true;
    return -1;
  }
  const int l = id - e0;
  return (id >= 0 && l >= 0 && l < El) ? l : -1;
}

// ---- f16 activation rows ------------------------------------------------------------------

// A token's row is scaled by 2^sigma before its conversion to f16, sigma chosen so the
// row's largest magnitude lands in [2^13, 2^14) (the conversion of bf16 values is then
// exact down to 2^-28 of the row maximum). mx: the largest magnitude's bf16 bits with the
// sign cleared (bf16_pair_maxbits over the row); 0 for a zero row.
__device__ __forceinline__ uint32_t bf16_pair_maxbits(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}
__device__ __forceinline__ int row_sigma(uint32_t mx) {
  if (mx == 0) return 0;
  const int sigma = 13 - ((int)((mx >> 7) & 0xFF) - 127);
  return sigma > 126 ? 126 : (sigma < -126 ? -126 : sigma);
}
// Two bf16 values (low half first) times sc = 2^sigma, rounded to f16.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float sc) {
  const __half2 hh = __floats2half2_rn(__uint_as_float(w << 16) * sc, __uint_as_float(w & 0xFFFF0000u) * sc);
  return *reinterpret_cast<const uint32_t*>(&hh);
}

// The two per-row factors of routed row p (local expert e, activation scaled by 2^sigma)
// that connect the normalised intermediates to true values:
//   gate_f[p] = g_gate * 2^(n_gate - sigma)
//   comb_f[p] = g_down * g_gate * g_up * 2^(n_gate + n_up + n_down + 6 - 2 sigma)
// The three tensor scales are split into mantissa and exponent first, so the product
// over- or underflows only if the result itself does. The combine's weight of route
// (t, j), wc[t*k + j] = w[t][j] * comb_f[p], is written too, indexed by the route, so the
// combine does not wait for inv before loading it.
struct RowFactors {
  const int32_t* idx;  // global expert ids [T][k]; the context's local expert is idx - e0
  int e0;
  const float* gu_global;
  const float* dn_global;
  const int32_t* norm_exp;
  float* gate_f;
  float* comb_f;
  const float* w;  // gate weights [T][k]
  float* wc;       // [T][k]
  __device__ __forceinline__ void write(int p, int route, int e, int sigma) const {
    const int32_t* n = norm_exp + 4 * e;
    int a, b, c;
    const float ma = frexpf(gu_global[2 * e], &a);
    const float mb = frexpf(gu_global[2 * e + 1], &b);
    const float mc = frexpf(dn_global[e], &c);
    gate_f[p] = ldexpf(gu_global[2 * e], n[0] - sigma);
    const float cf = ldexpf(ma * mb * mc, a + b + c + n[0] + n[1] + n[2] + kHStoreExp - 2 * sigma);
    comb_f[p] = cf;
    wc[route] = w[route] * cf;
  }
};

// ---- launchers (each enqueues its kernels on `s`) ----------------------------------

// Router split count for T tokens and the partial buffer size it needs.
int router_splits(const Shape& sh, int T, int sm_count);
size_t router_part_elems(const Shape& sh, int T_max, int sm_count);

cudaError_t launch_router(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const uint16_t* x, int T,
                          int sm_count, cudaStream_t s);
cudaError_t launch_router_reduce(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, int S,
                                 cudaStream_t s);
RouterTcPlan router_tc_plan(const Shape& sh, int T, int sm_count);
cudaError_t launch_router_split(const Shape& sh, const float* W, uint16_t* w3, cudaStream_t s);
cudaError_t launch_router_tc(const Shape& sh, const RouterTcPlan& pl, const CUtensorMap& mw, const CUtensorMap& mx,
                             const DeviceLayer& L, const Workspace& ws, int T, cudaStream_t s,
                             bool reduce = true);
cudaError_t launch_select(const Shape& sh, const float* logits, int32_t* idx, float* w, int T, cudaStream_t s);
// S1 reduce + S2 + S3 of a batch of at most kRouteSmallT tokens in one launch (E <= 1024,
// E % 4 == 0, k <= 32, router K splits <= 64).
constexpr int kRouteSmallT = 32;
inline bool route_small_ok(const Shape& sh, int T, int router_splits) {
  return T <= kRouteSmallT && sh.E <= 1024 && sh.E % 4 == 0 && sh.k <= 32 && router_splits <= 64 && sh.El <= 1024;
}
cudaError_t launch_route_small(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, int S, int nmax,
                               cudaStream_t s);
// nmax > 0 also emits the row chunks of at most nmax rows (ws.chunks, count in meta[2]);
// with cold_rows > 0 experts of at most cold_rows rows go as one chunk each to
// ws.chunks_cold instead (count in meta[3]); served (may be null) receives idx where the
// route is served by this context, else -1.
cudaError_t launch_permute(const Shape& sh, const Workspace& ws, const int32_t* idx, int T, cudaStream_t s,
                           int nmax = 0, int32_t* served = nullptr, int cold_rows = 0);

// LatentMoE block: the bf16 dense GEMMs part[S][T][M] = A[M][K] B[T][K]^T (the router's
// tensor-core kernel, A and B bf16 TMA maps in 64-element boxes of 128 / nt rows) and
// their finalize kernels (block.cu).
RouterTcPlan dense_tc_plan(int M, int K, int T, int sm_count);
cudaError_t launch_dense_tc(const RouterTcPlan& pl, const CUtensorMap& mw, const CUtensorMap& mx, int T, int M, int K,
                            float* part, uint32_t* err, cudaStream_t s);
// lat[t][j] = bf16(sum_s part[s][t][j]) for j < d; for i < Is the shared SwiGLU of rows
// d + 2i (gate) and d + 2i + 1 (up) into hcat[t][d + i] (row stride ldh).
cudaError_t launch_block_in_finalize(const float* part, int S, int T, int d, int Is, uint16_t* lat, uint16_t* hcat,
                                     int ldh, cudaStream_t s);
// out[t][c] = bf16(sum_s part[s][t][c]), c < H.
cudaError_t launch_block_out_finalize(const float* part, int S, int T, int H, uint16_t* out, cudaStream_t s);

// Large-shared-memory opt-in for the kernels that need it (call once per context).
cudaError_t tc_configure();
cudaError_t router_tc_configure();

TcPlan tc_plan(const Shape& sh, int T, int sm_count);
size_t tc_chunk_cap(const Shape& sh, int T, int sm_count);
// idx, w: the routing whose local routes are gathered and its gate weights (ws.idx and
// ws.w, or a caller's).
cudaError_t launch_gather_x(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const int32_t* idx,
                            const float* w, const uint16_t* x, int T, cudaStream_t s);
// map: activation rows in boxes of 16 rows; map64 / map128: the same tensor in boxes of 64 / 128 rows.
cudaError_t launch_gemm(const TcPlan& pl, const CUtensorMap& map, const CUtensorMap& map64, const CUtensorMap& map128,
                        const TcGemmParams& P, cudaStream_t s);
cudaError_t launch_swiglu_finalize(const Shape& sh, const Workspace& ws, const TcPlan& pl, int T, cudaStream_t s);
// Uses the per-route weights ws.wc the gather wrote.
cudaError_t launch_combine_tc(const Shape& sh, const Workspace& ws, const TcPlan& pl, uint16_t* out, int ldo, int T,
                              cudaStream_t s);
cudaError_t launch_debug_hy(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const TcPlan& pl, int T,
                            float* h, float* y, cudaStream_t s);
// Load time: largest block scale of each expert's gate, up and down tensors (raw E4M3 bytes in
// device memory) into maxb[3e..3e+2] (zeroed by the caller), then the normalisers from them.
cudaError_t launch_scale_max(const Shape& sh, int e, const uint8_t* gu_scales_raw, const uint8_t* dn_scales_raw,
                             uint32_t* maxb, cudaStream_t s);
cudaError_t launch_norms(const Shape& sh, const uint32_t* maxb, float* gu_norm, float* dn_norm, int32_t* norm_exp,
                         cudaStream_t s);
cudaError_t launch_repack_tc(const Shape& sh, int e, const uint8_t* gu_codes_raw, const uint8_t* gu_scales_raw,
                             const uint8_t* dn_codes_raw, const uint8_t* dn_scales_raw, uint8_t* gu_tc, uint8_t* dn_tc,
                             cudaStream_t s);

}  // namespace moe
