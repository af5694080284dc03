// C ABI: context, weight loading, the forward launch sequence, inspection hooks.
// The operations and their sources are documented in include/moe_gb300.h.
//
// Forward sequence (all on the caller's stream, no host synchronisation, no
// allocation, so it can be captured in a CUDA graph):
//   router_tc (+ reduce)  S1 logits            route.cu / router_tc.cu
//   select                S2 top-k, weights    route.cu
//   permute (3 kernels)   S3 offsets, perm, row chunks
//   gather                f16 activation rows in routed order
//   gate/up GEMM          S4 (+ K-split reduction with SwiGLU when split)
//   down GEMM             S5
//   combine               S6
// In a LatentMoE block (block.cu) the block-in GEMM (routed-down projection and shared
// experts' gate/up) runs after the routing and the experts read its latent; the combine
// writes the routed latent next to the shared SwiGLU rows and the block-out GEMM (routed-up
// projection plus shared down projection, one contraction) writes out.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "moe_internal.cuh"

using namespace moe;

thread_local bool moe::g_launch_pdl = false;

struct moe_ctx {
  moe_config cfg{};
  Shape sh{};
  int device = 0;
  int sm_count = 0;
  bool loaded = false;
  DeviceLayer L{};
  Workspace ws{};
  void* weights_mem = nullptr;
  size_t weights_bytes = 0;
  void* ws_mem = nullptr;
  size_t ws_bytes = 0;
  int64_t launches = 0;   // kernels enqueued so far
  CUtensorMap tmap_x{};   // f16 activation rows (B of the gate/up GEMM)
  CUtensorMap tmap_h{};   // f16 SwiGLU rows (B of the down GEMM)
  CUtensorMap tmap_x64{}; // the same two tensors in boxes of 64 and 128 rows
  CUtensorMap tmap_h64{};
  CUtensorMap tmap_x128{};
  CUtensorMap tmap_h128{};
  CUtensorMap tmap_w3{};  // bf16 three-term router weights (A of the router GEMM)
  CUtensorMap tmap_win{};   // LatentMoE block: [W_down ; shared gate/up interleaved] bf16 [d + 2Is][H]
  CUtensorMap tmap_wout{};  // LatentMoE block: [W_up | shared down] bf16 [H][d + Is]
  // profiling
  int prof_max = 0;
  int prof_calls = 0;
  std::vector<cudaEvent_t> prof_ev;  // [prof_max][kNumStages][2]
  std::vector<uint8_t> prof_rec;     // [prof_max][kNumStages]: the stage ran in that call
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// Programmatic dependent launch for the kernels one forward enqueues (decode sizes).
struct PdlScope {
  explicit PdlScope(bool on) { g_launch_pdl = on; }
  ~PdlScope() { g_launch_pdl = false; }
};

const char* kStageNames[kNumStages] = {"router", "select", "permute", "prep",     "gateup",
                                       "finalize", "down",  "combine", "block_in", "block_out"};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2D 16-bit tensor [rows][cols] read in boxes of 64 columns x box_rows rows with
// 128-byte swizzle. Host-only (no GPU work), so it may run during stream capture.
bool make_tmap_16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool bf16) {
  static EncodeTiledFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->flags != 0) return MOE_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->inter <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->expert_begin < 0 || c->expert_count < 0 || (c->expert_count == 0 && c->expert_begin != 0) ||
      (int64_t)c->expert_begin + c->expert_count > c->n_experts)
    return MOE_ERR_INVALID_ARG;
  if (c->hidden % 256 != 0 || c->inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->hidden > 14336) return MOE_ERR_UNSUPPORTED;
  if (c->latent < 0 || c->shared_inter < 0) return MOE_ERR_INVALID_ARG;
  if (c->latent % 256 != 0 || c->latent > 14336 || c->shared_inter % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->shared_inter > 0 && c->latent == 0) return MOE_ERR_UNSUPPORTED;  // shared experts ride on the block GEMMs
  // a block's projections and shared experts belong to the whole layer: range outputs would
  // each carry the shared experts and would not add up to the layer
  if (c->latent > 0 && c->expert_count != 0) return MOE_ERR_UNSUPPORTED;
  if (c->top_k > 32 || c->top_k > c->n_experts || c->n_experts > 1024) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->max_tokens * c->top_k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Bump allocation from one device block (256-byte aligned). With base == nullptr only
// the offsets are computed (the returned pointers are then never dereferenced).
struct Carver {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += (count * sizeof(T) + 255) & ~(size_t)255;
    return p;
  }
};

// The kernels' view of a configuration: the layer's E experts, of which the context
// holds [e0, e0 + El) (all of them when expert_count is 0).
Shape shape_of(const moe_config& c) {
  Shape sh{c.hidden, c.inter, c.n_experts, c.top_k};
  sh.e0 = c.expert_count ? c.expert_begin : 0;
  sh.El = c.expert_count ? c.expert_count : c.n_experts;
  sh.D = c.latent ? c.latent : c.hidden;
  return sh;
}

bool is_block(const moe_config& c) { return c.latent > 0; }

// The block GEMMs' shapes: block-in M = d + 2 Is over K = H, block-out M = H over K = d + Is.
int block_in_rows(const moe_config& c) { return c.latent + 2 * c.shared_inter; }
int block_width(const moe_config& c) { return c.latent + c.shared_inter; }

size_t workspace_layout(const moe_config& c, int sm_count, Workspace* ws, char* base) {
  const Shape sh = shape_of(c);
  const size_t T = c.max_tokens, E = c.n_experts, El = sh.El, k = c.top_k, H = c.hidden, I = c.inter, D = sh.D;
  const size_t C = (T + 31) / 32;
  // sizes that depend on the per-T plans: the maxima over every T <= max_tokens
  size_t rpart = 1, part1 = 1, ytc = T * k * D, ccap = 1, bpart = 1;
  for (int t = 1; t <= c.max_tokens; ++t) {
    const size_t rows = (size_t)t * k;
    rpart = std::max(rpart, (size_t)router_tc_plan(sh, t, sm_count).S * (size_t)t * E);
    const TcPlan pl = tc_plan(sh, t, sm_count);
    if (pl.S1 > 1) part1 = std::max(part1, (size_t)pl.S1 * rows * 2 * I);
    ytc = std::max(ytc, (size_t)pl.S2 * rows * D);
    ccap = std::max(ccap, tc_chunk_cap(sh, t, sm_count));
    if (is_block(c)) {
      const int Mi = block_in_rows(c), Kw = block_width(c);
      bpart = std::max(bpart, (size_t)dense_tc_plan(Mi, (int)H, t, sm_count).S * (size_t)t * Mi);
      bpart = std::max(bpart, (size_t)dense_tc_plan((int)H, Kw, t, sm_count).S * (size_t)t * H);
    }
  }
  Carver cv{base};
  Workspace w;
  w.router_part = cv.take<float>(rpart);
  w.logits = cv.take<float>(T * E);
  w.idx = cv.take<int32_t>(T * k);
  w.w = cv.take<float>(T * k);
  w.masks = cv.take<uint32_t>(C * El);
  w.chunk_base = cv.take<int32_t>(C * El);
  w.counts = cv.take<int32_t>(El);
  w.offsets = cv.take<int32_t>(El + 1);
  w.active = cv.take<int32_t>(El);
  w.meta = cv.take<int32_t>(4);
  w.perm = cv.take<int32_t>(T * k);
  w.slot = cv.take<int32_t>(T * k);
  w.inv = cv.take<int32_t>(T * k);
  w.x_stage = cv.take<uint16_t>(T * H);
  w.out_stage = cv.take<uint16_t>(T * H);
  w.err = cv.take<uint32_t>(1);
  w.ticket = cv.take<uint32_t>(1);
  w.xg = cv.take<uint16_t>(T * k * D);
  w.gate_f = cv.take<float>(T * k);
  w.comb_f = cv.take<float>(T * k);
  w.wc = cv.take<float>(T * k);
  w.h16 = cv.take<uint16_t>(T * k * I);
  w.part1 = cv.take<float>(part1);
  w.ytc = cv.take<uint16_t>(ytc);
  w.chunks = cv.take<TcChunk>(ccap);
  w.chunk_cap = (int)ccap;
  w.chunk_cap_cold = (int)std::min(El, T * k);  // one chunk per cold expert
  w.chunks_cold = cv.take<TcChunk>(w.chunk_cap_cold);
  if (is_block(c)) {
    w.lat = cv.take<uint16_t>(T * c.latent);
    w.hcat = cv.take<uint16_t>(T * block_width(c));
    w.blk_part = cv.take<float>(bpart);
  }
  if (ws) *ws = w;
  return cv.off;
}

struct WeightPtrs {
  float *router_w, *router_bias, *gu_global, *dn_global, *gu_norm, *dn_norm;
  int32_t* norm_exp;
  uint32_t* scale_max;
  uint16_t* w3;
  uint8_t *gu_tc, *dn_tc;
  uint16_t *w_in, *w_out;  // LatentMoE block weights (null otherwise)
};

size_t weights_layout(const moe_config& c, WeightPtrs* p, char* base) {
  const size_t E = c.n_experts, El = shape_of(c).El, H = c.hidden, I = c.inter, D = shape_of(c).D;
  Carver cv{base};
  WeightPtrs w;
  w.router_w = cv.take<float>(H * E);  // the router scores all E experts
  w.router_bias = cv.take<float>(E);
  w.gu_global = cv.take<float>(2 * El);  // expert tensors: the context's El experts
  w.dn_global = cv.take<float>(El);
  w.gu_norm = cv.take<float>(2 * El);
  w.dn_norm = cv.take<float>(El);
  w.norm_exp = cv.take<int32_t>(4 * El);
  w.scale_max = cv.take<uint32_t>(3 * El);
  w.w3 = cv.take<uint16_t>(((E + 127) / 128) * 128 * 3 * H);
  w.gu_tc = cv.take<uint8_t>(El * 2 * I * D * 9 / 16);  // codes (1/2 B) + scales (1/16 B) per weight
  w.dn_tc = cv.take<uint8_t>(El * D * I * 9 / 16);
  w.w_in = is_block(c) ? cv.take<uint16_t>((size_t)block_in_rows(c) * H) : nullptr;
  w.w_out = is_block(c) ? cv.take<uint16_t>(H * (size_t)block_width(c)) : nullptr;
  if (p) *p = w;
  return cv.off;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Events bracketing each stage of a profiled forward (no-ops when not armed).
struct StageTimer {
  moe_ctx* ctx;
  cudaStream_t s;
  int call = -1;
  unsigned flags = cudaEventRecordDefault;
  StageTimer(moe_ctx* c, cudaStream_t st) : ctx(c), s(st) {
    if (ctx->prof_max > 0 && ctx->prof_calls < ctx->prof_max) {
      call = ctx->prof_calls++;
      // under stream capture, external records become event nodes timed by every replay
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        flags = cudaEventRecordExternal;
    }
  }
  void begin(int stage) {
    if (call >= 0) cudaEventRecordWithFlags(ctx->prof_ev[((size_t)call * kNumStages + stage) * 2 + 0], s, flags);
  }
  void end(int stage) {
    if (call >= 0) {
      cudaEventRecordWithFlags(ctx->prof_ev[((size_t)call * kNumStages + stage) * 2 + 1], s, flags);
      ctx->prof_rec[(size_t)call * kNumStages + stage] = 1;
    }
  }
};

// S1..S3. nmax > 0 also emits the row chunks the expert GEMMs iterate over (and, with
// cold_rows > 0, the list of experts with at most cold_rows rows).
int run_route(moe_ctx* ctx, cudaStream_t s, const uint16_t* x, int T, StageTimer* tm, int nmax, int cold_rows = 0) {
  const Shape& sh = ctx->sh;
  if (tm) tm->begin(kStageRouter);
  const RouterTcPlan rp = router_tc_plan(sh, T, ctx->sm_count);
  CUtensorMap mx;
  if (!make_tmap_16(&mx, x, (uint64_t)T, (uint64_t)sh.H, (uint32_t)rp.nt, true)) return MOE_ERR_CUDA;
  const bool small = route_small_ok(sh, T, rp.S);
  if (launch_router_tc(sh, rp, ctx->tmap_w3, mx, ctx->L, ctx->ws, T, s, !small) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStageRouter);
  if (small) {  // reduce, select and permute in one CTA
    if (tm) tm->begin(kStageSelect);
    if (launch_route_small(sh, ctx->L, ctx->ws, T, rp.S, nmax, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (tm) tm->end(kStageSelect);
    ctx->launches += 2;
    return MOE_OK;
  }
  if (tm) tm->begin(kStageSelect);
  if (launch_select(sh, ctx->ws.logits, ctx->ws.idx, ctx->ws.w, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStageSelect);
  if (tm) tm->begin(kStagePermute);
  if (launch_permute(sh, ctx->ws, ctx->ws.idx, T, s, nmax, nullptr, cold_rows) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStagePermute);
  ctx->launches += 6;
  return MOE_OK;
}

// S4..S6 on the tensor cores, for the plan `pl` (the route must have used pl.nmax), with
// the routing idx (global expert ids) and gate weights w.
int run_experts(moe_ctx* ctx, cudaStream_t s, const uint16_t* x, uint16_t* out, int ldo, int T, const TcPlan& pl,
                StageTimer* tm, const int32_t* idx, const float* w) {
  const Shape& sh = ctx->sh;
  const Workspace& ws = ctx->ws;
  const int rows = T * sh.k;
  if (tm) tm->begin(kStagePrep);
  if (launch_gather_x(sh, ctx->L, ws, idx, w, x, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStagePrep);

  TcGemmParams P1;
  P1.w = ctx->L.gu_tc;
  P1.M = 2 * sh.I / 128;
  P1.KC = sh.D / 128;
  P1.S = pl.S1;
  P1.chunks = ws.chunks;
  P1.n_chunks = ws.meta + 2;
  P1.gscale = ctx->L.gu_norm;
  P1.gstride = 2;
  P1.gsel = 1;
  P1.gate_f = ws.gate_f;
  P1.mode = pl.S1 == 1 ? kTcModeSwiglu : kTcModePartial;
  P1.out = ws.part1;
  P1.out_slice = (size_t)rows * 2 * sh.I;
  P1.ldo = 2 * sh.I;
  P1.h16 = ws.h16;
  P1.I = sh.I;
  P1.err = ws.err;
  // prefill-sized calls: the cold experts' single chunks on the decode GEMM first
  TcPlan dp = pl;
  dp.prefill = false;
  dp.nmax = kTcDecodeN;
  dp.ctas_per_sm = 2;
  dp.grid = 2 * ctx->sm_count;
  dp.S1 = dp.S2 = 1;
  TcGemmParams P1c = P1;
  P1c.chunks = ws.chunks_cold;
  P1c.n_chunks = ws.meta + 3;
  if (tm) tm->begin(kStageGateUp);
  if (pl.cold_rows && launch_gemm(dp, ctx->tmap_x, ctx->tmap_x64, ctx->tmap_x128, P1c, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gemm(pl, ctx->tmap_x, ctx->tmap_x64, ctx->tmap_x128, P1, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStageGateUp);
  int n = 4;
  if (pl.S1 > 1) {
    if (tm) tm->begin(kStageFinalize);
    if (launch_swiglu_finalize(sh, ws, pl, T, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (tm) tm->end(kStageFinalize);
    ++n;
  }

  TcGemmParams P2;
  P2.w = ctx->L.dn_tc;
  P2.M = sh.D / 128;
  P2.KC = sh.I / 128;
  P2.S = pl.S2;
  P2.chunks = ws.chunks;
  P2.n_chunks = ws.meta + 2;
  P2.gscale = ctx->L.dn_norm;
  P2.gstride = 1;
  P2.gsel = 0;
  P2.gate_f = nullptr;
  P2.mode = kTcModeOutF16;
  P2.out16 = ws.ytc;
  P2.out_slice = (size_t)rows * sh.D;
  P2.ldo = sh.D;
  P2.I = sh.I;
  P2.err = ws.err;
  TcGemmParams P2c = P2;
  P2c.chunks = ws.chunks_cold;
  P2c.n_chunks = ws.meta + 3;
  if (tm) tm->begin(kStageDown);
  if (pl.cold_rows && launch_gemm(dp, ctx->tmap_h, ctx->tmap_h64, ctx->tmap_h128, P2c, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gemm(pl, ctx->tmap_h, ctx->tmap_h64, ctx->tmap_h128, P2, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStageDown);
  if (pl.cold_rows) n += 2;
  if (tm) tm->begin(kStageCombine);
  if (launch_combine_tc(sh, ws, pl, out, ldo, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (tm) tm->end(kStageCombine);
  ctx->launches += n;
  return MOE_OK;
}

// LatentMoE block-in: the routed latent (ws.lat) and the shared SwiGLU rows (ws.hcat[:, d:]).
int run_block_in(moe_ctx* ctx, cudaStream_t s, const uint16_t* x, int T, StageTimer* tm) {
  const moe_config& c = ctx->cfg;
  const int M = block_in_rows(c), d = c.latent, Is = c.shared_inter;
  const RouterTcPlan pl = dense_tc_plan(M, c.hidden, T, ctx->sm_count);
  CUtensorMap mx;
  if (!make_tmap_16(&mx, x, (uint64_t)T, (uint64_t)c.hidden, (uint32_t)pl.nt, true)) return MOE_ERR_CUDA;
  if (tm) tm->begin(kStageBlockIn);
  if (launch_dense_tc(pl, ctx->tmap_win, mx, T, M, c.hidden, ctx->ws.blk_part, ctx->ws.err, s) != cudaSuccess ||
      launch_block_in_finalize(ctx->ws.blk_part, pl.S, T, d, Is, ctx->ws.lat, ctx->ws.hcat, d + Is, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (tm) tm->end(kStageBlockIn);
  ctx->launches += 2;
  return MOE_OK;
}

// LatentMoE block-out: out = bf16([routed latent | shared SwiGLU] [W_up | W_shared_down]^T).
int run_block_out(moe_ctx* ctx, cudaStream_t s, uint16_t* out, int T, StageTimer* tm) {
  const moe_config& c = ctx->cfg;
  const int K = block_width(c);
  const RouterTcPlan pl = dense_tc_plan(c.hidden, K, T, ctx->sm_count);
  CUtensorMap mh;
  if (!make_tmap_16(&mh, ctx->ws.hcat, (uint64_t)T, (uint64_t)K, (uint32_t)pl.nt, true)) return MOE_ERR_CUDA;
  if (tm) tm->begin(kStageBlockOut);
  if (launch_dense_tc(pl, ctx->tmap_wout, mh, T, c.hidden, K, ctx->ws.blk_part, ctx->ws.err, s) != cudaSuccess ||
      launch_block_out_finalize(ctx->ws.blk_part, pl.S, T, c.hidden, out, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (tm) tm->end(kStageBlockOut);
  ctx->launches += 2;
  return MOE_OK;
}

// width: the row width of x and out (H for the layer, D for the expert stage alone).
int check_forward_args(moe_ctx* ctx, const void* x, const void* out, int32_t T, int width) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > ctx->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)T * width * 2;
  const char* xa = (const char*)x;
  const char* oa = (const char*)out;
  if (xa < oa + bytes && oa < xa + bytes) return MOE_ERR_INVALID_ARG;
  if (!ctx->loaded) return MOE_ERR_NOT_LOADED;
  return MOE_OK;
}

// A caller's kernel that consumes moe_forward's output, launched with programmatic stream
// serialisation: it waits on its grid dependency before its first read (what the header
// asks of such a kernel), then copies n16 16-byte units.
__global__ void pdl_consumer_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

extern "C" {

const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_ERR_NOT_LOADED: return "layer not loaded";
    case MOE_ERR_OOM: return "device out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_FLAG: return "device error flag raised";
    default: return "unknown status";
  }
}

int moe_create(const moe_config* cfg, int device, moe_ctx** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int st = check_config(cfg);
  if (st != MOE_OK) return st;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return MOE_ERR_CUDA;
  if (device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(device);
  moe_ctx* ctx = new moe_ctx();
  ctx->cfg = *cfg;
  ctx->sh = shape_of(*cfg);
  ctx->device = device;
  ctx->sm_count = prop.multiProcessorCount;
  ctx->ws_bytes = workspace_layout(*cfg, ctx->sm_count, nullptr, nullptr);
  if (cudaMalloc(&ctx->ws_mem, ctx->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return MOE_ERR_OOM;
  }
  workspace_layout(*cfg, ctx->sm_count, &ctx->ws, (char*)ctx->ws_mem);
  const uint64_t rows = (uint64_t)cfg->max_tokens * cfg->top_k;
  if (cudaMemset(ctx->ws.err, 0, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(ctx->ws.ticket, 0, sizeof(uint32_t)) != cudaSuccess ||
      !make_tmap_16(&ctx->tmap_x, ctx->ws.xg, rows, ctx->sh.D, 16, false) ||
      !make_tmap_16(&ctx->tmap_h, ctx->ws.h16, rows, cfg->inter, 16, false) ||
      !make_tmap_16(&ctx->tmap_x64, ctx->ws.xg, rows, ctx->sh.D, 64, false) ||
      !make_tmap_16(&ctx->tmap_h64, ctx->ws.h16, rows, cfg->inter, 64, false) ||
      !make_tmap_16(&ctx->tmap_x128, ctx->ws.xg, rows, ctx->sh.D, 128, false) ||
      !make_tmap_16(&ctx->tmap_h128, ctx->ws.h16, rows, cfg->inter, 128, false) || tc_configure() != cudaSuccess ||
      router_tc_configure() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(ctx->ws_mem);
    delete ctx;
    return MOE_ERR_CUDA;
  }
  *out = ctx;
  return MOE_OK;
}

int moe_load_layer(moe_ctx* ctx, const moe_layer_host* lh) {
  if (!ctx || !lh || !lh->router_w || !lh->gu_codes || !lh->gu_scales || !lh->gu_global || !lh->dn_codes ||
      !lh->dn_scales || !lh->dn_global)
    return MOE_ERR_INVALID_ARG;
  const moe_config& c = ctx->cfg;
  const size_t E = c.n_experts, El = ctx->sh.El, H = c.hidden, I = c.inter, D = ctx->sh.D;
  for (size_t e = 0; e < El; ++e)
    if (!lh->gu_codes[e] || !lh->gu_scales[e] || !lh->dn_codes[e] || !lh->dn_scales[e]) return MOE_ERR_INVALID_ARG;
  if (is_block(c) && (!lh->proj_down || !lh->proj_up)) return MOE_ERR_INVALID_ARG;
  if (c.shared_inter > 0 && (!lh->shared_gu || !lh->shared_dn)) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!ctx->weights_mem) {
    ctx->weights_bytes = weights_layout(c, nullptr, nullptr);
    if (cudaMalloc(&ctx->weights_mem, ctx->weights_bytes) != cudaSuccess) {
      cudaGetLastError();
      ctx->weights_mem = nullptr;
      return MOE_ERR_OOM;
    }
  }
  ctx->loaded = false;
  WeightPtrs W;
  weights_layout(c, &W, (char*)ctx->weights_mem);
  ctx->L.router_w = W.router_w;
  ctx->L.router_bias = W.router_bias;
  ctx->L.router_w3 = W.w3;
  ctx->L.gu_global = W.gu_global;
  ctx->L.dn_global = W.dn_global;
  ctx->L.gu_norm = W.gu_norm;
  ctx->L.dn_norm = W.dn_norm;
  ctx->L.norm_exp = W.norm_exp;
  ctx->L.gu_tc = W.gu_tc;
  ctx->L.dn_tc = W.dn_tc;
  const size_t gu_cb = 2 * I * (D / 2), gu_sb = 2 * I * (D / 16), dn_cb = D * (I / 2), dn_sb = D * (I / 16);
  uint8_t* staging = nullptr;
  if (cudaMalloc(&staging, gu_cb + gu_sb + dn_cb + dn_sb) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_OOM;
  }
  cudaStream_t s;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFree(staging);
    return MOE_ERR_CUDA;
  }
  int st = MOE_OK;
  do {
    if (cudaMemcpy(W.router_w, lh->router_w, H * E * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        (lh->router_bias
             ? cudaMemcpy(W.router_bias, lh->router_bias, E * sizeof(float), cudaMemcpyHostToDevice)
             : cudaMemset(W.router_bias, 0, E * sizeof(float))) != cudaSuccess ||
        cudaMemcpy(W.gu_global, lh->gu_global, 2 * El * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(W.dn_global, lh->dn_global, El * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(W.scale_max, 0, 3 * El * sizeof(uint32_t)) != cudaSuccess) {
      st = MOE_ERR_CUDA;
      break;
    }
    if (launch_router_split(ctx->sh, W.router_w, W.w3, s) != cudaSuccess ||
        !make_tmap_16(&ctx->tmap_w3, W.w3, ((E + 127) / 128) * 128, 3 * H, 128, true)) {
      st = MOE_ERR_CUDA;
      break;
    }
    if (is_block(c)) {
      // block-in weights: W_down rows, then the shared gate and up rows interleaved (row
      // d + 2i gate i, d + 2i + 1 up i) so a SwiGLU pair sits in adjacent accumulator lanes;
      // block-out weights: each row c is W_up[c][:] followed by W_shared_down[c][:]
      const size_t d = c.latent, Is = c.shared_inter, Kw = block_width(c), rb = H * 2;
      if (cudaMemcpy(W.w_in, lh->proj_down, d * rb, cudaMemcpyHostToDevice) != cudaSuccess ||
          (Is && (cudaMemcpy2D(W.w_in + d * H, 2 * rb, lh->shared_gu, rb, rb, Is, cudaMemcpyHostToDevice) !=
                      cudaSuccess ||
                  cudaMemcpy2D(W.w_in + (d + 1) * H, 2 * rb, lh->shared_gu + Is * H, rb, rb, Is,
                               cudaMemcpyHostToDevice) != cudaSuccess)) ||
          cudaMemcpy2D(W.w_out, Kw * 2, lh->proj_up, d * 2, d * 2, H, cudaMemcpyHostToDevice) != cudaSuccess ||
          (Is && cudaMemcpy2D(W.w_out + d, Kw * 2, lh->shared_dn, Is * 2, Is * 2, H, cudaMemcpyHostToDevice) !=
                     cudaSuccess) ||
          !make_tmap_16(&ctx->tmap_win, W.w_in, (uint64_t)block_in_rows(c), H, 128, true) ||
          !make_tmap_16(&ctx->tmap_wout, W.w_out, H, Kw, 128, true)) {
        st = MOE_ERR_CUDA;
        break;
      }
    }
    for (size_t e = 0; e < El && st == MOE_OK; ++e) {
      if (cudaStreamSynchronize(s) != cudaSuccess) {  // the staging buffer is free again
        st = MOE_ERR_CUDA;
        break;
      }
      uint8_t* sc = staging;
      uint8_t* ss = staging + gu_cb;
      uint8_t* dc = ss + gu_sb;
      uint8_t* ds = dc + dn_cb;
      if (cudaMemcpyAsync(sc, lh->gu_codes[e], gu_cb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
          cudaMemcpyAsync(ss, lh->gu_scales[e], gu_sb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
          cudaMemcpyAsync(dc, lh->dn_codes[e], dn_cb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
          cudaMemcpyAsync(ds, lh->dn_scales[e], dn_sb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
          launch_repack_tc(ctx->sh, (int)e, sc, ss, dc, ds, W.gu_tc, W.dn_tc, s) != cudaSuccess ||
          launch_scale_max(ctx->sh, (int)e, ss, ds, W.scale_max, s) != cudaSuccess) {
        st = MOE_ERR_CUDA;
        break;
      }
    }
    if (st == MOE_OK && launch_norms(ctx->sh, W.scale_max, W.gu_norm, W.dn_norm, W.norm_exp, s) != cudaSuccess)
      st = MOE_ERR_CUDA;
    if (st == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) st = MOE_ERR_CUDA;
  } while (0);
  cudaStreamDestroy(s);
  cudaFree(staging);
  if (st == MOE_OK) ctx->loaded = true;
  return st;
}

int moe_forward(moe_ctx* ctx, void* stream, const void* x, void* out, int32_t T) {
  int st = check_forward_args(ctx, x, out, T, ctx ? ctx->cfg.hidden : 0);
  if (st != MOE_OK || T == 0) return st;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  StageTimer tm(ctx, s);
  const TcPlan pl = tc_plan(ctx->sh, T, ctx->sm_count);
  PdlScope pdl(!pl.prefill);
  st = run_route(ctx, s, (const uint16_t*)x, T, &tm, pl.nmax, pl.cold_rows);
  if (st != MOE_OK) return st;
  if (!is_block(ctx->cfg))
    return run_experts(ctx, s, (const uint16_t*)x, (uint16_t*)out, ctx->cfg.hidden, T, pl, &tm, ctx->ws.idx,
                       ctx->ws.w);
  st = run_block_in(ctx, s, (const uint16_t*)x, T, &tm);
  if (st != MOE_OK) return st;
  st = run_experts(ctx, s, ctx->ws.lat, ctx->ws.hcat, block_width(ctx->cfg), T, pl, &tm, ctx->ws.idx, ctx->ws.w);
  if (st != MOE_OK) return st;
  return run_block_out(ctx, s, (uint16_t*)out, T, &tm);
}

int moe_forward_routed(moe_ctx* ctx, void* stream, const void* x, const int32_t* idx, const float* w, void* out,
                       int32_t T, int32_t* served) {
  int st = check_forward_args(ctx, x, out, T, ctx ? ctx->sh.D : 0);
  if (st != MOE_OK || T == 0) return st;
  if (!idx || !w || ((uintptr_t)idx & 3u) || ((uintptr_t)w & 3u) || ((uintptr_t)served & 3u))
    return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  StageTimer tm(ctx, s);
  const TcPlan pl = tc_plan(ctx->sh, T, ctx->sm_count);
  PdlScope pdl(!pl.prefill);
  tm.begin(kStagePermute);
  if (launch_permute(ctx->sh, ctx->ws, idx, T, s, pl.nmax, served, pl.cold_rows) != cudaSuccess) return MOE_ERR_CUDA;
  tm.end(kStagePermute);
  ctx->launches += 3;
  return run_experts(ctx, s, (const uint16_t*)x, (uint16_t*)out, ctx->sh.D, T, pl, &tm, idx, w);
}

int moe_forward_host(moe_ctx* ctx, void* stream, const void* x_host, void* out_host, int32_t T) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > ctx->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (!ctx->loaded) return MOE_ERR_NOT_LOADED;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)T * ctx->cfg.hidden * 2;
  if (cudaMemcpyAsync(ctx->ws.x_stage, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  int st = moe_forward(ctx, stream, ctx->ws.x_stage, ctx->ws.out_stage, T);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(out_host, ctx->ws.out_stage, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_destroy(moe_ctx* ctx) {
  if (!ctx) return MOE_OK;
  DeviceGuard g(ctx->device);
  for (cudaEvent_t ev : ctx->prof_ev) cudaEventDestroy(ev);
  if (ctx->weights_mem) cudaFree(ctx->weights_mem);
  if (ctx->ws_mem) cudaFree(ctx->ws_mem);
  delete ctx;
  return MOE_OK;
}

int moe_get_error(moe_ctx* ctx, uint32_t* bits) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  uint32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, ctx->ws.err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ctx->ws.err, 0, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits) *bits = v;
  return v ? MOE_ERR_DEVICE_FLAG : MOE_OK;
}

static int copy_route_outputs(moe_ctx* ctx, cudaStream_t s, int T, float* logits, int32_t* idx, float* w,
                              int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv) {
  const size_t E = ctx->cfg.n_experts, El = ctx->sh.El, k = ctx->cfg.top_k;
  struct Item {
    void* dst;
    const void* src;
    size_t bytes;
  } items[] = {{logits, ctx->ws.logits, (size_t)T * E * 4}, {idx, ctx->ws.idx, (size_t)T * k * 4},
               {w, ctx->ws.w, (size_t)T * k * 4},           {offsets, ctx->ws.offsets, (El + 1) * 4},
               {perm, ctx->ws.perm, (size_t)T * k * 4},     {slot, ctx->ws.slot, (size_t)T * k * 4},
               {inv, ctx->ws.inv, (size_t)T * k * 4}};
  for (const Item& it : items)
    if (it.dst && cudaMemcpyAsync(it.dst, it.src, it.bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_debug_route(moe_ctx* ctx, void* stream, const void* x, int32_t T, float* logits, int32_t* idx, float* w,
                    int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv) {
  if (!ctx || !x || T <= 0 || T > ctx->cfg.max_tokens || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (!ctx->loaded) return MOE_ERR_NOT_LOADED;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  int st = run_route(ctx, s, (const uint16_t*)x, T, nullptr, 0);
  if (st != MOE_OK) return st;
  return copy_route_outputs(ctx, s, T, logits, idx, w, offsets, perm, slot, inv);
}

int moe_debug_select(moe_ctx* ctx, void* stream, const float* logits, int32_t T, int32_t* idx, float* w,
                     int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv) {
  if (!ctx || !logits || T <= 0 || T > ctx->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_select(ctx->sh, logits, ctx->ws.idx, ctx->ws.w, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_permute(ctx->sh, ctx->ws, ctx->ws.idx, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  ctx->launches += 4;
  return copy_route_outputs(ctx, s, T, nullptr, idx, w, offsets, perm, slot, inv);
}

int moe_debug_experts(moe_ctx* ctx, void* stream, const void* x, int32_t T, float* h, float* y, void* lat) {
  if (!ctx || !x || T <= 0 || T > ctx->cfg.max_tokens || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (!ctx->loaded) return MOE_ERR_NOT_LOADED;
  DeviceGuard g(ctx->device);
  cudaStream_t s = (cudaStream_t)stream;
  const TcPlan pl = tc_plan(ctx->sh, T, ctx->sm_count);
  int st = run_route(ctx, s, (const uint16_t*)x, T, nullptr, pl.nmax, pl.cold_rows);
  if (st != MOE_OK) return st;
  const uint16_t* xin = (const uint16_t*)x;
  if (is_block(ctx->cfg)) {
    st = run_block_in(ctx, s, xin, T, nullptr);
    if (st != MOE_OK) return st;
    xin = ctx->ws.lat;
    if (lat && cudaMemcpyAsync(lat, ctx->ws.lat, (size_t)T * ctx->cfg.latent * 2, cudaMemcpyDeviceToDevice, s) !=
                   cudaSuccess)
      return MOE_ERR_CUDA;
  }
  st = run_experts(ctx, s, xin, ctx->ws.out_stage, ctx->sh.D, T, pl, nullptr, ctx->ws.idx, ctx->ws.w);
  if (st != MOE_OK) return st;
  return launch_debug_hy(ctx->sh, ctx->L, ctx->ws, pl, T, h, y, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_debug_pdl_copy(void* stream, const void* src, void* dst, int64_t bytes) {
  if (!src || !dst || bytes < 0 || (bytes & 15) || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
  const char* sa = (const char*)src;
  const char* da = (const char*)dst;
  if (sa < da + bytes && da < sa + bytes) return MOE_ERR_INVALID_ARG;
  if (bytes == 0) return MOE_OK;
  const int64_t n16 = bytes / 16;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(1024, (n16 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const uint4* s4 = (const uint4*)src;
  uint4* d4 = (uint4*)dst;
  return cudaLaunchKernelEx(&cfg, pdl_consumer_copy_kernel, s4, d4, n16) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_profile_stages(void) { return kNumStages; }

const char* moe_profile_stage_name(int i) { return (i >= 0 && i < kNumStages) ? kStageNames[i] : ""; }

int moe_profile_begin(moe_ctx* ctx, int32_t max_calls) {
  if (!ctx || max_calls < 0) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  for (cudaEvent_t ev : ctx->prof_ev) cudaEventDestroy(ev);
  ctx->prof_ev.assign((size_t)max_calls * kNumStages * 2, nullptr);
  ctx->prof_rec.assign((size_t)max_calls * kNumStages, 0);
  for (auto& ev : ctx->prof_ev)
    if (cudaEventCreate(&ev) != cudaSuccess) return MOE_ERR_CUDA;
  ctx->prof_max = max_calls;
  ctx->prof_calls = 0;
  return MOE_OK;
}

int moe_profile_end(moe_ctx* ctx, float* ms, int32_t* launches, int32_t n) {
  if (!ctx || n < 0 || n > kNumStages) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  for (int i = 0; i < n; ++i) {
    if (ms) ms[i] = 0.f;
    if (launches) launches[i] = 0;
  }
  for (int c = 0; c < ctx->prof_calls; ++c)
    for (int i = 0; i < n; ++i) {
      if (!ctx->prof_rec[(size_t)c * kNumStages + i]) continue;
      cudaEvent_t a = ctx->prof_ev[((size_t)c * kNumStages + i) * 2];
      cudaEvent_t b = ctx->prof_ev[((size_t)c * kNumStages + i) * 2 + 1];
      if (cudaEventSynchronize(b) != cudaSuccess) return MOE_ERR_CUDA;
      float t = 0.f;
      if (cudaEventElapsedTime(&t, a, b) != cudaSuccess) {
        // a captured call whose graph was never replayed leaves its events unrecorded:
        // not an error of the device, the call is just not counted
        cudaGetLastError();
        continue;
      }
      if (ms) ms[i] += t;
      if (launches) launches[i] += 1;
    }
  ctx->prof_max = 0;
  ctx->prof_calls = 0;
  return MOE_OK;
}

int moe_plan(const moe_config* cfg, int32_t sm_count, int32_t T, int64_t* plan) {
  const int st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!plan || sm_count < 1 || T < 1 || T > cfg->max_tokens) return MOE_ERR_INVALID_ARG;
  const Shape sh = shape_of(*cfg);
  const TcPlan pl = tc_plan(sh, T, sm_count);
  const RouterTcPlan rp = router_tc_plan(sh, T, sm_count);
  Workspace w;
  const size_t bytes = workspace_layout(*cfg, sm_count, &w, nullptr);
  plan[0] = pl.prefill ? 1 : 0;
  plan[1] = pl.nmax;
  plan[2] = pl.S1;
  plan[3] = pl.S2;
  plan[4] = pl.grid;
  plan[5] = rp.S;
  plan[6] = rp.grid;
  plan[7] = route_small_ok(sh, T, rp.S) ? 1 : 0;
  plan[8] = w.chunk_cap;
  plan[9] = (int64_t)bytes;
  plan[10] = pl.cold_rows;
  return MOE_OK;
}

int64_t moe_launch_count(const moe_ctx* ctx) { return ctx ? ctx->launches : 0; }

int64_t moe_device_bytes(const moe_ctx* ctx) {
  if (!ctx) return 0;
  return (int64_t)(ctx->weights_bytes + ctx->ws_bytes);
}

}  // extern "C"
