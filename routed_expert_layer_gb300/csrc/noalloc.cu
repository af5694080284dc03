// Routing step (router logits, top-k select, stable per-expert permutation) for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a serving engine that reserves its
// whole HBM budget once at start-up and forbids allocation on the request path, a
// plugin or custom-op host that only hands out the buffers it planned, or a decode
// loop that cannot afford the device-wide synchronisation an allocation may cause.
// This entry point needs no context and allocates nothing: its scratch (router
// partial sums, logits, per-chunk masks, counts) lives in one file-scope
// __device__ array that every GPU loading this library holds until the process
// exits. The caller passes the inputs and every output buffer.
//
// Set-up: the first call on a device (that device current) looks up the array's
// device address with cudaGetSymbolAddress and caches it together with the SM
// count; make that first call before any stream capture. The address belongs to the
// device's primary context (the one the CUDA runtime uses); a caller that makes another
// context current on the same device through the driver API is not supported. Every
// call on a device shares the one array and finds the previous call's contents in it;
// the parts that must start at zero are cleared on the call's stream. Two calls whose
// work overlaps on the GPU (different streams, no ordering between them) race on the
// array and corrupt each other's results.
//
// The logits come from the fp32 SIMT router (one product and one fp32 addition per
// element of H, in a fixed order), not from the forward path's three-term tensor-core
// router, so they may differ from moe_forward's in the last bits; two experts whose
// logits are that close may then be ordered differently.
#include <mutex>

#include "moe_internal.cuh"

using namespace moe;

namespace {

constexpr int kMaxTokens = MOE_NOALLOC_MAX_TOKENS;
constexpr int kMaxExperts = MOE_NOALLOC_MAX_EXPERTS;
constexpr size_t kPartWords = MOE_NOALLOC_MAX_PARTIALS;                // router partial sums
constexpr size_t kLogitWords = (size_t)kMaxTokens * kMaxExperts;        // logits
constexpr size_t kChunkWords = (size_t)(kMaxTokens / 32) * kMaxExperts;  // masks / chunk bases
// word offsets inside the array; each region starts on a 256-byte boundary
constexpr size_t kOffPart = 0;
constexpr size_t kOffLogits = kOffPart + kPartWords;
constexpr size_t kOffMasks = kOffLogits + kLogitWords;
constexpr size_t kOffBase = kOffMasks + kChunkWords;
constexpr size_t kOffCounts = kOffBase + kChunkWords;
constexpr size_t kOffActive = kOffCounts + kMaxExperts;
constexpr size_t kOffZeros = kOffActive + kMaxExperts;
constexpr size_t kOffMeta = kOffZeros + kMaxExperts;
constexpr size_t kOffErr = kOffMeta + 64;
constexpr size_t kWords = kOffErr + 64;
static_assert(kPartWords % 64 == 0 && kLogitWords % 64 == 0 && kChunkWords % 64 == 0 && kMaxExperts % 64 == 0,
              "regions must stay 256-byte aligned");

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  std::once_flag once;
  uint32_t* scratch = nullptr;  // device address of g_route_scratch on this device
  int sm_count = 0;
  int status = MOE_OK;
};

DeviceSetup g_setup[kMaxDevices];

}  // namespace

// The scratch. In host code this name is only a host-side stand-in for the symbol;
// kernels get the device address looked up in setup_device().
static __device__ __align__(256) uint32_t g_route_scratch[kWords];

static void setup_device(int dev, DeviceSetup* d) {
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    d->status = MOE_ERR_CUDA;
    return;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    d->status = MOE_ERR_UNSUPPORTED;
    return;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    d->status = MOE_ERR_CUDA;
    return;
  }
  d->scratch = static_cast<uint32_t*>(p);
  d->sm_count = prop.multiProcessorCount;
  d->status = MOE_OK;
}

extern "C" MOE_API int moe_route_noalloc(void* stream, const void* x, const float* router_w, const float* router_bias,
                                         int32_t H, int32_t E, int32_t k, int32_t T, int32_t* idx, float* w,
                                         int32_t* offsets, int32_t* perm, int32_t* slot, int32_t* inv,
                                         uint32_t* err) {
  if (!x || !router_w || !idx || !w || !offsets || !perm || !slot || !inv) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(err) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (H <= 0 || E <= 0 || k <= 0 || T <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED;
  if (T > kMaxTokens || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  DeviceSetup* d = &g_setup[dev];
  std::call_once(d->once, setup_device, dev, d);
  if (d->status != MOE_OK) return d->status;
  Shape sh{H, 0, E, k};
  sh.El = E;  // every expert is routed to (no expert range here)
  sh.D = H;
  if ((size_t)router_splits(sh, T, d->sm_count) * (size_t)T * (size_t)E > kPartWords) return MOE_ERR_UNSUPPORTED;

  uint32_t* base = d->scratch;
  Workspace ws;
  ws.router_part = reinterpret_cast<float*>(base + kOffPart);
  ws.logits = reinterpret_cast<float*>(base + kOffLogits);
  ws.masks = base + kOffMasks;
  ws.chunk_base = reinterpret_cast<int32_t*>(base + kOffBase);
  ws.counts = reinterpret_cast<int32_t*>(base + kOffCounts);
  ws.active = reinterpret_cast<int32_t*>(base + kOffActive);
  ws.meta = reinterpret_cast<int32_t*>(base + kOffMeta);
  ws.err = err ? err : base + kOffErr;
  ws.idx = idx;
  ws.w = w;
  ws.offsets = offsets;
  ws.perm = perm;
  ws.slot = slot;
  ws.inv = inv;
  float* zeros = reinterpret_cast<float*>(base + kOffZeros);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the internal error word (used when the caller passes none) accumulates with OR and a
  // missing bias reads zeros: both start at 0; a caller's error word is the caller's to clear
  if (!err && cudaMemsetAsync(ws.err, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!router_bias && cudaMemsetAsync(zeros, 0, (size_t)E * sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
  DeviceLayer L;
  L.router_w = router_w;
  L.router_bias = router_bias ? router_bias : zeros;
  if (launch_router(sh, L, ws, static_cast<const uint16_t*>(x), T, d->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_select(sh, ws.logits, idx, w, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_permute(sh, ws, idx, T, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
