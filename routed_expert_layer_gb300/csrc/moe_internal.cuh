// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

// Device error word bits (also documented in moe_get_error).
constexpr uint32_t kErrExpertRange = 1u;
constexpr uint32_t kErrCountOverflow = 2u;

// Profiled stages of one forward.
enum Stage { kStageRouter = 0, kStageSelect, kStagePermute, kStageGateUp, kStageDown, kStageCombine, kNumStages };

// Tokens per pass of the SIMT expert kernels and the SIMT tile shapes.
constexpr int kSimtNT = 4;        // token rows held in shared memory per pass
constexpr int kSimtWarps = 8;     // warps per CTA, splitting K
constexpr int kRouterTT = 16;     // router tile: tokens
constexpr int kRouterTE = 128;    // router tile: experts (one per thread)

// Repacked weight layout for the streaming kernels ("row tiles of 32"):
//   gate/up: tile rt covers gate features 16rt..16rt+15 (tile rows 0..15) and the
//   up features with the same indices (tile rows 16..31); for every 32-element K
//   chunk the 32 rows' 16-byte code chunks are contiguous (512 B), and for every
//   64-element K chunk the 32 rows' 4 scale bytes are contiguous (128 B).
//   down: tile rt covers output rows 32rt..32rt+31, same chunking along K = I.
struct DeviceLayer {
  const float* router_w = nullptr;    // [H][E]
  const float* router_bias = nullptr; // [E] (zeros when the caller gave none)
  const uint8_t* gu_codes = nullptr;  // [E][I/16][H/32][32][16]
  const uint8_t* gu_scales = nullptr; // [E][I/16][H/64][32][4]
  const float* gu_global = nullptr;   // [E][2]
  const uint8_t* dn_codes = nullptr;  // [E][H/32][I/32][32][16]
  const uint8_t* dn_scales = nullptr; // [E][H/32][I/64][32][4]
  const float* dn_global = nullptr;   // [E]
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
  int32_t* meta = nullptr;        // [4]: [0] number of touched experts, [1] max rows per expert
  int32_t* perm = nullptr;        // [T*k]
  int32_t* slot = nullptr;        // [T*k]
  int32_t* inv = nullptr;         // [T*k]
  float* h = nullptr;             // [T*k][I]
  float* y = nullptr;             // [T*k][H]
  uint16_t* x_stage = nullptr;    // [T][H] for moe_forward_host
  uint16_t* out_stage = nullptr;  // [T][H]
  uint32_t* err = nullptr;        // device error word
};

struct Shape {
  int H, I, E, k;
};

// ---- launchers (each enqueues its kernels on `s`) ----------------------------------

// Router split count for T tokens and the partial buffer size it needs.
int router_splits(const Shape& sh, int T, int sm_count);
size_t router_part_elems(const Shape& sh, int T_max, int sm_count);

cudaError_t launch_router(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const uint16_t* x, int T,
                          int sm_count, cudaStream_t s);
cudaError_t launch_select(const Shape& sh, const float* logits, int32_t* idx, float* w, int T, cudaStream_t s);
cudaError_t launch_permute(const Shape& sh, const Workspace& ws, const int32_t* idx, int T, cudaStream_t s);
cudaError_t launch_gateup_simt(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const uint16_t* x, int T,
                               cudaStream_t s);
cudaError_t launch_down_simt(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, cudaStream_t s);
cudaError_t launch_combine(const Shape& sh, const Workspace& ws, uint16_t* out, int T, cudaStream_t s);

// Load-time repack of one expert from raw (caller layout) device staging buffers.
cudaError_t launch_repack_expert(const Shape& sh, int e, const uint8_t* gu_codes_raw, const uint8_t* gu_scales_raw,
                                 const uint8_t* dn_codes_raw, const uint8_t* dn_scales_raw, uint8_t* gu_codes,
                                 uint8_t* gu_scales, uint8_t* dn_codes, uint8_t* dn_scales, cudaStream_t s);

}  // namespace moe
