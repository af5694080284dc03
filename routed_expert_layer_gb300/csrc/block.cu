// The two dense steps around the routed experts of a LatentMoE block, on the tensor cores
// through launch_dense_tc (router_tc.cu), and their finalize kernels.
//
// "Kimi K3 optimization on GB300, Part I", section "Routed-down projection: column sharding
// and latent assembly": every MoE block projects the 7,168-wide hidden state into a
// 3,584-wide routed latent (a [3584, 7168] BF16 weight) and back after the experts
// (section "Routed-up projection", same size). "Serving Kimi K3 End to End", section 3.3:
// the 2 shared experts, which every token uses; the first page's shape-aware projection
// routing section: the NVFP4 target's shared-expert projections are unquantized.
//
// On one GPU the block is two GEMMs around the expert stage:
//   block-in   A = [W_down ; W_shared_gate/up, rows interleaved] (d + 2 Is rows), B = x:
//              the routed latent (bf16, the experts' input) and the shared SwiGLU rows
//              (bf16, written next to where the combine leaves the routed latent);
//   block-out  A = [W_up | W_shared_down] (H rows, K = d + Is), B = [routed latent | shared
//              SwiGLU]: the up projection and the shared experts' down projection are
//              summed in the fp32 accumulator, then rounded once to bf16.
// (The sharded design on the pages injects the routed up-projection block into the shared
// experts' partial before one all-reduce; here the same sum is one contraction.)
#include "moe_internal.cuh"

namespace moe {

// Thread per (token, output column) of [lat | shared SwiGLU]; K splits added in ascending
// order.
__global__ void block_in_finalize_kernel(const float* __restrict__ part, int S, int T, int M, int d, int Is,
                                         uint16_t* __restrict__ lat, uint16_t* __restrict__ hcat, int ldh) {
  pdl_entry();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int W = d + Is;
  if (i >= (size_t)T * W) return;
  const int t = (int)(i / W), c = (int)(i % W);
  const size_t slice = (size_t)T * M;
  const float* row = part + (size_t)t * M;
  if (c < d) {
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += row[(size_t)s * slice + c];
    lat[(size_t)t * d + c] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    const int j = d + 2 * (c - d);
    float g = 0.f, u = 0.f;
    for (int s = 0; s < S; ++s) {
      const float2 v = *reinterpret_cast<const float2*>(row + (size_t)s * slice + j);
      g += v.x;
      u += v.y;
    }
    const float h = g / (1.f + expf(-g)) * u;
    hcat[(size_t)t * ldh + c] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
  }
}

__global__ void block_out_finalize_kernel(const float* __restrict__ part, int S, int T, int H,
                                          uint16_t* __restrict__ out) {
  pdl_entry();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t n = (size_t)T * H;
  if (i >= n) return;
  float v = 0.f;
  for (int s = 0; s < S; ++s) v += part[(size_t)s * n + i];
  out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

cudaError_t launch_block_in_finalize(const float* part, int S, int T, int d, int Is, uint16_t* lat, uint16_t* hcat,
                                     int ldh, cudaStream_t s) {
  const size_t n = (size_t)T * (d + Is);
  return launch_pdl(block_in_finalize_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, part, S, T,
                    d + 2 * Is, d, Is, lat, hcat, ldh);
}

cudaError_t launch_block_out_finalize(const float* part, int S, int T, int H, uint16_t* out, cudaStream_t s) {
  const size_t n = (size_t)T * H;
  return launch_pdl(block_out_finalize_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, part, S, T, H,
                    out);
}

}  // namespace moe
