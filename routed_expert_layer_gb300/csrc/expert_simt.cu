// Expert FFN on NVFP4 weights, streaming variant (S4 gate/up + SwiGLU, S5 down),
// and the weighted combine (S6).
//
// Every touched expert's bucket of routed rows is served by one pass over that
// expert's weights (SemiAnalysis essay, section 4: one expert weight load serves
// every activation in its bucket; section 15: the arithmetic intensity of an expert
// grows with the rows n assigned to it). Three matrices per expert and E2M1 values
// two per byte: "Serving Kimi-K3 ... with 8xB300 GPUs", section "The model, as the
// serving system sees it". An FP8 scale per 16 values plus a per-expert global scale:
// "Kimi-K3 NVFP4 station eight sparks", section "What has to be built".
//
// Layout (row tiles of 32, see DeviceLayer): lane r of a warp owns tile row r, and a
// warp-wide 16-byte load per lane reads 512 contiguous bytes = one 32-element K
// chunk of 32 rows. The 8 warps of a CTA split K; partial sums are reduced in shared
// memory in a fixed order, so results are deterministic.
#include "moe_internal.cuh"

namespace moe {

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Eight E2M1 codes (one 32-bit word, element i in bits 4i..4i+3) -> eight floats.
// The hardware conversion maps the low nibble of a byte to the low half of the f16x2.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t word, float* out) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(word));
  const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
  const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
  const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&h3));
  out[0] = f0.x; out[1] = f0.y; out[2] = f1.x; out[3] = f1.y;
  out[4] = f2.x; out[5] = f2.y; out[6] = f3.x; out[7] = f3.y;
}

// Two E4M3 scales (low byte -> first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two_bytes) {
  uint32_t h;
  const uint16_t b = (uint16_t)(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// One 32-element K chunk of one row against NT token rows held in shared memory.
template <int NT>
__device__ __forceinline__ void chunk_dot(const uint4 cw, const float2 s, const float* __restrict__ xs, int ldx,
                                          int k0, float* acc) {
  float wv[32];
  e2m1x8_to_f32(cw.x, wv + 0);
  e2m1x8_to_f32(cw.y, wv + 8);
  e2m1x8_to_f32(cw.z, wv + 16);
  e2m1x8_to_f32(cw.w, wv + 24);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float4* xr = reinterpret_cast<const float4*>(xs + t * ldx + k0);
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 xv = xr[q];
      p0 = fmaf(wv[4 * q + 0], xv.x, p0);
      p0 = fmaf(wv[4 * q + 1], xv.y, p0);
      p0 = fmaf(wv[4 * q + 2], xv.z, p0);
      p0 = fmaf(wv[4 * q + 3], xv.w, p0);
    }
#pragma unroll
    for (int q = 4; q < 8; ++q) {
      const float4 xv = xr[q];
      p1 = fmaf(wv[4 * q + 0], xv.x, p1);
      p1 = fmaf(wv[4 * q + 1], xv.y, p1);
      p1 = fmaf(wv[4 * q + 2], xv.z, p1);
      p1 = fmaf(wv[4 * q + 3], xv.w, p1);
    }
    acc[t] = fmaf(s.x, p0, acc[t]);
    acc[t] = fmaf(s.y, p1, acc[t]);
  }
}

// Warp-level K loop over this warp's chunks (kc = warp, warp + 8, ...).
template <int NT>
__device__ __forceinline__ void tile_k_loop(const uint4* __restrict__ codes, const uint32_t* __restrict__ scales,
                                            const float* __restrict__ xs, int ldx, int nkc, int warp, int lane,
                                            float* acc) {
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  int kc = warp;
  for (; kc + kSimtWarps < nkc; kc += 2 * kSimtWarps) {
    const uint4 c0 = ldg_stream(codes + (size_t)kc * 32 + lane);
    const uint4 c1 = ldg_stream(codes + (size_t)(kc + kSimtWarps) * 32 + lane);
    const uint32_t w0 = ldg_stream32(scales + (size_t)(kc >> 1) * 32 + lane);
    const uint32_t w1 = ldg_stream32(scales + (size_t)((kc + kSimtWarps) >> 1) * 32 + lane);
    chunk_dot<NT>(c0, e4m3x2_to_f32((kc & 1) ? (w0 >> 16) : w0), xs, ldx, kc * 32, acc);
    chunk_dot<NT>(c1, e4m3x2_to_f32(((kc + kSimtWarps) & 1) ? (w1 >> 16) : w1), xs, ldx, (kc + kSimtWarps) * 32, acc);
  }
  for (; kc < nkc; kc += kSimtWarps) {
    const uint4 c0 = ldg_stream(codes + (size_t)kc * 32 + lane);
    const uint32_t w0 = ldg_stream32(scales + (size_t)(kc >> 1) * 32 + lane);
    chunk_dot<NT>(c0, e4m3x2_to_f32((kc & 1) ? (w0 >> 16) : w0), xs, ldx, kc * 32, acc);
  }
}

// S4: grid (I/16 row tiles, touched-expert slots), 256 threads. For each pass of up
// to kSimtNT routed rows: x rows -> fp32 in shared memory, the 32 tile rows' dot
// products, a fixed-order reduction over the 8 warps, then h = silu(g) * u.
__global__ void __launch_bounds__(256) gateup_simt_kernel(DeviceLayer L, Shape sh, const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ active,
                                                          const int32_t* __restrict__ meta,
                                                          const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ perm, float* __restrict__ h) {
  extern __shared__ float smem[];
  const int a = blockIdx.y;
  if (a >= meta[0]) return;
  const int e = active[a];
  const int rt = blockIdx.x;
  const int H = sh.H, I = sh.I;
  const int p0 = offsets[e];
  const int n = offsets[e + 1] - p0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkc = H / 32;
  const uint4* codes =
      reinterpret_cast<const uint4*>(L.gu_codes + ((size_t)e * (I / 16) + rt) * (size_t)(H / 32) * 512);
  const uint32_t* scales =
      reinterpret_cast<const uint32_t*>(L.gu_scales + ((size_t)e * (I / 16) + rt) * (size_t)(H / 64) * 128);
  float* xs = smem;                      // [kSimtNT][H]
  float* red = smem + kSimtNT * H;       // [8 warps][32 rows][kSimtNT]
  const float gg = L.gu_global[2 * e], gu = L.gu_global[2 * e + 1];
  for (int g0 = 0; g0 < n; g0 += kSimtNT) {
    const int nt = min(kSimtNT, n - g0);
    for (int i = threadIdx.x; i < kSimtNT * (H / 2); i += 256) {
      const int r = i / (H / 2), c2 = i % (H / 2);
      uint32_t v = 0;
      if (r < nt) v = reinterpret_cast<const uint32_t*>(x + (size_t)perm[p0 + g0 + r] * H)[c2];
      xs[r * H + 2 * c2] = __uint_as_float(v << 16);
      xs[r * H + 2 * c2 + 1] = __uint_as_float(v & 0xFFFF0000u);
    }
    __syncthreads();
    float acc[kSimtNT];
    if (nt == 1) {
      tile_k_loop<1>(codes, scales, xs, H, nkc, warp, lane, acc);
    } else if (nt == 2) {
      tile_k_loop<2>(codes, scales, xs, H, nkc, warp, lane, acc);
    } else {
      tile_k_loop<kSimtNT>(codes, scales, xs, H, nkc, warp, lane, acc);
    }
#pragma unroll
    for (int t = 0; t < kSimtNT; ++t) red[(warp * 32 + lane) * kSimtNT + t] = (t < nt) ? acc[t] : 0.f;
    __syncthreads();
    if (threadIdx.x < 16 * kSimtNT) {
      const int r = threadIdx.x / kSimtNT, t = threadIdx.x % kSimtNT;
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kSimtWarps; ++w8) {
        g += red[(w8 * 32 + r) * kSimtNT + t];
        u += red[(w8 * 32 + r + 16) * kSimtNT + t];
      }
      if (t < nt) {
        g *= gg;
        u *= gu;
        h[(size_t)(p0 + g0 + t) * I + rt * 16 + r] = g / (1.f + expf(-g)) * u;
      }
    }
    __syncthreads();
  }
}

// S5: grid (H/32 row tiles, touched-expert slots). y[p][c] = dn_global * (W_d h[p])[c]
// (unweighted; the gate weight is applied in the combine).
__global__ void __launch_bounds__(256) down_simt_kernel(DeviceLayer L, Shape sh, const int32_t* __restrict__ active,
                                                        const int32_t* __restrict__ meta,
                                                        const int32_t* __restrict__ offsets,
                                                        const float* __restrict__ h, float* __restrict__ y) {
  extern __shared__ float smem[];
  const int a = blockIdx.y;
  if (a >= meta[0]) return;
  const int e = active[a];
  const int rt = blockIdx.x;
  const int H = sh.H, I = sh.I;
  const int p0 = offsets[e];
  const int n = offsets[e + 1] - p0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkc = I / 32;
  const uint4* codes =
      reinterpret_cast<const uint4*>(L.dn_codes + ((size_t)e * (H / 32) + rt) * (size_t)(I / 32) * 512);
  const uint32_t* scales =
      reinterpret_cast<const uint32_t*>(L.dn_scales + ((size_t)e * (H / 32) + rt) * (size_t)(I / 64) * 128);
  float* hs = smem;                 // [kSimtNT][I]
  float* red = smem + kSimtNT * I;  // [8][32][kSimtNT]
  const float gd = L.dn_global[e];
  for (int g0 = 0; g0 < n; g0 += kSimtNT) {
    const int nt = min(kSimtNT, n - g0);
    for (int i = threadIdx.x; i < kSimtNT * I; i += 256) {
      const int r = i / I;
      hs[i] = (r < nt) ? h[(size_t)(p0 + g0 + r) * I + (i % I)] : 0.f;
    }
    __syncthreads();
    float acc[kSimtNT];
    if (nt == 1) {
      tile_k_loop<1>(codes, scales, hs, I, nkc, warp, lane, acc);
    } else if (nt == 2) {
      tile_k_loop<2>(codes, scales, hs, I, nkc, warp, lane, acc);
    } else {
      tile_k_loop<kSimtNT>(codes, scales, hs, I, nkc, warp, lane, acc);
    }
#pragma unroll
    for (int t = 0; t < kSimtNT; ++t) red[(warp * 32 + lane) * kSimtNT + t] = (t < nt) ? acc[t] : 0.f;
    __syncthreads();
    if (threadIdx.x < 32 * kSimtNT) {
      const int r = threadIdx.x / kSimtNT, t = threadIdx.x % kSimtNT;
      float v = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kSimtWarps; ++w8) v += red[(w8 * 32 + r) * kSimtNT + t];
      if (t < nt) y[(size_t)(p0 + g0 + t) * H + rt * 32 + r] = v * gd;
    }
    __syncthreads();
  }
}

cudaError_t simt_configure(const Shape& sh) {
  const size_t s1 = (size_t)kSimtNT * sh.H * sizeof(float) + (size_t)kSimtWarps * 32 * kSimtNT * sizeof(float);
  const size_t s2 = (size_t)kSimtNT * sh.I * sizeof(float) + (size_t)kSimtWarps * 32 * kSimtNT * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(gateup_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
}

cudaError_t launch_gateup_simt(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const uint16_t* x, int T,
                               cudaStream_t s) {
  const int slots = min(sh.E, T * sh.k);
  const size_t smem = (size_t)kSimtNT * sh.H * sizeof(float) + (size_t)kSimtWarps * 32 * kSimtNT * sizeof(float);
  dim3 grid(sh.I / 16, slots);
  gateup_simt_kernel<<<grid, 256, smem, s>>>(L, sh, x, ws.active, ws.meta, ws.offsets, ws.perm, ws.h);
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, cudaStream_t s) {
  const int slots = min(sh.E, T * sh.k);
  const size_t smem = (size_t)kSimtNT * sh.I * sizeof(float) + (size_t)kSimtWarps * 32 * kSimtNT * sizeof(float);
  dim3 grid(sh.H / 32, slots);
  down_simt_kernel<<<grid, 256, smem, s>>>(L, sh, ws.active, ws.meta, ws.offsets, ws.h, ws.y);
  return cudaGetLastError();
}

// ---- S6 combine -----------------------------------------------------------------------------

// out[t][c] = bf16_rne( sum over j ascending of w[t][j] * y[inv[t*k + j]][c] ), fp32 sum.
__global__ void combine_kernel(const float* __restrict__ y, const float* __restrict__ w,
                               const int32_t* __restrict__ inv, uint16_t* __restrict__ out, int H, int k) {
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int p = inv[(size_t)t * k + j];
    if (p < 0) continue;
    const float wj = w[(size_t)t * k + j];
    const float4 v = reinterpret_cast<const float4*>(y + (size_t)p * H)[c4];
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + (size_t)t * H)[c4] = packed;
}

cudaError_t launch_combine(const Shape& sh, const Workspace& ws, uint16_t* out, int T, cudaStream_t s) {
  dim3 grid((sh.H / 4 + 127) / 128, T);
  combine_kernel<<<grid, 128, 0, s>>>(ws.y, ws.w, ws.inv, out, sh.H, sh.k);
  return cudaGetLastError();
}

// ---- load-time repack -----------------------------------------------------------------------

__global__ void repack_gu_kernel(const uint8_t* __restrict__ raw_c, const uint8_t* __restrict__ raw_s,
                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int H, int I) {
  const size_t nc = (size_t)(I / 16) * (H / 32) * 32;
  const size_t ns = (size_t)(I / 16) * (H / 64) * 32;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nc) {
    const int r = (int)(i % 32);
    const int kc = (int)((i / 32) % (H / 32));
    const int rt = (int)(i / (32 * (size_t)(H / 32)));
    const int R = (r < 16) ? rt * 16 + r : I + rt * 16 + (r - 16);
    reinterpret_cast<uint4*>(codes)[i] = *reinterpret_cast<const uint4*>(raw_c + (size_t)R * (H / 2) + kc * 16);
  }
  if (i < ns) {
    const int r = (int)(i % 32);
    const int kc2 = (int)((i / 32) % (H / 64));
    const int rt = (int)(i / (32 * (size_t)(H / 64)));
    const int R = (r < 16) ? rt * 16 + r : I + rt * 16 + (r - 16);
    reinterpret_cast<uint32_t*>(scales)[i] = *reinterpret_cast<const uint32_t*>(raw_s + (size_t)R * (H / 16) + kc2 * 4);
  }
}

__global__ void repack_dn_kernel(const uint8_t* __restrict__ raw_c, const uint8_t* __restrict__ raw_s,
                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int H, int I) {
  const size_t nc = (size_t)(H / 32) * (I / 32) * 32;
  const size_t ns = (size_t)(H / 32) * (I / 64) * 32;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nc) {
    const int r = (int)(i % 32);
    const int kc = (int)((i / 32) % (I / 32));
    const int rt = (int)(i / (32 * (size_t)(I / 32)));
    const int R = rt * 32 + r;
    reinterpret_cast<uint4*>(codes)[i] = *reinterpret_cast<const uint4*>(raw_c + (size_t)R * (I / 2) + kc * 16);
  }
  if (i < ns) {
    const int r = (int)(i % 32);
    const int kc2 = (int)((i / 32) % (I / 64));
    const int rt = (int)(i / (32 * (size_t)(I / 64)));
    const int R = rt * 32 + r;
    reinterpret_cast<uint32_t*>(scales)[i] = *reinterpret_cast<const uint32_t*>(raw_s + (size_t)R * (I / 16) + kc2 * 4);
  }
}

cudaError_t launch_repack_expert(const Shape& sh, int e, const uint8_t* gu_codes_raw, const uint8_t* gu_scales_raw,
                                 const uint8_t* dn_codes_raw, const uint8_t* dn_scales_raw, uint8_t* gu_codes,
                                 uint8_t* gu_scales, uint8_t* dn_codes, uint8_t* dn_scales, cudaStream_t s) {
  const int H = sh.H, I = sh.I;
  const size_t gu_c = (size_t)2 * I * (H / 2), gu_s = (size_t)2 * I * (H / 16);
  const size_t dn_c = (size_t)H * (I / 2), dn_s = (size_t)H * (I / 16);
  const size_t n1 = (size_t)(I / 16) * (H / 32) * 32;
  repack_gu_kernel<<<(unsigned)((n1 + 255) / 256), 256, 0, s>>>(gu_codes_raw, gu_scales_raw, gu_codes + e * gu_c,
                                                                gu_scales + e * gu_s, H, I);
  const size_t n2 = (size_t)(H / 32) * (I / 32) * 32;
  repack_dn_kernel<<<(unsigned)((n2 + 255) / 256), 256, 0, s>>>(dn_codes_raw, dn_scales_raw, dn_codes + e * dn_c,
                                                                dn_scales + e * dn_s, H, I);
  return cudaGetLastError();
}

}  // namespace moe
