// Expert FFN on the 5th-generation tensor cores (S4 gate/up + SwiGLU, S5 down, S6 combine).
//
// Every touched expert's bucket of routed rows is one grouped-GEMM problem
// (SemiAnalysis essay, section 4: one expert weight load serves the whole bucket;
// section 15: AI ~ 2nW / (B_W + n B_A + B_O) grows with the bucket size n). The
// weights are NVFP4 ("Kimi-K3 NVFP4 station eight sparks", section "What has to be
// built"): E2M1 codes with an E4M3 scale per 16 values along K and an fp32 scale
// per tensor.
//
// Design (swap-AB, A from tensor memory):
//   D[weight row][token] = sum_k A[row][k] * B[token][k]
//   A = dequantised weights, M = 128 rows per tile. The product e2m1 * e4m3 has at
//       most 6 significant bits and lies in [2^-10, 2688], so it is exact in f16.
//       Dequantisation warps read the codes (staged in shared memory by a bulk TMA
//       copy), convert them with the hardware e2m1x2 -> f16x2 conversion, multiply
//       by the block scale and write the f16 tile straight into tensor memory
//       (tcgen05.st); the MMA reads A from there, so the dequantised weights never
//       occupy shared-memory bandwidth.
//   B = the bucket's activation rows (tokens), f16, K-major, staged by 2D TMA with
//       128-byte swizzle in boxes of 16 rows; N = rows rounded up to 16.
//   D accumulates in fp32 in tensor memory; the epilogue applies the tensor and
//       row scales and either the SwiGLU (gate/up rows are interleaved in the tile)
//       or writes fp32 partial sums of a K split.
// Warp roles: warp 0 issues TMA, warp 1 issues MMAs (one thread), warps 2..9
// dequantise and run the epilogue (warp w may only touch TMEM lanes 32*(w%4)..).
// The kernel is persistent over a device-built list of work items
// (expert, row range, M tile, K split).
#include <cuda.h>

#include <algorithm>
#include <cmath>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kChunkK = 64;          // K elements per pipeline stage (4 MMAs of K=16)
constexpr int kRawBytes = 4608;      // one stage of A: 128 rows x 32 B codes + 128 x 4 B scales
constexpr int kRawSlot = 5120;       // raw slot rounded up to the 1024 B swizzle atom
constexpr int kBoxRows = 16;         // activation rows per TMA box
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kDequantWarps = 8;
constexpr int kThreads = (2 + kDequantWarps) * 32;
constexpr int kAStages = 4;          // A tiles in TMEM, 32 columns each

__host__ __device__ constexpr uint32_t tmem_cols(int nmax) {
  const uint32_t need = kAStages * 32 + nmax;
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

template <int NMAX, int NS>
constexpr size_t gemm_smem_bytes() {
  return 1024 /*alignment slack*/ + (size_t)NS * (kRawSlot + NMAX * 128) + 256 /*barriers*/;
}

__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                  uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  return h;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

}  // namespace

// Grouped GEMM over the work list. See the file comment for the roles.
template <int NMAX, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const TcGemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int kStage = kRawSlot + NMAX * 128;
  constexpr uint32_t kCols = tmem_cols(NMAX);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * kStage);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;
  uint64_t* aempty = afull + kAStages;
  uint64_t* accfull = aempty + kAStages;
  uint64_t* accempty = accfull + 1;
  uint64_t* drain = accempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDequantWarps + 1);
    }
    for (int a = 0; a < kAStages; ++a) {
      mbar_init(&afull[a], kDequantWarps);
      mbar_init(&aempty[a], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, kDequantWarps);
    mbar_init(drain, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t acc_col = kAStages * 32;
  const int n_items = *P.n_items;
  const int kc_per = P.KC / P.S;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const TcItem item = P.items[it];
        const int m = item.ms >> 8, s = item.ms & 0xFF;
        const int nb = (item.n + kBoxRows - 1) / kBoxRows;
        const uint8_t* wsrc = P.w + ((size_t)(item.e * P.M + m) * P.KC + (size_t)s * kc_per) * kRawBytes;
        for (int c = 0; c < kc_per; ++c, ++g) {
          const int st = g % NS;
          if (!mbar_wait(&empty[st], ((g / NS) & 1) ^ 1, P.err)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + (size_t)st * kStage;
          mbar_arrive_expect_tx(&full[st], kRawBytes + nb * kBoxBytes);
          bulk_g2s(sb, wsrc + (size_t)c * kRawBytes, kRawBytes, &full[st]);
          const int kx = (s * kc_per + c) * kChunkK;
          for (int b = 0; b < nb; ++b) tma_2d(sb + kRawSlot + b * kBoxBytes, &tmap_b, kx, item.p0 + b * kBoxRows,
                                              &full[st]);
        }
      }
      if (!ok) {
        s_fail = 1;
        // let copies already issued land before the CTA's shared memory goes away
        for (uint32_t j = (g > (uint32_t)NS ? g - NS : 0); j < g; ++j) mbar_wait(&full[j % NS], (j / NS) & 1, P.err);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      uint32_t g = 0;
      int local = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local) {
        const TcItem item = P.items[it];
        const uint32_t N = (uint32_t)((item.n + 15) / 16) * 16;
        const uint32_t idesc = idesc_f16(128, N);
        if (local > 0) {
          if (!mbar_wait(accempty, (local - 1) & 1, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int c = 0; c < kc_per; ++c, ++g) {
          const int st = g % NS;
          const int as = g % kAStages;
          if (!mbar_wait(&full[st], (g / NS) & 1, P.err) || !mbar_wait(&afull[as], (g / kAStages) & 1, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bsm = smem_u32(smem + (size_t)st * kStage + kRawSlot);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            mma_f16_ts(tmem + acc_col, tmem + as * 32 + kk * 8, desc_sw128(bsm + kk * 32), idesc,
                       (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[st]);
          mma_commit(&aempty[as]);
        }
        if (ok) mma_commit(accfull);
      }
      if (!ok) s_fail = 1;
      // drain: every MMA this thread issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, P.err);
    }
  } else {
    // ---- dequantisation + epilogue ----
    const int dw = warp - 2;
    const int q = warp & 3;        // TMEM lane quarter of this warp
    const int half = dw >> 2;      // which 32-element half of a 64-element chunk (and of N)
    const int r = 32 * q + lane;   // tile row owned by this thread
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    uint32_t g = 0;
    int local = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local) {
      const TcItem item = P.items[it];
      for (int c = 0; c < kc_per; ++c, ++g) {
        const int st = g % NS;
        const int as = g % kAStages;
        if (!mbar_wait(&full[st], (g / NS) & 1, P.err) || !mbar_wait(&aempty[as], ((g / kAStages) & 1) ^ 1, P.err)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + (size_t)st * kStage;
        const uint4 cw = *reinterpret_cast<const uint4*>(raw + (half * 128 + r) * 16);
        const uint16_t sw = *reinterpret_cast<const uint16_t*>(raw + 4096 + r * 4 + half * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        const uint32_t s2 = e4m3x2_to_f16x2(sw);
        const uint32_t sa = prmt(s2, s2, 0x1010u);  // (scale of block 0, same)
        const uint32_t sb = prmt(s2, s2, 0x3232u);  // (scale of block 1, same)
        uint32_t v[16];
        e2m1x8_to_f16x2x4(cw.x, v[0], v[1], v[2], v[3]);
        e2m1x8_to_f16x2x4(cw.y, v[4], v[5], v[6], v[7]);
        e2m1x8_to_f16x2x4(cw.z, v[8], v[9], v[10], v[11]);
        e2m1x8_to_f16x2x4(cw.w, v[12], v[13], v[14], v[15]);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = hmul2(v[i], sa);
#pragma unroll
        for (int i = 8; i < 16; ++i) v[i] = hmul2(v[i], sb);
        __syncwarp();
        tmem_st16(tmem + lane_base + (uint32_t)(as * 32 + half * 16), v);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[as]);
      }
      if (!ok) break;
      // ---- epilogue ----
      if (!mbar_wait(accfull, local & 1, P.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int N = ((item.n + 15) / 16) * 16;
      const int m = item.ms >> 8, s = item.ms & 0xFF;
      const int c_lo = half * (N / 2), c_hi = c_lo + N / 2;
      const float gsc = P.gscale[item.e * P.gstride + (P.gsel ? (r & 1) : 0)] * P.post_scale;
      for (int c0 = c_lo; c0 < c_hi; c0 += 8) {
        uint32_t v[8];
        __syncwarp();
        tmem_ld8(tmem + lane_base + acc_col + (uint32_t)c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          const int p = item.p0 + n;
          const float acc = __uint_as_float(v[i]);
          if (P.mode == kTcModeSwiglu) {
            // rows 2f (gate) and 2f+1 (up) sit in adjacent lanes
            const float other = __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
            const float o_gsc = __shfl_xor_sync(0xFFFFFFFFu, gsc, 1);
            if (n < item.n && (r & 1) == 0) {
              const float rs = P.row_scale[p];
              const float gv = acc * gsc * rs;
              const float uv = other * o_gsc * rs;
              const float hv = gv / (1.f + expf(-gv)) * uv * kHScaleInv;
              const int f = m * 64 + (r >> 1);
              P.h16[(size_t)p * P.I + f] = __half_as_ushort(__float2half_rn(fminf(fmaxf(hv, -65504.f), 65504.f)));
            }
          } else if (n < item.n) {
            const float rs = P.row_scale ? P.row_scale[p] : 1.f;
            P.out[(size_t)s * P.out_slice + (size_t)p * P.ldo + (size_t)m * 128 + r] = acc * gsc * rs;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty);
    }
    if (!ok) s_fail = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kCols);
  }
}

// ---- activation rows in f16 ---------------------------------------------------------------

// Routed row p <- token perm[p], converted to f16 after scaling by 2^sigma so the
// row's largest magnitude lands in [2^13, 2^14): the conversion of bf16 values is
// then exact (f16 has 11 significant bits) down to 2^-28 of the row maximum.
// row_scale[p] = 2^-sigma undoes it in the epilogue. One warp per routed row.
__global__ void gather_x_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                    uint16_t* __restrict__ xg, float* __restrict__ row_scale, int rows, int H) {
  const int p = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)perm[p] * H);
  const int n8 = H / 8;
  uint32_t mx = 0;
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  // bf16 magnitude bits: exponent field in bits 7..14
  int sigma = 0;
  if (mx != 0) {
    const int e = (int)((mx >> 7) & 0xFF) - 127;  // floor(log2(max)) for normal values
    sigma = 13 - e;
    sigma = sigma > 126 ? 126 : (sigma < -126 ? -126 : sigma);
  }
  const float sc = __int_as_float((sigma + 127) << 23);  // exactly 2^sigma
  if (lane == 0) row_scale[p] = __int_as_float((127 - sigma) << 23);
  uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)p * H);
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16) * sc;
      const float hi = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
      const __half2 hh = __floats2half2_rn(lo, hi);
      o[j] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---- work list ---------------------------------------------------------------------------

// One thread per touched expert: its rows are cut into chunks of at most nmax and
// every (chunk, M tile, K split) becomes an item, expert-major so that items
// sharing an activation tile run close together.
__global__ void __launch_bounds__(1024) worklist_kernel(const int32_t* __restrict__ active,
                                                        const int32_t* __restrict__ meta,
                                                        const int32_t* __restrict__ offsets, int nmax, int M1, int S1,
                                                        TcItem* __restrict__ items1, int32_t* __restrict__ n1, int cap1,
                                                        int M2, int S2, TcItem* __restrict__ items2,
                                                        int32_t* __restrict__ n2, int cap2, uint32_t* err) {
  __shared__ int warp_sums[32];
  __shared__ int totals[2];
  const int a = threadIdx.x;
  const int nact = meta[0];
  int e = 0, p0 = 0, ne = 0, nch = 0;
  if (a < nact) {
    e = active[a];
    p0 = offsets[e];
    ne = offsets[e + 1] - p0;
    nch = (ne + nmax - 1) / nmax;
  }
  int base[2];
  const int cnt[2] = {nch * M1 * S1, nch * M2 * S2};
  for (int which = 0; which < 2; ++which) {
    // block-wide exclusive scan of cnt[which]
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = cnt[which];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int ws = warp_sums[lane];
      int wi = ws;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
        if (lane >= off) wi += o;
      }
      warp_sums[lane] = wi - ws;
      if (lane == 31) totals[which] = wi;
    }
    __syncthreads();
    base[which] = warp_sums[wid] + incl - cnt[which];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int t1 = totals[0], t2 = totals[1];
    if (t1 > cap1 || t2 > cap2) atomicOr(err, kErrCountOverflow);
    *n1 = min(t1, cap1);
    *n2 = min(t2, cap2);
  }
  for (int which = 0; which < 2; ++which) {
    const int M = which ? M2 : M1, S = which ? S2 : S1, cap = which ? cap2 : cap1;
    TcItem* items = which ? items2 : items1;
    int idx = base[which];
    for (int ch = 0; ch < nch; ++ch)
      for (int m = 0; m < M; ++m)
        for (int s = 0; s < S; ++s, ++idx)
          if (idx < cap) items[idx] = TcItem{e, p0 + ch * nmax, min(nmax, ne - ch * nmax), (m << 8) | s};
  }
}

// ---- K-split reduction + SwiGLU, and the combine --------------------------------------

// h16[p][f] = f16( silu(sum_s P[s][p][2f]) * sum_s P[s][p][2f+1] * 2^-8 ) (partials already scaled).
__global__ void swiglu_finalize_kernel(const float* __restrict__ part, size_t slice, int S, int rows, int I,
                                       uint16_t* __restrict__ h16) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)rows * I) return;
  const size_t p = i / I, f = i % I;
  float g = 0.f, u = 0.f;
  for (int s = 0; s < S; ++s) {
    const float2 v = reinterpret_cast<const float2*>(part + (size_t)s * slice + p * 2 * I)[f];
    g += v.x;
    u += v.y;
  }
  const float hv = g / (1.f + expf(-g)) * u * kHScaleInv;
  h16[i] = __half_as_ushort(__float2half_rn(fminf(fmaxf(hv, -65504.f), 65504.f)));
}

// out[t][c] = bf16_rne( sum over j ascending of w[t][j] * sum over s of Y[s][inv[t*k+j]][c] ).
__global__ void combine_tc_kernel(const float* __restrict__ y, size_t slice, int S, const float* __restrict__ w,
                                  const int32_t* __restrict__ inv, uint16_t* __restrict__ out, int H, int k) {
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int p = inv[(size_t)t * k + j];
    if (p < 0) continue;
    const float wj = w[(size_t)t * k + j];
    float4 v = reinterpret_cast<const float4*>(y + (size_t)p * H)[c4];
    for (int s = 1; s < S; ++s) {
      const float4 u = reinterpret_cast<const float4*>(y + (size_t)s * slice + (size_t)p * H)[c4];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
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

// Inspection: h as fp32 (undoing the 2^-8 storage scale) and y summed over K splits.
__global__ void debug_hy_kernel(const uint16_t* __restrict__ h16, const float* __restrict__ ytc, size_t slice, int S,
                                int rows, int I, int H, float* __restrict__ h, float* __restrict__ y) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (h && i < (size_t)rows * I) h[i] = __half2float(__ushort_as_half(h16[i])) * kHScale;
  if (y && i < (size_t)rows * H) {
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += ytc[(size_t)s * slice + i];
    y[i] = v;
  }
}

cudaError_t launch_debug_hy(const Shape& sh, const Workspace& ws, const TcPlan& pl, int T, float* h, float* y,
                            cudaStream_t s) {
  const int rows = T * sh.k;
  const size_t n = (size_t)rows * std::max(sh.I, sh.H);
  debug_hy_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws.h16, ws.ytc, (size_t)rows * sh.H, pl.S2, rows, sh.I,
                                                                sh.H, h, y);
  return cudaGetLastError();
}

// ---- load-time repack into the tensor-core tile layout ------------------------------------------

// Tile layout: [M tiles][K chunks of 64][4608 B]: codes as [half (2)][row (128)][16 B],
// then scales as [row (128)][4 B]. Gate/up tiles interleave rows: tile row 2i is gate
// feature 64m+i, row 2i+1 is up feature 64m+i. Down tiles: row r is output 128m+r.
__global__ void repack_tc_kernel(const uint8_t* __restrict__ raw_c, const uint8_t* __restrict__ raw_s,
                                 uint8_t* __restrict__ out, int rows_total, int K, int M, int gateup, int half_rows) {
  const int KC = K / 64;
  const size_t units = (size_t)M * KC * (2 * 128 + 128);  // 16-byte code units + 4-byte scale units
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= units) return;
  const size_t tile = i / (384);
  const int u = (int)(i % 384);
  const int m = (int)(tile / KC), kc = (int)(tile % KC);
  uint8_t* dst = out + tile * kRawBytes;
  if (u < 256) {
    const int hf = u / 128, r = u % 128;
    const int R = gateup ? ((r & 1) ? half_rows + m * 64 + (r >> 1) : m * 64 + (r >> 1)) : m * 128 + r;
    *reinterpret_cast<uint4*>(dst + (hf * 128 + r) * 16) =
        *reinterpret_cast<const uint4*>(raw_c + (size_t)R * (K / 2) + kc * 32 + hf * 16);
  } else {
    const int r = u - 256;
    const int R = gateup ? ((r & 1) ? half_rows + m * 64 + (r >> 1) : m * 64 + (r >> 1)) : m * 128 + r;
    *reinterpret_cast<uint32_t*>(dst + 4096 + r * 4) =
        *reinterpret_cast<const uint32_t*>(raw_s + (size_t)R * (K / 16) + kc * 4);
  }
  (void)rows_total;
}

cudaError_t launch_repack_tc(const Shape& sh, int e, const uint8_t* gu_codes_raw, const uint8_t* gu_scales_raw,
                             const uint8_t* dn_codes_raw, const uint8_t* dn_scales_raw, uint8_t* gu_tc, uint8_t* dn_tc,
                             cudaStream_t s) {
  const int H = sh.H, I = sh.I;
  const int M1 = 2 * I / 128, M2 = H / 128;
  const size_t per1 = (size_t)M1 * (H / 64) * kRawBytes, per2 = (size_t)M2 * (I / 64) * kRawBytes;
  const size_t u1 = (size_t)M1 * (H / 64) * 384, u2 = (size_t)M2 * (I / 64) * 384;
  repack_tc_kernel<<<(unsigned)((u1 + 255) / 256), 256, 0, s>>>(gu_codes_raw, gu_scales_raw, gu_tc + e * per1, 2 * I,
                                                                H, M1, 1, I);
  repack_tc_kernel<<<(unsigned)((u2 + 255) / 256), 256, 0, s>>>(dn_codes_raw, dn_scales_raw, dn_tc + e * per2, H, I,
                                                                M2, 0, 0);
  return cudaGetLastError();
}

// ---- host-side launchers -------------------------------------------------------------------------

TcPlan tc_plan(const Shape& sh, int T, int sm_count) {
  TcPlan pl;
  const double avg = (double)T * sh.k / sh.E;
  pl.prefill = avg >= 8.0;
  pl.nmax = pl.prefill ? kTcPrefillN : kTcDecodeN;
  pl.ctas_per_sm = pl.prefill ? 1 : 2;
  pl.grid = sm_count * pl.ctas_per_sm;
  const int M1 = 2 * sh.I / 128, M2 = sh.H / 128, KC1 = sh.H / 64, KC2 = sh.I / 64;
  // expected touched experts for uniform routing
  const double d = sh.E * (1.0 - pow(1.0 - (double)sh.k / sh.E, (double)T));
  const double target = 4.0 * pl.grid;
  auto pick = [&](double items, int KC) {
    int want = (int)ceil(target / (items > 1 ? items : 1));
    int best = 1;
    for (int s = 1; s <= KC / 4 && s <= 64; ++s)
      if (KC % s == 0 && s <= want) best = s;
    return best;
  };
  pl.S1 = pl.prefill ? 1 : pick(d * M1, KC1);
  pl.S2 = pl.prefill ? 1 : pick(d * M2, KC2);
  return pl;
}

size_t tc_items_cap(const Shape& sh, int T, int which, int sm_count) {
  const TcPlan pl = tc_plan(sh, T, sm_count);
  const size_t rows = (size_t)T * sh.k;
  const size_t chunks = (size_t)std::min<size_t>(sh.E, rows) + rows / pl.nmax + 1;
  const int M = which == 1 ? 2 * sh.I / 128 : sh.H / 128;
  return chunks * M * (which == 1 ? pl.S1 : pl.S2);
}

cudaError_t launch_gather_x(const Shape& sh, const Workspace& ws, const uint16_t* x, int T, cudaStream_t s) {
  const int rows = T * sh.k;
  gather_x_f16_kernel<<<(rows + 7) / 8, 256, 0, s>>>(x, ws.perm, ws.xg, ws.row_scale, rows, sh.H);
  return cudaGetLastError();
}

cudaError_t launch_worklist(const Shape& sh, const Workspace& ws, const TcPlan& pl, cudaStream_t s) {
  worklist_kernel<<<1, 1024, 0, s>>>(ws.active, ws.meta, ws.offsets, pl.nmax, 2 * sh.I / 128, pl.S1, ws.items1,
                                     ws.n_items1, ws.cap1, sh.H / 128, pl.S2, ws.items2, ws.n_items2, ws.cap2, ws.err);
  return cudaGetLastError();
}

template <int NMAX, int NS>
static cudaError_t launch_gemm_t(const CUtensorMap& map, const TcGemmParams& P, int grid, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes<NMAX, NS>();
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<NMAX, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  grouped_gemm_kernel<NMAX, NS><<<grid, kThreads, smem, s>>>(map, P);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const TcPlan& pl, const CUtensorMap& map, const TcGemmParams& P, cudaStream_t s) {
  if (pl.prefill) return launch_gemm_t<kTcPrefillN, kTcPrefillStages>(map, P, pl.grid, s);
  return launch_gemm_t<kTcDecodeN, kTcDecodeStages>(map, P, pl.grid, s);
}

cudaError_t launch_swiglu_finalize(const Shape& sh, const Workspace& ws, const TcPlan& pl, int T, cudaStream_t s) {
  const int rows = T * sh.k;
  const size_t n = (size_t)rows * sh.I;
  swiglu_finalize_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws.part1, (size_t)rows * 2 * sh.I, pl.S1, rows,
                                                                      sh.I, ws.h16);
  return cudaGetLastError();
}

cudaError_t launch_combine_tc(const Shape& sh, const Workspace& ws, const TcPlan& pl, uint16_t* out, int T,
                              cudaStream_t s) {
  dim3 grid((sh.H / 4 + 127) / 128, T);
  combine_tc_kernel<<<grid, 128, 0, s>>>(ws.ytc, (size_t)T * sh.k * sh.H, pl.S2, ws.w, ws.inv, out, sh.H, sh.k);
  return cudaGetLastError();
}

}  // namespace moe
