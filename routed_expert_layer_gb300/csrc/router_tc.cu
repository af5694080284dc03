// Router logits on the tensor cores (S1): logit[t][e] = sum_h x[t][h] * W_r[h][e].
//
// The router multiplies every token with every expert ("Kimi-K3 NVFP4 station
// eight sparks", section "The number the project hangs on": attention, then a
// router, then 16 experts, then a sum). W_r is fp32; x is bf16. W_r is split once,
// at load time, into three bf16 terms W = W0 + W1 + W2 (each the bf16 rounding of
// what the previous terms left), which represent it to 2^-24 relative; every
// product of a bf16 x with a bf16 term is exact in fp32, so the MMA with fp32
// accumulation gives fp32-level logits. The three terms are laid side by side
// along K (A = [E][3H]) and x is read three times (B[t][tau*H + h] = x[t][h]), so
// one accumulation sums all of them. Experts are the M dimension (128 per tile),
// tokens the N dimension, and K is split across CTAs; the fixed-order reduction
// over splits (router_reduce_kernel) adds the bias.
//
// The same kernel is the bf16 dense GEMM of a LatentMoE block (launch_dense_tc): A is a
// bf16 weight [M][K], B bf16 activation rows [T][K], and the fp32 partial sums per K
// split go to the block's finalize kernels (block.cu).
#include <cuda.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kRThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kRK = 64;         // K elements per stage (one 128-byte swizzle row of bf16)

template <int NMAX>
constexpr int router_stages() {
  return NMAX <= 64 ? 8 : 4;
}

template <int NMAX>
constexpr size_t router_smem_bytes() {
  return 1024 + (size_t)router_stages<NMAX>() * (128 * 128 + NMAX * 128) + 256;
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Ring {
  int idx = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      ph ^= 1u;
    }
  }
};

}  // namespace

// Items (M tile of 128 experts, N tile of NT tokens, K split): partial logits
// part[s][t][e] for t < T, e < E.
template <int NMAX>
__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                     const RouterTcParams P) {
  constexpr int NS = router_stages<NMAX>();
  constexpr int kA = 128 * 128;
  constexpr int kStage = kA + NMAX * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * kStage);
  uint64_t* empty = full + NS;
  uint64_t* accfull = empty + NS;
  uint64_t* accempty = accfull + 1;
  uint64_t* drain = accempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  constexpr uint32_t kCols = NMAX <= 32 ? 32 : (NMAX <= 64 ? 64 : (NMAX <= 128 ? 128 : 256));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, 4);
    mbar_init(drain, 1);
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
  pdl_entry();
  const int KS = P.S;  // K splits
  const int n_items = P.m_tiles * P.n_tiles * KS;
  const int kc_per = P.kc_total / KS;
  const uint32_t nt = (uint32_t)P.nt;

  if (warp == 0) {
    if (lane == 0) {
      Ring rs;
      bool ok = true;
      uint32_t issued = 0;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int s = it % KS, mn = it / KS, m = mn % P.m_tiles, n = mn / P.m_tiles;
        for (int c = 0; c < kc_per; ++c) {
          if (!mbar_wait(&empty[rs.idx], rs.ph ^ 1u, P.err)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + (size_t)rs.idx * kStage;
          const int kx = (s * kc_per + c) * kRK;
          mbar_arrive_expect_tx(&full[rs.idx], kA + nt * 128);
          tma_2d(sb, &tmap_w, kx, m * 128, &full[rs.idx]);
          tma_2d(sb + kA, &tmap_x, kx % P.H, n * (int)nt, &full[rs.idx]);
          ++issued;
          rs.next(NS);
        }
      }
      if (!ok) {
        Ring w = rs;
        for (uint32_t j = 0; j < (issued < (uint32_t)NS ? issued : (uint32_t)NS); ++j) {
          if (w.idx == 0) {
            w.idx = NS;
            w.ph ^= 1u;
          }
          --w.idx;
          mbar_wait(&full[w.idx], w.ph, P.err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      Ring rs;
      int local = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(128, nt);
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local) {
        if (local > 0) {
          if (!mbar_wait(accempty, (uint32_t)(local - 1) & 1u, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int c = 0; c < kc_per; ++c) {
          if (!mbar_wait(&full[rs.idx], rs.ph, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + (size_t)rs.idx * kStage);
#pragma unroll
          for (int kk = 0; kk < kRK / 16; ++kk)
            mma_bf16_ss(tmem, desc_sw128(a + kk * 32), desc_sw128(a + kA + kk * 32), idesc,
                        (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[rs.idx]);
          rs.next(NS);
        }
        if (ok) mma_commit(accfull);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, P.err);
    }
  } else {
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int local = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
      if (!mbar_wait(accfull, (uint32_t)local & 1u, P.err)) break;
      tc_fence_after();
      const int s = it % KS, mn = it / KS, m = mn % P.m_tiles, n = mn / P.m_tiles;
      const int e = m * 128 + r;
      float* dst = P.part + (size_t)s * P.T * P.E;
      for (uint32_t c0 = 0; c0 < nt; c0 += 8) {
        uint32_t v[8];
        __syncwarp();
        tmem_ld8(tmem + lane_base + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = n * (int)nt + (int)c0 + i;
          if (t < P.T && e < P.E) dst[(size_t)t * P.E + e] = __uint_as_float(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kCols);
  }
}

// Three-term bf16 split of W_r [H][E] into A = [E_pad][3H] (term tau in columns tau*H..).
__global__ void router_split_kernel(const float* __restrict__ W, uint16_t* __restrict__ w3, int H, int E, int E_pad) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)E_pad * H) return;
  const int e = (int)(i / H), h = (int)(i % H);
  float rem = (e < E) ? W[(size_t)h * E + e] : 0.f;
  uint16_t* row = w3 + (size_t)e * 3 * H;
#pragma unroll
  for (int tau = 0; tau < 3; ++tau) {
    const __nv_bfloat16 b = __float2bfloat16_rn(rem);
    row[(size_t)tau * H + h] = __bfloat16_as_ushort(b);
    rem = rem - __bfloat162float(b);
  }
}

// Tiles and K splits of part[S][T][M] = A[M][K] B[T][K]^T: tokens in N tiles of 16..64
// (small T) or 128 / 256, M in tiles of 128, K in stages of 64.
static RouterTcPlan plan_mk(int M, int K, int T, int sm_count) {
  RouterTcPlan pl;
  const int t16 = ((T + 15) / 16) * 16;
  pl.nt = t16 <= 64 ? t16 : (T <= 1024 ? 128 : 256);
  if (pl.nt > 256) pl.nt = 256;
  pl.n_tiles = (T + pl.nt - 1) / pl.nt;
  pl.m_tiles = (M + 127) / 128;
  pl.kc_total = K / kRK;
  pl.small = pl.nt <= 64;
  const int base = pl.m_tiles * pl.n_tiles;
  const int grid_ctas = sm_count;  // one CTA per SM (shared memory)
  // few tiles: as many K splits as fill one wave; many tiles: about two waves
  const int want = base < grid_ctas ? grid_ctas / base : (2 * grid_ctas + base - 1) / base;
  int best = 1;
  for (int s = 1; s <= pl.kc_total / 4; ++s)
    if (pl.kc_total % s == 0 && s <= want) best = s;
  pl.S = best;
  pl.grid = std::min(grid_ctas, base * best);
  return pl;
}

RouterTcPlan router_tc_plan(const Shape& sh, int T, int sm_count) { return plan_mk(sh.E, 3 * sh.H, T, sm_count); }

RouterTcPlan dense_tc_plan(int M, int K, int T, int sm_count) { return plan_mk(M, K, T, sm_count); }

cudaError_t launch_router_split(const Shape& sh, const float* W, uint16_t* w3, cudaStream_t s) {
  const int E_pad = ((sh.E + 127) / 128) * 128;
  const size_t n = (size_t)E_pad * sh.H;
  router_split_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(W, w3, sh.H, sh.E, E_pad);
  return cudaGetLastError();
}

cudaError_t router_tc_configure() {
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)router_smem_bytes<64>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)router_smem_bytes<256>());
}

template <int NMAX>
static cudaError_t launch_router_tc_t(const CUtensorMap& mw, const CUtensorMap& mx, const RouterTcParams& P, int grid,
                                      cudaStream_t s) {
  return launch_pdl(router_tc_kernel<NMAX>, dim3(grid), dim3(kRThreads), router_smem_bytes<NMAX>(), s, mw, mx, P);
}

cudaError_t launch_dense_tc(const RouterTcPlan& pl, const CUtensorMap& mw, const CUtensorMap& mx, int T, int M, int K,
                            float* part, uint32_t* err, cudaStream_t s) {
  RouterTcParams P;
  P.T = T;
  P.E = M;
  P.H = K;  // B's K coordinate runs over all of K (no repetition)
  P.nt = pl.nt;
  P.n_tiles = pl.n_tiles;
  P.m_tiles = pl.m_tiles;
  P.kc_total = pl.kc_total;
  P.S = pl.S;
  P.part = part;
  P.err = err;
  return pl.small ? launch_router_tc_t<64>(mw, mx, P, pl.grid, s) : launch_router_tc_t<256>(mw, mx, P, pl.grid, s);
}

cudaError_t launch_router_tc(const Shape& sh, const RouterTcPlan& pl, const CUtensorMap& mw, const CUtensorMap& mx,
                             const DeviceLayer& L, const Workspace& ws, int T, cudaStream_t s, bool reduce) {
  RouterTcParams P;
  P.T = T;
  P.E = sh.E;
  P.H = sh.H;
  P.nt = pl.nt;
  P.n_tiles = pl.n_tiles;
  P.m_tiles = pl.m_tiles;
  P.kc_total = pl.kc_total;
  P.S = pl.S;
  P.part = ws.router_part;
  P.err = ws.err;
  cudaError_t e = pl.small ? launch_router_tc_t<64>(mw, mx, P, pl.grid, s) : launch_router_tc_t<256>(mw, mx, P, pl.grid, s);
  if (e != cudaSuccess || !reduce) return e;
  return launch_router_reduce(sh, L, ws, T, pl.S, s);
}

}  // namespace moe
