// Expert FFN on the 5th-generation tensor cores (S4 gate/up + SwiGLU, S5 down, S6 combine).
//
// Every touched expert's bucket of routed rows is one grouped-GEMM problem
// ("Computation and Data Movement for Inference", section 4: one expert weight load
// serves the whole bucket; section 15: the arithmetic intensity 2nW / (B_W + n B_A +
// B_O) grows with the bucket size n). The
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
// Warp roles: warp 0 issues the copies, one thread of each MMA warp issues MMAs, the
// other warps dequantise and run the epilogue (warp w may only touch TMEM lanes
// 32*(w%4)..). The kernels are persistent over a device-built list of work items
// (expert, row range, M tile(s), K split): the decode variant with two CTAs per SM and
// two MMA warps each, the prefill variant with one CTA per SM.
#include <cuda.h>

#include <algorithm>
#include <cmath>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kChunkK = 128;         // K elements per pipeline stage (8 MMAs of K=16)
constexpr int kSlice = 4608;         // one tile's 64-element K half: [2 units][128 rows][16 B] codes + [128][4 B] scales
constexpr int kRawBytes = 2 * kSlice;  // one tile's 128-element K chunk
constexpr int kRawSlot = 9216;       // raw slot (a multiple of the 1024 B swizzle atom)
constexpr int kBoxRows = 16;         // activation rows per TMA box (64 f16 = 128 B per row)
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kACols = 64;           // one A stage (128 rows x 128 K of f16) in TMEM columns

__host__ __device__ constexpr uint32_t tmem_cols(int a_stages, int nmax) {
  const uint32_t need = a_stages * kACols + nmax;
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

template <int NMAX, int NS>
constexpr size_t gemm_smem_bytes() {
  return 1024 /*alignment slack*/ + (size_t)NS * (kRawSlot + 2 * NMAX * 128) + 512 /*barriers*/;
}
static_assert(kTcDecodeAStages * kACols + 2 * 2 * kTcDecodeN <= 256, "two decode CTAs per SM must fit in TMEM");

__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* h) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_in_low16) {
  uint32_t h;
  const uint16_t two = (uint16_t)two_in_low16;
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

// 16 codes (one 16-byte unit, one E4M3 scale per 8 of them... two blocks) -> 8 f16x2.
__device__ __forceinline__ void dequant_unit(const uint4 cw, uint32_t s_lo, uint32_t s_hi, uint32_t* v) {
  e2m1x8_to_f16x2x4(cw.x, v + 0);
  e2m1x8_to_f16x2x4(cw.y, v + 4);
  e2m1x8_to_f16x2x4(cw.z, v + 8);
  e2m1x8_to_f16x2x4(cw.w, v + 12);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = hmul2(v[i], s_lo);
#pragma unroll
  for (int i = 8; i < 16; ++i) v[i] = hmul2(v[i], s_hi);
}

// f16 of a normalised intermediate; a value beyond the f16 range or not finite is stored
// as the conversion gives it (an infinity or NaN, never clamped) and marks `bad`, which the
// caller turns into one atomicOr of the error word per work item (report_range).
__device__ __forceinline__ uint16_t f16_checked(float v, bool& bad) {
  bad |= !(fabsf(v) <= 65504.f);
  return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ void report_range(bool bad, uint32_t* err) {
  if (bad) atomicOr(err, kErrF16Range);
}

// SwiGLU in normalised units: gn, un normalised gate and up sums, gv the true gate
// pre-activation; returns gn * un * sigmoid(gv) * 2^-6 (fast division: 2 ulp, and a
// denominator of +inf, from a very negative gv, gives 0).
__device__ __forceinline__ float swiglu_store(float gn, float un, float gv) {
  return __fdividef(gn * un * kHStore, 1.f + __expf(-gv));
}

struct Ring {  // stage index and phase parity of a circular buffer of n slots
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

// Grouped GEMM over the work items (chunk, M tile, K split), decode variant, two CTAs
// per SM. A thread issues one tcgen05.mma about every 50 cycles however small N is, so
// at decode (N <= 16) two warps issue MMAs: warp 1 takes the even K chunks of an item,
// warp 2 the odd ones, each into its own accumulator, and the epilogue adds the two in
// a fixed order. TMEM A stage a is free again once the MMA of the chunk that used it
// has completed, i.e. once that chunk's shared-memory stage has been released
// (`empty`), so each chunk needs a single commit; the dequantisation warps convert a
// chunk's weights first and wait for that release only before storing them into the
// A stage, so the conversion overlaps the MMAs still reading it. Warps: 0 TMA, 1-2 MMA, 3..10
// dequantisation (one per TMEM lane quarter and 64-element K half), 11..14 epilogue.
// Two accumulator sets let the MMAs of the next item overlap the epilogue of the last.
constexpr int kEpiWarps = 4;
constexpr int kDequantWarps = 8;
constexpr int kMmaWarps = 2;
constexpr int kThreadsD = (1 + kMmaWarps + kDequantWarps + kEpiWarps) * 32;

template <int NMAX, int NS>
__global__ void __launch_bounds__(kThreadsD, 2)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const TcGemmParams P) {
  constexpr int kAStages = kTcDecodeAStages;
  static_assert(NS > kAStages, "an A stage is recycled through an older shared-memory stage");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int kBSub = NMAX * 128;          // one 64-column K half of the activation tile
  constexpr int kStage = kRawSlot + 2 * kBSub;
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  constexpr uint32_t kCols = tmem_cols(kAStages, 2 * kMmaWarps * NMAX);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * kStage);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;
  uint64_t* accfull = afull + kAStages;   // [2]
  uint64_t* accempty = accfull + 2;       // [2]
  uint64_t* drain = accempty + 2;         // [kMmaWarps]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + kMmaWarps);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDequantWarps + 1);
    }
    for (int a = 0; a < kAStages; ++a) mbar_init(&afull[a], kDequantWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], kMmaWarps);
      mbar_init(&accempty[b], kEpiWarps);
    }
    for (int w = 0; w < kMmaWarps; ++w) mbar_init(&drain[w], 1);
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
  constexpr uint32_t acc_col = kAStages * kACols;
  const int MS = P.M * P.S;
  const int n_items = *P.n_chunks * MS;
  const int kc_per = P.KC / P.S;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      Ring rs;
      uint32_t issued = 0;
      bool ok = true;
      TcChunk nxt = blockIdx.x < n_items ? P.chunks[blockIdx.x / MS] : TcChunk{0, 0, 0, 0};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int ci = it / MS, rem = it - ci * MS, m = rem / P.S, s = rem - m * P.S;
        const TcChunk ch = nxt;  // record of this item, loaded one item ahead
        if (it + (int)gridDim.x < n_items) nxt = P.chunks[(it + gridDim.x) / MS];
        (void)ci;
        const int nb = (ch.n + kBoxRows - 1) / kBoxRows;
        // slice (m, kc, h) of expert e sits at (((e*M/2 + m/2)*KC + kc)*2 + h)*2 + m%2 slices
        const uint8_t* wsrc = P.w + ((size_t)(ch.e * (P.M / 2) + (m >> 1)) * P.KC + (size_t)s * kc_per) * 4 * kSlice +
                              (size_t)(m & 1) * kSlice;
        const uint32_t tx = kRawBytes + nb * 2 * kBoxBytes;
        for (int c = 0; c < kc_per; ++c) {
          if (!mbar_wait(&empty[rs.idx], rs.ph ^ 1u, P.err)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + (size_t)rs.idx * kStage;
          mbar_arrive_expect_tx(&full[rs.idx], tx);
          bulk_g2s(sb, wsrc + (size_t)c * 4 * kSlice, kSlice, &full[rs.idx]);
          bulk_g2s(sb + kSlice, wsrc + (size_t)c * 4 * kSlice + 2 * kSlice, kSlice, &full[rs.idx]);
          const int kx = (s * kc_per + c) * kChunkK;
          for (int b = 0; b < nb; ++b) {
            tma_2d(sb + kRawSlot + b * kBoxBytes, &tmap_b, kx, ch.p0 + b * kBoxRows, &full[rs.idx]);
            tma_2d(sb + kRawSlot + kBSub + b * kBoxBytes, &tmap_b, kx + 64, ch.p0 + b * kBoxRows, &full[rs.idx]);
          }
          ++issued;
          rs.next(NS);
        }
      }
      if (!ok) {
        // let copies already issued land before the CTA's shared memory goes away
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
  } else if (warp <= kMmaWarps) {
    // ---- MMA issuers: warp 1 + mw takes the chunks c = mw, mw + 2, ... of every item ----
    const int mw = warp - 1;
    if (lane == 0) {
      int local = 0;
      uint32_t g0 = 0;  // CTA-wide index of the item's first chunk
      bool ok = true;
      TcChunk nxt = blockIdx.x < n_items ? P.chunks[blockIdx.x / MS] : TcChunk{0, 0, 0, 0};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local, g0 += (uint32_t)kc_per) {
        const TcChunk ch = nxt;  // loaded one item ahead
        if (it + (int)gridDim.x < n_items) nxt = P.chunks[(it + gridDim.x) / MS];
        const uint32_t N = (uint32_t)((ch.n + 15) / 16) * 16;
        const uint32_t idesc = idesc_f16(128, N);
        const int b = local & 1;
        if (local >= 2) {  // the epilogue of item local-2 has drained this accumulator set
          if (!mbar_wait(&accempty[b], (uint32_t)((local - 2) >> 1) & 1u, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t acc = tmem + acc_col + (uint32_t)((mw * 2 + b) * NMAX);
        for (int c = mw; c < kc_per; c += kMmaWarps) {
          const uint32_t g = g0 + (uint32_t)c;
          const int si = (int)(g % NS), ai = (int)(g % kAStages);
          // the dequantisation warps signal A stage ai after waiting for chunk g's copies,
          // so its activation boxes have landed too
          if (!mbar_wait(&afull[ai], (g / kAStages) & 1u, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bsm = smem_u32(smem + (size_t)si * kStage + kRawSlot);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            mma_f16_ts(acc, tmem + ai * kACols + kk * 8, desc_sw128(bsm + (kk >> 2) * kBSub + (kk & 3) * 32),
                       idesc, (c >= kMmaWarps || kk > 0) ? 1u : 0u);
          mma_commit(&empty[si]);  // frees the shared-memory stage and, through it, the A stage
        }
        if (ok) mma_commit(&accfull[b]);
      }
      // drain: every MMA this thread issued has completed before TMEM is released
      mma_commit(&drain[mw]);
      mbar_wait(&drain[mw], 0, P.err);
    }
  } else if (warp <= kMmaWarps + kDequantWarps) {
    // ---- dequantisation ----
    const int dw = warp - 1 - kMmaWarps;
    const int q = warp & 3;        // TMEM lane quarter of this warp
    const int half = dw >> 2;      // which 64-element half of a 128-element stage
    const int r = 32 * q + lane;   // tile row owned by this thread
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int code_off0 = half * kSlice + r * 16;
    const int code_off1 = half * kSlice + (128 + r) * 16;
    const int scale_off = half * kSlice + 4096 + r * 4;
    uint32_t g = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      for (int c = 0; c < kc_per; ++c, ++g) {
        const int si = (int)(g % NS), ai = (int)(g % kAStages);
        if (!mbar_wait(&full[si], (g / NS) & 1u, P.err)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + (size_t)si * kStage;
        const uint4 c0 = *reinterpret_cast<const uint4*>(raw + code_off0);
        const uint4 c1 = *reinterpret_cast<const uint4*>(raw + code_off1);
        const uint32_t s4 = *reinterpret_cast<const uint32_t*>(raw + scale_off);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[si]);
        const uint32_t s01 = e4m3x2_to_f16x2(s4 & 0xFFFFu);
        const uint32_t s23 = e4m3x2_to_f16x2(s4 >> 16);
        uint32_t v[32];
        dequant_unit(c0, prmt(s01, s01, 0x1010u), prmt(s01, s01, 0x3232u), v);
        dequant_unit(c1, prmt(s23, s23, 0x1010u), prmt(s23, s23, 0x3232u), v + 16);
        // the weights are converted while the MMAs of chunk g - kAStages may still read A
        // stage ai; only the store into it waits for their release
        if (g >= (uint32_t)kAStages) {
          const uint32_t go = g - kAStages;
          if (!mbar_wait(&empty[go % NS], (go / NS) & 1u, P.err)) {
            ok = false;
            break;
          }
        }
        __syncwarp();
        tc_fence_after();
        tmem_st32(tmem + lane_base + (uint32_t)(ai * kACols + half * 32), v);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[ai]);
      }
    }
  } else {
    // ---- epilogue ----
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int local = 0;
    TcChunk nxt = blockIdx.x < n_items ? P.chunks[blockIdx.x / MS] : TcChunk{0, 0, 0, 0};
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
      const int b = local & 1;
      const TcChunk ch = nxt;  // loaded one item ahead
      if (it + (int)gridDim.x < n_items) nxt = P.chunks[(it + gridDim.x) / MS];
      if (!mbar_wait(&accfull[b], (uint32_t)(local >> 1) & 1u, P.err)) break;
      tc_fence_after();
      const int ci = it / MS, rem = it - ci * MS, m = rem / P.S, s = rem - m * P.S;
      (void)ci;
      const int N = ((ch.n + 15) / 16) * 16;
      uint32_t v[kMmaWarps][NMAX];
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w)
#pragma unroll
        for (int c0 = 0; c0 < NMAX; c0 += 8) {
          if (c0 < N && w < kc_per) {  // an item of one K chunk only has the first accumulator
            __syncwarp();
            tmem_ld8(tmem + lane_base + acc_col + (uint32_t)((w * 2 + b) * NMAX + c0),
                     *reinterpret_cast<uint32_t(*)[8]>(&v[w][c0]));
          }
        }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
      const float gsc = P.gscale[ch.e * P.gstride + (P.gsel ? (r & 1) : 0)];
      const float o_gsc = __shfl_xor_sync(0xFFFFFFFFu, gsc, 1);  // the partner row's normaliser
      bool bad = false;
#pragma unroll
      for (int n = 0; n < NMAX; ++n) {
        if (n >= N) break;
        const int p = ch.p0 + n;
        const float acc = kc_per > 1 ? __uint_as_float(v[0][n]) + __uint_as_float(v[1][n]) : __uint_as_float(v[0][n]);
        if (P.mode == kTcModeSwiglu) {
          // rows 2f (gate) and 2f+1 (up) sit in adjacent lanes
          const float other = __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
          if (n < ch.n && (r & 1) == 0) {
            const float gn = acc * gsc, un = other * o_gsc;
            const float hv = swiglu_store(gn, un, gn * P.gate_f[p]);
            const int f = m * 64 + (r >> 1);
            P.h16[(size_t)p * P.I + f] = f16_checked(hv, bad);
          }
        } else if (n < ch.n) {
          const size_t o = (size_t)s * P.out_slice + (size_t)p * P.ldo + (size_t)m * 128 + r;
          if (P.mode == kTcModeOutF16)
            P.out16[o] = f16_checked(acc * gsc, bad);
          else
            P.out[o] = acc * gsc;
        }
      }
      report_range(bad, P.err);
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

// ---- prefill and midfill variants: two weight tiles per activation tile ----------------

// Each CTA computes two adjacent 128-row weight tiles (M tiles 2mp and 2mp+1) of one
// row chunk, so every activation tile staged in shared memory feeds twice the MMA
// work; stages are KH x 64 elements of K (one 128-byte swizzle row per 64), NS deep.
// TMEM: kA2 A stages of KH x 2 x 32 columns and two fp32 accumulators of NMAX columns.
// Instances: prefill <192, 6, 2, 1>, midfill <128, 4, 2, 2> and <64, 6, 2, 2>. Warp 0 issues
// the copies; warps 1 and 2 issue the MMAs of tile 0 and tile 1 (one thread issues a
// tcgen05.mma about every 50 cycles, so two issuers halve the MMA part of the
// dequantise -> MMA -> release chain that paces each A stage; the conversion itself
// runs before the wait for the release and overlaps the MMAs). The MMA warps wait only
// for the dequantised A stage: the dequantisation warps signal it after they have waited
// for the stage's copies, so the activation tile of that stage has landed too. Sixteen
// dequantisation warps in two groups of eight (one per TMEM lane quarter and weight tile)
// take alternate stages, each thread converting the KH x 64 weights of its row of its
// tile per stage, so two stages are dequantised at a time; later each group runs the epilogue
// for half of the accumulator columns.
constexpr int kDequantWarpsP = 16;
constexpr int kMmaWarpsP = 2;
constexpr int kThreadsP = (1 + kMmaWarpsP + kDequantWarpsP) * 32;

// KH is the number of 64-element K halves per stage (1 or 2): a stage holds KH x 2 tiles'
// raw slices (one contiguous run of the tile-pair layout) and KH activation boxes, and an
// A stage in TMEM holds KH x 2 tiles x 32 columns. Larger stages mean more MMAs per wait
// of the MMA warps and more weights per wait of the dequantisation threads.
template <int NMAX, int NS, int kA2, int KH>
__global__ void __launch_bounds__(kThreadsP, 1)
    grouped_gemm_mt2_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_b64,
                            const __grid_constant__ CUtensorMap tmap_b128, const TcGemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  static_assert(KH == 1 || KH == 2, "64- or 128-element K stages");
  constexpr int kARaw = KH * 2 * kSlice;      // the stage's raw slices: [K half][tile][4608 B]
  constexpr int kASlot = (kARaw + 1023) / 1024 * 1024;  // padded to the 1024-B swizzle atom
  constexpr int kBHalf = NMAX * 128;          // one 64-element K half of the activation tile
  constexpr int kStage = kASlot + KH * kBHalf;
  constexpr int kACols = KH * 64;             // TMEM columns of one A stage (2 tiles)
  constexpr uint32_t kCols = 512;
  static_assert(kA2 * kACols + 2 * NMAX <= 512, "TMEM budget");
  static_assert(kA2 % 2 == 0 && NS % 2 == 0, "the two dequantisation groups own alternate A and shared stages");
  static_assert(NMAX == 64 || NMAX == 128 || NMAX == 192, "activation boxes cover 16, 64, 128 or 192 rows (<= NMAX)");
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * kStage);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;
  uint64_t* aempty = afull + kA2;
  uint64_t* accfull = aempty + kA2;
  uint64_t* accempty = accfull + 1;
  uint64_t* drain = accempty + 1;  // [kMmaWarpsP]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + kMmaWarpsP);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDequantWarpsP / 2 + kMmaWarpsP);  // one dequantisation group per stage
    }
    for (int a = 0; a < kA2; ++a) {
      mbar_init(&afull[a], kDequantWarpsP / 2);
      mbar_init(&aempty[a], kMmaWarpsP);
    }
    mbar_init(accfull, kMmaWarpsP);
    mbar_init(accempty, kDequantWarpsP);
    for (int w = 0; w < kMmaWarpsP; ++w) mbar_init(&drain[w], 1);
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
  constexpr uint32_t acc_col = kA2 * kACols;
  const int MP = P.M / 2;
  const int n_items = *P.n_chunks * MP;
  const int n64 = P.KC * 2 / KH;  // stages over the whole K (no K split in this variant)

  if (warp == 0) {
    if (lane == 0) {
      Ring rs;
      uint32_t issued = 0;
      bool ok = true;
      TcChunk nxt = blockIdx.x < n_items ? P.chunks[blockIdx.x / MP] : TcChunk{0, 0, 0, 0};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int ci = it / MP, mp = it - ci * MP;
        const TcChunk ch = nxt;  // loaded one item ahead
        if (it + (int)gridDim.x < n_items) nxt = P.chunks[(it + gridDim.x) / MP];
        (void)ci;
        // The activation tile in as few copies as possible (each copy instruction costs this
        // single issuing thread time): one box of 16, 64 or 128 rows, or 128 + 64 rows. Rows
        // past the chunk are loaded but never read by the MMA (N covers the chunk only);
        // rows past the tensor are zero-filled.
        const int nb = (ch.n + kBoxRows - 1) / kBoxRows;  // 16-row units of the activation tile
        const int rows_loaded = nb <= 1 ? 16 : (nb <= 4 ? 64 : (nb <= 8 ? 128 : 192));
        // the two tiles' slices of K half h are adjacent: one copy per stage
        const uint8_t* wsrc = P.w + (size_t)(ch.e * (P.M / 2) + mp) * P.KC * 4 * kSlice;
        const uint32_t tx = kARaw + (uint32_t)(KH * rows_loaded * 128);
        for (int c = 0; c < n64; ++c) {
          if (!mbar_wait(&empty[rs.idx], rs.ph ^ 1u, P.err)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + (size_t)rs.idx * kStage;
          mbar_arrive_expect_tx(&full[rs.idx], tx);
          bulk_g2s(sb, wsrc + (size_t)c * kARaw, kARaw, &full[rs.idx]);
#pragma unroll
          for (int h = 0; h < KH; ++h) {
            uint8_t* bd = sb + kASlot + h * kBHalf;
            const int kx = (c * KH + h) * 64;
            if (rows_loaded == 16) {
              tma_2d(bd, &tmap_b, kx, ch.p0, &full[rs.idx]);
            } else if (rows_loaded == 64) {
              tma_2d(bd, &tmap_b64, kx, ch.p0, &full[rs.idx]);
            } else {
              tma_2d(bd, &tmap_b128, kx, ch.p0, &full[rs.idx]);
              if (rows_loaded == 192) tma_2d(bd + 128 * 128, &tmap_b64, kx, ch.p0 + 128, &full[rs.idx]);
            }
          }
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
  } else if (warp <= kMmaWarpsP) {
    // ---- MMA issuers: warp 1 + t for weight tile t of every item ----
    const int t = warp - 1;
    if (lane == 0) {
      Ring rs, ra;
      int local = 0;
      bool ok = true;
      TcChunk nxt = blockIdx.x < n_items ? P.chunks[blockIdx.x / MP] : TcChunk{0, 0, 0, 0};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local) {
        const TcChunk ch = nxt;  // loaded one item ahead
        if (it + (int)gridDim.x < n_items) nxt = P.chunks[(it + gridDim.x) / MP];
        const uint32_t N = (uint32_t)((ch.n + 15) / 16) * 16;
        const uint32_t idesc = idesc_f16(128, N);
        if (local > 0) {
          if (!mbar_wait(accempty, (uint32_t)(local - 1) & 1u, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int c = 0; c < n64; ++c) {
          if (!mbar_wait(&afull[ra.idx], ra.ph, P.err)) {  // implies the stage's copies have landed
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bsm = smem_u32(smem + (size_t)rs.idx * kStage + kASlot);
#pragma unroll
          for (int h = 0; h < KH; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(tmem + acc_col + t * NMAX, tmem + ra.idx * kACols + t * (KH * 32) + h * 32 + kk * 8,
                         desc_sw128(bsm + h * kBHalf + kk * 32), idesc, (c > 0 || h > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[rs.idx]);
          mma_commit(&aempty[ra.idx]);
          rs.next(NS);
          ra.next(kA2);
        }
        if (ok) mma_commit(accfull);
      }
      // drain: every MMA this thread issued has completed before TMEM is released
      mma_commit(&drain[t]);
      mbar_wait(&drain[t], 0, P.err);
    }
  } else {
    const int dw = warp - 1 - kMmaWarpsP;
    const int q = warp & 3;          // TMEM lane quarter of this warp
    const int t = (dw >> 2) & 1;     // which of the two weight tiles this warp serves
    const int hh = dw >> 3;          // group: CTA-wide stages of parity hh; in the epilogue, half of the columns
    const int r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    // K half h of this row of tile t: codes of elements 0..31 and 32..63, then their four
    // E4M3 block scales, in slice (h * 2 + t) of the stage
    const int code_off0 = t * kSlice + r * 16;
    const int code_off1 = t * kSlice + (128 + r) * 16;
    const int scale_off = t * kSlice + 4096 + r * 4;
    uint32_t G = 0;  // CTA-wide index of the item's first stage
    int local = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++local, G += (uint32_t)n64) {
      // the group takes the stages g with g % 2 == hh, CTA-wide: then each A stage (g % kA2,
      // kA2 even) and each shared-memory stage (g % NS, NS even) only ever receives the
      // arrivals of one group, and every barrier's phases complete in the order its waiters
      // expect, whatever the number of stages per item
      for (int c = (hh ^ (int)(G & 1u)) & 1; c < n64; c += 2) {
        const uint32_t g = G + (uint32_t)c;
        const int si = (int)(g % NS), ai = (int)(g % kA2);
        // stage g's copies have landed
        if (!mbar_wait(&full[si], (g / NS) & 1u, P.err)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + (size_t)si * kStage;
        uint4 cw0[KH], cw1[KH];
        uint32_t s4[KH];
#pragma unroll
        for (int h = 0; h < KH; ++h) {
          cw0[h] = *reinterpret_cast<const uint4*>(raw + h * 2 * kSlice + code_off0);
          cw1[h] = *reinterpret_cast<const uint4*>(raw + h * 2 * kSlice + code_off1);
          s4[h] = *reinterpret_cast<const uint32_t*>(raw + h * 2 * kSlice + scale_off);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[si]);
        // all KH halves converted into one array and stored by one instruction (a
        // tcgen05.st may read its source registers until tcgen05.wait::st)
        uint32_t v[KH * 32];
#pragma unroll
        for (int h = 0; h < KH; ++h) {
          const uint32_t s01 = e4m3x2_to_f16x2(s4[h] & 0xFFFFu);
          const uint32_t s23 = e4m3x2_to_f16x2(s4[h] >> 16);
          dequant_unit(cw0[h], prmt(s01, s01, 0x1010u), prmt(s01, s01, 0x3232u), v + h * 32);
          dequant_unit(cw1[h], prmt(s23, s23, 0x1010u), prmt(s23, s23, 0x3232u), v + h * 32 + 16);
        }
        // converted while the MMAs of stage g - kA2 may still read A stage ai; the store
        // waits for their release
        if (!mbar_wait(&aempty[ai], ((g / kA2) & 1u) ^ 1u, P.err)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        if constexpr (KH == 2)
          tmem_st64(tmem + lane_base + (uint32_t)(ai * kACols + t * 64), v);
        else
          tmem_st32(tmem + lane_base + (uint32_t)(ai * kACols + t * 32), v);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[ai]);
      }
      if (!ok) break;
      if (!mbar_wait(accfull, (uint32_t)local & 1u, P.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int ci = it / MP, mp = it - ci * MP;
      const int m = 2 * mp + t;
      const TcChunk ch = P.chunks[ci];
      const int N = ((ch.n + 15) / 16) * 16;
      const float gsc = P.gscale[ch.e * P.gstride + (P.gsel ? (r & 1) : 0)];
      const float o_gsc = __shfl_xor_sync(0xFFFFFFFFu, gsc, 1);  // the partner row's normaliser
      bool bad = false;
      for (int c0 = hh * (N / 2); c0 < (hh + 1) * (N / 2); c0 += 8) {
        uint32_t v[8];
        float rs8[8];  // gate factors of the 8 rows, loaded ahead of the accumulator read
#pragma unroll
        for (int i = 0; i < 8; ++i)
          rs8[i] = (P.mode == kTcModeSwiglu && c0 + i < ch.n) ? P.gate_f[ch.p0 + c0 + i] : 1.f;
        __syncwarp();
        tmem_ld8(tmem + lane_base + acc_col + (uint32_t)(t * NMAX + c0), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          const int p = ch.p0 + n;
          const float acc = __uint_as_float(v[i]);
          if (P.mode == kTcModeSwiglu) {
            const float other = __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
            if (n < ch.n && (r & 1) == 0) {
              const float gn = acc * gsc, un = other * o_gsc;
              const float hv = swiglu_store(gn, un, gn * rs8[i]);
              const int f = m * 64 + (r >> 1);
              P.h16[(size_t)p * P.I + f] = f16_checked(hv, bad);
            }
          } else if (n < ch.n) {
            const size_t o = (size_t)p * P.ldo + (size_t)m * 128 + r;
            if (P.mode == kTcModeOutF16)
              P.out16[o] = f16_checked(acc * gsc, bad);
            else
              P.out[o] = acc * gsc;
          }
        }
      }
      report_range(bad, P.err);
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

// ---- activation rows in f16 ---------------------------------------------------------------

// Token t's row, converted to f16 after scaling by 2^sigma so the row's largest
// magnitude lands in [2^13, 2^14) (the conversion of bf16 values is then exact down to
// 2^-28 of the row maximum), is written to each of its k routed rows inv[t*k+j], with
// the row's factors. One warp per token: the row is read once into registers
// (H <= 14336 -> at most 56 uint4 per lane).
template <int MAXV>
__global__ void gather_x_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ inv,
                                    uint16_t* __restrict__ xg, const RowFactors rf, int T, int H, int k) {
  pdl_entry();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const int n8 = H / 8;
  uint4 v[MAXV];
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    v[i] = (c < n8) ? src[c] : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, bf16_pair_maxbits(w[j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  const int sigma = row_sigma(mx);
  const float sc = __int_as_float((sigma + 127) << 23);  // exactly 2^sigma
#pragma unroll
  for (int i = 0; i < MAXV; ++i)
    v[i] = make_uint4(bf16x2_to_f16x2_scaled(v[i].x, sc), bf16x2_to_f16x2_scaled(v[i].y, sc),
                      bf16x2_to_f16x2_scaled(v[i].z, sc), bf16x2_to_f16x2_scaled(v[i].w, sc));
  for (int j = 0; j < k; ++j) {
    const int p = inv[(size_t)t * k + j];
    if (p < 0) continue;
    if (lane == 0) rf.write(p, t * k + j, rf.idx[(size_t)t * k + j] - rf.e0, sigma);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)p * H);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = lane + 32 * i;
      if (c < n8) dst[c] = v[i];
    }
  }
}

// The same conversion with one warp per routed row p (token perm[p]): every row is
// produced in parallel, which is what small batches need; large batches use the
// per-token kernel above, which reads each token row once instead of k times.
// rows is the launch bound (T * k); *n_rows the routed rows actually present (fewer when
// routes are masked).
template <int MAXV>
__global__ void gather_rows_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                       const int32_t* __restrict__ slot, uint16_t* __restrict__ xg,
                                       const RowFactors rf, int rows, const int32_t* __restrict__ n_rows, int H,
                                       int k) {
  pdl_entry();
  const int p = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= rows || p >= *n_rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)perm[p] * H);
  const int n8 = H / 8;
  uint4 v[MAXV];
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    v[i] = (c < n8) ? src[c] : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, bf16_pair_maxbits(w[j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  const int sigma = row_sigma(mx);
  const float sc = __int_as_float((sigma + 127) << 23);  // exactly 2^sigma
  if (lane == 0) {
    const int route = perm[p] * k + slot[p];
    rf.write(p, route, rf.idx[route] - rf.e0, sigma);
  }
  uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)p * H);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    if (c < n8)
      dst[c] = make_uint4(bf16x2_to_f16x2_scaled(v[i].x, sc), bf16x2_to_f16x2_scaled(v[i].y, sc),
                          bf16x2_to_f16x2_scaled(v[i].z, sc), bf16x2_to_f16x2_scaled(v[i].w, sc));
  }
}

// ---- K-split reduction + SwiGLU, and the combine --------------------------------------

// h16[p][f] = f16( gn * un * sigmoid(gn * gate_f[p]) * 2^-6 ) with gn, un the normalised
// gate and up sums over the K splits s ascending.
__global__ void swiglu_finalize_kernel(const float* __restrict__ part, size_t slice, int S, int rows,
                                       const int32_t* __restrict__ n_rows, int I, const float* __restrict__ gate_f,
                                       uint16_t* __restrict__ h16, uint32_t* __restrict__ err) {
  pdl_entry();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)rows * I) return;
  const size_t p = i / I, f = i % I;
  if (p >= (size_t)*n_rows) return;
  float g = 0.f, u = 0.f;
  for (int s = 0; s < S; ++s) {
    const float2 v = reinterpret_cast<const float2*>(part + (size_t)s * slice + p * 2 * I)[f];
    g += v.x;
    u += v.y;
  }
  bool bad = false;
  h16[i] = f16_checked(swiglu_store(g, u, g * gate_f[p]), bad);
  report_range(bad, err);
}

// out[t][c] = bf16_rne( sum over j ascending of wc[t][j] * sum over s of Y[s][p][c] ),
// p = inv[t*k+j] (skipped when -1), fp32 sums; Y is stored in f16 in normalised units and
// wc[t][j] = w[t][j] * comb_f[p] restores the true down projection. Thread per 8 columns;
// the k rows' loads of a split are issued together.
__device__ __forceinline__ void acc_f16x8(const uint4 u, float wj, float* a) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    a[2 * i] = fmaf(wj, f.x, a[2 * i]);
    a[2 * i + 1] = fmaf(wj, f.y, a[2 * i + 1]);
  }
}

// KMAX >= k: the number of routes held in registers at once (16 covers top-16, 32 any k).
template <int KMAX>
__global__ void combine_tc_kernel(const uint16_t* __restrict__ y, size_t slice, int S, const float* __restrict__ wc,
                                  const int32_t* __restrict__ inv, uint16_t* __restrict__ out, int H, int ldo,
                                  int k) {
  pdl_entry();
  const int t = blockIdx.y;
  const int c8 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c8 * 8 >= H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (S == 1) {
    uint4 u[KMAX];
    float wj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const int p = inv[(size_t)t * k + j];
        wj[j] = (p < 0) ? 0.f : wc[(size_t)t * k + j];
        u[j] = (p < 0) ? make_uint4(0, 0, 0, 0) : reinterpret_cast<const uint4*>(y + (size_t)p * H)[c8];
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) acc_f16x8(u[j], wj[j], acc);
  } else {
    // eight routes at a time, so that their loads of one split are in flight together;
    // each route's splits are still added in ascending order before it is weighted
    for (int j0 = 0; j0 < k; j0 += 8) {
      int pj[8];
      float v[8][8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        pj[q] = j0 + q < k ? inv[(size_t)t * k + j0 + q] : -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[q][i] = 0.f;
      }
      for (int s = 0; s < S; ++s) {
        uint4 u[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          u[q] = pj[q] < 0 ? make_uint4(0, 0, 0, 0)
                           : reinterpret_cast<const uint4*>(y + (size_t)s * slice + (size_t)pj[q] * H)[c8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc_f16x8(u[q], 1.f, v[q]);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (pj[q] < 0) continue;
        const float wj = wc[(size_t)t * k + j0 + q];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[q][i], acc[i]);
      }
    }
  }
  uint4 packed;
  uint32_t* pk = reinterpret_cast<uint32_t*>(&packed);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    pk[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(out + (size_t)t * ldo)[c8] = packed;  // ldo: out's row stride
}

// Inspection: h and y in true units (fp32), y summed over K splits. Row p's stored h is
// converted by comb_f[p] / (g_down * 2^n_down) (the combine factor without the down
// projection's own scale), its stored y by comb_f[p].
__global__ void debug_hy_kernel(const uint16_t* __restrict__ h16, const uint16_t* __restrict__ ytc, size_t slice,
                                int S, int rows, const int32_t* __restrict__ n_rows, int I, int H,
                                const float* __restrict__ comb_f, const int32_t* __restrict__ perm,
                                const int32_t* __restrict__ slot, const int32_t* __restrict__ idx, int e0, int k,
                                const float* __restrict__ dn_global, const int32_t* __restrict__ norm_exp,
                                float* __restrict__ h, float* __restrict__ y) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t present = (size_t)*n_rows;  // rows beyond it (masked routes) read as zero
  if (h && i < (size_t)rows * I) {
    const int p = (int)(i / I);
    float v = 0.f;
    if ((size_t)p < present) {
      const int e = idx[(size_t)perm[p] * k + slot[p]] - e0;
      const float f = ldexpf(comb_f[p] / dn_global[e], -norm_exp[4 * e + 2]);
      v = __half2float(__ushort_as_half(h16[i])) * f;
    }
    h[i] = v;
  }
  if (y && i < (size_t)rows * H) {
    float v = 0.f;
    if (i / H < present) {
      for (int s = 0; s < S; ++s) v += __half2float(__ushort_as_half(ytc[(size_t)s * slice + i]));
      v *= comb_f[i / H];
    }
    y[i] = v;
  }
}

cudaError_t launch_debug_hy(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const TcPlan& pl, int T,
                            float* h, float* y, cudaStream_t s) {
  const int rows = T * sh.k;
  const size_t n = (size_t)rows * std::max(sh.I, sh.D);
  debug_hy_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws.h16, ws.ytc, (size_t)rows * sh.D, pl.S2, rows,
                                                                ws.offsets + sh.El, sh.I, sh.D, ws.comb_f, ws.perm,
                                                                ws.slot, ws.idx, sh.e0, sh.k, L.dn_global, L.norm_exp,
                                                                h, y);
  return cudaGetLastError();
}

// ---- load time: accumulator normalisers --------------------------------------------------------

// Largest block scale (as its E4M3 byte; positive bytes order like their values) of the
// gate rows, the up rows and the down tensor of one expert: maxb[0..2] via atomicMax. The
// sign bit is ignored and the NaN byte counts as the largest finite one (0x7E).
__global__ void scale_max_kernel(const uint8_t* __restrict__ gu, size_t n_half, const uint8_t* __restrict__ dn,
                                 size_t n_dn, uint32_t* __restrict__ maxb) {
  uint32_t m[3] = {0u, 0u, 0u};
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n_half + n_dn; i += stride) {
    const int which = i < n_half ? 0 : (i < 2 * n_half ? 1 : 2);
    uint32_t b = (which < 2 ? gu[i] : dn[i - 2 * n_half]) & 0x7Fu;
    if (b == 0x7Fu) b = 0x7Eu;
    m[which] = max(m[which], b);
  }
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    uint32_t v = m[w];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    if ((threadIdx.x & 31) == 0 && v) atomicMax(&maxb[w], v);
  }
}

cudaError_t launch_scale_max(const Shape& sh, int e, const uint8_t* gu_scales_raw, const uint8_t* dn_scales_raw,
                             uint32_t* maxb, cudaStream_t s) {
  const size_t n_half = (size_t)sh.I * (sh.D / 16), n_dn = (size_t)sh.D * (sh.I / 16);  // e is a local expert
  scale_max_kernel<<<64, 256, 0, s>>>(gu_scales_raw, n_half, dn_scales_raw, n_dn, maxb + 3 * (size_t)e);
  return cudaGetLastError();
}

// Value of a non-negative E4M3 ("fn") byte.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const int ex = (int)((b >> 3) & 15u), mt = (int)(b & 7u);
  return ex ? ldexpf(1.f + mt / 8.f, ex - 7) : ldexpf((float)mt, -9);
}

// Smallest n with 2^n >= v (v > 0), exactly.
__device__ __forceinline__ int ceil_log2(float v) {
  int ex;
  const float m = frexpf(v, &ex);  // v = m * 2^ex, m in [0.5, 1)
  return m == 0.5f ? ex - 1 : ex;
}

// Per expert: n_gate, n_up = ceil(log2(6 * M)) + 14 and n_down = ceil(log2(6 * M)), M the
// largest block scale (an all-zero tensor counts as 2^-9, the smallest E4M3 step).
__global__ void norms_kernel(const uint32_t* __restrict__ maxb, int E, float* __restrict__ gu_norm,
                             float* __restrict__ dn_norm, int32_t* __restrict__ norm_exp) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int n[3];
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    const uint32_t b = maxb[3 * e + w];
    const float M = b ? e4m3_value(b) : ldexpf(1.f, -9);
    n[w] = ceil_log2(6.f * M) + (w < 2 ? 14 : 0);
  }
  gu_norm[2 * e] = ldexpf(1.f, -n[0]);
  gu_norm[2 * e + 1] = ldexpf(1.f, -n[1]);
  dn_norm[e] = ldexpf(1.f, -n[2]);
  norm_exp[4 * e] = n[0];
  norm_exp[4 * e + 1] = n[1];
  norm_exp[4 * e + 2] = n[2];
  norm_exp[4 * e + 3] = 0;
}

cudaError_t launch_norms(const Shape& sh, const uint32_t* maxb, float* gu_norm, float* dn_norm, int32_t* norm_exp,
                         cudaStream_t s) {
  norms_kernel<<<(sh.El + 127) / 128, 128, 0, s>>>(maxb, sh.El, gu_norm, dn_norm, norm_exp);
  return cudaGetLastError();
}

// ---- load-time repack into the tensor-core tile layout ------------------------------------------

// Tile layout per expert: [M/2 tile pairs][K chunks of 128][K half h (2)][tile of the pair (2)][4608 B].
// A 4608-byte slice holds one tile's 64 elements of K for its 128 rows: codes as
// [unit (2)][row (128)][16 B] (unit u = elements 32u..32u+31 of the half), then the
// E4M3 scales as [row (128)][4 B]. So a 128-element chunk of one tile is two slices
// (K halves 0 and 1) and a 64-element half of a tile pair is one 9216-byte run.
// Gate/up tiles interleave rows: tile row 2i is gate feature 64m+i, row 2i+1 is up
// feature 64m+i. Down tiles: row r is output feature 128m+r.
__global__ void repack_tc_kernel(const uint8_t* __restrict__ raw_c, const uint8_t* __restrict__ raw_s,
                                 uint8_t* __restrict__ out, int K, int M, int gateup, int half_rows) {
  const int KC = K / kChunkK;
  const size_t units = (size_t)M * KC * 768;  // per (tile, chunk): 2 halves x (256 code units + 128 scale units)
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= units) return;
  const size_t tile = i / 768;
  const int u = (int)(i % 768);
  const int m = (int)(tile / KC), kc = (int)(tile % KC);
  const int h = u / 384, v = u % 384;
  const int r = (v < 256) ? (v % 128) : (v - 256);
  const int R = gateup ? ((r & 1) ? half_rows + m * 64 + (r >> 1) : m * 64 + (r >> 1)) : m * 128 + r;
  uint8_t* dst = out + ((((size_t)(m >> 1) * KC + kc) * 2 + h) * 2 + (m & 1)) * kSlice;
  if (v < 256) {
    const int unit = v / 128;
    *reinterpret_cast<uint4*>(dst + (unit * 128 + r) * 16) =
        *reinterpret_cast<const uint4*>(raw_c + (size_t)R * (K / 2) + kc * 64 + (2 * h + unit) * 16);
  } else {
    *reinterpret_cast<uint32_t*>(dst + 4096 + r * 4) =
        *reinterpret_cast<const uint32_t*>(raw_s + (size_t)R * (K / 16) + kc * 8 + h * 4);
  }
}

cudaError_t launch_repack_tc(const Shape& sh, int e, const uint8_t* gu_codes_raw, const uint8_t* gu_scales_raw,
                             const uint8_t* dn_codes_raw, const uint8_t* dn_scales_raw, uint8_t* gu_tc, uint8_t* dn_tc,
                             cudaStream_t s) {
  const int H = sh.D, I = sh.I;  // the experts' model width
  const int M1 = 2 * I / 128, M2 = H / 128;
  const size_t per1 = (size_t)M1 * (H / kChunkK) * kRawBytes, per2 = (size_t)M2 * (I / kChunkK) * kRawBytes;
  const size_t u1 = (size_t)M1 * (H / kChunkK) * 768, u2 = (size_t)M2 * (I / kChunkK) * 768;
  repack_tc_kernel<<<(unsigned)((u1 + 255) / 256), 256, 0, s>>>(gu_codes_raw, gu_scales_raw, gu_tc + e * per1, H, M1,
                                                                1, I);
  repack_tc_kernel<<<(unsigned)((u2 + 255) / 256), 256, 0, s>>>(dn_codes_raw, dn_scales_raw, dn_tc + e * per2, I, M2,
                                                                0, 0);
  return cudaGetLastError();
}

// ---- host-side launchers -------------------------------------------------------------------------

TcPlan tc_plan(const Shape& sh, int T, int sm_count) {
  TcPlan pl;
  const double avg = (double)T * sh.k / sh.E;
  pl.prefill = avg >= 8.0;
  pl.nmax = !pl.prefill ? kTcDecodeN
                        : (avg < kTcMid64MaxAvg ? kTcMid64N : (avg < kTcMidMaxAvg ? kTcMidN : kTcPrefillN));
  pl.ctas_per_sm = pl.prefill ? 1 : 2;
  pl.grid = sm_count * pl.ctas_per_sm;
  const int M1 = 2 * sh.I / 128, M2 = sh.D / 128, KC1 = sh.D / kChunkK, KC2 = sh.I / kChunkK;
  // expected touched experts of the context for uniform routing
  const double d = sh.El * (1.0 - pow(1.0 - (double)sh.k / sh.E, (double)T));
  // K splits: the divisor s of the chunk count (at most a third of it, at most 64) whose
  // critical path -- waves of items times chunks per item, ceil(items * s / grid) * KC / s
  // -- is shortest; a split must save at least kTcSplitMinGainPct percent of it over the
  // next smaller one (each split adds partial sums to write and add up).
  auto pick = [&](double items, int KC) {
    const double n = items > 1 ? items : 1;
    int best = 1;
    double best_cost = ceil(n / pl.grid) * KC;
    for (int s = 2; s <= KC / 3 && s <= 64; ++s) {
      if (KC % s) continue;
      const double cost = ceil(n * s / pl.grid) * (KC / s);
      if (cost < (1.0 - kTcSplitMinGainPct / 100.0) * best_cost) {
        best = s;
        best_cost = cost;
      }
    }
    return best;
  };
  pl.S1 = pl.prefill ? 1 : pick(d * M1, KC1);
  pl.S2 = pl.prefill ? 1 : pick(d * M2, KC2);
  pl.cold_rows = (pl.prefill && T > kRouteSmallT) ? kTcDecodeN : 0;
  return pl;
}

size_t tc_chunk_cap(const Shape& sh, int T, int sm_count) {
  const TcPlan pl = tc_plan(sh, T, sm_count);
  const size_t rows = (size_t)T * sh.k;
  return (size_t)std::min<size_t>(sh.El, rows) + rows / pl.nmax + 1;
}

cudaError_t launch_gather_x(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const int32_t* idx,
                            const float* w, const uint16_t* x, int T, cudaStream_t s) {
  cudaError_t e;
  const int n8 = sh.D / 8;
  const int maxv = n8 <= 32 * 8 ? 8 : (n8 <= 32 * 28 ? 28 : 56);
  const RowFactors rf{idx, sh.e0, L.gu_global, L.dn_global, L.norm_exp, ws.gate_f, ws.comb_f, w, ws.wc};
  const int32_t* n_rows = ws.offsets + sh.El;
  if (T < 1024) {  // one warp per routed row
    const int rows = T * sh.k;
    const dim3 grid((rows + 7) / 8), block(256);
    if (maxv == 8) e = launch_pdl(gather_rows_f16_kernel<8>, grid, block, 0, s, x, ws.perm, ws.slot, ws.xg, rf, rows, n_rows, sh.D, sh.k);
    else if (maxv == 28) e = launch_pdl(gather_rows_f16_kernel<28>, grid, block, 0, s, x, ws.perm, ws.slot, ws.xg, rf, rows, n_rows, sh.D, sh.k);
    else e = launch_pdl(gather_rows_f16_kernel<56>, grid, block, 0, s, x, ws.perm, ws.slot, ws.xg, rf, rows, n_rows, sh.D, sh.k);
  } else {  // one warp per token, its k rows written from registers
    const dim3 grid((T + 7) / 8), block(256);
    if (maxv == 8) e = launch_pdl(gather_x_f16_kernel<8>, grid, block, 0, s, x, ws.inv, ws.xg, rf, T, sh.D, sh.k);
    else if (maxv == 28) e = launch_pdl(gather_x_f16_kernel<28>, grid, block, 0, s, x, ws.inv, ws.xg, rf, T, sh.D, sh.k);
    else e = launch_pdl(gather_x_f16_kernel<56>, grid, block, 0, s, x, ws.inv, ws.xg, rf, T, sh.D, sh.k);
  }
  return e;
}

template <int NMAX, int NS>
static cudaError_t launch_gemm_t(const CUtensorMap& map, const TcGemmParams& P, int grid, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes<NMAX, NS>();
  return launch_pdl(grouped_gemm_kernel<NMAX, NS>, dim3(grid), dim3(kThreadsD), smem, s, map, P);
}

template <int NMAX, int NS, int KH>
constexpr size_t smem_mt2() {
  // alignment slack, NS stages of (padded raw slices + KH activation halves), barriers
  return 1024 + (size_t)NS * ((KH * 2 * kSlice + 1023) / 1024 * 1024 + KH * NMAX * 128) + 256;
}

// Opt the GEMM kernels into large dynamic shared memory (once, at context creation,
// outside any stream capture).
cudaError_t tc_configure() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kTcDecodeN, kTcDecodeStages>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem_bytes<kTcDecodeN, kTcDecodeStages>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_mt2_kernel<kTcMid64N, kTcMid64Stages, kTcMidAStages, kTcMidKH>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_mt2<kTcMid64N, kTcMid64Stages, kTcMidKH>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_mt2_kernel<kTcMidN, kTcMidStages, kTcMidAStages, kTcMidKH>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_mt2<kTcMidN, kTcMidStages, kTcMidKH>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_mt2_kernel<kTcPrefillN, kTcPrefillStages, kTcPrefillAStages, kTcPrefillKH>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_mt2<kTcPrefillN, kTcPrefillStages, kTcPrefillKH>());
}

template <int NMAX, int NS, int NA, int KH>
static cudaError_t launch_gemm_mt2_t(const CUtensorMap& map, const CUtensorMap& map64, const CUtensorMap& map128,
                                     const TcGemmParams& P, int grid, cudaStream_t s) {
  return launch_pdl(grouped_gemm_mt2_kernel<NMAX, NS, NA, KH>, dim3(grid), dim3(kThreadsP), smem_mt2<NMAX, NS, KH>(),
                    s, map, map64, map128, P);
}

cudaError_t launch_gemm(const TcPlan& pl, const CUtensorMap& map, const CUtensorMap& map64, const CUtensorMap& map128,
                        const TcGemmParams& P, cudaStream_t s) {
  if (pl.prefill && pl.nmax == kTcMid64N)
    return launch_gemm_mt2_t<kTcMid64N, kTcMid64Stages, kTcMidAStages, kTcMidKH>(map, map64, map128, P, pl.grid, s);
  if (pl.prefill && pl.nmax == kTcMidN)
    return launch_gemm_mt2_t<kTcMidN, kTcMidStages, kTcMidAStages, kTcMidKH>(map, map64, map128, P, pl.grid, s);
  if (pl.prefill)
    return launch_gemm_mt2_t<kTcPrefillN, kTcPrefillStages, kTcPrefillAStages, kTcPrefillKH>(map, map64, map128, P,
                                                                                              pl.grid, s);
  return launch_gemm_t<kTcDecodeN, kTcDecodeStages>(map, P, pl.grid, s);
}

cudaError_t launch_swiglu_finalize(const Shape& sh, const Workspace& ws, const TcPlan& pl, int T, cudaStream_t s) {
  const int rows = T * sh.k;
  const size_t n = (size_t)rows * sh.I;
  return launch_pdl(swiglu_finalize_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, ws.part1,
                    (size_t)rows * 2 * sh.I, pl.S1, rows, ws.offsets + sh.El, sh.I, ws.gate_f, ws.h16, ws.err);
}

cudaError_t launch_combine_tc(const Shape& sh, const Workspace& ws, const TcPlan& pl, uint16_t* out, int ldo, int T,
                              cudaStream_t s) {
  dim3 grid((sh.D / 8 + 127) / 128, T);
  if (sh.k <= 16)
    return launch_pdl(combine_tc_kernel<16>, grid, dim3(128), 0, s, ws.ytc, (size_t)T * sh.k * sh.D, pl.S2, ws.wc,
                      ws.inv, out, sh.D, ldo, sh.k);
  return launch_pdl(combine_tc_kernel<32>, grid, dim3(128), 0, s, ws.ytc, (size_t)T * sh.k * sh.D, pl.S2, ws.wc,
                    ws.inv, out, sh.D, ldo, sh.k);
}

}  // namespace moe
