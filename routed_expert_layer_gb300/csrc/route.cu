// Routing: router logits (S1), top-k select with renormalised softmax weights (S2),
// and the histogram / prefix-sum / stable permutation into per-expert groups (S3).
//
// S1: each token is scored against every expert ("Kimi-K3 NVFP4 station eight
//     sparks", section "The number the project hangs on": attention, then a router,
//     then 16 experts, then a sum). fp32 logits, deterministic: a fixed K split and
//     a fixed-order reduction of the partial sums.
// S2: 16 of 896 experts per token ("Serving Kimi-K3 ... with 8xB300 GPUs", section
//     "The model, as the serving system sees it"). Order: logit descending, expert
//     index ascending, -0 == +0; made total by a 64-bit key so the result is unique.
// S3: route records sorted by expert, stable in token order ("Computation and Data
//     Movement for Inference", sections 4 and 15: build records, count, permute, later
//     restore token order).
#include "moe_internal.cuh"

namespace moe {

// ---- S1 router -----------------------------------------------------------------------

int router_splits(const Shape& sh, int T, int sm_count) {
  const int tiles = ((T + kRouterTT - 1) / kRouterTT) * ((sh.E + kRouterTE - 1) / kRouterTE);
  const int max_s = sh.H / 64;
  int s = (2 * sm_count + tiles - 1) / tiles;
  if (s < 1) s = 1;
  if (s > max_s) s = max_s;
  if (s > 64) s = 64;
  // round the slice to whole 64-row chunks, then recount the splits
  const int ks = ((sh.H / s + 63) / 64) * 64;
  return (sh.H + ks - 1) / ks;
}

static int router_slice(const Shape& sh, int S) { return ((sh.H / S + 63) / 64) * 64; }

size_t router_part_elems(const Shape& sh, int T_max, int sm_count) {
  size_t best = 0;
  // splits shrink as T grows; the product S*T peaks where S first drops below its cap
  for (int T = 1; T <= T_max; T = (T < 64 ? T + 1 : T + kRouterTT)) {
    size_t v = (size_t)router_splits(sh, T, sm_count) * (size_t)T * (size_t)sh.E;
    if (v > best) best = v;
  }
  size_t v = (size_t)router_splits(sh, T_max, sm_count) * (size_t)T_max * (size_t)sh.E;
  return v > best ? v : best;
}

// grid (ceil(T/16), ceil(E/128), S), block 128: thread = expert column, 16 token rows
// held in registers; x is staged in shared memory 64 rows of K at a time.
__global__ void __launch_bounds__(kRouterTE) router_partial_kernel(const uint16_t* __restrict__ x,
                                                                    const float* __restrict__ W,
                                                                    float* __restrict__ part, int T, int H, int E,
                                                                    int KS) {
  pdl_entry();
  __shared__ float xs[64][kRouterTT];
  const int t0 = blockIdx.x * kRouterTT;
  const int e = blockIdx.y * kRouterTE + threadIdx.x;
  const int s = blockIdx.z;
  const int h0 = s * KS;
  const int h1 = min(H, h0 + KS);
  float acc[kRouterTT];
#pragma unroll
  for (int i = 0; i < kRouterTT; ++i) acc[i] = 0.f;
  for (int hc = h0; hc < h1; hc += 64) {
    for (int i = threadIdx.x; i < 64 * kRouterTT; i += kRouterTE) {
      const int tt = i / 64, r = i % 64;
      float v = 0.f;
      if (t0 + tt < T) {
        const uint32_t b = x[(size_t)(t0 + tt) * H + hc + r];
        v = __uint_as_float(b << 16);
      }
      xs[r][tt] = v;
    }
    __syncthreads();
    if (e < E) {
#pragma unroll 8
      for (int r = 0; r < 64; ++r) {
        const float wv = __ldg(W + (size_t)(hc + r) * E + e);
        const float4* xr = reinterpret_cast<const float4*>(&xs[r][0]);
#pragma unroll
        for (int q = 0; q < kRouterTT / 4; ++q) {
          const float4 xv = xr[q];
          acc[4 * q + 0] = fmaf(xv.x, wv, acc[4 * q + 0]);
          acc[4 * q + 1] = fmaf(xv.y, wv, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(xv.z, wv, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(xv.w, wv, acc[4 * q + 3]);
        }
      }
    }
    __syncthreads();
  }
  if (e < E) {
#pragma unroll
    for (int tt = 0; tt < kRouterTT; ++tt)
      if (t0 + tt < T) part[((size_t)s * T + t0 + tt) * E + e] = acc[tt];
  }
}

// logits[t][e] = sum over splits s ascending of part[s][t][e], plus bias[e].
__global__ void router_reduce_kernel(const float* __restrict__ part, const float* __restrict__ bias,
                                     float* __restrict__ logits, int T, int E, int S) {
  pdl_entry();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t n = (size_t)T * E;
  if (i >= n) return;
  float acc = 0.f;
  for (int s = 0; s < S; ++s) acc += part[(size_t)s * n + i];
  logits[i] = acc + bias[i % E];
}

cudaError_t launch_router_reduce(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, int S,
                                 cudaStream_t s) {
  const size_t n = (size_t)T * sh.E;
  return launch_pdl(router_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, ws.router_part,
                    L.router_bias, ws.logits, T, sh.E, S);
}

cudaError_t launch_router(const Shape& sh, const DeviceLayer& L, const Workspace& ws, const uint16_t* x, int T,
                          int sm_count, cudaStream_t s) {
  const int S = router_splits(sh, T, sm_count);
  const int KS = router_slice(sh, S);
  dim3 grid((T + kRouterTT - 1) / kRouterTT, (sh.E + kRouterTE - 1) / kRouterTE, S);
  router_partial_kernel<<<grid, kRouterTE, 0, s>>>(x, L.router_w, ws.router_part, T, sh.H, sh.E, KS);
  const size_t n = (size_t)T * sh.E;
  router_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws.router_part, L.router_bias, ws.logits, T,
                                                                    sh.E, S);
  return cudaGetLastError();
}

// ---- S2 select ---------------------------------------------------------------------------

// Order-preserving map of an fp32 logit to uint32 (larger float -> larger key);
// -0 is folded onto +0 so the two compare equal.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The logit a key was made from (a -0 logit comes back as +0, which gives the same
// softmax term: exp(+0 - m) == exp(-0 - m)).
__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// One warp per token. Each lane holds the keys of experts lane, lane+32, ... as
// (ordered logit << 32) | (0xFFFFFFFF - e): all keys distinct, the largest key is
// the largest logit with the lowest index. Each of the k rounds takes the warp-wide
// largest key with two warp reductions (largest high word, then the largest low word
// among the lanes holding it); only the lane that owned the winner clears it and
// recomputes its own largest key (a depth-5 tree over its 32 slots).
__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

__device__ __forceinline__ unsigned long long lane_best(const unsigned long long (&keys)[32]) {
  unsigned long long t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = max_u64(keys[2 * i], keys[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = max_u64(t[2 * i], t[2 * i + 1]);
  return t[0];
}

// Top-k of one token's logits l[0..E) by one warp; lanes j < k write idx_out[j], w_out[j]
// (and idx_sh[j] when given). L2 = true reads the logits at L2 (they were written by other
// CTAs of the same grid).
template <bool L2 = false>
__device__ __forceinline__ void select_token(const float* __restrict__ l, int E, int k, int lane,
                                             int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                             int32_t* idx_sh = nullptr) {
  unsigned long long keys[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    const float le = e < E ? (L2 ? __ldcg(l + e) : l[e]) : 0.f;
    keys[i] = (e < E) ? (((unsigned long long)ordered_bits(le) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e))
                      : 0ull;
  }
  unsigned long long best = lane_best(keys);
  int my_e = 0;
  uint32_t my_hi = 0;  // lane j < k: the ordered bits of the j-th largest logit
  for (int j = 0; j < k; ++j) {
    const uint32_t hi = (uint32_t)(best >> 32);
    const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? (uint32_t)best : 0u);
    const int e = (int)(0xFFFFFFFFu - mlo);
    if (lane == j) {
      my_e = e;
      my_hi = mhi;
    }
    if ((e & 31) == lane) {  // the owner drops the winner and finds its next best
      const unsigned long long win = ((unsigned long long)mhi << 32) | mlo;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (keys[i] == win) keys[i] = 0ull;
      best = lane_best(keys);
    }
  }
  const float v = (lane < k) ? from_ordered_bits(my_hi) : 0.f;
  const float m0 = __shfl_sync(0xFFFFFFFFu, v, 0);
  float p = (lane < k) ? expf(v - m0) : 0.f;
  float sum = p;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    idx_out[lane] = my_e;
    w_out[lane] = p / sum;
    if (idx_sh) idx_sh[lane] = my_e;
  }
}

__global__ void select_kernel(const float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ w,
                              int T, int E, int k) {
  pdl_entry();
  const int tok = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
  select_token(logits + (size_t)tok * E, E, k, lane, idx + (size_t)tok * k, w + (size_t)tok * k);
}

cudaError_t launch_select(const Shape& sh, const float* logits, int32_t* idx, float* w, int T, cudaStream_t s) {
  const int warps_per_block = 8;
  const int blocks = (T + warps_per_block - 1) / warps_per_block;
  return launch_pdl(select_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, s, logits, idx, w, T, sh.E, sh.k);
}

// ---- S3 histogram / prefix sum / permutation --------------------------------------------------

// Per 32-token chunk c and local expert l: mask[c][l] bit i set iff token 32c+i chose
// expert e0 + l (routes with id -1 or outside the context's range are masked). 256
// threads = 8 chunks; atomicOr makes the masks independent of thread order, and its old
// value shows a token that listed one expert twice.
__global__ void __launch_bounds__(256) perm_masks_kernel(const int32_t* __restrict__ idx, uint32_t* __restrict__ masks,
                                                         uint32_t* __restrict__ err, int T, int E, int e0, int El,
                                                         int k) {
  pdl_entry();
  extern __shared__ uint32_t msk[];  // [8][El]
  for (int i = threadIdx.x; i < 8 * El; i += 256) msk[i] = 0u;
  __syncthreads();
  const int cl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 256 + threadIdx.x;
  bool bad = false, dup = false;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int l = local_expert(idx[(size_t)t * k + j], E, e0, El, bad);
      if (l < 0) continue;
      dup |= (atomicOr(&msk[cl * El + l], 1u << lane) >> lane) & 1u;
    }
  }
  if (bad) atomicOr(err, kErrExpertRange);
  if (dup) atomicOr(err, kErrDuplicate);
  __syncthreads();
  const int C = (T + 31) / 32;
  for (int i = threadIdx.x; i < 8 * El; i += 256) {
    const int c = blockIdx.x * 8 + i / El;
    if (c < C) masks[(size_t)c * El + (i % El)] = msk[i];
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, at most 1024).
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int ws = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_sums[lane] = wi - ws;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[wid] + incl - v;
  __syncthreads();
  return r;
}

// One CTA of 1024 threads; thread e (a local expert; E here is the context's expert
// count) walks the chunks in order: chunk_base[c][e] = rows of e in chunks before c;
// counts, offsets (exclusive scan over e) and the ascending list of touched experts.
// With cold_rows > 0 an expert of at most cold_rows rows goes, as one chunk, to the
// second list `cold` (count in meta[3]) instead of the first (meta[2]).
__global__ void __launch_bounds__(1024) perm_scan_kernel(const uint32_t* __restrict__ masks,
                                                         int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                                                         int32_t* __restrict__ meta, int T, int E,
                                                         TcChunk* __restrict__ chunks, int nmax, int chunk_cap,
                                                         TcChunk* __restrict__ cold, int cold_rows, int cold_cap,
                                                         uint32_t* __restrict__ err) {
  pdl_entry();
  __shared__ int totals[4];
  __shared__ int max_rows;
  const int e = threadIdx.x;
  const int C = (T + 31) / 32;
  int run = 0;
  if (e < E) {
    for (int c = 0; c < C; ++c) {
      const uint32_t mk = masks[(size_t)c * E + e];
      chunk_base[(size_t)c * E + e] = run;
      run += __popc(mk);
    }
    counts[e] = run;
  }
  if (threadIdx.x == 0) max_rows = 0;
  __syncthreads();
  if (run > 0) atomicMax(&max_rows, run);
  const int off = block_exclusive_scan(run, &totals[0]);
  const int pos = block_exclusive_scan(run > 0 ? 1 : 0, &totals[1]);
  if (e < E) {
    offsets[e] = off;
    if (run > 0) active[pos] = e;
  }
  if (threadIdx.x == 0) {
    offsets[E] = totals[0];
    meta[0] = totals[1];
    meta[1] = max_rows;
  }
  if (chunks) {  // the expert's rows cut into runs of at most nmax (uniform branch)
    const bool is_cold = cold_rows > 0 && run <= cold_rows;
    const int nch = is_cold ? 0 : (run + nmax - 1) / nmax;
    const int cb = block_exclusive_scan(nch, &totals[2]);
    for (int j = 0; j < nch; ++j)
      if (cb + j < chunk_cap) chunks[cb + j] = TcChunk{e, off + j * nmax, min(nmax, run - j * nmax), 0};
    const int cc = block_exclusive_scan(is_cold && run > 0 ? 1 : 0, &totals[3]);
    if (is_cold && run > 0 && cc < cold_cap) cold[cc] = TcChunk{e, off, run, 0};
    if (threadIdx.x == 0) {
      if (totals[2] > chunk_cap || totals[3] > cold_cap) atomicOr(err, kErrCountOverflow);
      meta[2] = min(totals[2], chunk_cap);
      meta[3] = min(totals[3], cold_cap);
    }
  }
}

// Thread per (t, j): p = offsets[l] + rows of l in earlier chunks + earlier tokens of this
// chunk, for the route's local expert l; a masked route gets inv = -1 (and served = -1).
__global__ void perm_scatter_kernel(const int32_t* __restrict__ idx, const uint32_t* __restrict__ masks,
                                    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                                    int32_t* __restrict__ perm, int32_t* __restrict__ slot, int32_t* __restrict__ inv,
                                    int32_t* __restrict__ served, int T, int E, int e0, int El, int k) {
  pdl_entry();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * k) return;
  const int t = i / k, j = i % k;
  const int id = idx[i];
  bool bad = false;  // raised by perm_masks_kernel already
  const int l = local_expert(id, E, e0, El, bad);
  if (l < 0) {
    inv[i] = -1;
    if (served) served[i] = -1;
    return;
  }
  const int c = t >> 5, lane = t & 31;
  const uint32_t mk = masks[(size_t)c * El + l];
  const int p = offsets[l] + chunk_base[(size_t)c * El + l] + __popc(mk & ((1u << lane) - 1u));
  perm[p] = t;
  slot[p] = j;
  inv[i] = p;
  if (served) served[i] = id;
}

// ---- small batches: S1..S3 after the router GEMM in one CTA -------------------------------

// For T <= 32 tokens (one 32-token chunk) and E <= 1024 this kernel does what
// router_reduce_kernel, select_kernel, perm_masks_kernel, perm_scan_kernel and
// perm_scatter_kernel do, with the same arithmetic in the same order, in one launch:
//  1. every CTA adds the router's K-split partial sums of 128 logits in ascending split
//     order and adds the bias last (the partial sums are first staged in shared memory,
//     so each thread has all its loads in flight at once);
//  2. the CTA that finishes last (a ticket taken after a device-scope fence; no CTA
//     ever waits for another) takes the top-k of every token with select_token, then
//     counts, scans and scatters the routes exactly as for one chunk of 32 tokens
//     (thread i owns experts i and i + 512), and returns the ticket to zero.
constexpr int kRouteSmallThreads = 512;
constexpr int kRouteSmallGroups = 32;  // float4 groups of logits per CTA in step 1
constexpr int kRouteSmallMaxS = 64;    // router K splits staged in shared memory

__global__ void __launch_bounds__(kRouteSmallThreads) route_small_kernel(
    const float* __restrict__ part, const float* __restrict__ bias, int S, float* __restrict__ logits,
    int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ active, int32_t* __restrict__ meta, int32_t* __restrict__ perm, int32_t* __restrict__ slot,
    int32_t* __restrict__ inv, TcChunk* __restrict__ chunks, int nmax, int chunk_cap, uint32_t* __restrict__ err,
    uint32_t* __restrict__ ticket, int T, int E, int e0, int El, int k) {
  pdl_entry();
  constexpr int NT = kRouteSmallThreads, G = kRouteSmallGroups;
  __shared__ float4 stage[kRouteSmallMaxS][G];
  __shared__ uint32_t mask[2 * NT];  // bit t of mask[l]: token t chose local expert l
  __shared__ int32_t idx_s[kRouteSmallT * 32];  // the routes chosen here (T <= 32, k <= 32)
  __shared__ int off_s[2 * NT];
  __shared__ int totals[6];
  __shared__ int max_rows;
  __shared__ int last;
  const int tid = threadIdx.x;
  const size_t n = (size_t)T * E, n4 = n / 4;  // E % 4 == 0 (launcher)
  // 1. logits of this CTA's groups
  const float4* part4 = reinterpret_cast<const float4*>(part);
  const size_t g0 = (size_t)blockIdx.x * G;
  for (int i = tid; i < S * G; i += NT) {
    const int s = i / G, gl = i - s * G;
    if (g0 + gl < n4) stage[s][gl] = part4[(size_t)s * n4 + g0 + gl];
  }
  __syncthreads();
  if (tid < 4 * G) {
    const int gl = tid >> 2, c = tid & 3;
    if (g0 + gl < n4) {
      const float* st = reinterpret_cast<const float*>(&stage[0][gl]) + c;
      float acc = 0.f;
      for (int s = 0; s < S; ++s) acc += st[(size_t)s * G * 4];
      const size_t i = 4 * (g0 + gl) + c;
      logits[i] = acc + bias[i % E];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // 2. the last CTA: selection and permutation of all T tokens
  mask[tid] = 0u;
  mask[tid + NT] = 0u;
  if (tid == 0) {
    max_rows = 0;
    *ticket = 0u;  // every CTA has taken its ticket
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = warp; t < T; t += NT / 32)
    select_token<true>(logits + (size_t)t * E, E, k, lane, idx + (size_t)t * k, w + (size_t)t * k,
                       idx_s + t * k);
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < T * k; i += NT) {
    const int l = local_expert(idx_s[i], E, e0, El, bad);
    if (l >= 0) atomicOr(&mask[l], 1u << (i / k));
  }
  if (bad) atomicOr(err, kErrExpertRange);
  __syncthreads();
  // thread tid owns local experts l0 = tid and l1 = tid + NT
  const int l0 = tid, l1 = tid + NT;
  const int run0 = l0 < El ? __popc(mask[l0]) : 0;
  const int run1 = l1 < El ? __popc(mask[l1]) : 0;
  if (l0 < El) counts[l0] = run0;
  if (l1 < El) counts[l1] = run1;
  const int rmax = max(run0, run1);
  if (rmax > 0) atomicMax(&max_rows, rmax);
  const int off0 = block_exclusive_scan(run0, &totals[0]);
  const int off1 = block_exclusive_scan(run1, &totals[1]) + totals[0];
  const int pos0 = block_exclusive_scan(run0 > 0 ? 1 : 0, &totals[2]);
  const int pos1 = block_exclusive_scan(run1 > 0 ? 1 : 0, &totals[3]) + totals[2];
  off_s[l0] = off0;
  off_s[l1] = off1;
  if (l0 < El) {
    offsets[l0] = off0;
    if (run0 > 0) active[pos0] = l0;
  }
  if (l1 < El) {
    offsets[l1] = off1;
    if (run1 > 0) active[pos1] = l1;
  }
  if (tid == 0) {
    offsets[El] = totals[0] + totals[1];
    meta[0] = totals[2] + totals[3];
    meta[1] = max_rows;
  }
  if (chunks) {  // each expert's rows cut into runs of at most nmax (uniform branch)
    const int nch0 = (run0 + nmax - 1) / nmax, nch1 = (run1 + nmax - 1) / nmax;
    const int cb0 = block_exclusive_scan(nch0, &totals[4]);
    const int cb1 = block_exclusive_scan(nch1, &totals[5]) + totals[4];
    for (int j = 0; j < nch0; ++j)
      if (cb0 + j < chunk_cap) chunks[cb0 + j] = TcChunk{l0, off0 + j * nmax, min(nmax, run0 - j * nmax), 0};
    for (int j = 0; j < nch1; ++j)
      if (cb1 + j < chunk_cap) chunks[cb1 + j] = TcChunk{l1, off1 + j * nmax, min(nmax, run1 - j * nmax), 0};
    if (tid == 0) {
      const int tot = totals[4] + totals[5];
      if (tot > chunk_cap) atomicOr(err, kErrCountOverflow);
      meta[2] = min(tot, chunk_cap);
      meta[3] = 0;  // batches this small never split off cold experts
    }
  }
  __syncthreads();
  for (int i = tid; i < T * k; i += NT) {
    const int t = i / k, j = i - t * k;
    const int li = local_expert(idx_s[i], E, e0, El, bad);
    if (li < 0) {
      inv[i] = -1;
      continue;
    }
    const int p = off_s[li] + __popc(mask[li] & ((1u << t) - 1u));
    perm[p] = t;
    slot[p] = j;
    inv[i] = p;
  }
}

cudaError_t launch_route_small(const Shape& sh, const DeviceLayer& L, const Workspace& ws, int T, int S, int nmax,
                               cudaStream_t s) {
  const size_t n4 = (size_t)T * sh.E / 4;
  const unsigned grid = (unsigned)((n4 + kRouteSmallGroups - 1) / kRouteSmallGroups);
  return launch_pdl(route_small_kernel, dim3(grid), dim3(kRouteSmallThreads), 0, s, ws.router_part, L.router_bias, S,
                    ws.logits, ws.idx, ws.w, ws.counts, ws.offsets, ws.active, ws.meta, ws.perm, ws.slot, ws.inv,
                    nmax > 0 ? ws.chunks : nullptr, nmax > 0 ? nmax : 1, ws.chunk_cap, ws.err, ws.ticket, T, sh.E,
                    sh.e0, sh.El, sh.k);
}

cudaError_t launch_permute(const Shape& sh, const Workspace& ws, const int32_t* idx, int T, cudaStream_t s,
                           int nmax, int32_t* served, int cold_rows) {
  const int blocks = (T + 255) / 256;
  cudaError_t e = launch_pdl(perm_masks_kernel, dim3(blocks), dim3(256), 8 * sh.El * sizeof(uint32_t), s, idx,
                             ws.masks, ws.err, T, sh.E, sh.e0, sh.El, sh.k);
  if (e != cudaSuccess) return e;
  e = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, ws.masks, ws.chunk_base, ws.counts, ws.offsets,
                 ws.active, ws.meta, T, sh.El, nmax > 0 ? ws.chunks : nullptr, nmax > 0 ? nmax : 1, ws.chunk_cap,
                 ws.chunks_cold, cold_rows, ws.chunk_cap_cold, ws.err);
  if (e != cudaSuccess) return e;
  const int n = T * sh.k;
  return launch_pdl(perm_scatter_kernel, dim3((n + 255) / 256), dim3(256), 0, s, idx, ws.masks, ws.chunk_base,
                    ws.offsets, ws.perm, ws.slot, ws.inv, served, T, sh.E, sh.e0, sh.El, sh.k);
}

}  // namespace moe
