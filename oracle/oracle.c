/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY. A plain, slow, obviously correct CPU
 * restatement of the routed Mixture-of-Experts layer, in fp64, used to check
 * the CUDA path. Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it; the library never does. It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it computes, step by step, and the passages it follows:
 *
 *   S1 router      logit[t][e] = sum_h x[t][h] * W_r[h][e] (+ bias[e]).
 *                  "Kimi-K3 NVFP4 station eight sparks", section "The number
 *                  the project hangs on": each layer is attention, then a
 *                  router, then 16 experts, then a sum. The pages do not define
 *                  the score function; the reading used is an fp32 router
 *                  matrix with softmax scores.
 *   S2 select      per token the k experts of largest logit, ties to the lower
 *                  expert index, listed in that order; gate weights are the
 *                  softmax restricted to the selected logits (softmax over all
 *                  experts, then renormalised over the k -- the same numbers).
 *                  "Serving Kimi-K3 ... with 8xB300 GPUs", section "The model,
 *                  as the serving system sees it": each token visits 16 of 896
 *                  experts per layer.
 *   S3 permute     route records sorted by expert (stable in token order):
 *                  counts, exclusive offsets, perm[p] = token, slot[p] = j,
 *                  inv[t*k + j] = p. "Computation and Data Movement for
 *                  Inference" (Chinese translation),
 *                  section 4 (the prefill MoE flow: sort or queue route records
 *                  by expert so one weight load serves a whole bucket) and
 *                  section 15 (records are built, counted, permuted, and
 *                  restored to token order).
 *   S4 gate/up     g = W_g x, u = W_u x, h = silu(g) * u per routed row, with
 *                  W = e2m1(code) * e4m3(block scale) * fp32 tensor scale.
 *                  Three matrices per expert: "Serving Kimi-K3 ...", same
 *                  section (3 x 3584 x 3072 per expert). NVFP4: "Kimi-K3 NVFP4
 *                  station eight sparks", section "What has to be built" (an
 *                  FP8 scale per 16 values plus a per-expert global scale).
 *                  The activation is not named on the pages; SwiGLU is used.
 *   S5 down        y[p] = w[perm[p]][slot[p]] * (W_d h[p]).
 *   S6 combine     out[t] = sum over j ascending of y[inv[t*k + j]]: expert
 *                  outputs restored to token order, weighted and merged
 *                  ("Computation and Data Movement for Inference", section 4).
 *
 * Formats (decoded here from their definitions, not from any library):
 *   E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; codes 0..7 are
 *         0, 0.5, 1, 1.5, 2, 3, 4, 6 and codes 8..15 their negatives.
 *   E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, exponent 0 is
 *         subnormal (m * 2^-9), no infinities, 0x7F/0xFF are NaN, max 448.
 *   bf16: the top 16 bits of an IEEE binary32.
 *
 * All floating point is fp64. Every reduction runs in a fixed order, so the
 * results do not depend on the OpenMP thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats -------------------------------------------------------- */

double oracle_e2m1(unsigned code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7u];
  return (code & 8u) ? -v : v;
}

double oracle_e4m3(unsigned byte) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 15u && m == 7u) return NAN;
  double v = (e == 0u) ? (double)m * ldexp(1.0, -9) : (1.0 + (double)m / 8.0) * ldexp(1.0, (int)e - 7);
  return s ? -v : v;
}

double oracle_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* One dequantised NVFP4 row: W[c] = e2m1(code) * e4m3(scale[c/16]) * global. */
static void dequant_row(int64_t K, const uint8_t* codes, const uint8_t* scales, double global, double* row) {
  for (int64_t c = 0; c < K; ++c) {
    uint8_t byte = codes[c / 2];
    unsigned code = (c % 2 == 0) ? (byte & 15u) : (byte >> 4);
    row[c] = oracle_e2m1(code) * oracle_e4m3(scales[c / 16]) * global;
  }
}

/* Public for the pins: dequantise a [rows][K] NVFP4 tensor to fp64. */
void oracle_dequant(int64_t rows, int64_t K, const uint8_t* codes, const uint8_t* scales, double global,
                    double* out) {
  for (int64_t r = 0; r < rows; ++r) dequant_row(K, codes + r * (K / 2), scales + r * (K / 16), global, out + r * K);
}

/* ---- S1 router -------------------------------------------------------------- */

void oracle_router_logits(int64_t T, int64_t H, int64_t E, const uint16_t* x, const float* W_r, const float* bias,
                          double* logits) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* acc = logits + t * E;
    for (int64_t e = 0; e < E; ++e) acc[e] = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double xv = oracle_bf16(x[t * H + h]);
      const float* wr = W_r + h * E;
      for (int64_t e = 0; e < E; ++e) acc[e] += xv * (double)wr[e];
    }
    if (bias)
      for (int64_t e = 0; e < E; ++e) acc[e] += (double)bias[e];
  }
}

/* Also sum_h |x[t][h] * W_r[h][e]|: the scale of the rounding error any fp32 evaluation of the logit carries. */
void oracle_router_abs(int64_t T, int64_t H, int64_t E, const uint16_t* x, const float* W_r, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* acc = out + t * E;
    for (int64_t e = 0; e < E; ++e) acc[e] = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double xv = fabs(oracle_bf16(x[t * H + h]));
      const float* wr = W_r + h * E;
      for (int64_t e = 0; e < E; ++e) acc[e] += xv * fabs((double)wr[e]);
    }
  }
}

/* ---- S2 select -------------------------------------------------------------- */

/* k rounds of "largest remaining logit, lowest index among equals". -0 and +0
 * compare equal. w is the softmax over the k selected logits. */
void oracle_select(int64_t T, int64_t E, int64_t k, const double* logits, int32_t* idx, double* w) {
#pragma omp parallel
  {
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      const double* l = logits + t * E;
      memset(taken, 0, (size_t)E);
      for (int64_t j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
          if (taken[e]) continue;
          if (best < 0 || l[e] > l[best]) best = e;
        }
        taken[best] = 1;
        idx[t * k + j] = (int32_t)best;
      }
      double m = l[idx[t * k]];
      double s = 0.0;
      for (int64_t j = 0; j < k; ++j) {
        double p = exp(l[idx[t * k + j]] - m);
        w[t * k + j] = p;
        s += p;
      }
      for (int64_t j = 0; j < k; ++j) w[t * k + j] /= s;
    }
    free(taken);
  }
}

/* ---- S3 permute -------------------------------------------------------------- */

void oracle_permute(int64_t T, int64_t E, int64_t k, const int32_t* idx, int32_t* counts, int32_t* offsets,
                    int32_t* perm, int32_t* slot, int32_t* inv) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) counts[idx[i]]++;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc((size_t)E * sizeof(int32_t));
  for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t t = 0; t < T; ++t) /* ascending tokens: a stable sort by expert */
    for (int64_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      int32_t p = cursor[e]++;
      perm[p] = (int32_t)t;
      slot[p] = (int32_t)j;
      inv[t * k + j] = p;
    }
  free(cursor);
}

/* ---- S4 + S5 one expert over a bucket of n token rows ------------------------- */

typedef struct {
  int64_t H, I, E;
  const uint8_t* gu_codes;  /* [E][2I][H/2] */
  const uint8_t* gu_scales; /* [E][2I][H/16] */
  const float* gu_global;   /* [E][2] */
  const uint8_t* dn_codes;  /* [E][H][I/2] */
  const uint8_t* dn_scales; /* [E][H][I/16] */
  const float* dn_global;   /* [E] */
  const float* router_w;    /* [H][E] */
  const float* router_bias; /* [E] or NULL */
} oracle_layer;

/* xs[n][H] -> hs[n][I] (SwiGLU of the gate and up projections). */
void oracle_expert_gateup(const oracle_layer* L, int64_t e, int64_t n, const double* xs, double* hs) {
  const int64_t H = L->H, I = L->I;
  const uint8_t* codes = L->gu_codes + e * (2 * I) * (H / 2);
  const uint8_t* scales = L->gu_scales + e * (2 * I) * (H / 16);
  double* row = (double*)malloc((size_t)H * sizeof(double));
  double* g = (double*)malloc((size_t)n * sizeof(double));
  for (int64_t i = 0; i < I; ++i) {
    dequant_row(H, codes + i * (H / 2), scales + i * (H / 16), (double)L->gu_global[e * 2 + 0], row);
    for (int64_t r = 0; r < n; ++r) {
      double s = 0.0;
      for (int64_t c = 0; c < H; ++c) s += row[c] * xs[r * H + c];
      g[r] = s;
    }
    dequant_row(H, codes + (I + i) * (H / 2), scales + (I + i) * (H / 16), (double)L->gu_global[e * 2 + 1], row);
    for (int64_t r = 0; r < n; ++r) {
      double u = 0.0;
      for (int64_t c = 0; c < H; ++c) u += row[c] * xs[r * H + c];
      hs[r * I + i] = g[r] / (1.0 + exp(-g[r])) * u;
    }
  }
  free(g);
  free(row);
}

/* hs[n][I] -> ys[n][H] = W_d h (unweighted). */
void oracle_expert_down(const oracle_layer* L, int64_t e, int64_t n, const double* hs, double* ys) {
  const int64_t H = L->H, I = L->I;
  const uint8_t* codes = L->dn_codes + e * H * (I / 2);
  const uint8_t* scales = L->dn_scales + e * H * (I / 16);
  double* row = (double*)malloc((size_t)I * sizeof(double));
  for (int64_t c = 0; c < H; ++c) {
    dequant_row(I, codes + c * (I / 2), scales + c * (I / 16), (double)L->dn_global[e], row);
    for (int64_t r = 0; r < n; ++r) {
      double s = 0.0;
      for (int64_t i = 0; i < I; ++i) s += row[i] * hs[r * I + i];
      ys[r * H + c] = s;
    }
  }
  free(row);
}

/* ---- the whole layer ----------------------------------------------------------- */

/* Full layer over T tokens, in the method's order: route, sort by expert, one
 * pass over each touched expert for its whole bucket, restore token order and
 * merge. Any of idx/w/logits may be NULL. out[T][H] fp64. */
void oracle_moe_forward(const oracle_layer* L, int64_t T, int64_t k, const uint16_t* x, double* out,
                        int32_t* idx_out, double* w_out, double* logits_out) {
  const int64_t H = L->H, I = L->I, E = L->E;
  if (T <= 0) return;
  double* logits = logits_out ? logits_out : (double*)malloc((size_t)(T * E) * sizeof(double));
  int32_t* idx = idx_out ? idx_out : (int32_t*)malloc((size_t)(T * k) * sizeof(int32_t));
  double* w = w_out ? w_out : (double*)malloc((size_t)(T * k) * sizeof(double));
  oracle_router_logits(T, H, E, x, L->router_w, L->router_bias, logits);
  oracle_select(T, E, k, logits, idx, w);

  int32_t* counts = (int32_t*)malloc((size_t)E * sizeof(int32_t));
  int32_t* offsets = (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
  int32_t* perm = (int32_t*)malloc((size_t)(T * k) * sizeof(int32_t));
  int32_t* slot = (int32_t*)malloc((size_t)(T * k) * sizeof(int32_t));
  int32_t* inv = (int32_t*)malloc((size_t)(T * k) * sizeof(int32_t));
  oracle_permute(T, E, k, idx, counts, offsets, perm, slot, inv);

  double* y = (double*)malloc((size_t)(T * k * H) * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t e = 0; e < E; ++e) {
    int64_t n = counts[e];
    if (n == 0) continue;
    int64_t p0 = offsets[e];
    double* xs = (double*)malloc((size_t)(n * H) * sizeof(double));
    double* hs = (double*)malloc((size_t)(n * I) * sizeof(double));
    for (int64_t r = 0; r < n; ++r)
      for (int64_t c = 0; c < H; ++c) xs[r * H + c] = oracle_bf16(x[(int64_t)perm[p0 + r] * H + c]);
    oracle_expert_gateup(L, e, n, xs, hs);
    oracle_expert_down(L, e, n, hs, y + p0 * H);
    for (int64_t r = 0; r < n; ++r) {
      double g = w[(int64_t)perm[p0 + r] * k + slot[p0 + r]];
      for (int64_t c = 0; c < H; ++c) y[(p0 + r) * H + c] *= g;
    }
    free(xs);
    free(hs);
  }
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < H; ++c) {
      double s = 0.0;
      for (int64_t j = 0; j < k; ++j) s += y[(int64_t)inv[t * k + j] * H + c];
      out[t * H + c] = s;
    }
  free(y);
  free(counts);
  free(offsets);
  free(perm);
  free(slot);
  free(inv);
  if (!logits_out) free(logits);
  if (!idx_out) free(idx);
  if (!w_out) free(w);
}

/* The same layer evaluated one token at a time (each output row depends only on
 * its own token), for checking sampled rows of large batches. x_rows[n][H]. */
void oracle_moe_tokens(const oracle_layer* L, int64_t n, int64_t k, const uint16_t* x_rows, double* out,
                       int32_t* idx_out, double* w_out, double* logits_out) {
  const int64_t H = L->H, I = L->I, E = L->E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n; ++t) {
    double* logits = (double*)malloc((size_t)E * sizeof(double));
    int32_t* idx = (int32_t*)malloc((size_t)k * sizeof(int32_t));
    double* w = (double*)malloc((size_t)k * sizeof(double));
    double* xs = (double*)malloc((size_t)H * sizeof(double));
    double* hs = (double*)malloc((size_t)I * sizeof(double));
    double* ys = (double*)malloc((size_t)H * sizeof(double));
    const uint16_t* xr = x_rows + t * H;
    for (int64_t e = 0; e < E; ++e) logits[e] = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double xv = oracle_bf16(xr[h]);
      for (int64_t e = 0; e < E; ++e) logits[e] += xv * (double)L->router_w[h * E + e];
    }
    if (L->router_bias)
      for (int64_t e = 0; e < E; ++e) logits[e] += (double)L->router_bias[e];
    /* one token: the same selection rule as oracle_select */
    unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || logits[e] > logits[best])) best = e;
      taken[best] = 1;
      idx[j] = (int32_t)best;
    }
    free(taken);
    double m = logits[idx[0]], s = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      w[j] = exp(logits[idx[j]] - m);
      s += w[j];
    }
    for (int64_t j = 0; j < k; ++j) w[j] /= s;
    for (int64_t c = 0; c < H; ++c) xs[c] = oracle_bf16(xr[c]);
    double* o = out + t * H;
    for (int64_t c = 0; c < H; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      oracle_expert_gateup(L, idx[j], 1, xs, hs);
      oracle_expert_down(L, idx[j], 1, hs, ys);
      for (int64_t c = 0; c < H; ++c) o[c] += w[j] * ys[c];
    }
    if (idx_out)
      for (int64_t j = 0; j < k; ++j) idx_out[t * k + j] = idx[j];
    if (w_out)
      for (int64_t j = 0; j < k; ++j) w_out[t * k + j] = w[j];
    if (logits_out)
      for (int64_t e = 0; e < E; ++e) logits_out[t * E + e] = logits[e];
    free(logits);
    free(idx);
    free(w);
    free(xs);
    free(hs);
    free(ys);
  }
}

/* The expert stage on given routing for one worker that holds the experts
 * [e0, e0 + L->E) of a layer ("Kimi-K3 NVFP4 station eight sparks", section "What has
 * to be built": a worker takes each token's 16 global expert ids, -1 for a masked one,
 * and returns rows plus the ids it served). L holds the worker's experts only: local
 * expert l is global expert e0 + l; the router is not used.
 *   out[t] = sum over j ascending, where e0 <= idx[t][j] < e0 + L->E, of
 *            w[t][j] * FFN_{idx[t][j]}(x[t])          (zero if no route is served)
 *   served[t][j] = idx[t][j] for those routes, -1 for every other (may be NULL).
 * x[T][H] bf16 bits, idx[T][k], w[T][k], out[T][H]. */
void oracle_moe_routed(const oracle_layer* L, int64_t T, int64_t k, const uint16_t* x, const int32_t* idx,
                       const double* w, int64_t e0, double* out, int32_t* served) {
  const int64_t H = L->H, I = L->I, n_local = L->E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* xs = (double*)malloc((size_t)H * sizeof(double));
    double* hs = (double*)malloc((size_t)I * sizeof(double));
    double* ys = (double*)malloc((size_t)H * sizeof(double));
    for (int64_t c = 0; c < H; ++c) xs[c] = oracle_bf16(x[t * H + c]);
    double* o = out + t * H;
    for (int64_t c = 0; c < H; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      const int64_t id = idx[t * k + j];
      const int mine = id >= e0 && id < e0 + n_local;
      if (served) served[t * k + j] = mine ? (int32_t)id : -1;
      if (!mine) continue;
      oracle_expert_gateup(L, id - e0, 1, xs, hs);
      oracle_expert_down(L, id - e0, 1, hs, ys);
      for (int64_t c = 0; c < H; ++c) o[c] += w[t * k + j] * ys[c];
    }
    free(xs);
    free(hs);
    free(ys);
  }
}

/* ---- a LatentMoE block ----------------------------------------------------------- */

/* The dense parts of a LatentMoE block: bf16 bit patterns, row-major. */
typedef struct {
  int64_t hidden, d, Is;      /* row width of x and out, routed latent width, shared intermediate */
  const uint16_t* proj_down;  /* [d][hidden] */
  const uint16_t* proj_up;    /* [hidden][d] */
  const uint16_t* shared_gu;  /* [2 Is][hidden]: rows 0..Is-1 gate, Is..2Is-1 up (or NULL) */
  const uint16_t* shared_dn;  /* [hidden][Is] (or NULL) */
} oracle_block;

/* One MoE block of a LatentMoE model, one token at a time, in fp64:
 *   "Kimi K3 optimization on GB300, Part I", section "Routed-down projection": the
 *   block projects the hidden state into the routed latent with a [d][hidden] bf16
 *   weight; section "Routed-up projection": back with a weight of the same size after
 *   the experts; "Serving Kimi K3 End to End", section 3.3: 2 shared experts that every
 *   token uses (unquantized; all of them here as one SwiGLU of intermediate Is: two
 *   experts of width f side by side are one of width 2f).
 *   logits = x W_r (+ bias), x the hidden row; top-k and weights as oracle_select
 *   lat    = W_down x
 *   routed = sum over j ascending of w_j FFN_{idx_j}(lat)   (experts of width d = L->H)
 *   out    = W_up routed + W_sd (silu(W_sg x) * (W_su x))
 * L holds the experts (width d) and router_w [hidden][E]. */
void oracle_moe_block(const oracle_layer* L, const oracle_block* B, int64_t n, int64_t k, const uint16_t* x_rows,
                      double* out, int32_t* idx_out, double* w_out, double* logits_out) {
  const int64_t Hm = B->hidden, d = B->d, Is = B->Is, I = L->I, E = L->E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n; ++t) {
    double* xs = (double*)malloc((size_t)Hm * sizeof(double));
    double* logits = (double*)malloc((size_t)E * sizeof(double));
    double* lat = (double*)malloc((size_t)d * sizeof(double));
    double* routed = (double*)malloc((size_t)d * sizeof(double));
    double* hs = (double*)malloc((size_t)(I > Is ? I : Is) * sizeof(double));
    double* ys = (double*)malloc((size_t)d * sizeof(double));
    int32_t* idx = (int32_t*)malloc((size_t)k * sizeof(int32_t));
    double* w = (double*)malloc((size_t)k * sizeof(double));
    unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
    for (int64_t h = 0; h < Hm; ++h) xs[h] = oracle_bf16(x_rows[t * Hm + h]);
    /* router on the hidden row, top-k as oracle_select */
    for (int64_t e = 0; e < E; ++e) logits[e] = 0.0;
    for (int64_t h = 0; h < Hm; ++h)
      for (int64_t e = 0; e < E; ++e) logits[e] += xs[h] * (double)L->router_w[h * E + e];
    if (L->router_bias)
      for (int64_t e = 0; e < E; ++e) logits[e] += (double)L->router_bias[e];
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || logits[e] > logits[best])) best = e;
      taken[best] = 1;
      idx[j] = (int32_t)best;
    }
    double m = logits[idx[0]], ssum = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      w[j] = exp(logits[idx[j]] - m);
      ssum += w[j];
    }
    for (int64_t j = 0; j < k; ++j) w[j] /= ssum;
    /* routed-down projection */
    for (int64_t j = 0; j < d; ++j) {
      double a = 0.0;
      for (int64_t h = 0; h < Hm; ++h) a += oracle_bf16(B->proj_down[j * Hm + h]) * xs[h];
      lat[j] = a;
    }
    /* routed experts in the latent */
    for (int64_t c = 0; c < d; ++c) routed[c] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      oracle_expert_gateup(L, idx[j], 1, lat, hs);
      oracle_expert_down(L, idx[j], 1, hs, ys);
      for (int64_t c = 0; c < d; ++c) routed[c] += w[j] * ys[c];
    }
    /* routed-up projection plus the shared experts */
    for (int64_t i = 0; i < Is; ++i) {
      double g = 0.0, u = 0.0;
      for (int64_t h = 0; h < Hm; ++h) {
        g += oracle_bf16(B->shared_gu[i * Hm + h]) * xs[h];
        u += oracle_bf16(B->shared_gu[(Is + i) * Hm + h]) * xs[h];
      }
      hs[i] = g / (1.0 + exp(-g)) * u;
    }
    double* o = out + t * Hm;
    for (int64_t c = 0; c < Hm; ++c) {
      double a = 0.0;
      for (int64_t j = 0; j < d; ++j) a += oracle_bf16(B->proj_up[c * d + j]) * routed[j];
      double sh = 0.0;
      for (int64_t i = 0; i < Is; ++i) sh += oracle_bf16(B->shared_dn[c * Is + i]) * hs[i];
      o[c] = a + sh;
    }
    if (idx_out)
      for (int64_t j = 0; j < k; ++j) idx_out[t * k + j] = idx[j];
    if (w_out)
      for (int64_t j = 0; j < k; ++j) w_out[t * k + j] = w[j];
    if (logits_out)
      for (int64_t e = 0; e < E; ++e) logits_out[t * E + e] = logits[e];
    free(xs);
    free(logits);
    free(lat);
    free(routed);
    free(hs);
    free(ys);
    free(idx);
    free(w);
    free(taken);
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
