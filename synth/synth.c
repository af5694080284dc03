/*
 * synth.c -- seeded synthetic inputs for the routed expert layer.
 *
 * This module is shared by the oracle-side tests and by the CUDA-side tests and
 * benchmark. It holds none of the layer's arithmetic (no router, no top-k, no
 * dequantisation, no expert GEMM, no combine). It only produces input bytes:
 *
 *   - a counter-based generator: every value is a pure function of
 *     (seed, stream, index) through the SplitMix64 finaliser (Steele, Lea and
 *     Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), so
 *     the data do not depend on the number of threads that produced them;
 *   - standard normals by the Box-Muller transform (Box and Muller, 1958);
 *   - an NVFP4 *encoder* (E2M1 codes, one E4M3 block scale per 16 values along
 *     K, one fp32 scale per tensor) that turns Gaussian weights into the bytes
 *     the layer consumes;
 *   - a Zipf(s) router bias over a seeded permutation of the experts.
 *
 * Sources for the formats: "Serving Kimi-K3 ... with 8xB300 GPUs" (section
 * "The model, as the serving system sees it": E2M1 values, two per byte) and
 * "Kimi-K3 NVFP4 station eight sparks" (section "What has to be built": an FP8
 * scale per 16 values plus a per-expert global scale). The encoder's rounding
 * choices are a data-generation convention only: both the oracle and the CUDA
 * path read the same bytes.
 *
 * Built as a shared library with -ffp-contract=off so x86-64 and aarch64 give
 * the same bytes up to the host libm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define SYNTH_STREAM_X 1ull
#define SYNTH_STREAM_ROUTER 2ull
#define SYNTH_STREAM_GATE 3ull
#define SYNTH_STREAM_UP 4ull
#define SYNTH_STREAM_DOWN 5ull
#define SYNTH_STREAM_ZIPF 6ull
#define SYNTH_STREAM_LOGITS 7ull
#define SYNTH_STREAM_DENSE 8ull /* bf16 dense weights; the caller's stream id is added below it */

/* SplitMix64 finaliser applied to a counter built from (seed, stream, i). */
static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t synth_hash(uint64_t seed, uint64_t stream, uint64_t i) {
  uint64_t key = mix64(seed * 0x9E3779B97F4A7C15ull + 0x632BE59BD9B4E019ull);
  key = mix64(key ^ (stream * 0xD1B54A32D192ED03ull));
  return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}

/* Box-Muller on one pair of counters: element 2p gets r*cos, 2p+1 gets r*sin. */
static inline void normal_pair(uint64_t seed, uint64_t stream, uint64_t p, float* n0, float* n1) {
  uint64_t a = synth_hash(seed, stream, 2 * p);
  uint64_t b = synth_hash(seed, stream, 2 * p + 1);
  float u1 = (float)((a >> 40) + 1) * (1.0f / 16777216.0f); /* (0, 1] */
  float u2 = (float)(b >> 40) * (1.0f / 16777216.0f);       /* [0, 1) */
  float r = sqrtf(-2.0f * logf(u1));
  float th = 6.2831853071795864769f * u2;
  *n0 = r * cosf(th);
  *n1 = r * sinf(th);
}

double synth_normal(uint64_t seed, uint64_t stream, uint64_t i) {
  float n0, n1;
  normal_pair(seed, stream, i >> 1, &n0, &n1);
  return (i & 1) ? n1 : n0;
}

/* n normals (times scale) of one stream, written as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, float scale, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < (n + 1) / 2; ++p) {
    float n0, n1;
    normal_pair(seed, stream, (uint64_t)p, &n0, &n1);
    out[2 * p] = n0 * scale;
    if (2 * p + 1 < n) out[2 * p + 1] = n1 * scale;
  }
}

/* fp32 -> bf16 bits, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Activations x[T][H] ~ N(0, 1), stored as bf16 bits. */
void synth_x_bf16(uint64_t seed, int64_t T, int64_t H, uint16_t* out) {
  int64_t n = T * H;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < (n + 1) / 2; ++p) {
    float n0, n1;
    normal_pair(seed, SYNTH_STREAM_X, (uint64_t)p, &n0, &n1);
    out[2 * p] = f32_to_bf16_bits(n0);
    if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_bits(n1);
  }
}

/* Router weights W_r[H][E] ~ N(0, 1/H), fp32. */
void synth_router(uint64_t seed, int64_t H, int64_t E, float* out) {
  synth_normal_f32(seed, SYNTH_STREAM_ROUTER, H * E, (float)(1.0 / sqrt((double)H)), out);
}

/* A bf16 dense weight of n elements ~ N(0, scale^2), as bf16 bits (round to nearest even);
 * `which` tells the block's tensors apart (routed-down, routed-up, shared gate/up, shared
 * down). */
void synth_bf16_normal(uint64_t seed, uint64_t which, int64_t n, float scale, uint16_t* out) {
  const uint64_t stream = (SYNTH_STREAM_DENSE << 40) | which;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < (n + 1) / 2; ++p) {
    float n0, n1;
    normal_pair(seed, stream, (uint64_t)p, &n0, &n1);
    out[2 * p] = f32_to_bf16_bits(n0 * scale);
    if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_bits(n1 * scale);
  }
}

/* Logits[T][E] ~ N(0, 1), fp32, for exercising the selection step on its own. */
void synth_logits(uint64_t seed, int64_t T, int64_t E, float* out) {
  synth_normal_f32(seed, SYNTH_STREAM_LOGITS, T * E, 1.0f, out);
}

/* ---- NVFP4 encoder (data generation only) ---------------------------------- */

/* Nearest E4M3 ("fn" variant: bias 7, max 448, no infinities) to a
 * non-negative finite x, ties to even, saturating at 448. Returns the byte. */
uint8_t synth_e4m3_encode(double x) {
  if (!(x > 0.0)) return 0;
  if (x >= 448.0) return 0x7E;
  if (x < 0.015625) { /* below 2^-6: subnormal grid of step 2^-9 */
    double q = nearbyint(x * 512.0);
    return (uint8_t)q; /* q == 8 is the smallest normal, code 0x08 */
  }
  int e;
  double m = frexp(x, &e); /* x = m * 2^e, m in [0.5, 1) */
  e -= 1;                  /* x = (2m) * 2^e, 2m in [1, 2) */
  double mq = nearbyint((2.0 * m - 1.0) * 8.0);
  if (mq >= 8.0) {
    mq = 0.0;
    e += 1;
  }
  if (e > 8 || (e == 8 && mq > 6.0)) return 0x7E;
  return (uint8_t)(((e + 7) << 3) | (int)mq);
}

/* Value of an E4M3 byte, used by the encoder to divide by the stored scale. */
static double e4m3_value_for_encoder(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest E2M1 code to v (ties to the even code), saturating at +-6. */
uint8_t synth_e2m1_encode(double v) {
  static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double a = fabs(v);
  int c = 7;
  for (int i = 0; i < 7; ++i) {
    double mid = 0.5 * (grid[i] + grid[i + 1]);
    if (a < mid) { c = i; break; }
    if (a == mid) { c = (i % 2 == 0) ? i : i + 1; break; }
  }
  if (c == 0) return 0;
  return (uint8_t)(c | ((v < 0.0) ? 8 : 0));
}

/* Quantise w[rows][K] (K % 16 == 0) to NVFP4:
 *   G = amax(tensor) / (6 * 448);  per block of 16 along K: s = E4M3(amax(block) / 6 / G);
 *   code = E2M1(w / (s * G)).
 * codes[rows][K/2] (element k in byte k/2, low nibble = even k), scales[rows][K/16]. */
void synth_quantize_nvfp4(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                          float* global_scale) {
  double amax = 0.0;
  for (int64_t i = 0; i < rows * K; ++i) {
    double a = fabs((double)w[i]);
    if (a > amax) amax = a;
  }
  float G = (amax > 0.0) ? (float)(amax / (6.0 * 448.0)) : 1.0f;
  *global_scale = G;
  for (int64_t r = 0; r < rows; ++r) {
    const float* wr = w + r * K;
    for (int64_t b = 0; b < K / 16; ++b) {
      double bmax = 0.0;
      for (int j = 0; j < 16; ++j) {
        double a = fabs((double)wr[b * 16 + j]);
        if (a > bmax) bmax = a;
      }
      uint8_t sq = synth_e4m3_encode(bmax / 6.0 / (double)G);
      scales[r * (K / 16) + b] = sq;
      double sdec = e4m3_value_for_encoder(sq) * (double)G;
      for (int j = 0; j < 16; j += 2) {
        uint8_t lo = 0, hi = 0;
        if (sdec > 0.0) {
          lo = synth_e2m1_encode((double)wr[b * 16 + j] / sdec);
          hi = synth_e2m1_encode((double)wr[b * 16 + j + 1] / sdec);
        }
        codes[r * (K / 2) + (b * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

/* All experts of one layer. Gate and up are separate [I][H] tensors (each with
 * its own global scale) stored as rows 0..I-1 (gate) and I..2I-1 (up) of one
 * [2I][H] matrix; down is [H][I]. Weights ~ N(0, 1/fan_in) before quantisation,
 * fan_in = H for gate/up and I for down. */
void synth_experts(uint64_t seed, int64_t H, int64_t I, int64_t E, uint8_t* gu_codes, uint8_t* gu_scales,
                   float* gu_global, uint8_t* dn_codes, uint8_t* dn_scales, float* dn_global) {
  const float sg = (float)(1.0 / sqrt((double)H));
  const float sd = (float)(1.0 / sqrt((double)I));
#pragma omp parallel
  {
    float* buf = (float*)malloc((size_t)(I * H) * sizeof(float));
#pragma omp for schedule(dynamic, 1)
    for (int64_t e = 0; e < E; ++e) {
      uint8_t* gc = gu_codes + e * (2 * I) * (H / 2);
      uint8_t* gs = gu_scales + e * (2 * I) * (H / 16);
      for (int which = 0; which < 2; ++which) {
        uint64_t stream = ((which == 0 ? SYNTH_STREAM_GATE : SYNTH_STREAM_UP) << 40) | (uint64_t)e;
        for (int64_t p = 0; p < (I * H) / 2; ++p) {
          float n0, n1;
          normal_pair(seed, stream, (uint64_t)p, &n0, &n1);
          buf[2 * p] = n0 * sg;
          buf[2 * p + 1] = n1 * sg;
        }
        synth_quantize_nvfp4(buf, I, H, gc + which * I * (H / 2), gs + which * I * (H / 16),
                             &gu_global[e * 2 + which]);
      }
      uint64_t stream = (SYNTH_STREAM_DOWN << 40) | (uint64_t)e;
      for (int64_t p = 0; p < (H * I) / 2; ++p) {
        float n0, n1;
        normal_pair(seed, stream, (uint64_t)p, &n0, &n1);
        buf[2 * p] = n0 * sd;
        buf[2 * p + 1] = n1 * sd;
      }
      synth_quantize_nvfp4(buf, H, I, dn_codes + e * H * (I / 2), dn_scales + e * H * (I / 16), &dn_global[e]);
    }
    free(buf);
  }
}

/* Router bias for skewed routing: expert of popularity rank r (1-based, over a
 * seeded permutation) gets bias -s * ln(r), i.e. ln p with p proportional to r^-s. */
void synth_zipf_bias(uint64_t seed, int64_t E, double s, float* bias) {
  int64_t* perm = (int64_t*)malloc((size_t)E * sizeof(int64_t));
  for (int64_t i = 0; i < E; ++i) perm[i] = i;
  for (int64_t i = E - 1; i > 0; --i) { /* Fisher-Yates */
    int64_t j = (int64_t)(synth_hash(seed, SYNTH_STREAM_ZIPF, (uint64_t)i) % (uint64_t)(i + 1));
    int64_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  for (int64_t r = 0; r < E; ++r) bias[perm[r]] = (float)(-s * log((double)(r + 1)));
  free(perm);
}

int synth_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
