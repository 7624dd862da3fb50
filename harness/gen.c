/*
 * Seeded synthetic input generator for the quantized sparse MoE layer.
 *
 * Test and benchmark infrastructure only.  It produces the BYTES that both the
 * fp64 oracle and the CUDA path consume (activations, router weights, bias,
 * packed expert weights with their scales and zero-points).  It holds none of
 * the layer's forward arithmetic: no routing, no dequantisation, no FFN.
 *
 * Randomness: a counter-based generator.  Stream key = splitmix64 finaliser of
 * (seed, tag, a, b); draw i of a stream is the splitmix64 output for counter
 * i+1, so every value depends only on (seed, tag, a, b, i) and never on thread
 * order.  One 64-bit draw gives two 24-bit uniforms; Box-Muller turns them
 * into two normals.  The logarithm and sine/cosine in Box-Muller are this
 * file's own polynomial approximations (log via the atanh series, sin/cos via
 * Taylor series after quadrant reduction; absolute error < 1e-6), written so
 * that the compiler can vectorise them and so that results are identical on
 * every IEEE platform (only +, -, *, / and sqrt, no FMA contraction).
 *
 * Quantisers (the offline conversion step the pages describe as per-output-
 * channel scale + zero_point, "Colibri walkthrough" page, section 3.4):
 *   int4, groups of 128 inputs per output row: lo/hi = min/max of the group,
 *     s = fp16((hi-lo)/15) (round to nearest even), s==0 -> 1,
 *     z = clamp(rint(-lo/s), 0, 15), q = clamp(rint(w/s) + z, 0, 15).
 *   int8, per output row: same with 255 and an fp32 scale.
 * rint() rounds half to even (default FP environment).  Build with
 * -ffp-contract=off so results do not depend on FMA contraction.
 *
 * Packing (the layout the library's header documents):
 *   int4 q   : [N][K/2] bytes, byte j = q[2j] | q[2j+1] << 4 (low nibble = even k)
 *   int4 s   : [N][K/128] fp16 bit patterns
 *   int4 zp  : [N][ceil(K/256)] bytes, low nibble = even group
 *   int8 q   : [N][K] bytes;  s : [N] fp32;  zp : [N] bytes
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

#define GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t gen_stream_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b) {
  uint64_t k = mix64(seed + GOLDEN);
  k = mix64(k ^ (tag * GOLDEN + 1));
  k = mix64(k ^ (a * 0xD1B54A32D192ED03ULL + 2));
  k = mix64(k ^ (b * 0xAEF17502108EF2D9ULL + 3));
  return k;
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* two uniforms in (0,1) with 24-bit resolution */
static inline void unif2(uint64_t r, float* u1, float* u2) {
  *u1 = ((float)(r >> 40) + 0.5f) * (1.0f / 16777216.0f);
  *u2 = ((float)((r >> 16) & 0xFFFFFFu) + 0.5f) * (1.0f / 16777216.0f);
}

/* ln(u) for u in (0, 1]: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
   ln(m) = 2 atanh(f), f = (m-1)/(m+1), series to f^9 (|f| < 0.172) */
static inline float gen_logf(float u) {
  uint32_t b; memcpy(&b, &u, 4);
  int e = (int)((b >> 23) & 0xFF) - 127;
  uint32_t mb = (b & 0x7FFFFFu) | 0x3F800000u;
  float m; memcpy(&m, &mb, 4);                  /* m in [1, 2) */
  int big = m > 1.41421356f;
  m = big ? m * 0.5f : m;
  e += big;
  float f = (m - 1.0f) / (m + 1.0f), f2 = f * f;
  float p = 1.0f / 9.0f;
  p = p * f2 + 1.0f / 7.0f;
  p = p * f2 + 1.0f / 5.0f;
  p = p * f2 + 1.0f / 3.0f;
  p = p * f2 + 1.0f;
  return 2.0f * f * p + (float)e * 0.693147180559945f;
}

/* sin and cos of 2*pi*t for t in (0, 1): quadrant j = nearest quarter turn,
   remainder angle in [-pi/4, pi/4], Taylor series to degree 9 / 10 */
static inline void gen_sincos_turns(float t, float* sn, float* cs) {
  float j = (float)(int)(t * 4.0f + 0.5f);      /* 0..4 */
  float a = (t - 0.25f * j) * 6.28318530718f;   /* [-pi/4, pi/4] */
  float a2 = a * a;
  float sa = a - a * a2 * (1.0f / 6.0f - a2 * (1.0f / 120.0f - a2 * (1.0f / 5040.0f - a2 * (1.0f / 362880.0f))));
  float ca = 1.0f - a2 * (0.5f - a2 * (1.0f / 24.0f - a2 * (1.0f / 720.0f - a2 * (1.0f / 40320.0f - a2 * (1.0f / 3628800.0f)))));
  int q = ((int)j) & 3;                          /* rotate by q quarter turns */
  float s0 = q == 0 ? sa : (q == 1 ? ca : (q == 2 ? -sa : -ca));
  float c0 = q == 0 ? ca : (q == 1 ? -sa : (q == 2 ? -ca : sa));
  *sn = s0;
  *cs = c0;
}

/* normal number i of stream `key` (pairs share one draw) */
static inline float normal_at(uint64_t key, uint64_t i) {
  float u1, u2, sn, cs;
  unif2(draw(key, i >> 1), &u1, &u2);
  float r = sqrtf(-2.0f * gen_logf(u1));
  gen_sincos_turns(u2, &sn, &cs);
  return (i & 1) ? r * sn : r * cs;
}

void gen_normal_f32(uint64_t key, int64_t n, float mean, float std, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mean + std * normal_at(key, (uint64_t)i);
}

void gen_uniform_f32(uint64_t key, int64_t n, float lo, float hi, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float u1, u2;
    unif2(draw(key, (uint64_t)i), &u1, &u2);
    out[i] = lo + (hi - lo) * u1;
  }
}

/* random permutation of 0..n-1 (Fisher-Yates driven by the stream) */
void gen_permutation(uint64_t key, int32_t n, int32_t* out) {
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    int32_t j = (int32_t)(draw(key, (uint64_t)i) % (uint64_t)(i + 1));
    int32_t t = out[i]; out[i] = out[j]; out[j] = t;
  }
}

/* float -> IEEE binary16 bits, round to nearest even (software, no FP16 type) */
uint16_t gen_f32_to_f16_bits(float f) {
  uint32_t x; memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);           /* rounds to >= 65520: inf */
  if (ax < 0x38800000u) {                                              /* f16 subnormal or zero */
    if (ax < 0x33000000u) return (uint16_t)sign;                       /* < 2^-25: rounds to 0 */
    uint32_t e = ax >> 23, m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126 - e;                                          /* value = m * 2^(e-150); unit 2^-24 */
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) q++;
    return (uint16_t)(sign | q);
  }
  uint32_t e = (ax >> 23) - 112, m = ax & 0x7FFFFFu;
  uint32_t q = (e << 10) | (m >> 13), rem = m & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1))) q++;
  return (uint16_t)(sign | q);
}

static float f16_bits_to_f32(uint16_t h) {
  uint32_t s = (uint32_t)(h & 0x8000u) << 16, e = (h >> 10) & 0x1F, m = h & 0x3FF, x;
  if (e == 0) { float v = (float)m * (1.0f / 16777216.0f); return (h & 0x8000u) ? -v : v; }
  if (e == 31) x = s | 0x7F800000u | (m << 13);
  else x = s | ((e + 112) << 23) | (m << 13);
  float f; memcpy(&f, &x, 4); return f;
}

/* float -> bfloat16 bits, round to nearest even */
uint16_t gen_f32_to_bf16_bits(float f) {
  uint32_t x; memcpy(&x, &f, 4);
  if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  return (uint16_t)((x + 0x7FFFu + lsb) >> 16);
}

void gen_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f32_to_bf16_bits(in[i]);
}

void gen_f32_to_f16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f32_to_f16_bits(in[i]);
}

static inline float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* quantise one row of K floats to int4 groups of 128 */
static void quant_row_int4(const float* w, int K, uint8_t* q, uint16_t* s, uint8_t* z) {
  int G = K / 128;
  memset(z, 0, (size_t)(G + 1) / 2);
  for (int g = 0; g < G; ++g) {
    const float* wg = w + (size_t)g * 128;
    float lo = wg[0], hi = wg[0];
    for (int i = 1; i < 128; ++i) { lo = wg[i] < lo ? wg[i] : lo; hi = wg[i] > hi ? wg[i] : hi; }
    uint16_t sb = gen_f32_to_f16_bits((hi - lo) / 15.0f);
    float sc = f16_bits_to_f32(sb);
    if (!(sc > 0.0f)) { sb = 0x3C00u; sc = 1.0f; }
    s[g] = sb;
    int zz = (int)clampf(rintf(-lo / sc), 0.0f, 15.0f);
    z[g >> 1] |= (uint8_t)(zz << ((g & 1) * 4));
    for (int i = 0; i < 128; i += 2) {
      int q0 = (int)clampf(rintf(wg[i] / sc) + (float)zz, 0.0f, 15.0f);
      int q1 = (int)clampf(rintf(wg[i + 1] / sc) + (float)zz, 0.0f, 15.0f);
      q[((size_t)g * 128 + i) >> 1] = (uint8_t)(q0 | (q1 << 4));
    }
  }
}

static void quant_row_int8(const float* w, int K, uint8_t* q, float* s, uint8_t* z) {
  float lo = w[0], hi = w[0];
  for (int i = 1; i < K; ++i) { lo = w[i] < lo ? w[i] : lo; hi = w[i] > hi ? w[i] : hi; }
  float sc = (hi - lo) / 255.0f;
  if (!(sc > 0.0f)) sc = 1.0f;
  *s = sc;
  int zz = (int)clampf(rintf(-lo / sc), 0.0f, 255.0f);
  *z = (uint8_t)zz;
  for (int i = 0; i < K; ++i) q[i] = (uint8_t)(int)clampf(rintf(w[i] / sc) + (float)zz, 0.0f, 255.0f);
}

/* quantise a dense [N][K] matrix (used by tests that build weights by hand) */
void gen_quant_int4(const float* w, int N, int K, uint8_t* q, uint16_t* s, uint8_t* z) {
  int G = K / 128, ZB = (G + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n)
    quant_row_int4(w + (size_t)n * K, K, q + (size_t)n * (K / 2), s + (size_t)n * G, z + (size_t)n * ZB);
}

void gen_quant_int8(const float* w, int N, int K, uint8_t* q, float* s, uint8_t* z) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) quant_row_int8(w + (size_t)n * K, K, q + (size_t)n * K, s + n, z + n);
}

/* fill buf[0..K) with normals base..base+K-1 of stream `key` times std (base even) */
static void normal_row(uint64_t key, uint64_t base, int K, float std, float* buf) {
  int K2 = K / 2;
  for (int p = 0; p < K2; ++p) {
    float u1, u2, sn, cs;
    unif2(draw(key, (base >> 1) + (uint64_t)p), &u1, &u2);
    float r = std * sqrtf(-2.0f * gen_logf(u1));
    gen_sincos_turns(u2, &sn, &cs);
    buf[2 * p] = r * cs;
    buf[2 * p + 1] = r * sn;
  }
  if (K & 1) buf[K - 1] = std * normal_at(key, base + (uint64_t)(K - 1));
}

/*
 * Draw W[N][K] ~ N(0, std^2) from stream `key` (normal index n*K + k) and
 * quantise it row by row without materialising the float matrix.
 * qtype 0 = int4 group-128, 1 = int8 per-channel.  Returns 0, or -1 on bad K.
 */
int gen_quant_matrix(uint64_t key, int qtype, int N, int K, float std, uint8_t* q, void* s, uint8_t* z) {
  if ((qtype == 0 && (K % 128) != 0) || (K % 2) != 0 || K > 65536) return -1;
  int G = K / 128, ZB = (G + 1) / 2;
#pragma omp parallel
  {
    float buf[65536];
#pragma omp for schedule(static)
    for (int n = 0; n < N; ++n) {
      normal_row(key, (uint64_t)n * (uint64_t)K, K, std, buf);
      if (qtype == 0)
        quant_row_int4(buf, K, q + (size_t)n * (K / 2), (uint16_t*)s + (size_t)n * G, z + (size_t)n * ZB);
      else
        quant_row_int8(buf, K, q + (size_t)n * K, (float*)s + n, z + n);
    }
  }
  return 0;
}
