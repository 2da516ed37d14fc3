/*
 * tq_oracle.c -- plain, slow CPU oracle for TurboQuant speculative-verify
 * decode attention over a quantised paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library; both implement the same written spec.
 *
 * Sources (web pages, cited by title and section):
 *   [SD]  "spec-decode-intel-arc" (bryanvine.github.io/turboquant-xpu,
 *         2026-04-14): section "Context: TurboQuant, speculative decoding,
 *         and the gap" (the method: Walsh-Hadamard rotation, precomputed
 *         Lloyd-Max codebook for keys, uniform scalar quantisation for values;
 *         the presets k8v4 / k3v4_nc); section "Roofline" (196-byte k8v4 slot,
 *         16-token blocks); section "Part 3: The fused Triton kernel" (one K
 *         dequant per tile shared by all draft queries, online softmax,
 *         ATTN_SCALE); section "Part 4: The causal correction" (draft query n
 *         sees cached_len + n + 1 tokens); section "Part 6" (FP8 keys are a
 *         plain bitcast, k3v4_nc keys are centroid gathers + norm correction).
 *   [S3]  "sycl-three-attempts-arc-b70" (2026-04-15): section "Part 3:
 *         joint_matrix + split-KV" (NUM_KV_SPLITS partial attention, stage 2
 *         log-sum-exp reduction).
 *
 * Readings where the pages are silent (the GPU library follows the same ones):
 *   - codebook: 8-level (k3 presets), 16-level (k4v4_nc) or 4-level (k2v4_nc)
 *     Lloyd-Max for N(0, 1/D), derived in fp64 and rounded to fp16; decision
 *     boundaries are fp32 midpoints of adjacent centroids;
 *   - rotation: unnormalised Sylvester Walsh-Hadamard butterflies (h = 1, 2,
 *     4, ..., 64), no random signs; the rotated unit vector is H k / (|k| sqrt D);
 *   - norm correction: nc = |k| / |c_hat| stored as fp16;
 *   - values: asymmetric min/max, zero = min, scale = (max - min) / 15 rounded
 *     up to fp16, codes rounded half-to-even and clamped to [0, 15];
 *   - FP8 keys: e4m3, round-to-nearest-even, saturating to +-448, NaN -> 0x7F,
 *     no scale and no rotation;
 *   - bit order: key codes LSB-first in a little-endian stream; value codes
 *     coordinate-major (byte 8d + t/2, low nibble = even token t); the page for
 *     one (block, kv-head) is planar (below).
 *
 * Arithmetic: the encoder is fp32 in a fixed operation order (this file must be
 * compiled with -ffp-contract=off and without -ffast-math); the attention part
 * is fp64 over the decoded cache.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 128
#define BLK 16

enum {
  PRESET_K8V4 = 0,
  PRESET_K3V4_NC = 1,
  PRESET_K3V4 = 2,
  PRESET_K3V4_NC_RS = 3,
  PRESET_K4V4_NC = 4,
  PRESET_K2V4_NC = 5
};
/* k3v4_nc, k3v4 and k3v4_nc_rs share the key coding and the page; k3v4
 * stores the plain norm |k| as the key factor instead of the corrected
 * |k| / |c_hat|; k3v4_nc_rs rotates by H diag(s) instead of H, s a fixed
 * random sign vector.  k4v4_nc and k2v4_nc are k3v4_nc with 16- and 4-level
 * codebooks (the other widths of "3-4 bit" TurboQuant, [SD] "Context"). */
static int is_k3(int preset) {
  return preset == PRESET_K3V4_NC || preset == PRESET_K3V4 || preset == PRESET_K3V4_NC_RS;
}
/* bits per key code: 0 for the FP8 keys of k8v4 */
int oracle_key_bits(int preset) {
  if (is_k3(preset)) return 3;
  if (preset == PRESET_K4V4_NC) return 4;
  if (preset == PRESET_K2V4_NC) return 2;
  return 0;
}

/* SplitMix64 (Steele, Lea and Flood; the output function as published by
 * Vigna): output j of the generator seeded with seed is
 * mix(seed + (j + 1) * 0x9E3779B97F4A7C15). */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t j) {
  uint64_t z = seed + (j + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* The sign vector of preset k3v4_nc_rs: s_j = -1 where the top bit of output
 * j of SplitMix64 seeded with 0x54515F5349474E53 ("TQ_SIGNS") is set. */
#define RS_SEED 0x54515F5349474E53ull
int oracle_rs_sign(int j) { return (oracle_splitmix64(RS_SEED, (uint64_t)j) >> 63) ? -1 : 1; }

/* Planar page layout for one (block, kv-head), 16 tokens (value codes stored
 * coordinate-major: 128 coordinates x 8 bytes of 16 nibbles).  Byte budgets:
 * k8v4 slot = 128 (K) + 64 (V codes) + 2 (scale) + 2 (zero) = 196 B, which is
 * the slot_size_aligned the [SD] "Roofline" section multiplies out;
 * k3v4_nc slot = 48 (codes) + 2 (nc) + 64 + 2 + 2 = 118 B, aligned to 120 B,
 * the size that reproduces the 273.1 FLOP/B of the [SD] post-fusion profile. */
#define K8_K_OFF 0
#define K8_V_OFF 2048
#define K8_S_OFF 3072
#define K8_Z_OFF 3104
#define K8_PAGE 3136
#define K3_K_OFF 0
#define K3_NC_OFF 768
#define K3_V_OFF 800
#define K3_S_OFF 1824
#define K3_Z_OFF 1856
#define K3_PAGE 1920
/* k4v4_nc slot = 64 + 2 + 64 + 2 + 2 = 134 B and k2v4_nc slot = 32 + 2 + 64 +
 * 2 + 2 = 102 B, each rounded up to a multiple of 4 bytes like k3v4_nc's
 * (136 B and 104 B): the same planar page, 32 B of padding at the end */
#define K4_PAGE 2176
#define K2_PAGE 1664

/* Offsets of the planar page of a coded-key preset: codes [16][code_bytes]
 * @0, key factor fp16 [16], value codes [128][8], value scale fp16 [16],
 * value zero fp16 [16]. */
typedef struct {
  int code_bytes, nc_off, v_off, s_off, z_off, page;
} coded_layout;

static coded_layout coded_page(int preset) {
  coded_layout l;
  l.code_bytes = D * oracle_key_bits(preset) / 8;
  l.nc_off = BLK * l.code_bytes;
  l.v_off = l.nc_off + 2 * BLK;
  l.s_off = l.v_off + BLK * D / 2;
  l.z_off = l.s_off + 2 * BLK;
  l.page = preset == PRESET_K4V4_NC ? K4_PAGE : preset == PRESET_K2V4_NC ? K2_PAGE : K3_PAGE;
  return l;
}

long oracle_page_bytes(int preset) {
  if (preset == PRESET_K8V4) return K8_PAGE;
  if (oracle_key_bits(preset) > 0) return coded_page(preset).page;
  return -1;
}

/* ------------------------------------------------------------------ fp16 */

/* IEEE binary16 -> binary32, exact. */
float oracle_h2f(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  float v;
  if (e == 0)
    v = ldexpf((float)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexpf((float)(1024 + m), e - 25);
  return s ? -v : v;
}

/* binary64 -> binary16, round to nearest, ties to even (a float argument is
 * widened exactly first, so this is also the single-rounding float -> half). */
uint16_t oracle_d2h_rn(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return (uint16_t)(sign | 0x7E00);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);      /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;            /* a in [2^e, 2^(e+1)) */
  if (e < -14) {     /* subnormal range: step 2^-24 */
    double q = rint(a / ldexp(1.0, -24));
    return (uint16_t)(sign | (uint16_t)q); /* q == 1024 is the smallest normal */
  }
  double q = rint(a / ldexp(1.0, e - 10)); /* in [1024, 2048] */
  if (q == 2048.0) { q = 1024.0; e += 1; }
  if (e + 15 >= 31) return (uint16_t)(sign | 0x7C00);
  return (uint16_t)(sign | ((e + 15) << 10) | ((int)q - 1024));
}

uint16_t oracle_f2h_rn(float x) { return oracle_d2h_rn((double)x); }

/* ------------------------------------------------------------------ e4m3 */

/* e4m3 (OCP "fn" variant: no infinities, S.1111.111 is NaN) -> binary64. */
double oracle_e4m3_to_double(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* binary16 -> e4m3, round to nearest even, saturate to +-448, NaN -> 0x7F.
 * The key path of preset k8v4 ([SD] "Part 6": keys stored as FP8). */
uint8_t oracle_e4m3_from_half(uint16_t h) {
  float xf = oracle_h2f(h);
  if (isnan(xf)) return 0x7F;
  uint8_t sign = signbit(xf) ? 0x80 : 0;
  double a = fabs((double)xf);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  e -= 1;
  if (e < -6) { /* e4m3 subnormals: step 2^-9; q == 8 is the smallest normal */
    double q = rint(a / ldexp(1.0, -9));
    return (uint8_t)(sign | (uint8_t)q);
  }
  double q = rint(a / ldexp(1.0, e - 3)); /* in [8, 16] */
  if (q == 16.0) { q = 8.0; e += 1; }
  int code = ((e + 7) << 3) | ((int)q - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------- codebook */

static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
/* upper tail Q(x) = P(X > x) for X ~ N(0,1), stable for both signs */
static double qtail(double x) { return 0.5 * erfc(x / sqrt(2.0)); }

static double norm_quantile(double p) { /* bisection on the CDF */
  double lo = -40.0, hi = 40.0;
  for (int i = 0; i < 300; ++i) {
    double mid = 0.5 * (lo + hi);
    if (1.0 - qtail(mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

/* n-level Lloyd-Max quantiser of the standard normal, fp64 (n <= 16).
 * Lloyd's two conditions are iterated from the equiprobable quantile
 * midpoints: every decision boundary is the midpoint of its two neighbouring
 * levels, and every level is the conditional mean of N(0,1) over its cell,
 *   c = (phi(a) - phi(b)) / (Q(a) - Q(b)).
 * Returns the iteration count, or -1 if it did not converge.  ([SD] "Context":
 * a precomputed Lloyd-Max codebook for the rotated key coordinates.) */
int oracle_lloyd_max(int n, double* c_out) {
  double c[16];
  if (n < 2 || n > 16) return -1;
  for (int m = 0; m < n; ++m) c[m] = norm_quantile((m + 0.5) / n);
  for (int it = 1; it <= 200000; ++it) {
    double b[17];
    b[0] = -INFINITY;
    b[n] = INFINITY;
    for (int m = 0; m < n - 1; ++m) b[m + 1] = 0.5 * (c[m] + c[m + 1]);
    double delta = 0.0;
    for (int m = 0; m < n; ++m) {
      double lo = b[m], hi = b[m + 1];
      double pa = isinf(lo) ? 0.0 : phi(lo), pb = isinf(hi) ? 0.0 : phi(hi);
      double qa = isinf(lo) ? 1.0 : qtail(lo), qb = isinf(hi) ? 0.0 : qtail(hi);
      double nc = (pa - pb) / (qa - qb);
      double d = fabs(nc - c[m]);
      if (d > delta) delta = d;
      c[m] = nc;
    }
    if (delta < 1e-15) {
      memcpy(c_out, c, n * sizeof(double));
      return it;
    }
  }
  memcpy(c_out, c, n * sizeof(double));
  return -1;
}

int oracle_lloyd_max8(double c_out[8]) { return oracle_lloyd_max(8, c_out); }

/* The key codebook of an n-level preset: Lloyd-Max levels for N(0, 1/D)
 * rounded to fp16 (ascending).  Returned as fp16 bit patterns. */
int oracle_codebook_n(int n, uint16_t* out) {
  double c[16];
  int it = oracle_lloyd_max(n, c);
  double sigma = 1.0 / sqrt((double)D);
  for (int m = 0; m < n; ++m) out[m] = oracle_d2h_rn(c[m] * sigma);
  return it;
}

/* The 8-level codebook of the k3 presets. */
int oracle_codebook16(uint16_t out[8]) { return oracle_codebook_n(8, out); }

/* Number of key levels of a preset (0 for k8v4). */
int oracle_key_levels(int preset) {
  int b = oracle_key_bits(preset);
  return b ? 1 << b : 0;
}

/* -------------------------------------------------------------- encoder */

/* Unnormalised Walsh-Hadamard transform, Sylvester order, in place, fp32:
 * for h = 1, 2, 4, ..., 64 each pair (i, i + h) with (i & h) == 0 becomes
 * (t_i + t_{i+h}, t_i - t_{i+h}).  Equals H x with H_ij = (-1)^popcount(i & j).
 * ([SD] "Context": the Walsh-Hadamard rotation of keys.) */
void oracle_wht_f32(float t[D]) {
  for (int h = 1; h < D; h <<= 1)
    for (int i = 0; i < D; ++i)
      if (!(i & h)) {
        float a = t[i], b = t[i + h];
        t[i] = a + b;
        t[i + h] = a - b;
      }
}

void oracle_wht_f64(double t[D]) {
  for (int h = 1; h < D; h <<= 1)
    for (int i = 0; i < D; ++i)
      if (!(i & h)) {
        double a = t[i], b = t[i + h];
        t[i] = a + b;
        t[i + h] = a - b;
      }
}

/* The fixed fp32 summation order used for |k|^2 and |c_hat|^2: 32 partial
 * sums p_l = (a[4l] + a[4l+1]) + (a[4l+2] + a[4l+3]), then five pairwise
 * rounds p_l <- p_l + p_{l xor off} for off = 16, 8, 4, 2, 1. */
float oracle_tree_sum(const float a[D]) {
  float p[32], q[32];
  for (int l = 0; l < 32; ++l)
    p[l] = (a[4 * l] + a[4 * l + 1]) + (a[4 * l + 2] + a[4 * l + 3]);
  for (int off = 16; off >= 1; off >>= 1) {
    for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ off];
    memcpy(p, q, sizeof p);
  }
  return p[0];
}

/* Index of the cell of y in an n-level codebook: the number of decision
 * boundaries strictly below y (a tie goes to the lower cell). */
int oracle_quant_index_n(float y, const uint16_t* cb, int n) {
  int idx = 0;
  for (int m = 0; m < n - 1; ++m) {
    float bm = (oracle_h2f(cb[m]) + oracle_h2f(cb[m + 1])) / 2.0f;
    if (y > bm) ++idx;
  }
  return idx;
}

int oracle_quant_index(float y, const uint16_t cb[8]) { return oracle_quant_index_n(y, cb, 8); }

/* b-bit codes, LSB-first: bit (b j + i) of the (b D / 8)-byte little-endian
 * stream is bit i of idx[j]. */
void oracle_pack_bits(const uint8_t idx[D], int bits, uint8_t* out) {
  memset(out, 0, D * bits / 8);
  for (int j = 0; j < D; ++j)
    for (int b = 0; b < bits; ++b)
      if ((idx[j] >> b) & 1) {
        int bit = bits * j + b;
        out[bit >> 3] |= (uint8_t)(1u << (bit & 7));
      }
}

void oracle_unpack_bits(const uint8_t* in, int bits, uint8_t idx[D]) {
  for (int j = 0; j < D; ++j) {
    int v = 0;
    for (int b = 0; b < bits; ++b) {
      int bit = bits * j + b;
      v |= ((in[bit >> 3] >> (bit & 7)) & 1) << b;
    }
    idx[j] = (uint8_t)v;
  }
}

void oracle_pack3(const uint8_t idx[D], uint8_t out[48]) { oracle_pack_bits(idx, 3, out); }
void oracle_unpack3(const uint8_t in[48], uint8_t idx[D]) { oracle_unpack_bits(in, 3, idx); }

static void put_h(uint8_t* p, uint16_t h) { p[0] = (uint8_t)(h & 255); p[1] = (uint8_t)(h >> 8); }
static uint16_t get_h(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Coded-key encoder for one token-head with an n-level codebook (n = 2^bits):
 * norm, rotation, nearest centroid, bit packing, and the fp16 key factor:
 * |k| / |c_hat| (norm correction, the _nc presets) when corrected, else |k|
 * (preset k3v4).  Writes D bits / 8 code bytes and the factor. */
void oracle_encode_keyq(const uint16_t k[D], const uint16_t* cb, int bits, uint8_t* codes,
                        uint16_t* nc_out, int corrected, int signed_rotation) {
  int n = 1 << bits;
  float x[D], sq[D], t[D];
  for (int j = 0; j < D; ++j) {
    x[j] = oracle_h2f(k[j]);
    sq[j] = x[j] * x[j];
    t[j] = signed_rotation && oracle_rs_sign(j) < 0 ? -x[j] : x[j];
  }
  float ss = oracle_tree_sum(sq);
  float norm = sqrtf(ss);
  oracle_wht_f32(t);
  float denom = norm * sqrtf((float)D);
  uint8_t idx[D];
  float c2[D];
  for (int j = 0; j < D; ++j) {
    float y = (norm == 0.0f) ? 0.0f : t[j] / denom;
    idx[j] = (uint8_t)oracle_quant_index_n(y, cb, n);
    float c = oracle_h2f(cb[idx[j]]);
    c2[j] = c * c;
  }
  float cn2 = oracle_tree_sum(c2);
  if (!corrected) *nc_out = oracle_f2h_rn(norm);
  else *nc_out = (norm == 0.0f) ? 0 : oracle_f2h_rn(norm / sqrtf(cn2));
  oracle_pack_bits(idx, bits, codes);
}

void oracle_encode_key3_factor(const uint16_t k[D], const uint16_t cb[8], uint8_t codes[48],
                               uint16_t* nc_out, int corrected, int signed_rotation) {
  oracle_encode_keyq(k, cb, 3, codes, nc_out, corrected, signed_rotation);
}

/* k3v4_nc key encoder (norm correction). */
void oracle_encode_key3(const uint16_t k[D], const uint16_t cb[8], uint8_t codes[48],
                        uint16_t* nc_out) {
  oracle_encode_key3_factor(k, cb, codes, nc_out, 1, 0);
}

/* k8v4 key encoder: per-coordinate e4m3, coordinate order kept. */
void oracle_encode_key8(const uint16_t k[D], uint8_t out[D]) {
  for (int j = 0; j < D; ++j) out[j] = oracle_e4m3_from_half(k[j]);
}

/* 4-bit value encoder for one token-head ([SD] "Context": uniform scalar
 * quantisation of values with a scale and a zero).  Writes the 128 codes (one
 * per byte, 0..15) and the fp16 scale and zero. */
void oracle_encode_value4(const uint16_t v[D], uint8_t code[D], uint16_t* scale_out,
                          uint16_t* zero_out) {
  float lo = oracle_h2f(v[0]), hi = lo;
  for (int j = 1; j < D; ++j) {
    float f = oracle_h2f(v[j]);
    if (f < lo) lo = f;
    if (f > hi) hi = f;
  }
  uint16_t zh = oracle_f2h_rn(lo + 0.0f); /* -0 -> +0 */
  uint16_t sh = 0;
  if (hi != lo) {
    float r = (hi - lo) / 15.0f;
    sh = oracle_f2h_rn(r);
    if (oracle_h2f(sh) < r) sh = (uint16_t)(sh + 1); /* round the scale up */
  }
  float zf = oracle_h2f(zh), sf = oracle_h2f(sh);
  for (int j = 0; j < D; ++j) {
    int c = 0;
    if (sh != 0) {
      float q = rintf((oracle_h2f(v[j]) - zf) / sf);
      c = q < 0.0f ? 0 : (q > 15.0f ? 15 : (int)q);
    }
    code[j] = (uint8_t)c;
  }
  *scale_out = sh;
  *zero_out = zh;
}

/* Value codes in a page are stored coordinate-major: byte 8 * d + off / 2 of
 * the value region holds the code of coordinate d for token off (low nibble
 * for even off, high nibble for odd off). */
static void put_value_codes(uint8_t* vregion, int off, const uint8_t code[D]) {
  for (int d = 0; d < D; ++d) {
    uint8_t* b = vregion + 8 * d + off / 2;
    int sh = 4 * (off % 2);
    *b = (uint8_t)((*b & ~(0xF << sh)) | (code[d] << sh));
  }
}

static int get_value_code(const uint8_t* vregion, int off, int d) {
  return (vregion[8 * d + off / 2] >> (4 * (off % 2))) & 15;
}

/* Store T new tokens into the paged cache [num_blocks][Hk][page].  k, v are
 * fp16 [T][Hk][D]; slot = block * 16 + offset; a negative or out-of-range slot
 * is skipped.  ([SD] "Context": the fused store kernel.) */
int oracle_store(int preset, uint8_t* cache, int num_blocks, int Hk, const uint16_t* k,
                 const uint16_t* v, const int32_t* slot_mapping, int T) {
  long pb = oracle_page_bytes(preset);
  if (pb < 0) return -1;
  uint16_t cb[16];
  int bits = oracle_key_bits(preset);
  if (bits) oracle_codebook_n(1 << bits, cb);
  /* heads own disjoint pages, so they can be encoded in parallel; tokens of
   * one head share value-code bytes and are encoded in order */
#pragma omp parallel for schedule(static)
  for (int h = 0; h < Hk; ++h) {
    for (int t = 0; t < T; ++t) {
      int32_t slot = slot_mapping[t];
      if (slot < 0 || slot >= num_blocks * BLK) continue;
      int blk = slot / BLK, off = slot % BLK;
      uint8_t* page = cache + ((long)blk * Hk + h) * pb;
      const uint16_t* kk = k + ((long)t * Hk + h) * D;
      const uint16_t* vv = v + ((long)t * Hk + h) * D;
      uint16_t s, z;
      uint8_t code[D];
      oracle_encode_value4(vv, code, &s, &z);
      if (preset == PRESET_K8V4) {
        oracle_encode_key8(kk, page + K8_K_OFF + off * D);
        put_value_codes(page + K8_V_OFF, off, code);
        put_h(page + K8_S_OFF + 2 * off, s);
        put_h(page + K8_Z_OFF + 2 * off, z);
      } else {
        coded_layout l = coded_page(preset);
        uint16_t nc;
        oracle_encode_keyq(kk, cb, bits, page + off * l.code_bytes, &nc, preset != PRESET_K3V4,
                           preset == PRESET_K3V4_NC_RS);
        put_h(page + l.nc_off + 2 * off, nc);
        put_value_codes(page + l.v_off, off, code);
        put_h(page + l.s_off + 2 * off, s);
        put_h(page + l.z_off + 2 * off, z);
      }
    }
  }
  return 0;
}

/* --------------------------------------------------------------- decoder */

/* Decoded key of one cached token, fp64.  k8v4: the e4m3 value.  k3v4_nc:
 * k_hat = nc * H c_hat / sqrt(D) (H / sqrt(D) is symmetric and orthonormal, so
 * this inverts the rotation of the encoder). */
void oracle_decode_key(int preset, const uint8_t* page, int off, const uint16_t* cb,
                       double out[D]) {
  if (preset == PRESET_K8V4) {
    for (int j = 0; j < D; ++j) out[j] = oracle_e4m3_to_double(page[K8_K_OFF + off * D + j]);
    return;
  }
  coded_layout l = coded_page(preset);
  uint8_t idx[D];
  oracle_unpack_bits(page + off * l.code_bytes, oracle_key_bits(preset), idx);
  for (int j = 0; j < D; ++j) out[j] = (double)oracle_h2f(cb[idx[j]]);
  oracle_wht_f64(out);
  double nc = (double)oracle_h2f(get_h(page + l.nc_off + 2 * off));
  for (int j = 0; j < D; ++j) out[j] = nc * out[j] / sqrt((double)D);
  /* k3v4_nc_rs: the encoder rotated by H diag(s), whose inverse is diag(s) H / D */
  if (preset == PRESET_K3V4_NC_RS)
    for (int j = 0; j < D; ++j) out[j] *= (double)oracle_rs_sign(j);
}

/* Decoded value: v_hat = code * scale + zero, fp64. */
void oracle_decode_value(int preset, const uint8_t* page, int off, double out[D]) {
  coded_layout l = coded_page(preset);
  int vo = preset == PRESET_K8V4 ? K8_V_OFF : l.v_off;
  int so = preset == PRESET_K8V4 ? K8_S_OFF : l.s_off;
  int zo = preset == PRESET_K8V4 ? K8_Z_OFF : l.z_off;
  double s = (double)oracle_h2f(get_h(page + so + 2 * off));
  double z = (double)oracle_h2f(get_h(page + zo + 2 * off));
  for (int j = 0; j < D; ++j) out[j] = (double)get_value_code(page + vo, off, j) * s + z;
}

/* -------------------------------------------------------------- attention */

/* Source of decoded K/V rows for positions 0..L-1 of one (sequence, kv-head):
 * either the quantised paged cache or, for the quantisation-bypass mode, raw
 * fp16 arrays [L][D]. */
typedef struct {
  int preset;          /* -1: bypass (raw fp16 K/V) */
  const uint8_t* cache;
  int Hk, g, num_blocks;
  const int32_t* bt;   /* block table row of this sequence */
  int max_blocks;
  const uint16_t* raw_k;
  const uint16_t* raw_v;
  uint16_t cb[16];
} kv_source;

/* Returns 0 and fills out, or -1 when the position's block id is invalid. */
static int src_key(const kv_source* s, int p, double out[D]) {
  if (s->preset < 0) {
    for (int j = 0; j < D; ++j) out[j] = (double)oracle_h2f(s->raw_k[(long)p * D + j]);
    return 0;
  }
  int lb = p / BLK;
  if (lb >= s->max_blocks) return -1;
  int blk = s->bt[lb];
  if (blk < 0 || blk >= s->num_blocks) return -1;
  const uint8_t* page = s->cache + ((long)blk * s->Hk + s->g) * oracle_page_bytes(s->preset);
  oracle_decode_key(s->preset, page, p % BLK, s->cb, out);
  return 0;
}

static int src_value(const kv_source* s, int p, double out[D]) {
  if (s->preset < 0) {
    for (int j = 0; j < D; ++j) out[j] = (double)oracle_h2f(s->raw_v[(long)p * D + j]);
    return 0;
  }
  int lb = p / BLK;
  if (lb >= s->max_blocks) return -1;
  int blk = s->bt[lb];
  if (blk < 0 || blk >= s->num_blocks) return -1;
  const uint8_t* page = s->cache + ((long)blk * s->Hk + s->g) * oracle_page_bytes(s->preset);
  oracle_decode_value(s->preset, page, p % BLK, out);
  return 0;
}

/* Softmax attention of nr query rows over positions [lo_r, hi_r) of one
 * (sequence, kv-head), fp64, straight from the definition:
 *   s_p = (q . k_hat_p) / sqrt(D),  w = softmax(s),  out = sum_p w_p v_hat_p.
 * q: fp16 [nr][D].  Positions whose block id is invalid are left out.
 * Per row, out_o gets the normalised output and out_lse gets ln(sum_p
 * exp(s_p)) = m + ln l; a row with no position gets lse = -inf and out = 0.
 * ([SD] "Part 3": scores * ATTN_SCALE with ATTN_SCALE = 1/sqrt(D), softmax, P V.) */
static void attend_rows(const kv_source* src, int nr, const uint16_t* q, const int* lo,
                        const int* hi, double* out_o, double* out_lse) {
  int pmax = 0, pmin = 1 << 30;
  for (int r = 0; r < nr; ++r) {
    if (hi[r] > pmax) pmax = hi[r];
    if (lo[r] < pmin) pmin = lo[r];
  }
  if (pmin > pmax) pmin = pmax;
  int L = pmax - pmin;
  double* s = (double*)malloc(sizeof(double) * (size_t)nr * (size_t)(L > 0 ? L : 1));
  char* ok = (char*)malloc((size_t)(L > 0 ? L : 1));
  double* qd = (double*)malloc(sizeof(double) * (size_t)nr * D);
  for (int r = 0; r < nr; ++r)
    for (int j = 0; j < D; ++j) qd[(long)r * D + j] = (double)oracle_h2f(q[(long)r * D + j]);
  double kh[D], vh[D];
  const double scale = 1.0 / sqrt((double)D);
  /* pass 1: scores */
  for (int p = pmin; p < pmax; ++p) {
    ok[p - pmin] = (char)(src_key(src, p, kh) == 0);
    if (!ok[p - pmin]) continue;
    for (int r = 0; r < nr; ++r) {
      if (p < lo[r] || p >= hi[r]) continue;
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += qd[(long)r * D + j] * kh[j];
      s[(long)r * L + (p - pmin)] = acc * scale;
    }
  }
  /* row maxima and normalisers */
  double* m = (double*)malloc(sizeof(double) * nr);
  double* l = (double*)malloc(sizeof(double) * nr);
  for (int r = 0; r < nr; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0;
    for (int p = lo[r]; p < hi[r]; ++p)
      if (ok[p - pmin] && s[(long)r * L + (p - pmin)] > m[r]) m[r] = s[(long)r * L + (p - pmin)];
    for (int p = lo[r]; p < hi[r]; ++p)
      if (ok[p - pmin]) l[r] += exp(s[(long)r * L + (p - pmin)] - m[r]);
    for (int j = 0; j < D; ++j) out_o[(long)r * D + j] = 0.0;
  }
  /* pass 2: weighted values */
  for (int p = pmin; p < pmax; ++p) {
    if (!ok[p - pmin]) continue;
    int need = 0;
    for (int r = 0; r < nr; ++r)
      if (p >= lo[r] && p < hi[r]) need = 1;
    if (!need) continue;
    src_value(src, p, vh);
    for (int r = 0; r < nr; ++r) {
      if (p < lo[r] || p >= hi[r]) continue;
      double w = exp(s[(long)r * L + (p - pmin)] - m[r]) / l[r];
      for (int j = 0; j < D; ++j) out_o[(long)r * D + j] += w * vh[j];
    }
  }
  for (int r = 0; r < nr; ++r) out_lse[r] = (l[r] > 0.0) ? m[r] + log(l[r]) : -INFINITY;
  free(s);
  free(ok);
  free(qd);
  free(m);
  free(l);
}

/* Number of cache positions draft query n of a sequence of length L sees:
 * causal spec-verify ([SD] "Part 4": query n attends to cached_len + n + 1
 * tokens, cached_len = L - n_spec) or parallel completion (all see L). */
int oracle_visible(int L, int n_spec, int n, int causal) {
  int v = causal ? L - n_spec + n + 1 : L;
  return v < 0 ? 0 : v;
}

static void make_source(kv_source* src, int preset, const uint8_t* cache, int num_blocks,
                        int Hk, int g, const int32_t* bt_row, int max_blocks) {
  memset(src, 0, sizeof *src);
  src->preset = preset;
  src->cache = cache;
  src->num_blocks = num_blocks;
  src->Hk = Hk;
  src->g = g;
  src->bt = bt_row;
  src->max_blocks = max_blocks;
  if (oracle_key_bits(preset)) oracle_codebook_n(oracle_key_levels(preset), src->cb);
}

/* Spec-verify attention for a list of output rows.  Each row is (n, b, h):
 * draft n of sequence b, query head h; its kv-head is h / (Hq / Hk) (GQA).
 * q: fp16 [n_spec][B][Hq][D]; block_table int32 [B][max_blocks]; seq_lens [B]
 * counts the draft tokens already stored.  out: fp64 [nrows][D].
 * Rows of the same (b, kv-head) are evaluated together. */
int oracle_verify_rows(int preset, const uint8_t* cache, int num_blocks, int Hk,
                       const uint16_t* q, const int32_t* block_table, int max_blocks,
                       const int32_t* seq_lens, int n_spec, int B, int Hq, int causal,
                       int nrows, const int32_t* rows /* [nrows][3] = n, b, h */,
                       double* out) {
  if (Hk <= 0 || Hq % Hk) return -1;
  int group = Hq / Hk;
  int ngroups = B * Hk;
  int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bg = 0; bg < ngroups; ++bg) {
    int b = bg / Hk, g = bg % Hk;
    int cnt = 0;
    for (int i = 0; i < nrows; ++i)
      if (rows[3 * i + 1] == b && rows[3 * i + 2] / group == g) ++cnt;
    if (!cnt) continue;
    int* idx = (int*)malloc(sizeof(int) * cnt);
    int* lo = (int*)malloc(sizeof(int) * cnt);
    int* hi = (int*)malloc(sizeof(int) * cnt);
    uint16_t* qq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)cnt * D);
    double* oo = (double*)malloc(sizeof(double) * (size_t)cnt * D);
    double* ll = (double*)malloc(sizeof(double) * cnt);
    int c = 0;
    for (int i = 0; i < nrows; ++i) {
      int n = rows[3 * i], bb = rows[3 * i + 1], h = rows[3 * i + 2];
      if (bb != b || h / group != g) continue;
      idx[c] = i;
      lo[c] = 0;
      hi[c] = oracle_visible(seq_lens[b], n_spec, n, causal);
      memcpy(qq + (long)c * D, q + (((long)n * B + b) * Hq + h) * D, sizeof(uint16_t) * D);
      ++c;
    }
    kv_source src;
    make_source(&src, preset, cache, num_blocks, Hk, g, block_table + (long)b * max_blocks,
                max_blocks);
    attend_rows(&src, cnt, qq, lo, hi, oo, ll);
    for (int i = 0; i < cnt; ++i) memcpy(out + (long)idx[i] * D, oo + (long)i * D, sizeof(double) * D);
    free(idx); free(lo); free(hi); free(qq); free(oo); free(ll);
  }
  return rc;
}

/* All rows: out fp64 [n_spec][B][Hq][D]. */
int oracle_verify(int preset, const uint8_t* cache, int num_blocks, int Hk, const uint16_t* q,
                  const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                  int n_spec, int B, int Hq, int causal, double* out) {
  int nrows = n_spec * B * Hq;
  int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)nrows);
  int i = 0;
  for (int n = 0; n < n_spec; ++n)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < Hq; ++h, ++i) {
        rows[3 * i] = n;
        rows[3 * i + 1] = b;
        rows[3 * i + 2] = h;
      }
  int rc = oracle_verify_rows(preset, cache, num_blocks, Hk, q, block_table, max_blocks,
                              seq_lens, n_spec, B, Hq, causal, nrows, rows, out);
  free(rows);
  return rc;
}

/* Split-KV partials ([S3] "Part 3": NUM_KV_SPLITS partitions of the sequence).
 * Split s of sequence b covers positions [s*chunk, min((s+1)*chunk, visible))
 * with chunk = 16 * ceil(ceil(L_b / S) / 16).  Outputs, per (n, b, h, s):
 * o = the normalised attention over that range (fp64 [n_spec][B][Hq][S][D]) and
 * lse = ln(sum exp(scores)) ([n_spec][B][Hq][S]); an empty split has lse = -inf
 * and o = 0. */
int oracle_partials(int preset, const uint8_t* cache, int num_blocks, int Hk, const uint16_t* q,
                    const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                    int n_spec, int B, int Hq, int S, int causal, double* part_o,
                    double* part_lse) {
  if (Hk <= 0 || Hq % Hk || S <= 0) return -1;
  int group = Hq / Hk;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bg = 0; bg < B * Hk; ++bg) {
    int b = bg / Hk, g = bg % Hk;
    int L = seq_lens[b];
    int per = (L + S - 1) / S;
    int chunk = BLK * ((per + BLK - 1) / BLK);
    int nr = n_spec * group;
    uint16_t* qq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)nr * D);
    int* lo = (int*)malloc(sizeof(int) * nr);
    int* hi = (int*)malloc(sizeof(int) * nr);
    double* oo = (double*)malloc(sizeof(double) * (size_t)nr * D);
    double* ll = (double*)malloc(sizeof(double) * nr);
    kv_source src;
    make_source(&src, preset, cache, num_blocks, Hk, g, block_table + (long)b * max_blocks,
                max_blocks);
    for (int s = 0; s < S; ++s) {
      for (int n = 0; n < n_spec; ++n)
        for (int j = 0; j < group; ++j) {
          int r = n * group + j, h = g * group + j;
          memcpy(qq + (long)r * D, q + (((long)n * B + b) * Hq + h) * D, sizeof(uint16_t) * D);
          int vis = oracle_visible(L, n_spec, n, causal);
          lo[r] = s * chunk;
          hi[r] = (s + 1) * chunk < vis ? (s + 1) * chunk : vis;
          if (hi[r] < lo[r]) hi[r] = lo[r];
        }
      attend_rows(&src, nr, qq, lo, hi, oo, ll);
      for (int n = 0; n < n_spec; ++n)
        for (int j = 0; j < group; ++j) {
          int r = n * group + j, h = g * group + j;
          long row = (((long)n * B + b) * Hq + h) * S + s;
          memcpy(part_o + row * D, oo + (long)r * D, sizeof(double) * D);
          part_lse[row] = ll[r];
        }
    }
    free(qq); free(lo); free(hi); free(oo); free(ll);
  }
  return 0;
}

/* Stage 2: log-sum-exp merge of S partials per row ([SD] "Roofline" / [S3]
 * "Part 3": the stage-2 reduction).  out = sum_s e^(lse_s - M) o_s /
 * sum_s e^(lse_s - M) with M = max_s lse_s; a row whose splits are all empty
 * gives 0.  part_o [rows][S][D], part_lse [rows][S], out [rows][D]. */
void oracle_merge(const double* part_o, const double* part_lse, long nrows, int S, double* out) {
  for (long r = 0; r < nrows; ++r) {
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
      if (part_lse[r * S + s] > M) M = part_lse[r * S + s];
    for (int j = 0; j < D; ++j) out[r * D + j] = 0.0;
    if (isinf(M) && M < 0) continue;
    double den = 0.0;
    for (int s = 0; s < S; ++s) {
      double lse = part_lse[r * S + s];
      if (isinf(lse) && lse < 0) continue;
      double w = exp(lse - M);
      den += w;
      for (int j = 0; j < D; ++j) out[r * D + j] += w * part_o[(r * S + s) * D + j];
    }
    for (int j = 0; j < D; ++j) out[r * D + j] /= den;
  }
}

/* Quantisation-bypass mode: the same attention over raw fp16 K/V [L][D]
 * (positions [lo, hi) per row).  Used to pin the attention arithmetic against
 * an independent brute force. */
void oracle_attend_raw(const uint16_t* q, int nr, const uint16_t* k, const uint16_t* v,
                       const int32_t* lo, const int32_t* hi, double* out_o, double* out_lse) {
  kv_source src;
  memset(&src, 0, sizeof src);
  src.preset = -1;
  src.raw_k = k;
  src.raw_v = v;
  attend_rows(&src, nr, q, lo, hi, out_o, out_lse);
}
