/*
 * Four Over Six NVFP4 oracle: plain, slow, single-threaded C.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product path
 * (the CUDA kernels behind include/fos.h) shares no code with it.
 *
 * Sources, cited by page title and section:
 *   [FOS]  "Four Over Six" (Hugging Face Transformers docs; Russian, Arabic and
 *          English copies), first section: each NVFP4 block is scaled to
 *          either 4 or 6 to cut the error on near-maximal values; options RHT,
 *          2D block scaling, transposed inputs, stochastic rounding.
 *          Same page, "Training": the quantized linear layer has a backward pass.
 *          Same page, first section: older GPUs and CPUs fall back to a
 *          simulation with FP32 matrix multiplication (the GEMM reference here).
 *   [FP4]  "FP4" (Ultralytics glossary), section "FP4 Nasıl Çalışır": the E2M1
 *          layout and its value grid {0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6}; NVFP4
 *          groups 16 values under one FP8 E4M3 scale plus a second FP32
 *          per-tensor scale; a block's scale maps its largest magnitude to 6;
 *          the worked block-size MAE example.  Section "FP4 ile Çıkarım ve
 *          Eğitim": FP4 matmuls accumulate at higher precision; RHT and SR in
 *          NVFP4 training.
 *   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *          1, 2, 3", SC'11: Philox4x32 with 10 rounds.
 *   [OCP]  OCP 8-bit floating point specification: E4M3 ("fn" variant, bias 7,
 *          no infinities, S.1111.111 is NaN, max 448).
 *   [MX]   OCP Microscaling (MX) formats specification v1.0: the E8M0 scale
 *          and the shared exponent floor(log2(amax)) - emax(element).
 *
 * Fixed readings (the pages leave these steps open):
 *   R1  tensor scale s_t = amax / (6*448) in FP32, amax over the (transformed)
 *       tensor.  A block's candidate scale maps its maximum a_b to M (6 or 4):
 *       t_M = M * s_t and sf_M = E4M3_rne_satfinite(a_b / t_M), the product
 *       and the quotient each one FP32 rounding ([FOS] first section: the
 *       block maximum is scaled to 4 or to 6); sf_M = 0 when t_M = 0.
 *   R2  a candidate's squared error is evaluated in the scaled domain:
 *       E_M = (sum_j (q_j - g_j)^2) * eff_M^2, q_j = y_j * (1/eff_M), with the
 *       sum in the fixed order of sumsq16() / the 2D tree; a candidate whose
 *       E4M3 scale is 0 has E_M = sum_j y_j^2 (every value flushes to 0).
 *   R3  keep 4 iff E_4 < E_6 (ties go to 6).
 *   R4  E2M1 rounding: RNE with ties to the even code, |q| > 6 saturates to 6,
 *       the sign bit of q is kept (a negative value that rounds to 0 gives -0).
 *   R5  stochastic rounding: u = (w >> 8) * 2^-24, w = word (i mod 4) of
 *       Philox4x32-10(counter = (lo32(i/4), hi32(i/4), 0, 0), key = seed),
 *       i = r*cols + c the source element index; round up iff u < p.
 *   R6  RHT: per 16-block along the blocking dimension, y = 0.25 * H16 * (s . v)
 *       with H16 the Sylvester Hadamard matrix applied as butterflies of
 *       stride 1, 2, 4, 8 and s_j = 1 - 2*bit_j(word 0 of
 *       Philox4x32-10(counter = (0, 0, 0, 1), key = hadamard_seed)).
 *   R7  2D 16x16 tiles: one scale per tile, replicated into the tile's 16
 *       rows of the 1D scale layout; the tile error is the per-source-row
 *       sumsq16 combined by a pairwise tree over the 16 source rows.
 *   R8  transposed input: the output describes X^T; blocks run along the
 *       rows of X; the RHT runs along the blocking dimension.
 *   R12 MXFP4 ([FP4] "FP4 Nasıl Çalışır": 32 values under one 8-bit
 *       power-of-two scale; [MX] E8M0: byte b = X + 127 means 2^X, 0xFF is
 *       NaN; no tensor scale) with the 4/6 choice: the 6-candidate exponent is
 *       [MX]'s own, X6 = floor(log2 amax) - 2 (E2M1's largest exponent is 2),
 *       which maps the block maximum into [4, 8) and lets values above 6
 *       saturate; the 4-candidate is X4 = X6 + 1, which maps the maximum
 *       below 4 and saturates nothing (a candidate pair "maximum to 6" /
 *       "maximum to 4" cannot be formed from powers of two otherwise: with X6
 *       the smallest X whose 6 * 2^X covers amax, the 4-candidate's grid would
 *       lie inside the 6-candidate's and could never win).  Both are clamped to
 *       [-127, 127].  Each candidate's codes are the R4 roundings of
 *       q = y * 2^-X; S_M is the sum of (q - g)^2 in the R2 order over each
 *       16-value half, the halves then added; keep 4 iff 4 * S_4 < S_6 (the
 *       4-candidate's error in the 6-candidate's units, exact), ties to 6.
 *       An all-zero block gets byte 0 (2^-127) and zero codes.  A block that
 *       holds a NaN or an infinity gets the E8M0 NaN byte 0xFF ([MX]: a NaN
 *       scale makes every value of its block NaN; E2M1 itself has neither),
 *       zero codes and choice 0.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * FP32 arithmetic is IEEE binary32 round-to-nearest-even: every float
 * expression below is rounded where it is written; fmaf() is a fused
 * multiply-add with one rounding.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD 0)"
#endif

/* ---------------------------------------------------------------- formats */

/* [FP4] "FP4 Nasıl Çalışır": the eight non-negative E2M1 magnitudes, in code
 * order (code bits e1 e0 m); bit 3 of a code is the sign. */
static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float orc_e2m1_decode(uint8_t code) {
  double g = E2M1_GRID[code & 7];
  return (float)((code & 8) ? -g : g);
}

/* R4: round |q| to the nearest grid magnitude; on an exact tie between two
 * neighbours take the one with an even code; anything above 6 (and +inf)
 * saturates to 6.  The sign bit of q is kept. */
uint8_t orc_e2m1_rne(float q) {
  uint8_t s = signbit(q) ? 8 : 0;
  double a = fabs((double)q);
  if (isnan(q)) return 0; /* never reached by the quantizer (inputs finite) */
  if (a >= 6.0) return (uint8_t)(s | 7);
  int best = 0;
  double bestd = a;
  for (int k = 1; k < 8; ++k) {
    double d = fabs(a - E2M1_GRID[k]);
    if (d < bestd || (d == bestd && (k % 2) == 0)) {
      best = k;
      bestd = d;
    }
  }
  return (uint8_t)(s | best);
}

/* R5: stochastic rounding of |q| between its two grid neighbours lo <= |q| <
 * hi with P(up) = (|q| - lo) / (hi - lo); u = (w >> 8) * 2^-24. */
uint8_t orc_e2m1_sr(float q, uint32_t w) {
  uint8_t s = signbit(q) ? 8 : 0;
  double a = fabs((double)q);
  if (isnan(q)) return 0;
  if (a >= 6.0) return (uint8_t)(s | 7);
  int k = 0;
  while (k < 6 && E2M1_GRID[k + 1] <= a) ++k;
  double p = (a - E2M1_GRID[k]) / (E2M1_GRID[k + 1] - E2M1_GRID[k]);
  double u = (double)(w >> 8) * ldexp(1.0, -24);
  int idx = (u < p) ? k + 1 : k;
  return (uint8_t)(s | idx);
}

/* [OCP] E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal m * 2^-9; S.1111.111 is NaN; the largest finite value is 448. */
float orc_e4m3_decode(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = m * ldexp(1.0, -9);
  else
    v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return (float)(s ? -v : v);
}

/* Round to nearest E4M3, ties to even, saturating every magnitude above 448
 * (including +inf) to 448.  NaN maps to 0x7F. */
uint8_t orc_e4m3_rne_satfinite(float x) {
  uint8_t s = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return 0x7F;
  double a = fabs((double)x);
  if (a > 448.0) return (uint8_t)(s | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9; n == 8 is the smallest normal 0x08 */
    double n = rint(a * ldexp(1.0, 9));
    return (uint8_t)(s | (int)n);
  }
  int E;
  frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1; /* a in [2^e, 2^(e+1)) */
  double n = rint(a / ldexp(1.0, e - 3)); /* in [8, 16]; exact scaling */
  int code = ((e + 7) << 3) + ((int)n - 8); /* n == 16 carries into the exponent */
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(s | code);
}

/* ------------------------------------------------------------------ Philox */

/* [PHILOX] Philox4x32 with 10 rounds.  Round: multiply words 0 and 2 by the
 * two multipliers, cross the high halves with the other words and the key;
 * the key is bumped by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* R5: the random word for source element i. */
uint32_t orc_sr_word(uint64_t seed, uint64_t i) {
  uint64_t blk = i >> 2;
  uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[i & 3];
}

/* R6: the per-tensor sign mask (bit j set means s_j = -1). */
uint32_t orc_rht_sign_mask(uint64_t seed) {
  uint32_t ctr[4] = {0u, 0u, 0u, 1u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[0] & 0xFFFFu;
}

/* R6 / [FOS] first section ("random Hadamard transform"): in place on 16 values. */
void orc_rht16(float w[16], uint32_t sign_mask) {
  for (int j = 0; j < 16; ++j)
    if ((sign_mask >> j) & 1u) w[j] = -w[j];
  for (int h = 1; h < 16; h <<= 1)
    for (int j = 0; j < 16; ++j)
      if ((j & h) == 0) {
        float a = w[j], b = w[j + h];
        w[j] = a + b;
        w[j + h] = a - b;
      }
  for (int j = 0; j < 16; ++j) w[j] = w[j] * 0.25f;
}

/* R2: the fixed summation order for 16 squares: even and odd positions in
 * two fused-multiply-add chains, then one add. */
float orc_sumsq16(const float r[16]) {
  float a = 0.0f, b = 0.0f;
  for (int k = 0; k < 8; ++k) {
    a = fmaf(r[2 * k], r[2 * k], a);
    b = fmaf(r[2 * k + 1], r[2 * k + 1], b);
  }
  return a + b;
}

/* R7: pairwise adjacent tree over 16 per-row sums. */
static float tree16(const float s[16]) {
  float t[16];
  memcpy(t, s, sizeof(t));
  for (int n = 16; n > 1; n /= 2)
    for (int i = 0; i < n / 2; ++i) t[i] = t[2 * i] + t[2 * i + 1];
  return t[0];
}

/* --------------------------------------------------------- scale layouts */

/* Scale-factor layout consumed by the block-scaled tensor-core MMA: 128 rows x
 * 4 scale columns form one 512-byte tile; tiles are row-major over (row tile,
 * column tile); inside a tile (r, c) sits at (r%32)*16 + (r/32)*4 + c.
 * layout 1 is plain row-major [rows][nb]. */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t nb, int layout) {
  if (layout == 1) return r * nb + c;
  int64_t n_ct = (nb + 3) / 4;
  return ((r / 128) * n_ct + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

int64_t orc_sf_bytes(int64_t rows, int64_t nb, int layout) {
  if (layout == 1) return rows * nb;
  return ((rows + 127) / 128) * 128 * ((nb + 3) / 4) * 4;
}

/* --------------------------------------------------------------- quantize */

typedef struct {
  int32_t scale_rule; /* 0: 4/6, 1: always 6, 2: always 4 */
  int32_t rounding;   /* 0: RNE, 1: stochastic */
  int32_t block_2d;   /* 0: 1x16 blocks, 1: 16x16 tiles */
  int32_t transpose;  /* 1: output describes X^T */
  int32_t hadamard;   /* 1: apply the RHT */
  int32_t sf_layout;  /* 0: swizzled 128x4, 1: row-major */
  uint64_t sr_seed;
  uint64_t hadamard_seed;
  int32_t use_amax; /* 1: take amax from the field below */
  float amax;
  /* Source coordinates of x inside a larger matrix, for the stochastic-rounding
   * element index i = (src_row0 + r) * src_cols + c (src_cols 0: cols).  Lets a
   * caller quantize sampled rows of a big matrix with the big matrix's indices. */
  int64_t src_row0;
  int64_t src_cols;
} orc_options;

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* One candidate M for a block/tile: given a_b, compute sf, the codes and the
 * error E.  y, src are the candidate's n elements (16 or 256) in "source-row
 * major" order: element (i, j) = source row i, source column j of the tile,
 * for 2D; the 1D block is one row. */
typedef struct {
  uint8_t sf;
  float err;
} cand_t;

static cand_t eval_candidate(const float* y, const uint64_t* src, int nrows, float ab, float tM,
                             float s_t, const orc_options* o, uint8_t* codes_out) {
  cand_t c;
  /* R1: the block maximum divided by M * s_t, one IEEE division */
  float raw = (tM > 0.0f) ? ab / tM : 0.0f;
  c.sf = orc_e4m3_rne_satfinite(raw);
  float rowsum[16];
  if (c.sf == 0) {
    for (int i = 0; i < nrows * 16; ++i) codes_out[i] = orc_e2m1_rne(y[i] * 0.0f);
    for (int i = 0; i < nrows; ++i) rowsum[i] = orc_sumsq16(y + 16 * i);
  } else {
    float eff = orc_e4m3_decode(c.sf) * s_t;
    float inv = 1.0f / eff;
    if (inv > FLT_MAX) inv = FLT_MAX;
    for (int i = 0; i < nrows; ++i) {
      float r[16];
      for (int j = 0; j < 16; ++j) {
        float q = y[16 * i + j] * inv;
        uint8_t code = (o->rounding == 1) ? orc_e2m1_sr(q, orc_sr_word(o->sr_seed, src[16 * i + j]))
                                          : orc_e2m1_rne(q);
        codes_out[16 * i + j] = code;
        r[j] = q - orc_e2m1_decode(code);
      }
      rowsum[i] = orc_sumsq16(r);
    }
    float e2 = eff * eff;
    float S = (nrows == 1) ? rowsum[0] : tree16(rowsum);
    c.err = S * e2;
    return c;
  }
  c.err = (nrows == 1) ? rowsum[0] : tree16(rowsum);
  return c;
}

/*
 * Quantize a bf16 matrix X [rows, cols] (row stride ld elements) to NVFP4.
 * Output orientation: R_out x C_out = rows x cols, or cols x rows when
 * o->transpose.  codes: R_out rows of ld_codes bytes (two codes per byte, the
 * even element in the low nibble).  sf: orc_sf_bytes(R_out, C_out/16) bytes,
 * pad bytes written 0.  choice (may be NULL): R_out rows of ceil(nb/32) words,
 * bit b%32 of word b/32 set when block b kept the 4 candidate.
 * Returns 0, or -1 on a shape the options cannot take.
 */
int orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const orc_options* o,
                 uint8_t* codes, int64_t ld_codes, uint8_t* sf, float* tensor_scale,
                 uint32_t* choice) {
  int64_t R = o->transpose ? cols : rows;
  int64_t C = o->transpose ? rows : cols;
  /* shapes: cols % 16 == 0 always; rows % 16 == 0 when transposed or 2D */
  if (rows < 0 || cols < 0 || cols % 16 != 0) return -1;
  if ((o->transpose || o->block_2d) && rows % 16 != 0) return -1;
  int64_t nb = C / 16, nw = (nb + 31) / 32;

  /* step 1, R8: the output-oriented matrix and each element's source index */
  float* y = (float*)malloc(sizeof(float) * (size_t)(R * C > 0 ? R * C : 1));
  uint64_t* src = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(R * C > 0 ? R * C : 1));
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) {
      int64_t sr = o->transpose ? c : r, sc = o->transpose ? r : c;
      y[r * C + c] = bf16_to_f32(x[sr * ld + sc]);
      src[r * C + c] = (uint64_t)(o->src_row0 + sr) * (uint64_t)(o->src_cols ? o->src_cols : cols) + (uint64_t)sc;
    }
  /* step 2, R6 */
  if (o->hadamard) {
    uint32_t mask = orc_rht_sign_mask(o->hadamard_seed);
    for (int64_t r = 0; r < R; ++r)
      for (int64_t b = 0; b < nb; ++b) orc_rht16(y + r * C + 16 * b, mask);
  }
  /* step 3, R1 */
  float amax = 0.0f;
  if (o->use_amax)
    amax = o->amax;
  else
    for (int64_t i = 0; i < R * C; ++i)
      if (fabsf(y[i]) > amax) amax = fabsf(y[i]);
  float s_t = amax / 2688.0f;
  float t6 = 6.0f * s_t, t4 = 4.0f * s_t;
  *tensor_scale = s_t;

  memset(sf, 0, (size_t)orc_sf_bytes(R, nb, o->sf_layout));
  if (choice) memset(choice, 0, sizeof(uint32_t) * (size_t)(R * nw));
  for (int64_t r = 0; r < R; ++r) memset(codes + r * ld_codes, 0, (size_t)(C / 2));

  /* steps 4-7 per block (1D) or tile (2D) */
  int nrows = o->block_2d ? 16 : 1;
  int64_t rstep = nrows;
  float ty[256];
  uint64_t tsrc[256];
  uint8_t c6[256], c4[256];
  int64_t opos[256]; /* output linear position of each tile element */
  for (int64_t r0 = 0; r0 < R; r0 += rstep)
    for (int64_t b = 0; b < nb; ++b) {
      /* gather in source-row-major order */
      for (int i = 0; i < nrows; ++i)
        for (int j = 0; j < 16; ++j) {
          int64_t orow, ocol;
          if (nrows == 1) {
            orow = r0;
            ocol = 16 * b + j;
          } else if (!o->transpose) {
            orow = r0 + i;
            ocol = 16 * b + j;
          } else { /* source row i of the tile is output column 16b+i */
            orow = r0 + j;
            ocol = 16 * b + i;
          }
          ty[16 * i + j] = y[orow * C + ocol];
          tsrc[16 * i + j] = src[orow * C + ocol];
          opos[16 * i + j] = orow * C + ocol;
        }
      float ab = 0.0f;
      for (int i = 0; i < 16 * nrows; ++i)
        if (fabsf(ty[i]) > ab) ab = fabsf(ty[i]);
      cand_t e6 = eval_candidate(ty, tsrc, nrows, ab, t6, s_t, o, c6);
      cand_t e4 = eval_candidate(ty, tsrc, nrows, ab, t4, s_t, o, c4);
      int four;
      if (o->scale_rule == 1)
        four = 0;
      else if (o->scale_rule == 2)
        four = 1;
      else
        four = e4.err < e6.err;
      const uint8_t* cc = four ? c4 : c6;
      uint8_t s = four ? e4.sf : e6.sf;
      for (int i = 0; i < 16 * nrows; ++i) {
        int64_t orow = opos[i] / C, ocol = opos[i] % C;
        uint8_t* byte = codes + orow * ld_codes + ocol / 2;
        *byte = (uint8_t)(*byte | (cc[i] << ((ocol & 1) * 4)));
      }
      for (int i = 0; i < nrows; ++i) {
        sf[orc_sf_offset(r0 + i, b, nb, o->sf_layout)] = s;
        if (choice && four) choice[(r0 + i) * nw + b / 32] |= 1u << (b % 32);
      }
    }
  free(y);
  free(src);
  return 0;
}

/* Step 9: x_hat = g * (sf * s_t), each product rounded to FP32. */
void orc_dequantize(const uint8_t* codes, int64_t R, int64_t C, int64_t ld_codes, const uint8_t* sf,
                    int sf_layout, float s_t, float* out) {
  int64_t nb = C / 16;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) {
      uint8_t byte = codes[r * ld_codes + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      float eff = orc_e4m3_decode(sf[orc_sf_offset(r, c / 16, nb, sf_layout)]) * s_t;
      out[r * C + c] = orc_e2m1_decode(code) * eff;
    }
}

/* [FOS] first section (FP32 simulation) / [FP4] "FP4 ile Çıkarım ve Eğitim":
 * C = A_hat * W_hat^T with A_hat [M,K], W_hat [N,K] dequantized operands,
 * accumulated in double for the selected rows.  bound[i,n] = sum_k |a||w|. */
void orc_gemm_rows(const float* A, const float* W, int64_t N, int64_t K, const int64_t* rows,
                   int64_t n_rows, double* out, double* bound) {
  for (int64_t i = 0; i < n_rows; ++i) {
    const float* a = A + rows[i] * K;
    for (int64_t n = 0; n < N; ++n) {
      const float* w = W + n * K;
      double s = 0.0, b = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        s += (double)a[k] * (double)w[k];
        b += fabs((double)a[k] * (double)w[k]);
      }
      out[i * N + n] = s;
      bound[i * N + n] = b;
    }
  }
}

/* [FP4] "FP4 Nasıl Çalışır", the worked example: one FP32 scale amax/6 per
 * block of `block` values, each |x|/scale sent to the nearest grid value (the
 * first one on a tie), dequantized back; returns the mean absolute error. */
double orc_mae_nearest_grid(const float* x, int64_t n, int64_t block) {
  double err = 0.0;
  for (int64_t b0 = 0; b0 < n; b0 += block) {
    float amax = 0.0f;
    for (int64_t i = b0; i < b0 + block; ++i)
      if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    float scale = amax / 6.0f;
    for (int64_t i = b0; i < b0 + block; ++i) {
      float a = fabsf(x[i]) / scale;
      int best = 0;
      float bestd = fabsf(a - (float)E2M1_GRID[0]);
      for (int k = 1; k < 8; ++k) {
        float d = fabsf(a - (float)E2M1_GRID[k]);
        if (d < bestd) {
          best = k;
          bestd = d;
        }
      }
      float sgn = (x[i] > 0.0f) ? 1.0f : ((x[i] < 0.0f) ? -1.0f : 0.0f);
      float deq = (float)E2M1_GRID[best] * sgn * scale;
      err += fabs((double)deq - (double)x[i]);
    }
  }
  return err / (double)n;
}

/* ------------------------------------------------------------- MXFP4 */

/* R12: E8M0 byte -> 2^(b - 127); 0xFF is NaN. */
float orc_e8m0_decode(uint8_t b) {
  if (b == 0xFF) return NAN;
  return (float)ldexp(1.0, (int)b - 127);
}

/* R12: the candidate exponent for amax a > 0 (finite): X6 = floor(log2 a) - 2
 * for M = 6, X4 = X6 + 1 for M = 4, clamped to [-127, 127]. */
int orc_mx_exponent(float a, int M) {
  int e2;
  frexp((double)a, &e2); /* a = m * 2^e2 with m in [0.5, 1), so floor(log2 a) = e2 - 1 */
  int X = (e2 - 1) - 2 + (M == 4 ? 1 : 0);
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

/* One candidate of a 32-value block: codes, and S (R2 order per 16-value
 * half, then the halves added). */
static float mx_candidate(const float y[32], int X, uint8_t codes[32]) {
  const float inv = (float)ldexp(1.0, -X); /* exact: X in [-127, 127] */
  float r[32];
  for (int j = 0; j < 32; ++j) {
    float q = y[j] * inv;
    codes[j] = orc_e2m1_rne(q);
    r[j] = q - orc_e2m1_decode(codes[j]);
  }
  return orc_sumsq16(r) + orc_sumsq16(r + 16);
}

/* R12: MXFP4 4/6 quantization of a bf16 matrix [rows, cols] (row stride ld
 * elements, cols % 32 == 0) along its rows.  codes: rows x ld_codes bytes (two
 * per byte, even element low); scales: rows x cols/32 E8M0 bytes; choice (may
 * be NULL): rows x cols/32 bytes, 1 when the block kept the 4-candidate.
 * scale_rule 0: 4/6, 1: 6 only, 2: 4 only. */
int orc_quantize_mx(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int scale_rule, uint8_t* codes,
                    int64_t ld_codes, uint8_t* scales, uint8_t* choice) {
  if (cols % 32 != 0) return 1;
  const int64_t nb = cols / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      float y[32], a = 0.0f;
      int finite = 1;
      for (int j = 0; j < 32; ++j) {
        y[j] = bf16_to_f32(x[r * ld + 32 * b + j]);
        if (!isfinite(y[j])) finite = 0;
        if (fabsf(y[j]) > a) a = fabsf(y[j]);
      }
      if (!finite) { /* R12: the NaN scale, zero codes */
        for (int j = 0; j < 16; ++j) codes[r * ld_codes + 16 * b + j] = 0;
        scales[r * nb + b] = 0xFF;
        if (choice) choice[r * nb + b] = 0;
        continue;
      }
      uint8_t c6[32], c4[32];
      int X6, X4;
      if (a == 0.0f) {
        X6 = X4 = -127;
      } else {
        X6 = orc_mx_exponent(a, 6);
        X4 = orc_mx_exponent(a, 4);
      }
      float S6 = mx_candidate(y, X6, c6);
      float S4 = mx_candidate(y, X4, c4);
      /* X4 is X6 + 1 (or equal at the clamp): bring S4 into the 6-candidate's units */
      const float S4u = (X4 > X6) ? S4 * 4.0f : S4;
      int four = (scale_rule == 2) || (scale_rule == 0 && S4u < S6);
      const uint8_t* c = four ? c4 : c6;
      for (int j = 0; j < 16; ++j) codes[r * ld_codes + 16 * b + j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
      scales[r * nb + b] = (uint8_t)((four ? X4 : X6) + 127);
      if (choice) choice[r * nb + b] = (uint8_t)four;
    }
  return 0;
}

/* R12: x_hat = g * 2^X, exact in FP32. */
void orc_dequantize_mx(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols, int64_t ld_codes,
                       float* out) {
  const int64_t nb = cols / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = codes[r * ld_codes + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      out[r * cols + c] = orc_e2m1_decode(code) * orc_e8m0_decode(scales[r * nb + c / 32]);
    }
}

/* ------------------------------------------- array helpers for the tests */

void orc_e2m1_rne_n(const float* q, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_rne(q[i]);
}

void orc_e2m1_sr_n(const float* q, const uint32_t* w, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_sr(q[i], w[i]);
}

void orc_e4m3_rne_satfinite_n(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_rne_satfinite(x[i]);
}

void orc_sr_words_n(uint64_t seed, const uint64_t* idx, int64_t n, uint32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_sr_word(seed, idx[i]);
}

void orc_rht16_n(float* w, int64_t n_blocks, uint32_t sign_mask) {
  for (int64_t b = 0; b < n_blocks; ++b) orc_rht16(w + 16 * b, sign_mask);
}
