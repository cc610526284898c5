/*
 * Plain CPU oracle for the forward pass of Beam's Mixture-of-Experts block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (sources are the five web pages about Reflection's Beam):
 *   - "Hugging Face releases Beam ..." (deliver-ai.xyz), third paragraph:
 *     256 experts per layer, each a SwiGLU MLP with intermediate size 2,560;
 *     the router keeps the top 4 of 8 groups (32 experts each) and selects
 *     the top 8 experts inside them.
 *   - "Reflection Releases Beam ..." (telohudelo.online), section "Where Beam
 *     Saves and Where the Memory Bill Comes In": sigmoid scores, DeepSeek-V3
 *     style group limits, no shared expert, normalised and scaled by 2.5.
 *   - "Beam 1.0" (interestana.com digest): auxiliary-loss-free balancing with
 *     a per-expert bias.
 * The pages leave several steps open; the readings taken here are:
 *   - group score = sum of the two largest biased scores in the group;
 *   - experts are selected on biased scores s+b, weighted by unbiased s;
 *   - the 8 weights are normalised to sum to 1, then multiplied by 2.5;
 *   - experts outside the kept groups are excluded (never selected), not
 *     given a score of 0;
 *   - ties go to the lower group index, then to the lower expert index; the
 *     output order of the k experts is descending biased score.
 *
 * Precision: every decision value (logit, sigmoid score, biased score, group
 * score) is held in fp32, the precision the GPU path decides in; each is
 * computed in fp64 and rounded once to fp32, except s+b and top1+top2 which
 * are single fp32 additions.  The expert path (SwiGLU MLP and the weighted
 * sum) runs entirely in fp64.
 *
 * Parity pins for every function are in tests/test_oracle_*.py.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* ---- scalar decoders (from the formats' definitions) ------------------- */

/* bf16 is the upper half of an IEEE binary32. */
static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/nan. */
double oracle_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* FP8 E4M3 (the "fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * exponent 15 with mantissa 7 is NaN, there is no infinity. */
double oracle_e4m3_value(uint8_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp(m / 8.0, -6);
  else mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* ---- routing ----------------------------------------------------------- */

/*
 * Router of one MoE block, for T tokens.
 *   x         bf16 [T, H]   token activations (row-major)
 *   w_router  fp32 [E, H]   router weight, one row per expert
 *   bias      fp32 [E]      per-expert selection bias
 *   topk_idx  int32 [T, k]  selected experts, descending biased score
 *   topk_w    fp32 [T, k]   routed weights (sum to routed_scale)
 * Optional outputs (NULL to skip): logits/scores/biased [T, E] fp32,
 * group_score [T, G] fp32, group_kept [T, G] uint8.
 */
int oracle_route(int T, int H, int E, int n_group, int topk_group, int top_k,
                 float routed_scale, const uint16_t *x, const float *w_router,
                 const float *bias, int32_t *topk_idx, float *topk_w,
                 float *logits_out, float *scores_out, float *biased_out,
                 float *group_score_out, uint8_t *group_kept_out) {
  if (T < 0 || H <= 0 || E <= 0 || n_group <= 0 || E % n_group != 0) return ORACLE_BAD_ARG;
  const int gsize = E / n_group;
  if (gsize < 2 || topk_group <= 0 || topk_group > n_group) return ORACLE_BAD_ARG;
  if (top_k <= 0 || top_k > topk_group * gsize) return ORACLE_BAD_ARG;

  int bad = 0;
#pragma omp parallel
  {
    float *logit = (float *)malloc(sizeof(float) * E);
    float *s = (float *)malloc(sizeof(float) * E);
    float *sb = (float *)malloc(sizeof(float) * E);
    float *gs = (float *)malloc(sizeof(float) * n_group);
    uint8_t *kept = (uint8_t *)malloc(n_group);
    if (!logit || !s || !sb || !gs || !kept) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (size_t)t * H;
        /* logits: fp64 products and sum, one rounding to fp32 */
        for (int e = 0; e < E; ++e) {
          const float *we = w_router + (size_t)e * H;
          double acc = 0.0;
          for (int h = 0; h < H; ++h) acc += bf16_value(xt[h]) * (double)we[h];
          logit[e] = (float)acc;
        }
        /* sigmoid affinity, and the biased score used only for selection */
        for (int e = 0; e < E; ++e) {
          s[e] = (float)(1.0 / (1.0 + exp(-(double)logit[e])));
          sb[e] = s[e] + bias[e];
        }
        /* group score: the two largest biased scores of the group, added */
        for (int j = 0; j < n_group; ++j) {
          float a1 = -INFINITY, a2 = -INFINITY;
          for (int i = 0; i < gsize; ++i) {
            float v = sb[j * gsize + i];
            if (v > a1) { a2 = a1; a1 = v; }
            else if (v > a2) { a2 = v; }
          }
          gs[j] = a1 + a2;
        }
        /* keep a group when fewer than topk_group groups beat it; a group
         * beats another with a larger score, or an equal one and a lower index */
        for (int j = 0; j < n_group; ++j) {
          int rank = 0;
          for (int j2 = 0; j2 < n_group; ++j2)
            if (gs[j2] > gs[j] || (gs[j2] == gs[j] && j2 < j)) ++rank;
          kept[j] = rank < topk_group;
        }
        /* expert rank among the candidates (experts of kept groups) */
        int32_t *idx = topk_idx + (size_t)t * top_k;
        for (int e = 0; e < E; ++e) {
          if (!kept[e / gsize]) continue;
          int rank = 0;
          for (int e2 = 0; e2 < E; ++e2) {
            if (!kept[e2 / gsize]) continue;
            if (sb[e2] > sb[e] || (sb[e2] == sb[e] && e2 < e)) ++rank;
          }
          if (rank < top_k) idx[rank] = e;
        }
        /* weights from the unbiased scores, normalised, times routed_scale */
        double sum = 0.0;
        for (int k = 0; k < top_k; ++k) sum += (double)s[idx[k]];
        for (int k = 0; k < top_k; ++k)
          topk_w[(size_t)t * top_k + k] =
              (float)((double)routed_scale * (double)s[idx[k]] / sum);

        if (logits_out) memcpy(logits_out + (size_t)t * E, logit, sizeof(float) * E);
        if (scores_out) memcpy(scores_out + (size_t)t * E, s, sizeof(float) * E);
        if (biased_out) memcpy(biased_out + (size_t)t * E, sb, sizeof(float) * E);
        if (group_score_out) memcpy(group_score_out + (size_t)t * n_group, gs, sizeof(float) * n_group);
        if (group_kept_out) memcpy(group_kept_out + (size_t)t * n_group, kept, n_group);
      }
    }
    free(logit); free(s); free(sb); free(gs); free(kept);
  }
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* ---- rounding to the narrow formats (NVFP4 activation quantiser) -------- */

/* fp32 -> FP4 E2M1 code, round to nearest, ties to the code whose mantissa
 * bit is 0; magnitudes above 6 saturate to 6.  The sign bit is the value's
 * sign, so a negative value that rounds to zero gives the code of -0. */
uint8_t oracle_e2m1_rne(float v) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = signbit(v) ? 8 : 0;
  const double a = fabs((double)v);
  if (a >= 6.0) return sign | 7;
  int c = 0;
  while (mag[c + 1] <= a) ++c; /* mag[c] <= a < mag[c+1] */
  const double dlo = a - mag[c], dhi = mag[c + 1] - a;
  int code = (dlo < dhi) ? c : (dhi < dlo) ? c + 1 : ((c & 1) ? c + 1 : c);
  return sign | (uint8_t)code;
}

/* fp32 -> FP8 E4M3 code, round to nearest, ties to the even code; magnitudes
 * at or above 448 saturate to 448 (code 0x7E).  Same sign rule as above. */
uint8_t oracle_e4m3_rne(float v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int c = 0; /* codes 0..126 are the finite magnitudes in increasing order */
  while (oracle_e4m3_value((uint8_t)(c + 1)) <= a) ++c;
  const double lo = oracle_e4m3_value((uint8_t)c), hi = oracle_e4m3_value((uint8_t)(c + 1));
  const double dlo = a - lo, dhi = hi - a;
  int code = (dlo < dhi) ? c : (dhi < dlo) ? c + 1 : ((c & 1) ? c + 1 : c);
  return sign | (uint8_t)code;
}

/*
 * NVFP4 quantisation of activations with a given fp32 global scale g > 0
 * (the reading of "NVFP4" for activations: the weights' two-level format, a
 * static global scale per tensor and one E4M3 scale per 16 consecutive
 * values of a row).  For every block of 16 values v of a row, in fp32:
 *   amax = max |v|,  s = e4m3_rne(amax / (6 * g)),  scale = e4m3(s) * g,
 *   code_i = e2m1_rne(v_i / scale)            (all codes 0 when scale == 0).
 * v is fp32 [rows, cols] (cols % 16 == 0); q is uint8 [rows, cols/2] with
 * the even column in the low nibble; s is uint8 [rows, cols/16].
 * The value a code stands for is e2m1(code) * e4m3(s) * g.
 */
int oracle_quantize_nvfp4(int rows, int cols, const float *v, float g, uint8_t *q, uint8_t *s) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || !(g > 0.0f)) return ORACLE_BAD_ARG;
  const float six_g = 6.0f * g;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < cols / 16; ++b) {
      const float *blk = v + (size_t)r * cols + 16 * b;
      float amax = 0.0f;
      for (int i = 0; i < 16; ++i)
        if (fabsf(blk[i]) > amax) amax = fabsf(blk[i]);
      const uint8_t sc = oracle_e4m3_rne(amax / six_g);
      const float scale = (float)oracle_e4m3_value(sc) * g;
      s[(size_t)r * (cols / 16) + b] = sc;
      uint8_t *qb = q + (size_t)r * (cols / 2) + 8 * b;
      for (int i = 0; i < 16; i += 2) {
        const uint8_t c0 = scale == 0.0f ? 0 : oracle_e2m1_rne(blk[i] / scale);
        const uint8_t c1 = scale == 0.0f ? 0 : oracle_e2m1_rne(blk[i + 1] / scale);
        qb[i / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
  return ORACLE_OK;
}

/* ---- expert weights ---------------------------------------------------- */

/* One weight matrix [N, K] (out x in, K contiguous) of one expert.
 * dtype 0: bf16, data is uint16 [N, K].
 * dtype 1: NVFP4, data is uint8 [N, K/2] (low nibble = even k), scales is
 *          e4m3 uint8 [N, K/16], and the value is e2m1 * e4m3 * global.
 * dtype 2: FP8, data is e4m3 uint8 [N, K], row_scale is fp32 [N], and the
 *          value is e4m3 * row_scale[n] (one scale per output row). */
typedef struct {
  int dtype;
  const void *data;
  const uint8_t *scales;
  double global;
  const float *row_scale; /* FP8 only */
  double e2m1[16];  /* value of every e2m1 code (NVFP4 only) */
  double e4m3[256]; /* value of every e4m3 code (NVFP4 only) */
} oracle_matrix;

static oracle_matrix make_matrix(int dtype, const void *data, const uint8_t *scales, double global) {
  oracle_matrix m;
  m.dtype = dtype;
  m.data = data;
  m.scales = scales;
  m.global = global;
  m.row_scale = (const float *)scales; /* FP8: the scales argument carries fp32 [N] */
  for (int c = 0; c < 16; ++c) m.e2m1[c] = oracle_e2m1_value((uint8_t)c);
  for (int c = 0; c < 256; ++c) m.e4m3[c] = oracle_e4m3_value((uint8_t)c);
  return m;
}

static void decode_row(const oracle_matrix *m, int K, int row, double *out) {
  if (m->dtype == 0) {
    const uint16_t *r = (const uint16_t *)m->data + (size_t)row * K;
    for (int k = 0; k < K; ++k) out[k] = bf16_value(r[k]);
  } else if (m->dtype == 2) {
    const uint8_t *q = (const uint8_t *)m->data + (size_t)row * K;
    const double rs = (double)m->row_scale[row];
    for (int k = 0; k < K; ++k) out[k] = m->e4m3[q[k]] * rs;
  } else {
    const uint8_t *q = (const uint8_t *)m->data + (size_t)row * (K / 2);
    const uint8_t *sc = m->scales + (size_t)row * (K / 16);
    for (int k = 0; k < K; ++k) {
      uint8_t byte = q[k / 2];
      uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      out[k] = m->e2m1[code] * m->e4m3[sc[k / 16]] * m->global;
    }
  }
}

/* Dequantise (or widen) a whole matrix to fp64 [N, K]. */
int oracle_decode_matrix(int dtype, int N, int K, const void *data,
                         const uint8_t *scales, double global, double *out) {
  if (N <= 0 || K <= 0 || (dtype == 1 && K % 16 != 0)) return ORACLE_BAD_ARG;
  oracle_matrix m = make_matrix(dtype, data, scales, global);
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) decode_row(&m, K, n, out + (size_t)n * K);
  return ORACLE_OK;
}

/*
 * One SwiGLU expert applied to n rows:
 *   o[r] = W_down . ( silu(W_gate . x[r]) * (W_up . x[r]) ),   silu(z) = z / (1 + e^-z)
 *   x      bf16 [n, H]
 *   W_gate [I, H], W_up [I, H], W_down [H, I]  (bf16 or NVFP4, see oracle_matrix)
 *   o      fp64 [n, H]
 * All arithmetic in fp64.
 */
int oracle_expert_swiglu(int n, int H, int I, const uint16_t *x,
                         int dtype, const void *wg, const uint8_t *sg, double gg,
                         const void *wu, const uint8_t *su, double gu,
                         const void *wd, const uint8_t *sd, double gd,
                         double *o) {
  if (n < 0 || H <= 0 || I <= 0) return ORACLE_BAD_ARG;
  if (n == 0) return ORACLE_OK;
  oracle_matrix mg = make_matrix(dtype, wg, sg, gg), mu = make_matrix(dtype, wu, su, gu),
                md = make_matrix(dtype, wd, sd, gd);
  double *xd = (double *)malloc(sizeof(double) * (size_t)n * H);
  double *act = (double *)malloc(sizeof(double) * (size_t)n * I);
  if (!xd || !act) { free(xd); free(act); return ORACLE_BAD_ARG; }
  for (size_t i = 0; i < (size_t)n * H; ++i) xd[i] = bf16_value(x[i]);

#pragma omp parallel
  {
    double *rg = (double *)malloc(sizeof(double) * H);
    double *ru = (double *)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
    for (int i = 0; i < I; ++i) {
      decode_row(&mg, H, i, rg);
      decode_row(&mu, H, i, ru);
      for (int r = 0; r < n; ++r) {
        const double *xr = xd + (size_t)r * H;
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) { g += rg[h] * xr[h]; u += ru[h] * xr[h]; }
        act[(size_t)r * I + i] = g / (1.0 + exp(-g)) * u;
      }
    }
    free(rg); free(ru);
  }
#pragma omp parallel
  {
    double *rd = (double *)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
    for (int j = 0; j < H; ++j) {
      decode_row(&md, I, j, rd);
      for (int r = 0; r < n; ++r) {
        const double *ar = act + (size_t)r * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += rd[i] * ar[i];
        o[(size_t)r * H + j] = acc;
      }
    }
    free(rd);
  }
  free(xd); free(act);
  return ORACLE_OK;
}

/*
 * The same expert with NVFP4 weights and NVFP4 activations (W4A4):
 *   x_hat = dequant(quantize(x, gx))                 (x: bf16 rows, exact in fp32)
 *   g, u  = W_gate . x_hat, W_up . x_hat             (fp64)
 *   h     = fp32( silu(g) * u )                      (one rounding to fp32)
 *   h_hat = dequant(quantize(h, gh))
 *   o     = W_down . h_hat                           (fp64)
 * with quantize/dequant as in oracle_quantize_nvfp4 (blocks of 16 along H for
 * x and along I for h).  Weights are NVFP4 as in oracle_matrix (dtype 1).
 */
int oracle_expert_swiglu_w4a4(int n, int H, int I, const uint16_t *x,
                              const void *wg, const uint8_t *sg, double gg,
                              const void *wu, const uint8_t *su, double gu,
                              const void *wd, const uint8_t *sd, double gd,
                              float gx, float gh, double *o) {
  if (n < 0 || H <= 0 || I <= 0 || H % 16 || I % 16 || !(gx > 0.0f) || !(gh > 0.0f))
    return ORACLE_BAD_ARG;
  if (n == 0) return ORACLE_OK;
  oracle_matrix mg = make_matrix(1, wg, sg, gg), mu = make_matrix(1, wu, su, gu),
                md = make_matrix(1, wd, sd, gd);
  float *xf = (float *)malloc(sizeof(float) * (size_t)n * H);
  float *hf = (float *)malloc(sizeof(float) * (size_t)n * I);
  uint8_t *xq = (uint8_t *)malloc((size_t)n * H / 2), *xs = (uint8_t *)malloc((size_t)n * H / 16);
  uint8_t *hq = (uint8_t *)malloc((size_t)n * I / 2), *hs = (uint8_t *)malloc((size_t)n * I / 16);
  double *xd = (double *)malloc(sizeof(double) * (size_t)n * H);
  double *hd = (double *)malloc(sizeof(double) * (size_t)n * I);
  if (!xf || !hf || !xq || !xs || !hq || !hs || !xd || !hd) {
    free(xf); free(hf); free(xq); free(xs); free(hq); free(hs); free(xd); free(hd);
    return ORACLE_BAD_ARG;
  }
  for (size_t i = 0; i < (size_t)n * H; ++i) xf[i] = (float)bf16_value(x[i]);
  oracle_quantize_nvfp4(n, H, xf, gx, xq, xs);
  for (int r = 0; r < n; ++r)
    for (int h = 0; h < H; ++h) {
      const uint8_t byte = xq[(size_t)r * (H / 2) + h / 2];
      const uint8_t code = (h & 1) ? (byte >> 4) : (byte & 15);
      xd[(size_t)r * H + h] = mg.e2m1[code] * mg.e4m3[xs[(size_t)r * (H / 16) + h / 16]] * (double)gx;
    }
#pragma omp parallel
  {
    double *rg = (double *)malloc(sizeof(double) * H);
    double *ru = (double *)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
    for (int i = 0; i < I; ++i) {
      decode_row(&mg, H, i, rg);
      decode_row(&mu, H, i, ru);
      for (int r = 0; r < n; ++r) {
        const double *xr = xd + (size_t)r * H;
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) { g += rg[h] * xr[h]; u += ru[h] * xr[h]; }
        hf[(size_t)r * I + i] = (float)(g / (1.0 + exp(-g)) * u);
      }
    }
    free(rg); free(ru);
  }
  oracle_quantize_nvfp4(n, I, hf, gh, hq, hs);
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < I; ++i) {
      const uint8_t byte = hq[(size_t)r * (I / 2) + i / 2];
      const uint8_t code = (i & 1) ? (byte >> 4) : (byte & 15);
      hd[(size_t)r * I + i] = md.e2m1[code] * md.e4m3[hs[(size_t)r * (I / 16) + i / 16]] * (double)gh;
    }
#pragma omp parallel
  {
    double *rd = (double *)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
    for (int j = 0; j < H; ++j) {
      decode_row(&md, I, j, rd);
      for (int r = 0; r < n; ++r) {
        const double *ar = hd + (size_t)r * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += rd[i] * ar[i];
        o[(size_t)r * H + j] = acc;
      }
    }
    free(rd);
  }
  free(xf); free(hf); free(xq); free(xs); free(hq); free(hs); free(xd); free(hd);
  return ORACLE_OK;
}

/*
 * Weighted combine: y[t] = sum over k = 0..top_k-1, in that order, of
 * topk_w[t,k] * o[t,k,:].  o is fp64 [T, top_k, H]; y is fp64 [T, H].
 * There is no shared expert, so nothing else enters y.
 */
int oracle_combine(int T, int top_k, int H, const float *topk_w, const double *o, double *y) {
  if (T < 0 || top_k <= 0 || H <= 0) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double *yt = y + (size_t)t * H;
    for (int h = 0; h < H; ++h) yt[h] = 0.0;
    for (int k = 0; k < top_k; ++k) {
      double w = (double)topk_w[(size_t)t * top_k + k];
      const double *ok = o + ((size_t)t * top_k + k) * H;
      for (int h = 0; h < H; ++h) yt[h] += w * ok[h];
    }
  }
  return ORACLE_OK;
}

/* ---- auxiliary-loss-free balancing ------------------------------------ */

/*
 * One update of the per-expert selection bias ("Beam 1.0": DeepSeek-V3's
 * auxiliary-loss-free balancing with a cosine decay of the bias updates).
 * Readings: an expert's load is the number of (token, slot) entries routed
 * to it in the batch; the mean load is T*k/E; the step size is
 *   gamma_t = gamma_max * (1 + cos(pi * step / total_steps)) / 2,
 * step clamped to [0, total_steps]; and
 *   bias[e] += gamma_t * sign(mean_load - load_e)     (sign(0) = 0),
 * i.e. underloaded experts are raised, overloaded ones lowered.  gamma_t is
 * computed in fp64 and rounded once to fp32; each update is one fp32 addition.
 * Returns gamma_t (as used, fp32).
 */
float oracle_bias_update(int T, int top_k, int E, const int32_t *topk_idx, float *bias,
                         double gamma_max, int step, int total_steps) {
  double frac = total_steps > 0 ? (double)step / (double)total_steps : 1.0;
  if (frac < 0.0) frac = 0.0;
  if (frac > 1.0) frac = 1.0;
  const float gamma = (float)(gamma_max * 0.5 * (1.0 + cos(M_PI * frac)));
  long *load = (long *)calloc((size_t)E, sizeof(long));
  if (!load) return NAN;
  for (long n = 0; n < (long)T * top_k; ++n) {
    int e = topk_idx[n];
    if (e >= 0 && e < E) load[e] += 1;
  }
  const double mean = (double)T * top_k / (double)E;
  for (int e = 0; e < E; ++e) {
    const double diff = mean - (double)load[e];
    const float sgn = diff > 0 ? 1.0f : (diff < 0 ? -1.0f : 0.0f);
    bias[e] = bias[e] + gamma * sgn;
  }
  free(load);
  return gamma;
}
