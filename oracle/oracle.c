/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, single-threaded fp64 CPU statement of the routed
 * Mixture-of-Experts FFN layer with IQ4_NL expert weights and a sigmoid
 * router.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only at the raw input arrays.
 *
 * Sources (page title, then section):
 *   [EPQ]  HelloSun/xing4_0-29b-IQ4_NL_EPQ model card, "模型與路由"
 *          (router: sigmoid, expert_weights_norm = yes, scale 2.0, top-4 of
 *          64, one shared expert) and "對純 NumPy：單一 expert / 整層"
 *          (IQ4_NL dequantised as a 16-entry nonlinear table times one fp16
 *          scale per block; the layer re-computed as sigmoid, top-4,
 *          normalise by the sum, times routed_scaling_factor, weighted sum of
 *          the 4 experts).
 *   [REC]  PocketLLM "Xing4.0-29B-A4B: the design record", section 2 (the
 *          routed sum and the shared expert are added in wide precision;
 *          silu(gate) * up is handed to the down projection wide) and
 *          section 4 (routes sorted by expert, top-k summed per token).
 *   [ZHU]  zhuai.tech feed, "FFN: feature processing inside each layer"
 *          (gated MLP: y = W_down(act(x W_gate) * (x W_up)), act = SiLU).
 *
 * Readings where the pages are silent (each is restated in the design notes):
 *   - the 16 codebook values are the ones given with the synthetic workload
 *     definition (the pages do not print them);
 *   - inside an 18-byte block (fp16 scale, then 16 bytes), weight j (0..15)
 *     is the low nibble of byte j and weight j+16 is its high nibble;
 *   - experts are selected by descending sigmoid score, equal scores going
 *     to the lower expert id; a logit bias, when given, is added to the
 *     logit before the sigmoid and so enters both selection and weights;
 *   - the shared expert is added with weight 1.
 *
 * All arithmetic is IEEE fp64, compiled without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32
#define BLOCK_BYTES 18

/* IQ4_NL's 16-entry nonlinear codebook (integers; the weight is d * code). */
static const double kCodebook[16] = {
    -127.0, -104.0, -83.0, -65.0, -49.0, -35.0, -22.0, -10.0,
    1.0, 13.0, 25.0, 38.0, 53.0, 69.0, 89.0, 113.0};

/* IEEE-754 binary16 -> double, exact (normals, subnormals, inf, nan). */
double oracle_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 31;
  int man = h & 1023;
  double v;
  if (ex == 0) {
    v = ldexp((double)man, -24);
  } else if (ex == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + man), ex - 25);
  }
  return sign ? -v : v;
}

/* Dequantise n_blocks consecutive IQ4_NL blocks into 32*n_blocks doubles. */
void oracle_iq4nl_dequant(const uint8_t *blocks, int64_t n_blocks, double *w) {
  for (int64_t b = 0; b < n_blocks; ++b) {
    const uint8_t *blk = blocks + BLOCK_BYTES * b;
    double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 16; ++j) {
      w[QK * b + j] = d * kCodebook[qs[j] & 15];
      w[QK * b + j + 16] = d * kCodebook[qs[j] >> 4];
    }
  }
}

/* Encode 32*n_blocks weights with the given fp16 scales: each weight takes
 * the codebook index nearest to w/d (ties to the lower index).  Used to check
 * that decode followed by encode returns the original bytes. */
void oracle_iq4nl_quantize(const double *w, const uint16_t *d_bits,
                           int64_t n_blocks, uint8_t *blocks) {
  for (int64_t b = 0; b < n_blocks; ++b) {
    uint8_t *blk = blocks + BLOCK_BYTES * b;
    double d = oracle_fp16_to_double(d_bits[b]);
    blk[0] = (uint8_t)(d_bits[b] & 0xFF);
    blk[1] = (uint8_t)(d_bits[b] >> 8);
    uint8_t idx[QK];
    for (int j = 0; j < QK; ++j) {
      int best = 0;
      double best_err = fabs(w[QK * b + j] - d * kCodebook[0]);
      for (int c = 1; c < 16; ++c) {
        double e = fabs(w[QK * b + j] - d * kCodebook[c]);
        if (e < best_err) {
          best_err = e;
          best = c;
        }
      }
      idx[j] = (uint8_t)best;
    }
    for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(idx[j] | (idx[j + 16] << 4));
  }
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/*
 * Router [EPQ "模型與路由"]: logits l = x Wr^T (+ bias), scores s = sigmoid(l),
 * the k largest scores selected in descending order, weights
 * w = scale * s / (sum of the selected s).
 *   x [T x H], wr [E x H], bias [T x E] with row stride bias_stride (0: one
 *   row shared by all tokens) or NULL; logits [T x E] may be NULL.
 * Returns 0, or -1 on invalid sizes.
 */
int oracle_route(int64_t T, int64_t H, int64_t E, int64_t k, double scale,
                 const double *x, const double *wr, const double *bias,
                 int64_t bias_stride, double *logits, int32_t *ids,
                 double *weights) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return -1;
  double *l = (double *)malloc(sizeof(double) * (size_t)E);
  double *s = (double *)malloc(sizeof(double) * (size_t)E);
  char *taken = (char *)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) acc += x[t * H + h] * wr[e * H + h];
      if (bias) acc += bias[t * bias_stride + e];
      l[e] = acc;
      s[e] = sigmoid(acc);
      taken[e] = 0;
      if (logits) logits[t * E + e] = acc;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || s[e] > s[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
      sum += s[best];
    }
    for (int64_t j = 0; j < k; ++j) weights[t * k + j] = scale * s[ids[t * k + j]] / sum;
  }
  free(l);
  free(s);
  free(taken);
  return 0;
}

/*
 * Router with a selection-only score bias (noaux_tc) [EPQ "模型與路由":
 * "sigmoid + ffn_exp_probs_b (noaux_tc)"; the bias is a per-expert vector
 * added to the sigmoid probabilities].  Per token t:
 *   l_e = x_t . Wr_e                  s_e = 1 / (1 + exp(-l_e))
 *   the k experts with the largest s_e + b[t, e], in descending order of
 *   that sum, equal sums going to the lower expert id
 *   w_e = scale * s_e / sum over the selected of s   (the unbiased scores)
 * b[t, e] = bias[t * bias_stride + e] (bias_stride 0: one vector for all).
 * logits (may be NULL) receive l.  Returns 0, or -1 on invalid sizes.
 */
int oracle_route_selbias(int64_t T, int64_t H, int64_t E, int64_t k, double scale,
                         const double *x, const double *wr, const double *bias,
                         int64_t bias_stride, double *logits, int32_t *ids,
                         double *weights) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || !bias) return -1;
  double *prob = (double *)malloc(sizeof(double) * (size_t)E);
  double *choice = (double *)malloc(sizeof(double) * (size_t)E);
  char *taken = (char *)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) acc += x[t * H + h] * wr[e * H + h];
      prob[e] = sigmoid(acc);
      choice[e] = prob[e] + bias[t * bias_stride + e];
      taken[e] = 0;
      if (logits) logits[t * E + e] = acc;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || choice[e] > choice[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
      sum += prob[best];
    }
    for (int64_t j = 0; j < k; ++j) weights[t * k + j] = scale * prob[ids[t * k + j]] / sum;
  }
  free(prob);
  free(choice);
  free(taken);
  return 0;
}

/*
 * Layer forward with given routes [EPQ "整層"; REC section 2; ZHU "FFN"]:
 *   out[t] = sum_j weights[t,j] * FFN_{ids[t,j]}(x[t]) + FFN_shared(x[t])
 *   FFN(x) = W_down (silu(W_gate x) * (W_up x)),  silu(g) = g / (1 + e^-g)
 * Each expert matrix is dequantised explicitly into fp64, one matrix at a
 * time, and only for experts that some token selected.
 *   x [T x H]; ids, weights [T x k];
 *   up, gate: [E][F][H/32] blocks; down: [E][H][F/32] blocks;
 *   sh_*: the shared expert's three matrices (ignored when n_shared == 0).
 * Returns 0, -1 on invalid sizes, -2 on an expert id outside [0, E).
 */
int oracle_moe_forward(int64_t T, int64_t H, int64_t E, int64_t k, int64_t F,
                       int64_t n_shared, const double *x, const int32_t *ids,
                       const double *weights, const uint8_t *up,
                       const uint8_t *gate, const uint8_t *down,
                       const uint8_t *sh_up, const uint8_t *sh_gate,
                       const uint8_t *sh_down, double *out) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || F <= 0 || H % QK || F % QK) return -1;
  for (int64_t i = 0; i < T * k; ++i)
    if (ids[i] < 0 || ids[i] >= E) return -2;
  memset(out, 0, sizeof(double) * (size_t)(T * H));
  if (T == 0) return 0;

  const int64_t up_blocks = F * (H / QK);   /* blocks in one [F x H] matrix */
  const int64_t down_blocks = H * (F / QK); /* blocks in one [H x F] matrix */
  double *wu = (double *)malloc(sizeof(double) * (size_t)(F * H));
  double *wg = (double *)malloc(sizeof(double) * (size_t)(F * H));
  double *wd = (double *)malloc(sizeof(double) * (size_t)(H * F));
  double *h = (double *)malloc(sizeof(double) * (size_t)F);
  /* an expert may be named in several slots of one token, so it can hold up
   * to T * k routes (and the shared expert T <= T * k) */
  int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T * k));
  double *wt = (double *)malloc(sizeof(double) * (size_t)(T * k));

  for (int64_t e = 0; e < E + n_shared; ++e) {
    const int shared = (e == E);
    int64_t n = 0;
    if (shared) {
      for (int64_t t = 0; t < T; ++t) {
        tok[n] = t;
        wt[n] = 1.0;
        ++n;
      }
    } else {
      for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < k; ++j)
          if (ids[t * k + j] == e) {
            tok[n] = t;
            wt[n] = weights[t * k + j];
            ++n;
          }
    }
    if (n == 0) continue;
    const uint8_t *bu = shared ? sh_up : up + (size_t)(e * up_blocks * BLOCK_BYTES);
    const uint8_t *bg = shared ? sh_gate : gate + (size_t)(e * up_blocks * BLOCK_BYTES);
    const uint8_t *bd = shared ? sh_down : down + (size_t)(e * down_blocks * BLOCK_BYTES);
    oracle_iq4nl_dequant(bu, up_blocks, wu);
    oracle_iq4nl_dequant(bg, up_blocks, wg);
    oracle_iq4nl_dequant(bd, down_blocks, wd);
    for (int64_t i = 0; i < n; ++i) {
      const double *xt = x + tok[i] * H;
      for (int64_t f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int64_t c = 0; c < H; ++c) {
          g += wg[f * H + c] * xt[c];
          u += wu[f * H + c] * xt[c];
        }
        h[f] = g * sigmoid(g) * u;
      }
      double *ot = out + tok[i] * H;
      for (int64_t r = 0; r < H; ++r) {
        double y = 0.0;
        for (int64_t f = 0; f < F; ++f) y += wd[r * F + f] * h[f];
        ot[r] += wt[i] * y;
      }
    }
  }
  free(wu);
  free(wg);
  free(wd);
  free(h);
  free(tok);
  free(wt);
  return 0;
}

/* Unweighted RMS normalisation of each row: u = r / sqrt(mean(r^2) + eps). */
void oracle_rmsnorm(int64_t T, int64_t H, const double *r, double eps, double *u) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t c = 0; c < H; ++c) ss += r[t * H + c] * r[t * H + c];
    double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t c = 0; c < H; ++c) u[t * H + c] = r[t * H + c] * inv;
  }
}
