/*
 * maskllm_oracle.c -- plain, slow, single-threaded CPU definition of the
 * MaskLLM differentiable 2:4 mask layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant generator with the
 * CUDA library; it was written from the method's description, not from the
 * kernels.
 *
 * Sources (titles of the pages the method is described on):
 *  [MaskLLM]  "MaskLLM: Learnable Semi-Structured Sparsity for Large Language
 *             Models" (project page), Abstract, Fig. 3 caption (per-group
 *             categorical distribution over candidate masks, Gumbel softmax,
 *             weighted averaging, all differentiable), Fig. 5 caption (scaling
 *             factor kappa), Table 2 caption (prior masks), Table 3 caption
 *             (weight regularisation).
 *  [ASDNN]    "Accelerating Sparse Deep Neural Networks" (Mishra et al.),
 *             Sec. 1 and 3 (2:4 = at least two zeros in every four consecutive
 *             values), Sec. 3.1 (two values per group + 2-bit position
 *             metadata; ~44%/~38% storage saving), Sec. 4.1 (magnitude
 *             pruning keeps the two largest of four).
 *  [Philox]   Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
 *             as 1, 2, 3", SC'11 -- the Philox4x32 bijection, 10 rounds.
 *  [CPERM]    "Channel Permutations for N:M Sparsity" (abstract: a quality
 *             metric to judge permutations, a search for good ones); with
 *             [ASDNN] Sec. 4.1 (permuting weight columns before pruning raises
 *             the magnitude that 2:4 pruning keeps, Fig. 5: 83.7 -> 102.9).
 *
 * The layer, per group of 4 consecutive weights w[0..3] of a row of W:
 *   candidates  S_c, c = 0..5: the kept index pairs in lexicographic order
 *               (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
 *   noise       g_c: Gumbel(0,1) drawn from Philox4x32-10, keyed by the seed,
 *               counter = (group index, step, tensor id); see orc_noise_words
 *   probs       p = softmax((kappa*L + g) / tau)
 *   soft mask   M_j = sum_c p_c S_cj
 *   output      W'_j = bf16(w_j * M_j);  row_sq[r] = sum_j (w_j M_j)^2
 *   backward    dL/dlogits from dL/dW' (straight through the bf16 rounding)
 *   hard mask   argmax_c L_c, packed as 2 kept values + 2-bit positions
 *
 * Precision.  The logits are fp32 tensors, and the noisy logit
 *   z_c = fl( fl( fl(kappa*L_c) + g_c ) * rho ),  rho = fl32(1/tau)
 * is formed in fp32 in exactly this order: with kappa/tau in the thousands one
 * ulp of z moves p far beyond any useful tolerance, so this rounding sequence
 * is part of the definition (both sides must form z identically).  Likewise
 * the magnitude prior is formed in fp32 as fl(s * fl(|w_i| + |w_j|)).  Every
 * later step (softmax, soft mask, products, sums, gradients) is computed here
 * in double and rounded only where the output type demands it (W' to bf16 by
 * round-to-nearest-even directly from the double product).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math (no FMA
 * contraction, so every fp32 statement below is one IEEE operation).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_NCAND 6
#define ORC_TABLE_BITS 14
#define ORC_TABLE_SIZE (1 << ORC_TABLE_BITS)

/* The six 2:4 candidates as kept index pairs, lexicographic order [ASDNN
 * Sec. 3; MaskLLM Fig. 3: "candidate masks" of each group of M=4]. */
static const int ORC_PAIR[ORC_NCAND][2] = {
    {0, 1}, {0, 2}, {0, 3}, {1, 2}, {1, 3}, {2, 3}};

int orc_candidate_pair(int c, int which) {
  if (c < 0 || c >= ORC_NCAND || which < 0 || which > 1) return -1;
  return ORC_PAIR[c][which];
}

/* S_cj: 1 when position j of a group is kept by candidate c. */
int orc_candidate_keeps(int c, int j) {
  return ORC_PAIR[c][0] == j || ORC_PAIR[c][1] == j;
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> binary64                                                          */
/* ------------------------------------------------------------------------ */

double orc_bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bfloat16 (ties to even), in one rounding.
 * bfloat16: 1 sign, 8 exponent (bias 127), 7 stored fraction bits; normal
 * values have 8 significant bits, subnormals a fixed spacing of 2^-133. */
uint16_t orc_double_to_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
  int spacing_exp = e - 8;     /* ulp of an 8-significant-bit value in [2^(e-1), 2^e) */
  if (spacing_exp < -133) spacing_exp = -133;  /* subnormal range */
  double q = ldexp(a, -spacing_exp);            /* exact: power-of-two scaling */
  double r = nearbyint(q);                      /* default mode: nearest, ties even */
  double v = ldexp(r, spacing_exp);             /* exact */
  /* Largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds above it
   * overflows to infinity. */
  const double bf16_max = ldexp(255.0, 120);
  if (v > bf16_max) return (uint16_t)(sign | 0x7F80u);
  float f = (float)v;                           /* exact: v has <= 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

static float orc_bf16_to_float(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Counter-based RNG: Philox4x32-10 [Philox].                                  */
/* ------------------------------------------------------------------------ */

/* One application of the Philox4x32 bijection with 10 rounds.  Each round
 * multiplies counter words 0 and 2 by the two Philox multipliers, swaps the
 * high halves across and xors in the round key; the key advances by the two
 * Weyl constants (golden ratio and sqrt(3)-1 scaled to 32 bits) per round. */
void orc_philox4x32_10(const uint32_t key[2], const uint32_t ctr[4], uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t k0 = key[0], k1 = key[1];
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  for (int round = 0; round < 10; ++round) {
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    k0 += weyl0;
    k1 += weyl1;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The four noise words of one group: key = (seed low, seed high), counter =
 * (group index low, group index high, step, tensor id).  The group index is
 * the row-major index of the group within its matrix: row * (cols/4) + k. */
void orc_group_words(uint64_t seed, uint32_t step, uint32_t tensor_id,
                     uint64_t group, uint32_t words[4]) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)group, (uint32_t)(group >> 32), step, tensor_id};
  orc_philox4x32_10(key, ctr, words);
}

void orc_noise_words(uint64_t seed, uint32_t step, uint32_t tensor_id,
                     int64_t group_begin, int64_t n, uint32_t* out4) {
  for (int64_t i = 0; i < n; ++i)
    orc_group_words(seed, step, tensor_id, (uint64_t)(group_begin + i), out4 + 4 * i);
}

/* ------------------------------------------------------------------------ */
/* Gumbel noise.                                                              */
/* ------------------------------------------------------------------------ */

/* Table of Gumbel(0,1) quantiles at the midpoints of 2^14 equal cells of
 * (0,1): T[i] = -ln(-ln(u_i)), u_i = (i + 1/2) / 2^14, computed in double and
 * rounded once to fp32.  Inverse-CDF sampling of Gumbel(0,1): if
 * u ~ U(0,1) then -ln(-ln u) ~ Gumbel(0,1). */
void orc_gumbel_table(float* table) {
  for (int i = 0; i < ORC_TABLE_SIZE; ++i) {
    double u = ((double)i + 0.5) / (double)ORC_TABLE_SIZE;
    table[i] = (float)(-log(-log(u)));
  }
}

/* Candidate c takes the 16-bit half (c & 1) of word (c >> 1) -- the low half
 * for even c -- and uses its top 14 bits as the table cell.  Word 3 is not
 * used. */
int orc_gumbel_cell(const uint32_t words[4], int c) {
  uint32_t half = (words[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
  return (int)(half >> 2);
}

/* ------------------------------------------------------------------------ */
/* One group: probabilities, soft mask.                                       */
/* ------------------------------------------------------------------------ */

/* p = softmax((kappa*L + g)/tau) for one group [MaskLLM Fig. 3, Fig. 5].
 * exact == 0: z formed in fp32 as in the header (the definition used for
 *             parity).
 * exact != 0: z formed in double without intermediate rounding; used only by
 *             the finite-difference checks, which need a smooth function of
 *             the logits.
 * The softmax itself is in double. */
void orc_group_probs(const float logits[6], const float gumbel[6], float kappa,
                     float tau, int exact, double p[6], double z_out[6]) {
  double z[ORC_NCAND];
  if (exact) {
    for (int c = 0; c < ORC_NCAND; ++c)
      z[c] = ((double)kappa * (double)logits[c] + (double)gumbel[c]) / (double)tau;
  } else {
    const float rho = (float)(1.0 / (double)tau);
    for (int c = 0; c < ORC_NCAND; ++c) {
      float a = kappa * logits[c];
      float s = a + gumbel[c];
      float zc = s * rho;
      z[c] = (double)zc;
    }
  }
  double m = z[0];
  for (int c = 1; c < ORC_NCAND; ++c)
    if (z[c] > m) m = z[c];
  double e[ORC_NCAND], sum = 0.0;
  for (int c = 0; c < ORC_NCAND; ++c) {
    e[c] = exp(z[c] - m);
    sum += e[c];
  }
  for (int c = 0; c < ORC_NCAND; ++c) p[c] = e[c] / sum;
  if (z_out)
    for (int c = 0; c < ORC_NCAND; ++c) z_out[c] = z[c];
}

/* M_j = sum_c p_c S_cj: the weighted average of the candidate masks
 * [MaskLLM Fig. 3 "weighted averaging"]. */
void orc_soft_mask(const double p[6], double mask[4]) {
  for (int j = 0; j < 4; ++j) {
    double s = 0.0;
    for (int c = 0; c < ORC_NCAND; ++c)
      if (orc_candidate_keeps(c, j)) s += p[c];
    mask[j] = s;
  }
}

/* dl/dlogits of one group, given the upstream gradient t_j = dl/dx_j of the
 * unrounded masked weights x_j = w_j M_j.  With h_j = t_j w_j = dl/dM_j,
 * dl/dp_c = sum_j S_cj h_j, and the softmax Jacobian gives
 * dl/dz_c = p_c (dl/dp_c - sum_d p_d dl/dp_d); dz_c/dL_c = kappa*rho. */
void orc_group_backward(const double p[6], const double w[4], const double t[4],
                        double dz_dlogit, double dlogits[6]) {
  double h[4];
  for (int j = 0; j < 4; ++j) h[j] = t[j] * w[j];
  double dp[ORC_NCAND], r = 0.0;
  for (int c = 0; c < ORC_NCAND; ++c) {
    dp[c] = h[ORC_PAIR[c][0]] + h[ORC_PAIR[c][1]];
    r += p[c] * dp[c];
  }
  for (int c = 0; c < ORC_NCAND; ++c) dlogits[c] = dz_dlogit * p[c] * (dp[c] - r);
}

/* ------------------------------------------------------------------------ */
/* Whole matrices (rows [row_begin, row_begin + rows) of a [*, cols] matrix;  */
/* pointers address the first processed row).                                */
/* ------------------------------------------------------------------------ */

static float orc_table_cache[ORC_TABLE_SIZE];
static int orc_table_ready = 0;

static const float* orc_table(void) {
  if (!orc_table_ready) {
    orc_gumbel_table(orc_table_cache);
    orc_table_ready = 1;
  }
  return orc_table_cache;
}

static void orc_group_noise(const float* table, uint64_t seed, uint32_t step,
                            uint32_t tensor_id, uint64_t group, float g[6]) {
  uint32_t words[4];
  orc_group_words(seed, step, tensor_id, group, words);
  for (int c = 0; c < ORC_NCAND; ++c) g[c] = table[orc_gumbel_cell(words, c)];
}

/* The Gumbel noise g[n, 6] of n consecutive groups starting at group_begin. */
void orc_gumbel_noise(uint64_t seed, uint32_t step, uint32_t tensor_id,
                      int64_t group_begin, int64_t n, float* out6) {
  const float* table = orc_table();
  for (int64_t i = 0; i < n; ++i)
    orc_group_noise(table, seed, step, tensor_id, (uint64_t)(group_begin + i), out6 + 6 * i);
}

/* Magnitude prior [MaskLLM Table 2: prior masks initialise the logits;
 * ASDNN Sec. 4.1: magnitude pruning keeps the two largest |w| of four]:
 * L_c = fl32(scale * fl32(|w_i| + |w_j|)) for the kept pair (i, j) of c. */
void orc_prior_init(const uint16_t* W, int64_t rows, int64_t cols, float scale,
                    float* logits) {
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < gpr; ++k) {
      const uint16_t* w = W + r * cols + 4 * k;
      float* L = logits + (r * gpr + k) * ORC_NCAND;
      for (int c = 0; c < ORC_NCAND; ++c) {
        float a = fabsf(orc_bf16_to_float(w[ORC_PAIR[c][0]]));
        float b = fabsf(orc_bf16_to_float(w[ORC_PAIR[c][1]]));
        float sum = a + b;
        L[c] = scale * sum;
      }
    }
}

/* Forward [MaskLLM Fig. 3; Table 3 for the row regulariser].  Outputs:
 *   W_out  bf16 [rows, cols]     W' = bf16_rne(w * M)
 *   row_sq double [rows]         sum over the row of (w * M)^2  (nullable)
 *   probs  double [rows, cols/4, 6]                             (nullable)
 *   masks  double [rows, cols]   the soft mask M                (nullable) */
void orc_forward(const uint16_t* W, const float* logits, int64_t rows, int64_t cols,
                 int64_t row_begin, float tau, float kappa, uint64_t seed,
                 uint32_t step, uint32_t tensor_id, uint16_t* W_out,
                 double* row_sq, double* probs, double* masks) {
  const float* table = orc_table();
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r) {
    double sq = 0.0;
    for (int64_t k = 0; k < gpr; ++k) {
      const uint64_t group = (uint64_t)((row_begin + r) * gpr + k);
      const float* L = logits + (r * gpr + k) * ORC_NCAND;
      float g[ORC_NCAND];
      orc_group_noise(table, seed, step, tensor_id, group, g);
      double p[ORC_NCAND], M[4];
      orc_group_probs(L, g, kappa, tau, 0, p, NULL);
      orc_soft_mask(p, M);
      for (int j = 0; j < 4; ++j) {
        const int64_t idx = r * cols + 4 * k + j;
        double x = orc_bf16_to_double(W[idx]) * M[j];
        W_out[idx] = orc_double_to_bf16(x);
        sq += x * x;
        if (masks) masks[idx] = M[j];
      }
      if (probs)
        for (int c = 0; c < ORC_NCAND; ++c) probs[(r * gpr + k) * ORC_NCAND + c] = p[c];
    }
    if (row_sq) row_sq[r] = sq;
  }
}

/* Backward [MaskLLM Fig. 3: every step is differentiable; Table 3: weight
 * regularisation].  The loss seen by the layer is
 *   l = <G, W'> + reg * sum (w M)^2
 * with the bf16 rounding of W' passed straight through.  So
 * t_j = G_j + 2 reg x_j, and the noise is a constant.  Output
 * dlogits double [rows, cols/4, 6]. */
void orc_backward(const uint16_t* W, const float* logits, const uint16_t* grad_out,
                  int64_t rows, int64_t cols, int64_t row_begin, float tau,
                  float kappa, uint64_t seed, uint32_t step, uint32_t tensor_id,
                  float reg_coeff, int exact, double* dlogits) {
  const float* table = orc_table();
  const int64_t gpr = cols / 4;
  const double dz_dlogit = exact ? (double)kappa / (double)tau
                                 : (double)kappa * (double)(float)(1.0 / (double)tau);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < gpr; ++k) {
      const uint64_t group = (uint64_t)((row_begin + r) * gpr + k);
      const float* L = logits + (r * gpr + k) * ORC_NCAND;
      float g[ORC_NCAND];
      orc_group_noise(table, seed, step, tensor_id, group, g);
      double p[ORC_NCAND], M[4], w[4], t[4];
      orc_group_probs(L, g, kappa, tau, exact, p, NULL);
      orc_soft_mask(p, M);
      for (int j = 0; j < 4; ++j) {
        const int64_t idx = r * cols + 4 * k + j;
        w[j] = orc_bf16_to_double(W[idx]);
        double x = w[j] * M[j];
        t[j] = orc_bf16_to_double(grad_out[idx]) + 2.0 * (double)reg_coeff * x;
      }
      orc_group_backward(p, w, t, dz_dlogit, dlogits + (r * gpr + k) * ORC_NCAND);
    }
}

/* The smooth loss the backward differentiates, for finite differences:
 * l = sum G_j x_j + reg * sum x_j^2, x = w * M(L), z formed in double
 * (exact mode), same noise. */
double orc_loss_exact(const uint16_t* W, const float* logits, const uint16_t* grad_out,
                      int64_t rows, int64_t cols, int64_t row_begin, float tau,
                      float kappa, uint64_t seed, uint32_t step, uint32_t tensor_id,
                      float reg_coeff) {
  const float* table = orc_table();
  const int64_t gpr = cols / 4;
  double loss = 0.0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < gpr; ++k) {
      const uint64_t group = (uint64_t)((row_begin + r) * gpr + k);
      const float* L = logits + (r * gpr + k) * ORC_NCAND;
      float g[ORC_NCAND];
      orc_group_noise(table, seed, step, tensor_id, group, g);
      double p[ORC_NCAND], M[4];
      orc_group_probs(L, g, kappa, tau, 1, p, NULL);
      orc_soft_mask(p, M);
      for (int j = 0; j < 4; ++j) {
        const int64_t idx = r * cols + 4 * k + j;
        double x = orc_bf16_to_double(W[idx]) * M[j];
        loss += orc_bf16_to_double(grad_out[idx]) * x + (double)reg_coeff * x * x;
      }
    }
  return loss;
}

/* Hard mask: the candidate with the largest raw logit (no noise; kappa and
 * tau play no part), lowest index on ties; a NaN logit never wins and a group
 * of six NaNs selects candidate 0 [MaskLLM: the learned distribution's most
 * likely mask is the deployed mask]. */
int orc_hard_index(const float logits[6]) {
  int best = -1;
  for (int c = 0; c < ORC_NCAND; ++c) {
    if (isnan(logits[c])) continue;
    if (best < 0 || logits[c] > logits[best]) best = c;
  }
  return best < 0 ? 0 : best;
}

/* 2:4 compressed storage [ASDNN Sec. 3.1: only the two kept values of each
 * group of four are stored, plus 2 bits per kept value giving its position].
 * Layout (row-major, one row at a time):
 *   values [rows, cols/2] bf16: group k of row r keeps w[i], w[j] (i < j) at
 *          values[r, 2k] and values[r, 2k+1];
 *   meta   [rows, cols/32] u32: group k's 4-bit code (i | j << 2) sits at
 *          bits 4*(k % 8) .. 4*(k % 8)+3 of meta[r, k / 8];
 *   idx    [rows, cols/4] u8: the chosen candidate (nullable). */
void orc_hard_compress(const uint16_t* W, const float* logits, int64_t rows, int64_t cols,
                       uint16_t* values, uint32_t* meta, uint8_t* idx) {
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t m = 0; m < cols / 32; ++m) meta[r * (cols / 32) + m] = 0u;
    for (int64_t k = 0; k < gpr; ++k) {
      const int c = orc_hard_index(logits + (r * gpr + k) * ORC_NCAND);
      const int i = ORC_PAIR[c][0], j = ORC_PAIR[c][1];
      values[r * (cols / 2) + 2 * k] = W[r * cols + 4 * k + i];
      values[r * (cols / 2) + 2 * k + 1] = W[r * cols + 4 * k + j];
      const uint32_t code = (uint32_t)(i | (j << 2));
      meta[r * (cols / 32) + k / 8] |= code << (4 * (k % 8));
      if (idx) idx[r * gpr + k] = (uint8_t)c;
    }
  }
}

/* Inverse of the storage above: kept values back in place, +0 (0x0000)
 * elsewhere. */
void orc_decompress(const uint16_t* values, const uint32_t* meta, int64_t rows,
                    int64_t cols, uint16_t* W_out) {
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < gpr; ++k) {
      const uint32_t code = (meta[r * (cols / 32) + k / 8] >> (4 * (k % 8))) & 0xFu;
      const int i = (int)(code & 3u), j = (int)(code >> 2);
      for (int q = 0; q < 4; ++q) W_out[r * cols + 4 * k + q] = 0u;
      W_out[r * cols + 4 * k + i] = values[r * (cols / 2) + 2 * k];
      W_out[r * cols + 4 * k + j] = values[r * (cols / 2) + 2 * k + 1];
    }
}

/* Bytes of the compressed form of a [rows, cols] operand with elem_bytes-wide
 * elements: half the values plus 4 bits of metadata per group of four. */
int64_t orc_compressed_bytes(int64_t rows, int64_t cols, int64_t elem_bytes) {
  return rows * (cols / 2) * elem_bytes + rows * (cols / 4) / 2;
}

/* ------------------------------------------------------------------------ */
/* Prior from a given mask and the convergence diagnostics.                   */
/* ------------------------------------------------------------------------ */

/* The candidate whose kept pair (i, j) has metadata code i | j << 2, or -1
 * for a code that names no candidate. */
int orc_candidate_of_code(uint32_t code) {
  for (int c = 0; c < ORC_NCAND; ++c)
    if ((uint32_t)(ORC_PAIR[c][0] | (ORC_PAIR[c][1] << 2)) == code) return c;
  return -1;
}

/* Logits that start from a given mask [MaskLLM Table 2: learned masks use a
 * prior mask for initialisation; transfer of masks across tasks]: for every
 * group, `high` on the candidate its 4-bit code names and `low` on the other
 * five; a code naming no candidate gives `low` everywhere.  meta is the 2:4
 * metadata layout of orc_hard_compress. */
void orc_prior_from_mask(const uint32_t* meta, int64_t rows, int64_t cols, float high,
                         float low, float* logits) {
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < gpr; ++k) {
      const uint32_t code = (meta[r * (cols / 32) + k / 8] >> (4 * (k % 8))) & 0xFu;
      const int c_prior = orc_candidate_of_code(code);
      for (int c = 0; c < ORC_NCAND; ++c)
        logits[(r * gpr + k) * ORC_NCAND + c] = (c == c_prior) ? high : low;
    }
}

/* Convergence diagnostics of one step [MaskLLM Fig. 5: (a) the L1 distance
 * of sampled masks between adjacent training steps; (b) the maximum
 * probability of the mask distribution; kappa sets the randomness].
 *   sample   the candidate drawn at this step: the first maximum of the noisy
 *            logits z (fp32, as in orc_group_probs) -- the mask the soft mask
 *            tends to as tau -> 0;
 *   l1       per row, sum over groups of |S_sample - S_prev|_1 (0, 2 or 4 per
 *            group) against the previous step's samples prev_idx (nullable:
 *            then l1 is not computed);
 *   maxprob  per row, sum over groups of max_c softmax(fl32(kappa * L))_c,
 *            the categorical distribution the draw samples from (no noise).
 * Outputs: idx_out u8 [rows, cols/4] (nullable), l1_row int64 [rows]
 * (nullable), maxprob_row double [rows] (nullable). */
void orc_mask_stats(const float* logits, int64_t rows, int64_t cols, int64_t row_begin,
                    float tau, float kappa, uint64_t seed, uint32_t step, uint32_t tensor_id,
                    const uint8_t* prev_idx, uint8_t* idx_out, int64_t* l1_row,
                    double* maxprob_row) {
  const float* table = orc_table();
  const int64_t gpr = cols / 4;
  for (int64_t r = 0; r < rows; ++r) {
    int64_t l1 = 0;
    double mp = 0.0;
    for (int64_t k = 0; k < gpr; ++k) {
      const uint64_t group = (uint64_t)((row_begin + r) * gpr + k);
      const float* L = logits + (r * gpr + k) * ORC_NCAND;
      float g[ORC_NCAND];
      orc_group_noise(table, seed, step, tensor_id, group, g);
      double p[ORC_NCAND], z[ORC_NCAND];
      orc_group_probs(L, g, kappa, tau, 0, p, z);
      int s = 0;
      for (int c = 1; c < ORC_NCAND; ++c)
        if (z[c] > z[s]) s = c;
      if (idx_out) idx_out[r * gpr + k] = (uint8_t)s;
      if (prev_idx) {
        const int q = prev_idx[r * gpr + k];
        for (int j = 0; j < 4; ++j) l1 += orc_candidate_keeps(s, j) != orc_candidate_keeps(q, j);
      }
      double y[ORC_NCAND], m = -INFINITY, sum = 0.0;
      for (int c = 0; c < ORC_NCAND; ++c) {
        float a = kappa * L[c];
        y[c] = (double)a;
        if (y[c] > m) m = y[c];
      }
      for (int c = 0; c < ORC_NCAND; ++c) sum += exp(y[c] - m);
      mp += 1.0 / sum;   /* the largest term is exp(0) = 1 */
    }
    if (l1_row) l1_row[r] = l1;
    if (maxprob_row) maxprob_row[r] = mp;
  }
}

/* ------------------------------------------------------------------------ */
/* Channel permutation before pruning [CPERM; ASDNN Sec. 4.1].                 */
/* ------------------------------------------------------------------------ */
/*
 * A permutation perm of the cols input channels puts channel perm[i] into
 * column ("slot") i:  W_perm[r, i] = W[r, perm[i]].  (The layer producing
 * those channels permutes its output rows the same way, so the product is
 * unchanged; that is the caller's business.)
 *
 * Quality metric: the total magnitude that 2:4 magnitude pruning keeps after
 * the permutation, sum over rows and groups of the two largest |W_perm| of
 * each group of four.
 *
 * Search: steepest ascent over channel swaps.  A swap exchanges the channels
 * of two slots in different groups; each step applies the swap that raises
 * the metric most (ties: the smallest first slot a, then the smallest second
 * slot b, a < b), and the search stops when no swap raises it or after
 * max_swaps swaps.  (The pages name two further devices for escaping local
 * optima without describing them; they are not part of this definition.)
 *
 * Exact comparison.  The search compares swaps on fixed-point magnitudes
 *   q(w) = floor(|w| * 2^k),  k = 31 - ceil(log2 rows) - floor(log2 max|w|)
 * (k = 0 for an all-zero matrix), so that any column sum of q over the rows is
 * below 2^32 and every gain is an exact integer, whatever the order of the
 * additions.  The float metric is also given, in double.
 */

/* floor(log2 x) for a finite x > 0. */
static int orc_floor_log2(double x) {
  int e;
  (void)frexp(x, &e);   /* x = f * 2^e, f in [0.5, 1) */
  return e - 1;
}

/* The fixed-point shift k of a matrix, or INT32_MIN when a weight is not
 * finite. */
int32_t orc_perm_shift(const uint16_t* W, int64_t rows, int64_t cols) {
  double mx = 0.0;
  for (int64_t i = 0; i < rows * cols; ++i) {
    const double a = fabs(orc_bf16_to_double(W[i]));
    if (!isfinite(a)) return INT32_MIN;
    if (a > mx) mx = a;
  }
  if (mx == 0.0) return 0;
  int lr = 0;
  while (((int64_t)1 << lr) < rows) ++lr;   /* ceil(log2 rows) */
  return 31 - lr - orc_floor_log2(mx);
}

/* q(w) = floor(|w| * 2^k): exact in double (a power-of-two scaling of a value
 * with 8 significant bits), then truncated. */
uint32_t orc_perm_fixed(uint16_t w, int32_t shift) {
  return (uint32_t)floor(ldexp(fabs(orc_bf16_to_double(w)), shift));
}

/* The two largest of four. */
static double orc_top2(double a, double b, double c, double d) {
  double v[4] = {a, b, c, d};
  for (int i = 0; i < 2; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (v[j] > v[i]) {
        const double t = v[i];
        v[i] = v[j];
        v[j] = t;
      }
  return v[0] + v[1];
}

/* Kept fixed-point magnitude of the group of slots 4g..4g+3 of row r. */
static uint64_t orc_group_kept_fixed(const uint16_t* W, int64_t cols, const int32_t* perm,
                                     int32_t shift, int64_t r, int64_t g) {
  double q[4];
  for (int j = 0; j < 4; ++j) q[j] = (double)orc_perm_fixed(W[r * cols + perm[4 * g + j]], shift);
  return (uint64_t)orc_top2(q[0], q[1], q[2], q[3]);
}

/* Metric of a permutation in fixed point (exact). */
uint64_t orc_perm_metric_fixed(const uint16_t* W, int64_t rows, int64_t cols,
                               const int32_t* perm, int32_t shift) {
  uint64_t total = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < cols / 4; ++g) total += orc_group_kept_fixed(W, cols, perm, shift, r, g);
  return total;
}

/* Metric of a permutation: kept magnitude, in double. */
double orc_perm_metric(const uint16_t* W, int64_t rows, int64_t cols, const int32_t* perm) {
  double total = 0.0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < cols / 4; ++g) {
      double a[4];
      for (int j = 0; j < 4; ++j) a[j] = fabs(orc_bf16_to_double(W[r * cols + perm[4 * g + j]]));
      total += orc_top2(a[0], a[1], a[2], a[3]);
    }
  return total;
}

/* Fixed-point gain of exchanging the channels of slots a and b: the change of
 * the two groups' kept magnitude, summed over the rows (0 within a group). */
int64_t orc_perm_swap_gain(const uint16_t* W, int64_t rows, int64_t cols, int32_t* perm,
                           int32_t shift, int64_t a, int64_t b) {
  const int64_t ga = a / 4, gb = b / 4;
  if (ga == gb) return 0;
  int64_t before = 0, after = 0;
  for (int64_t r = 0; r < rows; ++r)
    before += (int64_t)(orc_group_kept_fixed(W, cols, perm, shift, r, ga) +
                        orc_group_kept_fixed(W, cols, perm, shift, r, gb));
  int32_t t = perm[a];
  perm[a] = perm[b];
  perm[b] = t;
  for (int64_t r = 0; r < rows; ++r)
    after += (int64_t)(orc_group_kept_fixed(W, cols, perm, shift, r, ga) +
                       orc_group_kept_fixed(W, cols, perm, shift, r, gb));
  perm[b] = perm[a];
  perm[a] = t;
  return after - before;
}

/* Steepest-ascent channel-swap search from perm (updated in place).  Swap s
 * is logged as slots swaps[2s], swaps[2s+1] and its gain gains[s] (both
 * nullable).  Returns the number of swaps applied. */
int32_t orc_perm_search(const uint16_t* W, int64_t rows, int64_t cols, int32_t* perm,
                        int32_t shift, int32_t max_swaps, int32_t* swaps, int64_t* gains) {
  int32_t n = 0;
  while (n < max_swaps) {
    int64_t best = 0, ba = -1, bb = -1;
    for (int64_t a = 0; a < cols; ++a)
      for (int64_t b = a + 1; b < cols; ++b) {
        const int64_t g = orc_perm_swap_gain(W, rows, cols, perm, shift, a, b);
        if (g > best) {
          best = g;
          ba = a;
          bb = b;
        }
      }
    if (ba < 0) break;
    const int32_t t = perm[ba];
    perm[ba] = perm[bb];
    perm[bb] = t;
    if (swaps) {
      swaps[2 * n] = (int32_t)ba;
      swaps[2 * n + 1] = (int32_t)bb;
    }
    if (gains) gains[n] = best;
    ++n;
  }
  return n;
}
