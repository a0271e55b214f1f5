/*
 * Plain fp64 CPU oracle for the speculative accept/reject step that follows a verify pass.
 *
 * TEST INFRASTRUCTURE ONLY, like attention.c: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the CUDA library never loads or calls it, and the
 * two share no code.
 *
 * Sources (web pages, cited by title and section):
 *   [tinydecode/spec]  "tinydecode", section "speculative decoding": acceptance is the usual
 *       min(1, p_t / p_d) per draft token; the extra token comes from the residual
 *       (p_t - p_d)+ at the first rejection, or from the bonus row when every draft token
 *       went through; at temperature 0 this is "accept while the argmax matches".
 *   [flashspec]  "FlashSpec", sections "What is FlashSpec?" and "How it works" (the
 *       "Correctness" paragraph): the test is u_i < min(1, p(x_i) / q(x_i)), computed in
 *       log space to avoid underflow; a rejected position samples its token from
 *       max(0, p - q) / ||max(0, p - q)||_1 (Leviathan et al. 2023, Algorithm 1); greedy
 *       decoding takes the longest prefix matching the target's argmax.
 *
 * Layouts: target logits [B, G+1, V] (row i: the target's next-token logits after the
 * prefix and the first i draft tokens); draft logits [B, G, V] (row i: the distribution
 * draft token i was drawn from); draft tokens [B, G]; uniforms [B, G+1] in [0, 1): entry i
 * < G decides draft token i, entry G draws the extra token. Probabilities are
 * softmax(logits / temperature); temperature 0 is greedy.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - the extra token is drawn by inverse CDF: the smallest k whose running weight sum
 *     exceeds u * (total weight);
 *   - a residual whose weights are all zero (p = q at that row, reachable only through
 *     rounding) falls back to p;
 *   - a draft token outside [0, V) counts as rejected and raises a status bit;
 *   - argmax ties go to the lowest token id.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

#define ORC_BAD_TOKEN 64u

/* ln sum_k exp(row[k] / T) in fp64 (-inf for an all -inf row). */
static double row_lse(const float *row, int V, double T) {
  double m = -INFINITY;
  for (int k = 0; k < V; ++k) m = fmax(m, (double)row[k] / T);
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int k = 0; k < V; ++k) s += exp((double)row[k] / T - m);
  return m + log(s);
}

/* Lowest index of the largest entry. */
static int row_argmax(const float *row, int V) {
  int best = 0;
  for (int k = 1; k < V; ++k)
    if (row[k] > row[best]) best = k;
  return best;
}

/* Inverse-CDF draw from nonnegative weights w[0..V): the smallest k with
 * w[0] + ... + w[k] > u * W. A draw that rounding pushes past the end takes the last
 * index of positive weight. */
static int draw(const double *w, int V, double u) {
  double W = 0.0;
  for (int k = 0; k < V; ++k) W += w[k];
  const double target = u * W;
  double run = 0.0;
  int last = 0;
  for (int k = 0; k < V; ++k) {
    if (w[k] > 0.0) last = k;
    run += w[k];
    if (run > target) return k;
  }
  return last;
}

/* One accept/reject step for each of the B sequences; see the header for the layouts.
 * Writes n_accepted[b] (0..G) and next_token[b]; returns status bits. */
unsigned orc_spec_accept(const float *target, const float *draft, const int32_t *tokens, const double *uniforms,
                         int B, int G, int V, double temperature, int32_t *n_accepted, int32_t *next_token) {
  unsigned status = 0;
  double *w = (double *)malloc((size_t)V * sizeof(double));
  for (int b = 0; b < B; ++b) {
    const float *tb = target + (size_t)b * (G + 1) * V;
    const float *db = draft ? draft + (size_t)b * G * V : NULL;
    const double *ub = uniforms ? uniforms + (size_t)b * (G + 1) : NULL;
    int n = 0;
    for (; n < G; ++n) {
      const int x = tokens[(size_t)b * G + n];
      if (x < 0 || x >= V) {
        status |= ORC_BAD_TOKEN;
        break;
      }
      const float *trow = tb + (size_t)n * V;
      if (temperature == 0.0) {
#if ORC_MUTANT == 18
        if (db != NULL && x != row_argmax(db + (size_t)n * V, V)) break; /* planted: the draft's argmax */
#else
        if (x != row_argmax(trow, V)) break;
#endif
        continue;
      }
      const float *drow = db + (size_t)n * V;
      const double logp = (double)trow[x] / temperature - row_lse(trow, V, temperature);
      const double logq = (double)drow[x] / temperature - row_lse(drow, V, temperature);
#if ORC_MUTANT == 16
      if (!(log(ub[n]) < logq - logp)) break; /* planted: the ratio inverted */
#else
      if (!(log(ub[n]) < logp - logq)) break;
#endif
    }
    n_accepted[b] = n;
    const float *trow = tb + (size_t)n * V;
    if (temperature == 0.0) {
      next_token[b] = row_argmax(trow, V);
      continue;
    }
    const double lt = row_lse(trow, V, temperature);
    double W = 0.0;
    if (n < G) {
      /* rejected at draft token n: the residual max(0, p - q) of that row */
      const float *drow = db + (size_t)n * V;
      const double ld = row_lse(drow, V, temperature);
      for (int k = 0; k < V; ++k) {
        const double p = exp((double)trow[k] / temperature - lt), q = exp((double)drow[k] / temperature - ld);
#if ORC_MUTANT == 17
        w[k] = fmax(0.0, q - p); /* planted: the residual of the draft */
#else
        w[k] = fmax(0.0, p - q);
#endif
        W += w[k];
      }
    }
    if (n == G || !(W > 0.0)) /* the bonus row, or a residual with no weight: p itself */
      for (int k = 0; k < V; ++k) w[k] = exp((double)trow[k] / temperature - lt);
    next_token[b] = draw(w, V, ub[G]);
  }
  free(w);
  return status;
}
