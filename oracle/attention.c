/*
 * Plain fp64 CPU oracle for split-KV decode attention over a static KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers. The CUDA library never loads, links or calls
 * this file, and the two share no code: this file is the definition the GPU kernels
 * are checked against, written as directly as the sources allow.
 *
 * Sources (web pages, cited by title and section):
 *   [tinydecode/decode]  "tinydecode", section "how the decode step is put together":
 *       the KV cache is static and preallocated; per-sequence lengths (seq_lens) live on
 *       the device; the new key/value row is written at position seq_lens (an index_put_);
 *       attention masks keys by j < seq_len; the decode kernel gives each block one chunk
 *       of the cache, computes scores -> softmax statistics -> p @ V for that chunk and
 *       writes (m, l, acc); a second kernel merges the chunks with log-sum-exp; a query
 *       head is mapped to its key/value head in the index math (grouped-query attention).
 *   [tinydecode/spec]    "tinydecode", section "speculative decoding": the verify pass is
 *       chunk attention over k+1 new tokens on top of the cache, causal among themselves;
 *       rollback is a rewrite of seq_lens, and entries past it are never read.
 *   [llm-decode-cuda/split]  "llm-decode-cuda", the split-KV ("flash-decoding") attention
 *       section: the context is split into chunks, one block per (kv head, chunk) serves
 *       every query head sharing that kv head and computes a partial softmax, and the chunks
 *       are merged with the log-sum-exp trick.
 *   [rope]  "tinydecode" lists an in-place rope kernel for its llama models (loaded from
 *       Hugging Face llama checkpoints); "llm-decode-cuda" fuses "RoPE + KV-cache write"
 *       into its decode step. Neither prints the rotation; the reading taken is the llama
 *       checkpoints' layout (pairs (i, i + D/2), "rotate half"), with the angles given as
 *       cos/sin tables indexed by position.
 *
 * Layouts (row-major, contiguous):
 *   q, out      [B, Hq, T, D]      (T = 1 for single-token decode)
 *   k, v cache  [B, Hkv, Smax, D]
 *   lse         [B, Hq, T]
 *   partials    m, l [B, Hq*T, NS];  acc [B, Hq*T, NS, D]   (row index = hq*T + t)
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - query head hq reads kv head hq / (Hq/Hkv): contiguous groups.
 *   - seq_lens[b] > Smax is clamped to Smax, a negative length counts as 0 (status bits).
 *   - row t of a T-token chunk sees keys j < L - T + t + 1, where L counts the T new tokens.
 *   - a row that sees no key has out = 0 and lse = -inf.
 *   - partial acc is stored unnormalised (the pages name the triple (m, l, acc)).
 *   - a rotated row is evaluated exactly and rounded once, to nearest even, to the stored
 *     type (the rotated key is what the cache holds; the rotated query is what attends).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_MUTANT
#define ORC_MUTANT 0 /* >0 only in the test that plants mistakes to show the pins catch them */
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2

#define ORC_SEQLEN_CLAMPED 1u
#define ORC_APPEND_OVERFLOW 2u
#define ORC_VERIFY_SHORT 4u
#define ORC_NEGATIVE_SEQLEN 8u

int orc_mutant(void) { return ORC_MUTANT; }

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads later parallel loops use (n >= 1); for timing the oracle single-threaded and on all
 * cores. No effect on the arithmetic: each row is computed by one thread in a fixed order. */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Element i of a stored array, widened exactly to fp64. A bf16 number is the upper half of
 * an IEEE binary32 number: widening places its 16 bits above 16 zero bits. */
static double widen(int dtype, const void *base, int64_t i) {
  if (dtype == ORC_F32) return (double)((const float *)base)[i];
  if (dtype == ORC_BF16) {
    uint16_t h = ((const uint16_t *)base)[i];
#if ORC_MUTANT == 13
    /* planted: reads the 16 bits as IEEE half precision */
    int e = (h >> 10) & 31, mnt = h & 1023;
    double mag = e ? ldexp(1.0 + mnt / 1024.0, e - 15) : ldexp(mnt / 1024.0, -14);
    return (h & 0x8000) ? -mag : mag;
#else
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
#endif
  }
  return ((const double *)base)[i];
}

/* Attended length of sequence b: seq_lens[b] clamped into [0, Smax]. */
static int64_t attended_length(const int32_t *seq_lens, int b, int Smax, unsigned *status) {
  int64_t L = seq_lens[b];
  if (L < 0) {
    if (status) *status |= ORC_NEGATIVE_SEQLEN;
    L = 0;
  }
  if (L > Smax) {
    if (status) *status |= ORC_SEQLEN_CLAMPED;
    L = Smax;
  }
  return L;
}

/* Keys visible to row t of a T-token query chunk when the cache holds L rows (the T new
 * tokens included): positions 0 .. L-T+t, i.e. n = L - T + t + 1 of them [tinydecode/spec].
 * For T = 1 this is the decode mask j < seq_len [tinydecode/decode]. */
static int64_t visible_keys(int64_t L, int T, int t, int Smax) {
  int64_t n = L - T + t + 1;
#if ORC_MUTANT == 3
  n -= 1; /* planted: drops the newest key */
#endif
#if ORC_MUTANT == 4
  if (T > 1) n += 1; /* planted: verify row sees one future token */
#endif
#if ORC_MUTANT == 12
  if (T == 1) n = L + 1; /* planted: decode reads one row past seq_len */
#endif
  if (n < 0) n = 0;
  if (n > Smax) n = Smax; /* only a planted mistake can reach past L */
  return n;
}

/* kv head that query head hq reads: heads are grouped contiguously, g = Hq / Hkv. */
static int kv_head_of(int hq, int Hq, int Hkv) {
#if ORC_MUTANT == 1
  (void)Hq;
  return hq % Hkv; /* planted: strided instead of contiguous groups */
#else
  return hq / (Hq / Hkv);
#endif
}

static int64_t cache_index(int b, int h, int64_t j, int d, int Hkv, int Smax, int D) {
#if ORC_MUTANT == 9
  /* planted: treats each head's block as [D][Smax] */
  return (((int64_t)b * Hkv + h) * Smax) * D + (int64_t)d * Smax + j;
#else
  return (((int64_t)b * Hkv + h) * Smax + j) * D + d;
#endif
}

static int v_head(int kvh, int Hkv) {
#if ORC_MUTANT == 6
  return (kvh + 1) % Hkv; /* planted: value rows from the neighbouring head */
#else
  (void)Hkv;
  return kvh;
#endif
}

/* s_j = scale * sum_d q[d] k[j][d] */
static double score(int dtype, const void *q, int64_t q_off, const void *k, int b, int kvh, int64_t j,
                    int Hkv, int Smax, int D, double scale) {
  double dot = 0.0;
  for (int d = 0; d < D; ++d)
    dot += widen(dtype, q, q_off + d) * widen(dtype, k, cache_index(b, kvh, j, d, Hkv, Smax, D));
#if ORC_MUTANT == 2
  (void)scale;
  return dot; /* planted: scale dropped */
#else
  return scale * dot;
#endif
}

/* Exact attention, the definition the split-KV kernel reaches faster:
 *   s_j = scale * q . k_j for j < n;  M = max_j s_j;  w_j = exp(s_j - M);
 *   out = sum_j w_j v_j / sum_j w_j;  lse = M + ln sum_j w_j.
 * Returns the status bits for data errors (clamped / negative lengths, short verify). */
unsigned orc_attention(int dtype, const void *q, const void *k, const void *v, const int32_t *seq_lens, int B,
                       int Hq, int Hkv, int T, int Smax, int D, double scale, double *out, double *lse) {
  unsigned status = 0;
  for (int b = 0; b < B; ++b) {
    int64_t L = attended_length(seq_lens, b, Smax, &status);
    if (T > 1 && L < T) status |= ORC_VERIFY_SHORT;
  }
  const int64_t rows = (int64_t)B * Hq * T;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    const int b = (int)(r / ((int64_t)Hq * T));
    const int hq = (int)((r / T) % Hq);
    const int t = (int)(r % T);
    const int kvh = kv_head_of(hq, Hq, Hkv);
    const int64_t L = attended_length(seq_lens, b, Smax, NULL);
    const int64_t n = visible_keys(L, T, t, Smax);
    double *o = out + r * D;
    if (n == 0) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (lse) lse[r] = -INFINITY;
      continue;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double M = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      s[j] = score(dtype, q, r * D, k, b, kvh, j, Hkv, Smax, D, scale);
      if (s[j] > M) M = s[j];
    }
    double Z = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const double w = exp(s[j] - M);
      Z += w;
      for (int d = 0; d < D; ++d) o[d] += w * widen(dtype, v, cache_index(b, v_head(kvh, Hkv), j, d, Hkv, Smax, D));
    }
    for (int d = 0; d < D; ++d) o[d] /= Z;
#if ORC_MUTANT == 5
    if (lse) lse[r] = log(Z); /* planted: max term forgotten */
#else
    if (lse) lse[r] = M + log(Z);
#endif
    free(s);
  }
  return status;
}

/* The split step [tinydecode/decode], [llm-decode-cuda/split]: for split s of size S the
 * row's keys j in [s*S, min((s+1)*S, n)) give
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  acc = sum_j exp(s_j - m) v_j   (unnormalised).
 * A split with no key gives m = -inf, l = 0, acc = 0. */
unsigned orc_split_partials(int dtype, const void *q, const void *k, const void *v, const int32_t *seq_lens, int B,
                            int Hq, int Hkv, int T, int Smax, int D, double scale, int S, int NS, double *m,
                            double *l, double *acc) {
  unsigned status = 0;
  for (int b = 0; b < B; ++b) {
    int64_t L = attended_length(seq_lens, b, Smax, &status);
    if (T > 1 && L < T) status |= ORC_VERIFY_SHORT;
  }
  const int64_t rows = (int64_t)B * Hq * T;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    const int b = (int)(r / ((int64_t)Hq * T));
    const int hq = (int)((r / T) % Hq);
    const int t = (int)(r % T);
    const int kvh = kv_head_of(hq, Hq, Hkv);
    const int64_t n = visible_keys(attended_length(seq_lens, b, Smax, NULL), T, t, Smax);
    for (int s = 0; s < NS; ++s) {
      const int64_t p = r * NS + s; /* [B, Hq*T, NS] flattened: r already counts b */
      double *a = acc + p * D;
      const int64_t lo = (int64_t)s * S;
      const int64_t hi = lo + S < n ? lo + S : n;
      for (int d = 0; d < D; ++d) a[d] = 0.0;
      if (lo >= hi) {
        m[p] = -INFINITY;
        l[p] = 0.0;
        continue;
      }
      double mx = -INFINITY;
      for (int64_t j = lo; j < hi; ++j) {
        const double sj = score(dtype, q, r * D, k, b, kvh, j, Hkv, Smax, D, scale);
        if (sj > mx) mx = sj;
      }
      double sum = 0.0;
      for (int64_t j = lo; j < hi; ++j) {
        const double w = exp(score(dtype, q, r * D, k, b, kvh, j, Hkv, Smax, D, scale) - mx);
        sum += w;
        for (int d = 0; d < D; ++d) a[d] += w * widen(dtype, v, cache_index(b, v_head(kvh, Hkv), j, d, Hkv, Smax, D));
      }
#if ORC_MUTANT == 8
      for (int d = 0; d < D; ++d) a[d] /= sum; /* planted: normalised partial */
#endif
      m[p] = mx;
      l[p] = sum;
    }
  }
  return status;
}

/* The merge step [tinydecode/decode], [llm-decode-cuda/split]: over the active splits
 * s < min(NS, ceil(L_b / split)) that saw a key (l_s > 0),
 *   M = max_s m_s;  Lsum = sum_s l_s exp(m_s - M);
 *   out = sum_s acc_s exp(m_s - M) / Lsum;  lse = M + ln Lsum.
 * A row with no such split gets out = 0, lse = -inf. */
void orc_lse_merge(const double *m, const double *l, const double *acc, const int32_t *seq_lens, int B, int rows,
                   int NS, int D, int split, double *out, double *lse) {
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b] < 0 ? 0 : seq_lens[b];
    int64_t active = (L + split - 1) / split;
    if (active > NS) active = NS;
    for (int r = 0; r < rows; ++r) {
      const int64_t base = ((int64_t)b * rows + r) * NS;
      double *o = out + ((int64_t)b * rows + r) * D;
      double M = -INFINITY;
      for (int64_t s = 0; s < active; ++s)
        if (l[base + s] > 0.0 && m[base + s] > M) M = m[base + s];
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (M == -INFINITY) {
        if (lse) lse[(int64_t)b * rows + r] = -INFINITY;
        continue;
      }
      double Lsum = 0.0;
      for (int64_t s = 0; s < active; ++s) {
        if (!(l[base + s] > 0.0)) continue;
        const double f = exp(m[base + s] - M);
        Lsum += l[base + s] * f;
        for (int d = 0; d < D; ++d) {
#if ORC_MUTANT == 7
          o[d] += acc[(base + s) * D + d]; /* planted: partial not rescaled */
#else
          o[d] += acc[(base + s) * D + d] * f;
#endif
        }
      }
      for (int d = 0; d < D; ++d) o[d] /= Lsum;
      if (lse) lse[(int64_t)b * rows + r] = M + log(Lsum);
    }
  }
}

/* The cache write [tinydecode/decode]: new rows [B, Hkv, T, D] are copied bit for bit to
 * rows L_b .. L_b+T-1 of the cache, L_b = seq_lens[b]; with advance, seq_lens[b] += T.
 * A sequence whose rows would not fit (L_b < 0 or L_b + T > Smax) is left untouched and
 * flagged. elem_bytes is the stored element size (the copy never looks at the values). */
unsigned orc_kv_append(int elem_bytes, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance) {
  unsigned status = 0;
  const size_t row = (size_t)D * (size_t)elem_bytes;
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    if (L < 0 || L + T > Smax) {
      status |= ORC_APPEND_OVERFLOW;
      continue;
    }
#if ORC_MUTANT == 10
    if (L + T < Smax) L += 1; /* planted: writes one row late */
#endif
    for (int h = 0; h < Hkv; ++h)
      for (int t = 0; t < T; ++t) {
        const size_t src = (((size_t)b * Hkv + h) * T + t) * row;
        const size_t dst = (((size_t)b * Hkv + h) * Smax + (size_t)(L + t)) * row;
        memcpy((char *)k_cache + dst, (const char *)k_new + src, row);
        memcpy((char *)v_cache + dst, (const char *)v_new + src, row);
      }
#if ORC_MUTANT != 11 /* planted (11): advance forgotten */
    if (advance) seq_lens[b] += T;
#endif
  }
  return status;
}

/* An exact value rounded to the stored element type, to nearest with ties to even. fp32 by
 * the C conversion (the default rounding mode); bf16 directly from the fp64 value: 8
 * significant bits in the binary32 exponent range (multiples of 2^-133 below 2^-126). */
static void narrow(int dtype, void *base, int64_t i, double x) {
  if (dtype == ORC_F32) {
    ((float *)base)[i] = (float)x;
    return;
  }
  if (dtype == ORC_F64) {
    ((double *)base)[i] = x;
    return;
  }
  uint16_t h;
  const uint16_t sign = signbit(x) ? 0x8000u : 0u;
  const double a = fabs(x);
  if (isnan(x)) {
    h = 0x7FC0u;
  } else if (a == 0.0) {
    h = sign;
  } else {
    double y;
    if (a < ldexp(1.0, -126)) {
      y = ldexp(nearbyint(ldexp(a, 133)), -133);
    } else {
      int e;
      const double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
      y = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    if (y >= ldexp(1.0, 128)) {
      h = (uint16_t)(sign | 0x7F80u); /* infinity */
    } else {
      const float f = (float)y; /* exact: at most 8 significant bits */
      uint32_t u;
      memcpy(&u, &f, sizeof u);
      h = (uint16_t)(sign | (u >> 16));
    }
  }
  ((uint16_t *)base)[i] = h;
}

/* Rotary position embedding [rope] of `rows` rows of D elements, row r at position pos[r]:
 * for i < D/2 the pair (x[i], x[i + D/2]) turns by the angle whose cosine and sine are
 * cos_t[pos][i] and sin_t[pos][i] (fp32 tables [positions][D/2]):
 *   y[i]       = x[i] cos - x[i + D/2] sin
 *   y[i + D/2] = x[i + D/2] cos + x[i] sin
 * evaluated in fp64 from the stored inputs and rounded once to the stored type. */
void orc_rope(int dtype, const void *x, int64_t rows, int D, const int32_t *pos, const float *cos_t,
              const float *sin_t, void *y) {
  const int half = D / 2;
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t p = pos[r];
    for (int i = 0; i < half; ++i) {
#if ORC_MUTANT == 15
      /* planted: neighbouring elements (2i, 2i + 1) taken as the pair */
      const int64_t a = r * D + 2 * i, b = r * D + 2 * i + 1;
#else
      const int64_t a = r * D + i, b = r * D + i + half;
#endif
      const double c = (double)cos_t[p * half + i], s = (double)sin_t[p * half + i];
      const double x0 = widen(dtype, x, a), x1 = widen(dtype, x, b);
#if ORC_MUTANT == 14
      /* planted: turns the other way */
      narrow(dtype, y, a, x0 * c + x1 * s);
      narrow(dtype, y, b, x1 * c - x0 * s);
#else
      narrow(dtype, y, a, x0 * c - x1 * s);
      narrow(dtype, y, b, x1 * c + x0 * s);
#endif
    }
  }
}

/* Symmetric 8-bit quantisation of cache rows, one scale per row (the quantised KV cache:
 * "llm-decode-cuda" quantises its weights to INT8, one scale per row, dequantised in
 * registers after the load; the same scheme is read here for the K and V rows, which bound
 * the decode step). For each row of D elements, in fp32 (the precision the kernels decide
 * the codes in, so both sides reach the same integers):
 *   amax  = max_i |x_i|
 *   scale = amax / 127                      (IEEE division, rounded to nearest)
 *   code  = clamp(rint(x_i / scale), -127, 127), 0 when scale == 0
 * and the row reads back as code_i * scale. */
void orc_quantize_q8(int dtype, const void *x, int64_t rows, int D, int8_t *codes, float *scales) {
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int i = 0; i < D; ++i) {
      const float v = (float)widen(dtype, x, r * D + i);
      const float a = v < 0.0f ? -v : v;
      if (a > amax) amax = a;
    }
#if ORC_MUTANT == 19
    const float scale = amax / 128.0f; /* planted: the wrong full-scale code */
#else
    const float scale = amax / 127.0f;
#endif
    scales[r] = scale;
    for (int i = 0; i < D; ++i) {
      float c = 0.0f;
      if (scale > 0.0f) {
        const float q = (float)widen(dtype, x, r * D + i) / scale;
#if ORC_MUTANT == 20
        c = truncf(q); /* planted: truncation instead of rounding */
#else
        c = nearbyintf(q);
#endif
        if (c > 127.0f) c = 127.0f;
        if (c < -127.0f) c = -127.0f;
      }
      codes[r * D + i] = (int8_t)c;
    }
  }
}
