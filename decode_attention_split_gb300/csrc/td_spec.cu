// Speculative accept/reject on the device: the step after a verify pass.
//
// Method ("tinydecode", section "speculative decoding"; "FlashSpec", sections "What is
// FlashSpec?" and "How it works", after Leviathan et al. 2023, Algorithm 1): draft token i
// is kept while u_i < min(1, p_i(x_i) / q_i(x_i)), tested in log space; at the first
// rejection the extra token is drawn from the residual max(0, p - q) / ||max(0, p - q)||_1
// of that row, and when every draft token is kept it is drawn from the target's bonus row.
// At temperature 0: keep while the draft token is the target's argmax; the extra token is
// the target's argmax after the kept prefix. p = softmax(target logits / T),
// q = softmax(draft logits / T).
//
// GB300 design. Reading the logits is the whole cost (every target and draft row once), and
// one SM streams only a small share of HBM bandwidth, so each sequence's vocabulary is cut
// into 1024-entry slices, one CTA each, across the whole GPU; two launches, chained by
// programmatic dependent launch, meet through a small workspace with completion tickets (no
// CTA ever waits for another):
//  A. rows_kernel: each CTA reduces its slice of every row (a warp per row, eight 16-byte
//     loads in flight per lane): running (max, sum of exp) in base 2, or (argmax, lowest
//     index) at temperature 0. The CTA that completes a sequence merges the slices' partials
//     in slice order, takes the decisions and, when sampling, records the chosen row and its
//     normalisers for B.
//  B. draw_kernel (sampling only): each CTA sums the weights of its slice of the chosen row
//     (residual and plain p); the CTA that completes a sequence finds, in slice order, the
//     slice whose share of the running total holds u * total, and walks that slice.
// Every weight is recomputed from the logits with the same expression wherever it is used.
#include <math.h>

#include "td_device.cuh"
#include "td_internal.h"

namespace td {

namespace {

constexpr int kSpecThreads = 256;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kSlice = 1024;  // vocabulary entries per CTA
constexpr int kRowsMax = 2 * kMaxDraft + 1;

struct SpecParams {
  const float *target;    // [B, G+1, V]
  const float *draft;     // [B, G, V] (null when greedy)
  const int32_t *tokens;  // [B, G]
  const float *uniforms;  // [B, G+1] (null when greedy)
  int B, G, V, P;         // P slices per sequence
  float t2;               // log2(e) / temperature (0: greedy)
  int32_t *n_out, *tok_out;
  uint32_t *status;
  // workspace
  int *tick;              // [B][2] completion tickets (zero between calls)
  float2 *part;           // [B][rows][P] per-slice row partials
  float2 *sums;           // [B][P] per-slice (residual, p) weights of the chosen row
  float4 *info;           // [B]: (chosen row, its target and draft normalisers, -)
};

// Combines two (max, sum 2^(x - max)) pairs.
__device__ __forceinline__ void lse2_merge(float &m, float &s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * exp2f(m - M) + s2 * exp2f(m2 - M);
  m = M;
}

// Adds four values (base-2 units; -inf for none) to a running (max, sum 2^(x - max)).
__device__ __forceinline__ void lse2_add4(float &m, float &s, float a, float b, float c, float d) {
  const float mb = fmaxf(fmaxf(a, b), fmaxf(c, d));
  if (mb == -INFINITY) return;
  if (mb > m) {
    s *= exp2f(m - mb);
    m = mb;
  }
  s += exp2f(a - m) + exp2f(b - m) + exp2f(c - m) + exp2f(d - m);
}

// Keeps the larger value, the lower index on ties.
__device__ __forceinline__ void arg_merge(float &v, int &i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ const float *row_ptr(const SpecParams &p, int b, int r) {
  return r <= p.G ? p.target + ((size_t)b * (p.G + 1) + r) * p.V
                  : p.draft + ((size_t)b * p.G + (r - p.G - 1)) * p.V;
}

// A warp's reduction of entries [v0, v1) of one row: (max, sum) in base 2, or (argmax value,
// index) when greedy. 16-byte loads when rows are 16-byte aligned.
__device__ void warp_row(const SpecParams &p, const float *row, int v0, int v1, bool greedy, float &m, float &s,
                         int &bi) {
  const int lane = threadIdx.x & 31;
  m = -INFINITY;
  s = 0.f;
  bi = p.V;
  if ((p.V & 3) == 0) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int e0 = v0 / 4, e1 = v1 / 4;  // v0 and v1 are multiples of 4 here
    float4 x[kSlice / 128];
#pragma unroll
    for (int j = 0; j < kSlice / 128; ++j) {
      const int e = e0 + lane + 32 * j;
      x[j] = e < e1 ? r4[e] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int j = 0; j < kSlice / 128; ++j) {
      const int k = 4 * (e0 + lane + 32 * j);
      if (greedy) {
        arg_merge(m, bi, x[j].x, k);
        arg_merge(m, bi, x[j].y, k + 1);
        arg_merge(m, bi, x[j].z, k + 2);
        arg_merge(m, bi, x[j].w, k + 3);
      } else {
        lse2_add4(m, s, x[j].x * p.t2, x[j].y * p.t2, x[j].z * p.t2, x[j].w * p.t2);
      }
    }
  } else {
    for (int base = v0 + lane; base < v1; base += 32 * 8) {
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = base + 32 * j;
        x[j] = k < v1 ? row[k] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (greedy) arg_merge(m, bi, x[j], base + 32 * j);
        else lse2_add4(m, s, x[j] * p.t2, -INFINITY, -INFINITY, -INFINITY);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (greedy) arg_merge(m, bi, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, bi, o));
    else lse2_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  }
}

__global__ void __launch_bounds__(kSpecThreads) rows_kernel(const SpecParams p) {
  __shared__ float s_lse[kRowsMax];  // whole rows: base-2 log-sum-exp (argmax value when greedy)
  __shared__ int s_arg[kRowsMax];
  __shared__ float s_lt[kMaxDraft], s_ld[kMaxDraft];
  __shared__ int s_tok[kMaxDraft];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / p.P, c = blockIdx.x % p.P;
  const int G = p.G, V = p.V;
  const bool greedy = p.t2 == 0.f;
  const int rows = greedy ? G + 1 : 2 * G + 1;
  const int v0 = c * kSlice, v1 = min(v0 + kSlice, V);
  griddep_wait();
  griddep_launch_dependents();
  for (int r = warp; r < rows; r += kSpecWarps) {
    float m, s;
    int bi;
    warp_row(p, row_ptr(p, b, r), v0, v1, greedy, m, s, bi);
    if (lane == 0) p.part[((size_t)b * rows + r) * p.P + c] = make_float2(m, greedy ? __int_as_float(bi) : s);
  }
  __syncthreads();  // every partial of this CTA is written before its ticket
  if (tid == 0) s_last = ticket_acq_rel(&p.tick[2 * b]) == p.P - 1;
  __syncthreads();
  if (!s_last) return;

  // the CTA that completes sequence b: whole rows, in slice order (a warp per row)
  for (int r = warp; r < rows; r += kSpecWarps) {
    float m = -INFINITY, s = 0.f;
    int bi = V;
    for (int q = lane; q < p.P; q += 32) {
      const float2 v = p.part[((size_t)b * rows + r) * p.P + q];
      if (greedy) arg_merge(m, bi, v.x, __float_as_int(v.y));
      else lse2_merge(m, s, v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      if (greedy) arg_merge(m, bi, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, bi, o));
      else lse2_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    }
    if (lane == 0) {
      s_lse[r] = greedy ? m : (s > 0.f ? m + log2f(s) : -INFINITY);
      s_arg[r] = bi;
    }
  }
  if (tid < G) {  // the draft tokens and their own logits
    const int x = p.tokens[(size_t)b * G + tid];
    s_tok[tid] = x;
    if (!greedy && x >= 0 && x < V) {
      s_lt[tid] = row_ptr(p, b, tid)[x] * p.t2;
      s_ld[tid] = row_ptr(p, b, G + 1 + tid)[x] * p.t2;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0;
    uint32_t bits = 0;
    for (; n < G; ++n) {
      const int x = s_tok[n];
      if (x < 0 || x >= V) {
        bits |= TD_DEV_BAD_TOKEN;
        break;
      }
      if (greedy) {
        if (x != s_arg[n]) break;
      } else {
        const float lp = s_lt[n] - s_lse[n], lq = s_ld[n] - s_lse[G + 1 + n];  // log2 p(x), log2 q(x)
        if (!(log2f(p.uniforms[(size_t)b * (G + 1) + n]) < lp - lq)) break;
      }
    }
    p.n_out[b] = n;
    if (bits) report(p.status, bits);
    if (greedy) p.tok_out[b] = s_arg[n];
    else p.info[b] = make_float4(__int_as_float(n), s_lse[n], n < G ? s_lse[G + 1 + n] : 0.f, 0.f);
    p.tick[2 * b] = 0;  // every CTA of this sequence has taken its ticket
  }
}

// Weights of entries [k, k + 4) of the chosen row (the residual, or p when `use_p` or on the
// bonus row).
__device__ __forceinline__ void weights4(const SpecParams &p, const float *trow, const float *drow, float lt,
                                         float ld, bool use_p, int k, int v1, float *w) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float x = 0.f;
    if (k + j < v1) {
      const float pk = exp2f(trow[k + j] * p.t2 - lt);
      x = (drow != nullptr && !use_p) ? fmaxf(0.f, pk - exp2f(drow[k + j] * p.t2 - ld)) : pk;
    }
    w[j] = x;
  }
}

// Block-wide inclusive scan of one value per thread in thread order; returns this thread's
// inclusive sum and the block total in *total (s_w holds kSpecWarps floats).
__device__ float block_scan(float v, float *s_w, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  float before = 0.f, all = 0.f;
  for (int w = 0; w < kSpecWarps; ++w) {
    if (w < warp) before += s_w[w];
    all += s_w[w];
  }
  *total = all;
  __syncthreads();  // s_w may be reused
  return before + x;
}

__global__ void __launch_bounds__(kSpecThreads) draw_kernel(const SpecParams p) {
  __shared__ float s_w[kSpecWarps];
  __shared__ int s_last, s_pick, s_hit;
  __shared__ float s_before;
  const int tid = threadIdx.x;
  const int b = blockIdx.x / p.P, c = blockIdx.x % p.P;
  const int G = p.G, V = p.V;
  griddep_wait();  // the chosen row comes from rows_kernel
  griddep_launch_dependents();
  const float4 info = p.info[b];
  const int n = __float_as_int(info.x);
  const float lt = info.y, ld = info.z;
  const float *trow = row_ptr(p, b, n);
  const float *drow = n < G ? row_ptr(p, b, G + 1 + n) : nullptr;
  // this CTA's slice, four entries per thread in thread order
  const int v0 = c * kSlice, v1 = min(v0 + kSlice, V);
  const int k = v0 + 4 * tid;
  float wr[4], wp[4];
  weights4(p, trow, drow, lt, ld, false, k, v1, wr);
  weights4(p, trow, drow, lt, ld, true, k, v1, wp);
  float tr, tp;
  block_scan(wr[0] + wr[1] + wr[2] + wr[3], s_w, &tr);
  block_scan(wp[0] + wp[1] + wp[2] + wp[3], s_w, &tp);
  if (tid == 0) {
    p.sums[(size_t)b * p.P + c] = make_float2(tr, tp);
    s_last = ticket_acq_rel(&p.tick[2 * b + 1]) == p.P - 1;
  }
  __syncthreads();
  if (!s_last) return;

  // the CTA that completes sequence b: the slice holding u * total, in slice order. Totals
  // first (a thread per slice, 256 slices at a time), then a scan over the slices finds the
  // one whose share of the running total holds the target.
  float totr = 0.f, totp = 0.f;
  for (int q0 = 0; q0 < p.P; q0 += kSpecThreads) {
    const int q = q0 + tid;
    const float2 v = q < p.P ? p.sums[(size_t)b * p.P + q] : make_float2(0.f, 0.f);
    float cr, cp;
    block_scan(v.x, s_w, &cr);
    block_scan(v.y, s_w, &cp);
    totr += cr;
    totp += cp;
  }
  const bool use_p = !(totr > 0.f);  // a residual with no weight (p = q up to rounding) falls back to p
  const float target = p.uniforms[(size_t)b * (G + 1) + G] * (use_p ? totp : totr);
  if (tid == 0) {
    s_pick = -1;
    s_hit = -1;
    s_last = -1;  // reused: the last slice with weight
  }
  __syncthreads();
  float carry = 0.f;
  for (int q0 = 0; q0 < p.P; q0 += kSpecThreads) {
    const int q = q0 + tid;
    const float2 v = q < p.P ? p.sums[(size_t)b * p.P + q] : make_float2(0.f, 0.f);
    const float wq = use_p ? v.y : v.x;
    float chunk;
    const float incl = carry + block_scan(wq, s_w, &chunk);
    if (q < p.P && incl - wq <= target && incl > target) {  // at most one slice
      s_pick = q;
      s_before = incl - wq;
    }
    if (q < p.P && wq > 0.f) atomicMax(&s_last, q);
    __syncthreads();
    if (s_pick >= 0) break;  // the same in every thread
    carry += chunk;
  }
  if (s_pick < 0) {  // rounding pushed the target past the end: the last slice with weight
    const int last = max(s_last, 0);
    float before = 0.f;
    for (int q0 = 0; q0 < last; q0 += kSpecThreads) {
      const int q = q0 + tid;
      const float2 v = q < last ? p.sums[(size_t)b * p.P + q] : make_float2(0.f, 0.f);
      float chunk;
      block_scan(use_p ? v.y : v.x, s_w, &chunk);
      before += chunk;
    }
    if (tid == 0) {
      s_pick = last;
      s_before = before;
    }
    __syncthreads();
  }
  if (tid == 0) p.tick[2 * b + 1] = 0;  // every CTA of this sequence has taken its ticket
  // walk the picked slice: the thread whose four entries hold the target
  const int pv0 = s_pick * kSlice, pv1 = min(pv0 + kSlice, V);
  const int pk = pv0 + 4 * tid;
  float w[4];
  weights4(p, trow, drow, lt, ld, use_p, pk, pv1, w);
  const float mine = w[0] + w[1] + w[2] + w[3];
  float tot;
  const float incl = s_before + block_scan(mine, s_w, &tot);
  float acc = incl - mine;
  if (acc <= target && incl > target) {
    for (int j = 0; j < 4; ++j) {
      if (acc + w[j] > target) {
        s_hit = pk + j;
        break;
      }
      acc += w[j];
    }
  }
  __syncthreads();
  if (s_hit < 0) {  // no entry holds it (rounding): the slice's last entry with weight
    int lastk = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (w[j] > 0.f) lastk = pk + j;
    if (lastk >= 0) atomicMax(&s_hit, lastk);
    __syncthreads();
  }
  if (tid == 0) p.tok_out[b] = s_hit >= 0 ? s_hit : pv0;
}

}  // namespace

int spec_slices(int V) { return (V + kSlice - 1) / kSlice; }

size_t spec_workspace_bytes(int B, int G, int V) {
  const size_t P = (size_t)spec_slices(V);
  const auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return a256((size_t)B * 2 * sizeof(int)) + a256((size_t)B * sizeof(float4)) +
         a256((size_t)B * (2 * G + 1) * P * sizeof(float2)) + a256((size_t)B * P * sizeof(float2));
}

cudaError_t launch_spec_accept(const float *target, const float *draft, const int32_t *tokens, const float *uniforms,
                               int B, int G, int V, float temperature, int32_t *n_out, int32_t *tok_out,
                               uint32_t *status, void *workspace, cudaStream_t stream) {
  SpecParams p;
  p.target = target;
  p.draft = draft;
  p.tokens = tokens;
  p.uniforms = uniforms;
  p.B = B;
  p.G = G;
  p.V = V;
  p.P = spec_slices(V);
  p.t2 = temperature > 0.f ? 1.4426950408889634f / temperature : 0.f;
  p.n_out = n_out;
  p.tok_out = tok_out;
  p.status = status;
  const auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  p.tick = reinterpret_cast<int *>(ws);
  ws += a256((size_t)B * 2 * sizeof(int));
  p.info = reinterpret_cast<float4 *>(ws);
  ws += a256((size_t)B * sizeof(float4));
  p.part = reinterpret_cast<float2 *>(ws);
  ws += a256((size_t)B * (2 * G + 1) * p.P * sizeof(float2));
  p.sums = reinterpret_cast<float2 *>(ws);
  const dim3 grid((unsigned)(B * p.P));
  cudaError_t e = launch_pdl(rows_kernel, grid, dim3(kSpecThreads), 0, stream, p);
  if (e == cudaSuccess && temperature > 0.f) e = launch_pdl(draw_kernel, grid, dim3(kSpecThreads), 0, stream, p);
  return e;
}

}  // namespace td
