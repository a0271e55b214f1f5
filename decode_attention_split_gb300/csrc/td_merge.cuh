// Log-sum-exp merge of per-split partial softmax results ("tinydecode", section "how the
// decode step is put together": each split writes (m, l, acc) and a second step merges them;
// "llm-decode-cuda", split-KV attention section: chunks merged with the log-sum-exp trick).
//
// For one row with partials s < nc (only those with l_s > 0 count):
//   M = max_s m_s,  Lsum = sum_s l_s exp(m_s - M),
//   out = sum_s acc_s exp(m_s - M) / Lsum,  lse = M + ln Lsum.
// m is in natural-log units; acc is unnormalised (relative to exp(score - m_s)).
#pragma once

#include "td_device.cuh"

namespace td {

constexpr int kMergeBlock = 128;  // splits whose factors are staged in shared memory at a time

// Shared scratch (in floats) merge_rows<R> needs: factors, per-row stats and the row tables.
template <int R>
constexpr int merge_scratch_floats() {
  return R * kMergeBlock + 2 * R + 4 * R;  // + 2 x R long long row tables
}

// Merges up to R rows with the threads of one CTA (NT threads, a multiple of 32); each thread
// holds at most PAIRS (row, dim) sums, so the caller guarantees R * D <= PAIRS * NT.
//   rowbase[r]  (shared) offset of row r's first partial in m/l (in units of one split), or -1 to
//               skip the row; its acc rows start at rowbase[r] * D.
//   out_row[r]  (shared) output row index (out + out_row[r] * D, lse[out_row[r]]).
// Scratch: factors R * kMergeBlock floats, stats 2 * R floats.
// Partials are read with ld.global.cg: they may have been written by other CTAs of the
// same launch (made visible by a fence before their completion ticket).
template <int R, int NT, int PAIRS, typename OutE>
__device__ void merge_rows(const float *m, const float *l, const float *acc, const long long *rowbase,
                           const long long *out_row, int nc, int D, OutE *out, float *lse, float *factors,
                           float *stats) {
  constexpr int kWarpsM = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // phase 1: per-row maximum and normaliser
  for (int r = warp; r < R; r += kWarpsM) {
    float M = -INFINITY, Ls = 0.f;
    const long long base = rowbase[r];
    if (base >= 0) {
      for (int s = lane; s < nc; s += 32) {
        const float ls = __ldcg(l + base + s);
        if (ls > 0.f) M = fmaxf(M, __ldcg(m + base + s));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (M != -INFINITY) {
        for (int s = lane; s < nc; s += 32) {
          const float ls = __ldcg(l + base + s);
          if (ls > 0.f) Ls += ls * expf(__ldcg(m + base + s) - M);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      }
    }
    if (lane == 0) {
      stats[r] = M;
      stats[R + r] = Ls;
    }
  }
  __syncthreads();
  // phase 2: weighted sum of the unnormalised accumulators. Factors exp(m_s - M) / Lsum are
  // staged per block of splits; (row, dim) pairs are processed 8 per thread at a time.
  constexpr int kGroup = 8;
  constexpr int kGroups = (PAIRS + kGroup - 1) / kGroup;
  const int nblk = (nc + kMergeBlock - 1) / kMergeBlock;
  for (int pg = 0; pg < kGroups; ++pg) {
    float sum[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) sum[i] = 0.f;
    for (int sb = 0; sb < nc; sb += kMergeBlock) {
      const int nb = min(kMergeBlock, nc - sb);
      if (nblk > 1 || pg == 0) {
        for (int idx = tid; idx < R * kMergeBlock; idx += NT) {
          const int r = idx / kMergeBlock, s = idx % kMergeBlock;
          float f = 0.f;
          const long long base = rowbase[r];
          if (base >= 0 && s < nb && stats[r] != -INFINITY) {
            const float ls = __ldcg(l + base + sb + s);
            if (ls > 0.f) f = expf(__ldcg(m + base + sb + s) - stats[r]) / stats[R + r];
          }
          factors[idx] = f;
        }
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < kGroup; ++i) {
        const int idx = tid + (pg * kGroup + i) * NT;
        if (idx < R * D) {
          const int r = idx / D, d = idx % D;
          const long long base = rowbase[r];
          if (base >= 0) {
            const float *a = acc + (base + sb) * (long long)D + d;
            const float *f = factors + r * kMergeBlock;
            float x = sum[i];
#pragma unroll 4
            for (int s = 0; s < nb; ++s) x = fmaf(__ldcg(a + (long long)s * D), f[s], x);
            sum[i] = x;
          }
        }
      }
      if (nblk > 1) __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const int idx = tid + (pg * kGroup + i) * NT;
      if (idx < R * D) {
        const int r = idx / D, d = idx % D;
        if (rowbase[r] >= 0) {
          store_elem<OutE>(out + out_row[r] * D + d, sum[i]);
          if (d == 0 && lse != nullptr)
            lse[out_row[r]] = stats[r] == -INFINITY ? -INFINITY : stats[r] + logf(stats[R + r]);
        }
      }
    }
  }
}

}  // namespace td
