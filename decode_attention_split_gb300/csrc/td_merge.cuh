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

// Merges up to R rows with the threads of one CTA (nthreads, a multiple of 32).
//   rowbase[r]  offset of row r's first partial in m/l (in units of one split), or -1 to skip;
//               its acc rows start at rowbase[r] * D.
//   out_row[r]  output row index (out + out_row[r] * D, lse[out_row[r]]).
// Shared scratch: factors R * kMergeBlock floats, stats 2 * R floats.
// Partials are read with ld.global.cg: they may have been written by other CTAs of the
// same launch (made visible by a fence before their completion ticket).
template <int R, typename OutE>
__device__ void merge_rows(const float *m, const float *l, const float *acc, const long long (&rowbase)[R],
                           const long long (&out_row)[R], int nc, int D, OutE *out, float *lse, float *factors,
                           float *stats) {
  const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
  // phase 1: per-row maximum and normaliser
  for (int r = warp; r < R; r += nwarps) {
    float M = -INFINITY, Ls = 0.f;
    if (rowbase[r] >= 0) {
      for (int s = lane; s < nc; s += 32) {
        const float ls = __ldcg(l + rowbase[r] + s);
        if (ls > 0.f) M = fmaxf(M, __ldcg(m + rowbase[r] + s));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (M != -INFINITY) {
        for (int s = lane; s < nc; s += 32) {
          const float ls = __ldcg(l + rowbase[r] + s);
          if (ls > 0.f) Ls += ls * expf(__ldcg(m + rowbase[r] + s) - M);
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
  // phase 2: weighted sum of the unnormalised accumulators, factors staged per block of splits
  constexpr int kMaxPairs = 8;  // (row, dim) pairs a thread owns; R * D <= kMaxPairs * nthreads
  float sum[kMaxPairs];
#pragma unroll
  for (int i = 0; i < kMaxPairs; ++i) sum[i] = 0.f;
  for (int sb = 0; sb < nc; sb += kMergeBlock) {
    const int nb = min(kMergeBlock, nc - sb);
    for (int idx = tid; idx < R * kMergeBlock; idx += nthreads) {
      const int r = idx / kMergeBlock, s = idx % kMergeBlock;
      float f = 0.f;
      if (rowbase[r] >= 0 && s < nb && stats[r] != -INFINITY) {
        const float ls = __ldcg(l + rowbase[r] + sb + s);
        if (ls > 0.f) f = expf(__ldcg(m + rowbase[r] + sb + s) - stats[r]) / stats[R + r];
      }
      factors[idx] = f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxPairs; ++i) {
      const int idx = tid + i * nthreads;
      if (idx < R * D) {
        const int r = idx / D, d = idx % D;
        if (rowbase[r] >= 0) {
          const float *a = acc + (rowbase[r] + sb) * (long long)D + d;
          const float *f = factors + r * kMergeBlock;
          float x = sum[i];
          for (int s = 0; s < nb; ++s) {
            if (f[s] != 0.f) x = fmaf(__ldcg(a + (long long)s * D), f[s], x);
          }
          sum[i] = x;
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kMaxPairs; ++i) {
    const int idx = tid + i * nthreads;
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

}  // namespace td
