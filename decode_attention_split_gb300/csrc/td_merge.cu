// Stand-alone log-sum-exp merge of per-split partials (the same device routine the fused
// split-attention kernel runs in the CTA that completes a sequence's last chunk).
#include "td_internal.h"
#include "td_merge.cuh"

namespace td {

namespace {

constexpr int kMergeThreads = 128;

template <int R, typename OutE>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const float *m, const float *l, const float *acc,
                                                                   const int32_t *seq_lens, int rows, int NS, int D,
                                                                   int split, OutE *out, float *lse) {
  __shared__ float factors[R * kMergeBlock];
  __shared__ float stats[2 * R];
  __shared__ long long rowbase[R], out_row[R];
  const int b = blockIdx.y;
  griddep_wait();  // partials may come from the previous kernel in the stream
  griddep_launch_dependents();
  const long long L = seq_lens[b] < 0 ? 0 : seq_lens[b];
  long long nc = (L + split - 1) / split;
  if (nc > NS) nc = NS;
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    const int row = blockIdx.x * R + r;
    out_row[r] = (long long)b * rows + row;
    rowbase[r] = row < rows ? out_row[r] * NS : -1;
  }
  __syncthreads();
  // at most 8 (row, dim) pairs per thread: R * D <= 8 * kMergeThreads (D <= 256 for R = 4, 1024 for R = 1)
  merge_rows<R, kMergeThreads, 8, OutE>(m, l, acc, rowbase, out_row, (int)nc, D, out, lse, factors, stats);
}

template <int R>
void launch_r(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows, int NS,
              int D, int split, td_dtype out_dtype, void *out, float *lse, cudaStream_t stream) {
  const dim3 grid((rows + R - 1) / R, B);
  if (out_dtype == TD_F32)
    launch_pdl(lse_merge_kernel<R, float>, grid, dim3(kMergeThreads), 0, stream, m, l, acc, seq_lens, rows, NS, D,
               split, static_cast<float *>(out), lse);
  else
    launch_pdl(lse_merge_kernel<R, __nv_bfloat16>, grid, dim3(kMergeThreads), 0, stream, m, l, acc, seq_lens, rows,
               NS, D, split, static_cast<__nv_bfloat16 *>(out), lse);
}

}  // namespace

cudaError_t launch_merge(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows,
                         int NS, int D, int split, td_dtype out_dtype, void *out, float *lse, cudaStream_t stream) {
  // merge_rows gives each thread at most 8 (row, dim) pairs: R * D <= 8 * kMergeThreads
  if (D <= 256)
    launch_r<4>(m, l, acc, seq_lens, B, rows, NS, D, split, out_dtype, out, lse, stream);
  else
    launch_r<1>(m, l, acc, seq_lens, B, rows, NS, D, split, out_dtype, out, lse, stream);
  return cudaGetLastError();
}

}  // namespace td
