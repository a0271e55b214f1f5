// KV-cache append ("tinydecode", section "how the decode step is put together": the new key
// and value rows are written into the static cache at position seq_lens, which stays on the
// device). One CTA per sequence reads seq_lens[b] once, copies the sequence's T new rows of
// every kv head with 16-byte vector moves, then advances seq_lens[b] itself: no other CTA
// reads that length, so the advance cannot race with a read.
#include "td_device.cuh"
#include "td_internal.h"

namespace td {

namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const uint4 *k_new, const uint4 *v_new,
                                                                   uint4 *k_cache, uint4 *v_cache, int32_t *seq_lens,
                                                                   int Hkv, int T, int Smax, int vec_per_row,
                                                                   int advance, uint32_t *status) {
  __shared__ int s_start;
  const int b = blockIdx.x;
  griddep_wait();  // the cache and lengths may come from the previous kernel in the stream
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    const long long L = seq_lens[b];
    const bool fits = L >= 0 && L + T <= Smax;
    if (!fits) report(status, TD_DEV_APPEND_OVERFLOW);
    s_start = fits ? (int)L : -1;
  }
  __syncthreads();
  const int L = s_start;
  if (L < 0) return;
  const long long per_seq = (long long)Hkv * T * vec_per_row;
  for (long long idx = threadIdx.x; idx < per_seq; idx += kAppendThreads) {
    const long long row = idx / vec_per_row;  // (h, t) pair
    const int vec = (int)(idx % vec_per_row);
    const int h = (int)(row / T), t = (int)(row % T);
    const long long src = ((long long)b * Hkv * T + row) * vec_per_row + vec;
    const long long dst = (((long long)b * Hkv + h) * Smax + L + t) * vec_per_row + vec;
    k_cache[dst] = k_new[src];
    v_cache[dst] = v_new[src];
  }
  if (advance && threadIdx.x == 0) seq_lens[b] = L + T;
}

}  // namespace

cudaError_t launch_append(size_t elem_bytes, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                          uint32_t *dev_status, cudaStream_t stream) {
  const int vec_per_row = (int)((size_t)D * elem_bytes / 16);
  return launch_pdl(kv_append_kernel, dim3(B), dim3(kAppendThreads), 0, stream, static_cast<const uint4 *>(k_new),
                    static_cast<const uint4 *>(v_new), static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                    seq_lens, Hkv, T, Smax, vec_per_row, advance, dev_status);
}

}  // namespace td
