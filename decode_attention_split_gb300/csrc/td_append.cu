// KV-cache append ("tinydecode", section "how the decode step is put together": the new key
// and value rows are written into the static cache at position seq_lens, which stays on the
// device). One CTA per sequence reads seq_lens[b] once, copies the sequence's T new rows of
// every kv head with 16-byte vector moves, then advances seq_lens[b] itself: no other CTA
// reads that length, so the advance cannot race with a read.
#include "td_device.cuh"
#include "td_internal.h"
#include "td_rope.cuh"

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

// The same write with the new keys (and, when q is given, the T query rows of every query
// head) rotated to their positions L + t first (td_rope.cuh). Rotated rows are worked on as
// pairs of 16-byte vectors (i, i + D/2); value rows are copied. One CTA per sequence.
template <typename E>
__global__ void __launch_bounds__(kAppendThreads)
    rope_append_kernel(const uint4 *q, uint4 *q_out, int Hq, const uint4 *k_new, const uint4 *v_new, const float *cos_t,
                       const float *sin_t, uint4 *k_cache, uint4 *v_cache, int32_t *seq_lens, int Hkv, int T,
                       int Smax, int D, int advance, uint32_t *status) {
  constexpr int VE = 16 / sizeof(E);
  __shared__ int s_start;
  const int b = blockIdx.x;
  const int NV = D / VE;  // 16-byte vectors per row
  const int NH = NV / 2;  // rotated vector pairs per row
  const int half = D / 2;
  griddep_wait();
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
  // keys: rotate and write
  const long long k_items = (long long)Hkv * T * NH;
  for (long long idx = threadIdx.x; idx < k_items; idx += kAppendThreads) {
    const long long row = idx / NH;  // (h, t)
    const int v = (int)(idx % NH);
    const int h = (int)(row / T), t = (int)(row % T);
    const long long src = ((long long)b * Hkv * T + row) * NV;
    const long long dst = (((long long)b * Hkv + h) * Smax + L + t) * NV;
    uint4 lo = k_new[src + v], hi = k_new[src + v + NH];
    const long long tab = (long long)(L + t) * half + v * VE;
    rope_vec16<E>(lo, hi, cos_t + tab, sin_t + tab);
    k_cache[dst + v] = lo;
    k_cache[dst + v + NH] = hi;
  }
  // values: copy
  const long long v_items = (long long)Hkv * T * NV;
  for (long long idx = threadIdx.x; idx < v_items; idx += kAppendThreads) {
    const long long row = idx / NV;
    const int v = (int)(idx % NV);
    const int h = (int)(row / T), t = (int)(row % T);
    v_cache[(((long long)b * Hkv + h) * Smax + L + t) * NV + v] = v_new[((long long)b * Hkv * T + row) * NV + v];
  }
  // queries: rotate into q_out (which may be q itself: each thread reads both vectors of a
  // pair before writing them)
  if (q != nullptr) {
    const long long q_items = (long long)Hq * T * NH;
    for (long long idx = threadIdx.x; idx < q_items; idx += kAppendThreads) {
      const long long row = idx / NH;  // (hq, t)
      const int v = (int)(idx % NH);
      const int t = (int)(row % T);
      const long long off = ((long long)b * Hq * T + row) * NV;
      uint4 lo = q[off + v], hi = q[off + v + NH];
      const long long tab = (long long)(L + t) * half + v * VE;
      rope_vec16<E>(lo, hi, cos_t + tab, sin_t + tab);
      q_out[off + v] = lo;
      q_out[off + v + NH] = hi;
    }
  }
  if (advance && threadIdx.x == 0) seq_lens[b] = L + T;  // L was read once, into shared memory
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

cudaError_t launch_rope_append(size_t elem_bytes, const void *q, void *q_out, int Hq, const void *k_new,
                               const void *v_new, const float *cos_t, const float *sin_t, void *k_cache,
                               void *v_cache, int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                               uint32_t *dev_status, cudaStream_t stream) {
  const auto *qv = static_cast<const uint4 *>(q);
  auto *qo = static_cast<uint4 *>(q_out);
  const auto *kn = static_cast<const uint4 *>(k_new);
  const auto *vn = static_cast<const uint4 *>(v_new);
  auto *kc = static_cast<uint4 *>(k_cache);
  auto *vc = static_cast<uint4 *>(v_cache);
  if (elem_bytes == 2)
    return launch_pdl(rope_append_kernel<__nv_bfloat16>, dim3(B), dim3(kAppendThreads), 0, stream, qv, qo, Hq, kn,
                      vn, cos_t, sin_t, kc, vc, seq_lens, Hkv, T, Smax, D, advance, dev_status);
  return launch_pdl(rope_append_kernel<float>, dim3(B), dim3(kAppendThreads), 0, stream, qv, qo, Hq, kn, vn, cos_t,
                    sin_t, kc, vc, seq_lens, Hkv, T, Smax, D, advance, dev_status);
}

}  // namespace td
