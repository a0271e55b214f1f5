// Per-row int8 quantisation of cache rows, and the cache append that quantises its new rows.
//
// The scheme ("llm-decode-cuda" quantises its weights to INT8 with one scale per row,
// dequantised in registers after the load; here the same is read for the K and V rows):
// for a row x of D elements, in fp32 with IEEE division,
//   scale = max_i |x_i| / 127,   code_i = clamp(rint(x_i / scale), -127, 127)  (0 if scale == 0),
// read back as code_i * scale. One warp per row.
#include <math.h>

#include "td_device.cuh"
#include "td_internal.h"

namespace td {

namespace {

constexpr int kQuantThreads = 256;

// Quantises one row of D elements (warp-wide; the row's lanes stride by 32).
template <typename E>
__device__ __forceinline__ void quantize_row(const E *x, int D, int8_t *codes, float *scale_out) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
  for (int i = lane; i < D; i += 32) amax = fmaxf(amax, fabsf(widen_elem(x[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = __fdiv_rn(amax, 127.f);
  for (int i = lane; i < D; i += 32) {
    float c = 0.f;
    if (scale > 0.f) c = fminf(fmaxf(rintf(__fdiv_rn(widen_elem(x[i]), scale)), -127.f), 127.f);
    codes[i] = (int8_t)(int)c;
  }
  if (lane == 0) *scale_out = scale;
}

template <typename E>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const E *x, long long rows, int D, int8_t *codes,
                                                                 float *scales) {
  griddep_wait();
  griddep_launch_dependents();
  const long long warps = (long long)gridDim.x * (kQuantThreads / 32);
  for (long long r = (long long)blockIdx.x * (kQuantThreads / 32) + threadIdx.x / 32; r < rows; r += warps)
    quantize_row<E>(x + r * D, D, codes + r * D, scales + r);
}

// td_kv_append's rules for an int8 cache: one CTA per sequence reads seq_lens[b] once,
// quantises the sequence's T new key and value rows of every kv head into rows L .. L+T-1,
// then advances the length itself.
template <typename E>
__global__ void __launch_bounds__(kQuantThreads)
    append_q8_kernel(const E *k_new, const E *v_new, int8_t *k_codes, float *k_scales, int8_t *v_codes,
                     float *v_scales, int32_t *seq_lens, int Hkv, int T, int Smax, int D, int advance,
                     uint32_t *status) {
  __shared__ int s_start;
  const int b = blockIdx.x;
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
  const int rows = Hkv * T;
  for (int r = threadIdx.x / 32; r < 2 * rows; r += kQuantThreads / 32) {
    const bool isv = r >= rows;
    const int rr = isv ? r - rows : r;  // (h, t)
    const int h = rr / T, t = rr % T;
    const long long src = ((long long)b * Hkv * T + rr) * D;
    const long long dst = ((long long)b * Hkv + h) * Smax + L + t;
    quantize_row<E>((isv ? v_new : k_new) + src, D, (isv ? v_codes : k_codes) + dst * D,
                    (isv ? v_scales : k_scales) + dst);
  }
  __syncthreads();  // every read of L is done
  if (advance && threadIdx.x == 0) seq_lens[b] = L + T;
}

}  // namespace

cudaError_t launch_quantize_q8(size_t elem_bytes, const void *x, long long rows, int D, int8_t *codes, float *scales,
                               cudaStream_t stream) {
  long long blocks = (rows + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  if (blocks > 65535) blocks = 65535;
  if (elem_bytes == 2)
    return launch_pdl(quantize_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(kQuantThreads), 0, stream,
                      static_cast<const __nv_bfloat16 *>(x), rows, D, codes, scales);
  return launch_pdl(quantize_kernel<float>, dim3((unsigned)blocks), dim3(kQuantThreads), 0, stream,
                    static_cast<const float *>(x), rows, D, codes, scales);
}

cudaError_t launch_append_q8(size_t elem_bytes, const void *k_new, const void *v_new, int8_t *k_codes,
                             float *k_scales, int8_t *v_codes, float *v_scales, int32_t *seq_lens, int B, int Hkv,
                             int T, int Smax, int D, int advance, uint32_t *dev_status, cudaStream_t stream) {
  if (elem_bytes == 2)
    return launch_pdl(append_q8_kernel<__nv_bfloat16>, dim3(B), dim3(kQuantThreads), 0, stream,
                      static_cast<const __nv_bfloat16 *>(k_new), static_cast<const __nv_bfloat16 *>(v_new), k_codes,
                      k_scales, v_codes, v_scales, seq_lens, Hkv, T, Smax, D, advance, dev_status);
  return launch_pdl(append_q8_kernel<float>, dim3(B), dim3(kQuantThreads), 0, stream, static_cast<const float *>(k_new),
                    static_cast<const float *>(v_new), k_codes, k_scales, v_codes, v_scales, seq_lens, Hkv, T, Smax,
                    D, advance, dev_status);
}

}  // namespace td
