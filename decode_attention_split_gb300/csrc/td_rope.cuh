// Rotary position embedding on 16-byte vectors, shared by the rope + append kernel and the
// fused rope + append + attention kernels so both produce the same bits.
//
// Layout ("tinydecode" lists an in-place rope kernel for its llama models, loaded from
// Hugging Face llama checkpoints; "llm-decode-cuda" fuses "RoPE + KV-cache write" into its
// decode step; neither prints the rotation, so the llama checkpoints' layout is used): for
// i < D/2 the pair (x[i], x[i + D/2]) of a row at position p turns by the angle whose cosine
// and sine are cos_t[p][i] and sin_t[p][i] (fp32 tables [positions][D/2]):
//   y[i] = x[i] cos - x[i + D/2] sin,   y[i + D/2] = x[i + D/2] cos + x[i] sin,
// in fp32 with a fixed operation order (one product, one fused multiply-add), then rounded
// to nearest even into the element type.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace td {

__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float &y0, float &y1) {
  y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
  y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}

// Rotates the elements held in two 16-byte vectors: `lo` holds x[i .. i+VE) and `hi` holds
// x[i + D/2 .. i + D/2 + VE), VE = 16 / sizeof(E); c and s point at cos_t[p][i] and
// sin_t[p][i] (16-byte aligned).
template <typename E>
__device__ __forceinline__ void rope_vec16(uint4 &lo, uint4 &hi, const float *c, const float *s);

template <>
__device__ __forceinline__ void rope_vec16<__nv_bfloat16>(uint4 &lo, uint4 &hi, const float *c, const float *s) {
  const float4 c0 = *reinterpret_cast<const float4 *>(c), c1 = *reinterpret_cast<const float4 *>(c + 4);
  const float4 s0 = *reinterpret_cast<const float4 *>(s), s1 = *reinterpret_cast<const float4 *>(s + 4);
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t *a = reinterpret_cast<uint32_t *>(&lo);
  uint32_t *b = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 xa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a[w]));
    const float2 xb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&b[w]));
    float ya0, yb0, ya1, yb1;
    rope_pair(xa.x, xb.x, cc[2 * w], ss[2 * w], ya0, yb0);
    rope_pair(xa.y, xb.y, cc[2 * w + 1], ss[2 * w + 1], ya1, yb1);
    const __nv_bfloat162 ra = __floats2bfloat162_rn(ya0, ya1);
    const __nv_bfloat162 rb = __floats2bfloat162_rn(yb0, yb1);
    a[w] = *reinterpret_cast<const uint32_t *>(&ra);
    b[w] = *reinterpret_cast<const uint32_t *>(&rb);
  }
}

template <>
__device__ __forceinline__ void rope_vec16<float>(uint4 &lo, uint4 &hi, const float *c, const float *s) {
  const float4 c0 = *reinterpret_cast<const float4 *>(c);
  const float4 s0 = *reinterpret_cast<const float4 *>(s);
  float4 &a = reinterpret_cast<float4 &>(lo);
  float4 &b = reinterpret_cast<float4 &>(hi);
  float4 ya, yb;
  rope_pair(a.x, b.x, c0.x, s0.x, ya.x, yb.x);
  rope_pair(a.y, b.y, c0.y, s0.y, ya.y, yb.y);
  rope_pair(a.z, b.z, c0.z, s0.z, ya.z, yb.z);
  rope_pair(a.w, b.w, c0.w, s0.w, ya.w, yb.w);
  a = ya;
  b = yb;
}

}  // namespace td
