// Split-KV attention over an 8-bit quantised KV cache (per-row scales).
//
// Method: the split attention of split_attn_mma_kernel ("tinydecode", section "how the
// decode step is put together"; "llm-decode-cuda", split-KV attention section) over a cache
// whose K and V rows are stored as int8 codes with one fp32 scale per row (the per-row INT8
// scheme "llm-decode-cuda" applies to its weights, read here for the K/V bytes that bound
// the decode step): a row reads back as code * scale.
//
// GB300 design: the bytes streamed from HBM halve. Stages of 64 rows cross by TMA as int8
// tiles plus their 64 + 64 scales (tensor maps with zero fill past Smax). Each stage is
// widened once, in shared memory, into the 16-bit tile layout the tensor-core step reads. The
// step runs in fp16 here: an int8 code becomes an fp16 value exactly with one byte permute
// and half a packed subtraction per value (bf16's 8 significant bits leave no such trick),
// and the query is rounded to fp16 once per item. The scales are not applied to the tiles:
// the key scale multiplies each score and the value scale multiplies each probability
// before the P V product (warp_keys16). Everything else (planning, chunking, the fused
// merge) is the persistent kernel's.
#pragma once

#include "td_split_mma.cuh"

namespace td {

template <int D, int NST_>
struct Q8Cfg {
  static constexpr int NST = NST_;
  static constexpr int TK = 64;
  static constexpr int CODE_BYTES = TK * D;                    // one int8 tile
  // the scales of a stage's rows are fetched from the 16-byte boundary at or below its first
  // row (a TMA load's inner coordinate must be 16-byte aligned): 68 values, the stage's 64
  // starting at index (first row & 3)
  static constexpr int SCALE_BOX = TK + 4;
  static constexpr int SCALE_SLOT = 384;                       // bytes kept per scale box (128-aligned)
  static constexpr int STAGE_BYTES = 2 * CODE_BYTES + 2 * SCALE_SLOT;  // K, V codes, then K, V scales
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  static constexpr int WORK_BYTES = 2 * TK * D * 2;            // the widened bf16 K and V tiles
  static constexpr int WORK_OFF = (RING_BYTES + 1023) / 1024 * 1024;
  static constexpr int SMEM_BYTES = WORK_OFF + WORK_BYTES + 1024;  // + alignment slack
  static_assert(CODE_BYTES % 128 == 0, "tiles keep 128-byte alignment");
  static_assert(kWarps * kMmaRows * (D + 2) * 4 <= WORK_OFF + WORK_BYTES, "combine area fits");
};

template <int D>
constexpr int kQ8Stages = 4;

struct Q8Args {
  CUtensorMap kmap, vmap;    // int8 codes [B*Hkv][Smax][D]
  CUtensorMap ksmap, vsmap;  // fp32 scales [B*Hkv][Smax]
  SplitParams p;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Sixteen int8 codes -> sixteen fp16 values, exactly: with the sign bit flipped a code c is
// the byte c + 128; placed under the exponent byte 0x64 it forms the fp16 value 1024 + c + 128,
// and one packed subtraction of 1152 leaves c (two values per instruction).
__device__ __forceinline__ void widen_codes16(const uint4 v, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = __byte_perm(w[i], 0x64646464u, 0x4140);  // bytes 0, 1 under 0x64
    const uint32_t b = __byte_perm(w[i], 0x64646464u, 0x4342);  // bytes 2, 3
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    out[2 * i] = *reinterpret_cast<const uint32_t *>(&ha);
    out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&hb);
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// Eight bf16 values -> eight fp16 values (rounded to nearest even; exact for queries whose
// magnitudes lie in fp16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
    out[i] = pack_f16x2(f.x, f.y);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Streams keys [c0, c1) of (b, kvh) for row block rb, as stream_chunk does for bf16 caches,
// leaving the same combine area (at the start of `smem`).
template <int D, int NST>
__device__ bool stream_chunk_q8(const Q8Args &a, unsigned char *smem, uint64_t *s_bars, float *s_ks, float *s_vs,
                                uint32_t &seq, int b, int kvh, int rb, int L, int c0, int c1) {
  using C = Q8Cfg<D, NST>;
  constexpr int NCH = D * 2 / 16;  // 16-byte chunks per bf16 row
  const SplitParams &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2;
  const uint32_t sbase = smem_u32(smem);
  unsigned char *work = smem + C::WORK_OFF;
  const uint32_t kt = sbase + C::WORK_OFF, vt = kt + C::TK * D * 2;
  const int GT = p.G * p.T;
  const int nstages = (c1 - c0 + C::TK - 1) / C::TK;
  const int zc = b * p.Hkv + kvh;
  const uint64_t policy = l2_evict_first_policy();

  auto issue = [&](int sidx) {
    const int buf = (seq + sidx) % NST;
    const uint32_t bar = smem_u32(&s_bars[buf]);
    const uint32_t dst = sbase + buf * C::STAGE_BYTES;
    const int y = c0 + sidx * C::TK;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * C::CODE_BYTES + 2 * C::SCALE_BOX * 4);
    tma_load_3d(dst, &a.kmap, 0, y, zc, bar, policy);
    tma_load_3d(dst + C::CODE_BYTES, &a.vmap, 0, y, zc, bar, policy);
    tma_load_2d(dst + 2 * C::CODE_BYTES, &a.ksmap, y & ~3, zc, bar, policy);
    tma_load_2d(dst + 2 * C::CODE_BYTES + C::SCALE_SLOT, &a.vsmap, y & ~3, zc, bar, policy);
  };
  // the query rows, as fp16, go to the work K tile, read into registers before the first
  // widening
  for (int idx = tid; idx < kMmaRows * NCH; idx += kThreads) {
    const int r = idx / NCH, ch = idx % NCH;
    const int gr = rb * p.R + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < p.R && gr < GT) {
      const int hq = kvh * p.G + gr / p.T, t = gr % p.T;
      v = bf16x8_to_f16x8(static_cast<const uint4 *>(p.q)[(((size_t)b * p.Hq + hq) * p.T + t) * NCH + ch]);
    }
    *reinterpret_cast<uint4 *>(work + swz<D * 2>(r, ch)) = v;
  }
  if (tid == 0) {
    for (int s2 = 0; s2 < min(NST, nstages); ++s2) issue(s2);
  }
  int lim[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = gid + 8 * h;
    const int gr = rb * p.R + r;
    const bool valid = r < p.R && gr < GT;
    lim[h] = valid ? min(max(L - p.T + gr % p.T + 1, 0), c1) : 0;
  }
  uint32_t qa[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  int consumed = 0;
  bool ok = true;
  for (int st = 0; st < nstages; ++st) {
    const int buf = (seq + st) % NST;
    const bool landed = mbar_wait_bounded(smem_u32(&s_bars[buf]), ((seq + st) / NST) & 1u);
    // every warp has finished the previous stage with the work tiles; one decision for all
    if (!__syncthreads_and(landed)) {
      ok = false;
      break;
    }
    if (st == 0) {
#pragma unroll
      for (int j = 0; j < D / 16; ++j)
        ldmatrix_x4(qa[j], kt + swz<D * 2>(((lane >> 3) & 1) * 8 + (lane & 7), 2 * j + (lane >> 4)));
      __syncthreads();  // the query tile is read before the work tiles are overwritten
    }
    const int j0 = c0 + st * C::TK;
    const int valid = min(C::TK, c1 - j0);
    // widen this stage's codes into the work tiles (value rows past the chunk: zero)
    const unsigned char *k8 = smem + buf * C::STAGE_BYTES;
    const unsigned char *v8 = k8 + C::CODE_BYTES;
    for (int idx = tid; idx < 2 * C::TK * (D / 16); idx += kThreads) {
      const bool isv = idx >= C::TK * (D / 16);
      const int i = isv ? idx - C::TK * (D / 16) : idx;
      const int r = i / (D / 16), c = i % (D / 16);
      uint4 lo, hi;
      if (isv && r >= valid) {
        lo = hi = make_uint4(0u, 0u, 0u, 0u);
      } else {
        widen_codes16(*reinterpret_cast<const uint4 *>((isv ? v8 : k8) + r * D + c * 16), lo, hi);
      }
      unsigned char *tile = work + (isv ? C::TK * D * 2 : 0);
      *reinterpret_cast<uint4 *>(tile + tma_swz<C::TK>(r, 2 * c)) = lo;
      *reinterpret_cast<uint4 *>(tile + tma_swz<C::TK>(r, 2 * c + 1)) = hi;
    }
    if (tid < 2 * C::TK) {
      const bool isv = tid >= C::TK;
      const float *sc = reinterpret_cast<const float *>(k8 + 2 * C::CODE_BYTES + (isv ? C::SCALE_SLOT : 0));
      (isv ? s_vs : s_ks)[tid % C::TK] = sc[(j0 & 3) + tid % C::TK];
    }
    __syncthreads();  // work tiles and scales ready; this ring buffer is free
    if (tid == 0 && st + NST < nstages) issue(st + NST);
    const int kr = warp * 16;
    const int key0 = j0 + kr;
    if (key0 < c1) warp_keys16<D, true>(qa, kt, vt, kr, key0, lim, p.qscale, s_ks, s_vs, o, m_run, l_run);
    consumed = st + 1;
  }
  if (!ok) {
    const int issued = min(nstages, consumed + NST);
    for (int st = consumed; st < issued; ++st)
      mbar_wait_bounded(smem_u32(&s_bars[(seq + st) % NST]), ((seq + st) / NST) & 1u);
    if (tid == 0) report(p.status, TD_DEV_WAIT_TIMEOUT);
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
  }
  seq += nstages;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  __syncthreads();  // ring and work tiles idle: reuse them as the combine area
  float *combine = reinterpret_cast<float *>(smem);
  float *cm = combine;
  float *cl = combine + kWarps * kMmaRows;
  float *ca = combine + 2 * kWarps * kMmaRows;
  const int tig = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = gid + 8 * h;
    if (tig == 0) {
      cm[warp * kMmaRows + r] = m_run[h];
      cl[warp * kMmaRows + r] = l_run[h];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
      *reinterpret_cast<float2 *>(&ca[(warp * kMmaRows + r) * D + nt * 8 + 2 * tig]) =
          make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
  }
  __syncthreads();
  return ok;
}

// Persistent kernel over an int8 cache: the same items, chunks and fused merge as
// split_attn_mma_kernel.
template <int D>
__global__ void __launch_bounds__(kThreads, 2) split_attn_q8_kernel(const __grid_constant__ Q8Args a) {
  constexpr int NST = kQ8Stages<D>;
  using C = Q8Cfg<D, NST>;
  using E = __nv_bfloat16;
  static_assert((merge_fixed_floats<D, kMmaRows>() + part_block_floats(kMmaRows, D)) * 4 <= C::WORK_OFF + C::WORK_BYTES,
                "merge stages at least one chunk");
  const SplitParams &p = a.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_len[TD_MAX_BATCH];
  __shared__ int s_prefix[TD_MAX_BATCH + 1];
  __shared__ long long s_red[2 * kWarps];
  __shared__ int s_chunk, s_last;
  __shared__ __align__(8) uint64_t s_merge_bar;
  __shared__ __align__(8) uint64_t s_bars[NST];
  __shared__ float s_ks[64], s_vs[64];

  const int tid = threadIdx.x;
  unsigned char *smem = align1024(smem_raw);
  float *combine = reinterpret_cast<float *>(smem);
  if (tid == 0) {
    mbar_init(smem_u32(&s_merge_bar), 1);
#pragma unroll
    for (int i = 0; i < NST; ++i) mbar_init(smem_u32(&s_bars[i]), 1);
    fence_mbar_init();
  }
  uint32_t merge_phase = 0;
  uint32_t seq = 0;
  griddep_wait();
  griddep_launch_dependents();
  plan_items(p, s_len, s_prefix, &s_chunk, s_red);
  const int S = s_chunk;
  const int W = s_prefix[p.B];
  const int rows = p.Hq * p.T;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (s_len[b] != 0) continue;
    for (int idx = tid; idx < rows * D; idx += kThreads)
      store_elem<E>(static_cast<E *>(p.out) + (long long)b * rows * D + idx, 0.f);
    if (p.lse != nullptr)
      for (int r = tid; r < rows; r += kThreads) p.lse[(long long)b * rows + r] = -INFINITY;
  }
  for (int item = blockIdx.x; item < W; item += gridDim.x) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int L = s_len[b];
    const int NC = (L + S - 1) / S;
    const int local = item - s_prefix[b];
    const int c = local % NC;
    const int rest = local / NC;
    const int rb = rest % p.RB;
    const int kvh = rest / p.RB;
    const int c0 = c * S;
    const bool ok = stream_chunk_q8<D, NST>(a, smem, s_bars, s_ks, s_vs, seq, b, kvh, rb, L, c0, min(c0 + S, L));
    finish_item<E, D, kMmaRows, kWarps>(p, combine, (C::WORK_OFF + C::WORK_BYTES) / 4, &s_merge_bar, merge_phase, b,
                                        kvh, rb, c, NC, &s_last);
    fence_proxy_async_smem();
    __syncthreads();
    if (!ok) break;
  }
}

}  // namespace td
