// Split-KV attention over an 8-bit quantised KV cache (per-row scales).
//
// Method: the split attention of split_attn_mma_kernel ("tinydecode", section "how the
// decode step is put together"; "llm-decode-cuda", split-KV attention section) over a cache
// whose K and V rows are stored as int8 codes with one fp32 scale per row (the per-row INT8
// scheme "llm-decode-cuda" applies to its weights, read here for the K/V bytes that bound
// the decode step): a row reads back as code * scale.
//
// GB300 design: the bytes streamed from HBM halve. Stages of 128 rows cross by TMA as int8
// tiles (with the 128-byte swizzle for 128-byte rows, the 64-byte one for 64-byte rows) plus
// their scales (tensor maps with zero fill past Smax); each of the 4 warps takes 32 keys of a
// stage. The tensor-core step runs in fp16 and takes its B operands straight from the int8
// tiles: ldmatrix moves 16-bit words (two codes), and in registers one byte permute places a
// code c (sign bit flipped: c + 128) under the exponent byte 0x64, which reads as the exact
// fp16 value 1152 + c. The constant 1152 is not subtracted per value: it adds 1152 * sum(q)
// to every score of a query row and 1152 * sum(p) to every output of a row, and both are
// taken off afterwards from products of the same operands with a tile of 1152s (an fp32
// cancellation of about 2^-24 * 1279 * sum|q| per score, far below the query's own rounding
// to fp16). bf16's 8 significant bits leave no such trick. For the scores the order of the
// head dimensions is free: each thread's four dims are whichever four consecutive codes its
// word holds, and the query fragments (fp16, exact for bf16 queries) take the same order.
// For P V the transposed load gives each thread two adjacent output dims of two keys: the
// even dims form one 8-wide output tile and the odd dims another, put back in order when the
// partial results are written. The scales are not applied to the codes: the key scale
// multiplies each score and the value scale each probability before the P V product.
// Everything else (planning, chunking, the fused merge) is the persistent kernel's.
#pragma once

#include "td_split_mma.cuh"

namespace td {

template <int D, int NST_>
struct Q8Cfg {
  static constexpr int NST = NST_;
  static constexpr int TK = 128;                               // keys per stage, 32 per warp
  static constexpr int CODE_BYTES = TK * D;                    // one int8 tile
  static constexpr int CODES_STAGE = 2 * CODE_BYTES;           // K then V codes
  // the scales of a stage's rows are fetched from the 16-byte boundary at or below its first
  // row (a TMA load's inner coordinate must be 16-byte aligned): TK + 4 values, the stage's
  // starting at index (first row & 3)
  static constexpr int SCALE_BOX = TK + 4;
  static constexpr int SCALE_SLOT = 640;                       // bytes kept per scale box (128-aligned)
  static constexpr int SCALE_OFF = NST * CODES_STAGE;          // K, V scale slots of every stage
  static constexpr int RING_BYTES = SCALE_OFF + NST * 2 * SCALE_SLOT;
  static constexpr int SMEM_BYTES = RING_BYTES + 1024;         // + alignment slack
  static_assert(CODE_BYTES % 1024 == 0, "code tiles keep the swizzle's 1024-byte alignment");
  static_assert(SCALE_BOX * 4 <= SCALE_SLOT && (SCALE_BOX * 4) % 16 == 0, "scale box");
  static_assert(kWarps * kMmaRows * (D + 6) * 4 <= RING_BYTES, "combine area fits (rows D + 4 floats apart)");
};

// Ring depth: two CTAs per SM, NST - 1 stages in flight while one is read.
template <int D>
constexpr int kQ8Stages = D == 128 ? 3 : 6;

// Byte offset of 16-byte chunk `ch` of row `row` in an int8 tile of D-byte rows as the TMA
// unit writes it: 128-byte swizzle for D = 128 (chunk c ^ (row & 7)), 64-byte swizzle for
// D = 64 (chunk c ^ ((row >> 1) & 3)); either way the 8 rows one ldmatrix reads fall in 8
// different bank groups.
template <int D>
__device__ __forceinline__ uint32_t q8_swz(int row, int ch) {
  if constexpr (D == 128) {
    return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
  } else {
    return (uint32_t)(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
  }
}

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

// Two int8 codes of a word (sign bits already flipped) -> the fp16 values 1152 + code: `sel`
// places the chosen bytes under the exponent byte 0x64.
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t flipped, uint32_t sel) {
  return __byte_perm(flipped, 0x64646464u, sel);
}
constexpr uint32_t kFlip = 0x80808080u;
constexpr uint32_t kF16x2_1152 = 0x64806480u;           // two fp16 1152s
constexpr uint32_t kSelB01 = 0x4140, kSelB23 = 0x4342;  // bytes 0, 1 / bytes 2, 3
constexpr uint32_t kSelB02 = 0x4240, kSelB13 = 0x4341;  // bytes 0, 2 / bytes 1, 3

// One warp's step over 32 keys (rows kr .. kr+31 of the stage's code tiles kt / vt; keys
// key0 ..): S = Q K^T with the key scales, online softmax in base 2, then
// O += (P * value scale) V, where O and `ob` (the rows' 1152 * sum(p) terms) both carry the
// code bias. qb: the rows' score bias 1152 * sum(q), the scores' starting value negated;
// qscale = scale * log2(e) multiplies each key scale. ks / vs point at the
// stage's scales (index = row in the stage). MASK: some key of the step lies at or past a
// row's limit `lim` or the sequence's end `kend` (otherwise no key is masked: rows that do
// not exist compute finite values nobody reads). Fragment orders (mma m16n8k16, g = lane / 4, c = lane % 4):
//  - scores: ldmatrix gives thread (g, c) codes 4c .. 4c+3 of a 16-dim block of key g; the
//    k slots 2c, 2c+1, 2c+8, 2c+9 hold those four dims, and so do the query fragments;
//  - P V: the transposed ldmatrix gives thread (g, c) dims 2g, 2g+1 of keys 2c, 2c+1; o[2j]
//    takes the even dims of 16-dim block j and o[2j+1] the odd ones, so thread (g, c) holds
//    dims 16j + 4c .. 16j + 4c + 3 of its rows as o[2j][0], o[2j+1][0], o[2j][1], o[2j+1][1].
template <int D, bool MASK>
__device__ __forceinline__ void warp_keys32_q8(const uint32_t (&qa)[D / 16][4], const float (&qb)[2], uint32_t kt,
                                               uint32_t vt, int kr, int key0, int kend, const int (&lim)[2],
                                               float qscale, const float *ks, const float *vs, float (&o)[D / 8][4],
                                               float (&ob)[4], float (&m_run)[2], float (&l_run)[2]) {
  constexpr int NX = D / 32;  // ldmatrix.x4 per 16 keys: 16 keys x 32 dims
  const int lane = threadIdx.x & 31, tig = lane & 3;
  const int lrow = kr + (lane & 7) + ((lane >> 3) & 1) * 8, lch = lane >> 4;
  float sc[4][4];  // n tiles of 8 keys, starting from minus the rows' score bias
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    sc[nt][0] = sc[nt][1] = -qb[0];
    sc[nt][2] = sc[nt][3] = -qb[1];
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      uint32_t r[4];  // keys 0-7 / 8-15 of dims 32i .. 32i+15, then of dims 32i+16 .. 32i+31
      ldmatrix_x4(r, kt + q8_swz<D>(lrow + 16 * hf, 2 * i + lch));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t f = r[e] ^ kFlip;
        mma_f16_16816(sc[2 * hf + (e & 1)], qa[2 * i + (e >> 1)], codes_f16x2(f, kSelB01), codes_f16x2(f, kSelB23));
      }
    }
  float kss[4][2], vss[4][2];  // scales of this thread's eight keys
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = kr + nt * 8 + 2 * tig + e;
      kss[nt][e] = ks[r] * qscale;
      // keys past the sequence: a stale scale must not meet a zero probability
      vss[nt][e] = !MASK || key0 + nt * 8 + 2 * tig + e < kend ? vs[r] : 0.f;
    }
  float alpha[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + nt * 8 + 2 * tig + e;
        const float v = !MASK || key < lim[h] ? sc[nt][2 * h + e] * kss[nt][e] : -INFINITY;
        sc[nt][2 * h + e] = v;
        mx = fmaxf(mx, v);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // lazy reference maximum (see warp_keys16): rows with no visible key are never rescaled
    const bool move = mx > m_run[h] + kMaxGap;
    alpha[h] = move ? exp2_approx(m_run[h] - mx) : 1.f;
    if (move) m_run[h] = mx;
    const float base = m_run[h] == -INFINITY ? 0.f : m_run[h];
    float ps = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pv = exp2_approx(sc[nt][2 * h + e] - base);
        sc[nt][2 * h + e] = pv * vss[nt][e];
        ps += pv;
      }
    l_run[h] = l_run[h] * alpha[h] + ps;
  }
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
    ob[0] *= alpha[0];
    ob[1] *= alpha[0];
    ob[2] *= alpha[1];
    ob[3] *= alpha[1];
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const uint32_t pa[4] = {pack_f16x2(sc[2 * hf][0], sc[2 * hf][1]), pack_f16x2(sc[2 * hf][2], sc[2 * hf][3]),
                            pack_f16x2(sc[2 * hf + 1][0], sc[2 * hf + 1][1]),
                            pack_f16x2(sc[2 * hf + 1][2], sc[2 * hf + 1][3])};
    mma_f16_16816(ob, pa, kF16x2_1152, kF16x2_1152);
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      uint32_t r[4];  // transposed: keys 0-7 / 8-15 of dims 32i .. 32i+15, then of 32i+16 ..
      ldmatrix_x4_trans(r, vt + q8_swz<D>(lrow + 16 * hf, 2 * i + lch));
#pragma unroll
      for (int d2 = 0; d2 < 2; ++d2) {
        const uint32_t lo = r[2 * d2] ^ kFlip, hi = r[2 * d2 + 1] ^ kFlip;
        const int j = 2 * i + d2;  // 16-dim block
        mma_f16_16816(o[2 * j], pa, codes_f16x2(lo, kSelB02), codes_f16x2(hi, kSelB02));
        mma_f16_16816(o[2 * j + 1], pa, codes_f16x2(lo, kSelB13), codes_f16x2(hi, kSelB13));
      }
    }
  }
}

// The same step for at most 8 query rows with keys and rows swapped, as warp_keys16_n8 does
// for bf16 caches: S^T = K Q^T (m: 16 keys, n: the rows) and O^T += V^T P'^T (m: 16 output
// dims, k: 16 keys), for each 16-key half of the warp's 32 keys. Fragment orders
// (g = lane / 4, c = lane % 4):
//  - scores: ldmatrix gives thread (g, c) codes 4c .. 4c+3 of a 16-dim block of keys g and
//    g + 8; they fill k slots 2c, 2c+1, 2c+8, 2c+9 of the A fragment, and qn (the query rows
//    as B fragments) holds row g's dims 4c .. 4c+3 in the same slots. The accumulators start
//    at minus the rows' score bias qbn (rows 2c, 2c+1);
//  - P V: the transposed ldmatrix gives thread (g, c) dims 2g, 2g+1 of keys 2c, 2c+1; bytes
//    0, 2 (dim 2g) fill the A fragment of the even-dim tile o[2i], bytes 1, 3 the odd one
//    o[2i+1]. Tile rows m < 8 are dims 32i + 2m (+1), rows m >= 8 dims 32i + 16 + 2(m - 8)
//    (+1), so thread (g, c) holds dims 32i + 2g, +1 (rows 2c, 2c+1 in o[2i][0..1], o[2i+1][0..1])
//    and 32i + 16 + 2g, +1 (in [2..3]);
//  - ob: 1152 * sum(P') of rows 2c, 2c+1 (the output's code bias), from the same B operands.
template <int D, bool MASK>
__device__ __forceinline__ void warp_keys32_q8_n8(const uint32_t (&qn)[D / 16][2], const float (&qbn)[2], uint32_t kt,
                                                  uint32_t vt, int kr, int key0, int kend, const int (&lim)[2],
                                                  float qscale, const float *ks, const float *vs,
                                                  float (&o)[D / 16][4], float (&ob)[4], float (&m_run)[2],
                                                  float (&l_run)[2]) {
  constexpr int NX = D / 32;  // ldmatrix.x4 per 16 keys: 16 keys x 32 dims
  const int lane = threadIdx.x & 31, gid = lane >> 2;
  const int lrow = kr + (lane & 7) + ((lane >> 3) & 1) * 8, lch = lane >> 4;
  const uint32_t c1152[4] = {kF16x2_1152, kF16x2_1152, kF16x2_1152, kF16x2_1152};
  float sc[2][4];  // per 16-key half: keys gid, gid + 8 of rows 2c, 2c+1
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    sc[hf][0] = sc[hf][2] = -qbn[0];
    sc[hf][1] = sc[hf][3] = -qbn[1];
  }
#pragma unroll
  for (int i = 0; i < NX; ++i)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t r[4];  // keys 0-7 / 8-15 of dims 32i .. 32i+15, then of dims 32i+16 .. 32i+31
      ldmatrix_x4(r, kt + q8_swz<D>(lrow + 16 * hf, 2 * i + lch));
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint32_t f0 = r[2 * blk] ^ kFlip, f1 = r[2 * blk + 1] ^ kFlip;
        const uint32_t ak[4] = {codes_f16x2(f0, kSelB01), codes_f16x2(f1, kSelB01), codes_f16x2(f0, kSelB23),
                                codes_f16x2(f1, kSelB23)};
        mma_f16_16816(sc[hf], ak, qn[2 * i + blk][0], qn[2 * i + blk][1]);
      }
    }
  float alpha[2];
  float vss[2][2];  // value scales of keys gid, gid + 8 of each half
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int hk = 0; hk < 2; ++hk) {
      const int r = kr + 16 * hf + 8 * hk + gid;
      const float kss = ks[r] * qscale;
      const int key = key0 + 16 * hf + 8 * hk + gid;
      // keys past the sequence: a stale scale must not meet a zero probability
      vss[hf][hk] = !MASK || key < kend ? vs[r] : 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = sc[hf][2 * hk + e] * kss;
        sc[hf][2 * hk + e] = !MASK || key < lim[e] ? v : -INFINITY;
      }
    }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float mx = fmaxf(fmaxf(sc[0][e], sc[0][2 + e]), fmaxf(sc[1][e], sc[1][2 + e]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const bool move = mx > m_run[e] + kMaxGap;
    alpha[e] = move ? exp2_approx(m_run[e] - mx) : 1.f;
    if (move) m_run[e] = mx;
    const float base = m_run[e] == -INFINITY ? 0.f : m_run[e];
    float ps = 0.f;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        const float pv = exp2_approx(sc[hf][2 * hk + e] - base);
        sc[hf][2 * hk + e] = pv * vss[hf][hk];
        ps += pv;
      }
    l_run[e] = l_run[e] * alpha[e] + ps;  // this thread's keys; lanes summed at the end
  }
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int t = 0; t < D / 16; ++t) {
      o[t][0] *= alpha[0];
      o[t][1] *= alpha[1];
      o[t][2] *= alpha[0];
      o[t][3] *= alpha[1];
    }
    ob[0] *= alpha[0];
    ob[1] *= alpha[1];
    ob[2] *= alpha[0];
    ob[3] *= alpha[1];
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    // P'^T as the B operand: keys 2c, 2c+1 (+8) of row gid
    const uint32_t pb0 = movmatrix_trans(pack_f16x2(sc[hf][0], sc[hf][1]));
    const uint32_t pb1 = movmatrix_trans(pack_f16x2(sc[hf][2], sc[hf][3]));
    mma_f16_16816(ob, c1152, pb0, pb1);
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      uint32_t r[4];  // transposed: keys 0-7 / 8-15 of dims 32i .. 32i+15, then of 32i+16 ..
      ldmatrix_x4_trans(r, vt + q8_swz<D>(lrow + 16 * hf, 2 * i + lch));
      const uint32_t f0 = r[0] ^ kFlip, f1 = r[1] ^ kFlip, f2 = r[2] ^ kFlip, f3 = r[3] ^ kFlip;
      const uint32_t ae[4] = {codes_f16x2(f0, kSelB02), codes_f16x2(f2, kSelB02), codes_f16x2(f1, kSelB02),
                              codes_f16x2(f3, kSelB02)};
      const uint32_t ao[4] = {codes_f16x2(f0, kSelB13), codes_f16x2(f2, kSelB13), codes_f16x2(f1, kSelB13),
                              codes_f16x2(f3, kSelB13)};
      mma_f16_16816(o[2 * i], ae, pb0, pb1);
      mma_f16_16816(o[2 * i + 1], ao, pb0, pb1);
    }
  }
}

// Streams keys [c0, c1) of (b, kvh) for row block rb, as stream_chunk does for bf16 caches,
// leaving the same combine area (at the start of `smem`).
template <int D, int NST, bool NARROW = false>
__device__ bool stream_chunk_q8(const Q8Args &a, unsigned char *smem, uint64_t *s_bars, uint32_t &seq, int b, int kvh,
                                int rb, int L, int c0, int c1) {
  using C = Q8Cfg<D, NST>;
  const SplitParams &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t sbase = smem_u32(smem);
  const int GT = p.G * p.T;
  const int nstages = (c1 - c0 + C::TK - 1) / C::TK;
  const int zc = b * p.Hkv + kvh;
  const uint64_t policy = l2_evict_first_policy();

  auto issue = [&](int sidx) {
    const int buf = (seq + sidx) % NST;
    const uint32_t bar = smem_u32(&s_bars[buf]);
    const uint32_t dst = sbase + buf * C::CODES_STAGE;
    const uint32_t sdst = sbase + C::SCALE_OFF + buf * 2 * C::SCALE_SLOT;
    const int y = c0 + sidx * C::TK;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, C::CODES_STAGE + 2 * C::SCALE_BOX * 4);
    tma_load_3d(dst, &a.kmap, 0, y, zc, bar, policy);
    tma_load_3d(dst + C::CODE_BYTES, &a.vmap, 0, y, zc, bar, policy);
    tma_load_2d(sdst, &a.ksmap, y & ~3, zc, bar, policy);
    tma_load_2d(sdst + C::SCALE_SLOT, &a.vsmap, y & ~3, zc, bar, policy);
  };
  if (tid == 0) {
    for (int s2 = 0; s2 < min(NST - 1, nstages); ++s2) issue(s2);
  }
  // query rows gid and gid + 8 of this row block as fp16 A fragments (exact: a bf16 value in
  // fp16's range is an fp16 value; the scale stays out of them, its product would round),
  // dims in the order the key fragments take (slots 2c, 2c+1 <- dims 4c, 4c+1; slots 2c+8,
  // 2c+9 <- dims 4c+2, 4c+3)
  // (narrow layout: row gid as B fragments qa[ks][0..1], limits of rows 2c, 2c+1)
  uint32_t qa[D / 16][NARROW ? 2 : 4];
  int lim[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int lr = NARROW ? 2 * tig + h : gid + 8 * h;  // the row whose limit this thread applies
    const int lgr = rb * p.R + lr;
    lim[h] = lr < p.R && lgr < GT ? min(max(L - p.T + lgr % p.T + 1, 0), c1) : 0;
    if (NARROW && h == 1) break;  // one query row per thread in the narrow layout
    const int r = NARROW ? gid : gid + 8 * h;
    const int gr = rb * p.R + r;
    const bool valid = r < p.R && gr < GT;
    const int hq = kvh * p.G + (valid ? gr / p.T : 0), t = valid ? gr % p.T : 0;
    const uint2 *qrow = reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.q) +
                                                        (((size_t)b * p.Hq + hq) * p.T + t) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint2 w = valid ? qrow[ks * 4 + tig] : make_uint2(0u, 0u);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
      if constexpr (NARROW) {
        qa[ks][0] = pack_f16x2(lo.x, lo.y);
        qa[ks][1] = pack_f16x2(hi.x, hi.y);
      } else {
        qa[ks][h] = pack_f16x2(lo.x, lo.y);
        qa[ks][2 + h] = pack_f16x2(hi.x, hi.y);
      }
    }
  }
  // the rows' score bias 1152 * sum(q), from the same fragments (narrow: rows 2c, 2c+1)
  float qb[2];
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (NARROW) {
      const uint32_t c1152[4] = {kF16x2_1152, kF16x2_1152, kF16x2_1152, kF16x2_1152};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) mma_f16_16816(acc, c1152, qa[ks][0], qa[ks][1]);
      qb[0] = acc[0];
      qb[1] = acc[1];
    } else {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) mma_f16_16816(acc, qa[ks], kF16x2_1152, kF16x2_1152);
      qb[0] = acc[0];
      qb[1] = acc[2];
    }
  }
  // keys every existing row of the block sees (a warp-uniform bound for the unmasked step)
  int lim_all = c1;
  for (int r = 0; r < min(p.R, GT - rb * p.R); ++r) lim_all = min(lim_all, max(L - p.T + (rb * p.R + r) % p.T + 1, 0));
  constexpr int NO = NARROW ? D / 16 : D / 8;  // output tiles
  float o[NO][4], ob[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NO; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  int consumed = 0;
  bool ok = true;
  for (int st = 0; st < nstages; ++st) {
    const int buf = (seq + st) % NST;
    const bool landed = mbar_wait_bounded(smem_u32(&s_bars[buf]), ((seq + st) / NST) & 1u);
    // every warp has finished the previous stage, whose buffer is refilled next; one decision
    // for the whole CTA
    if (!__syncthreads_and(landed)) {
      ok = false;
      break;
    }
    if (tid == 0 && st + NST - 1 < nstages) issue(st + NST - 1);
    const int j0 = c0 + st * C::TK;
    const int kr = warp * 32;
    const int key0 = j0 + kr;
    if (key0 < c1) {
      const uint32_t kt = sbase + buf * C::CODES_STAGE;
      const float *scl = reinterpret_cast<const float *>(smem + C::SCALE_OFF + buf * 2 * C::SCALE_SLOT) + (j0 & 3);
      if constexpr (NARROW) {
        if (key0 + 32 <= lim_all)
          warp_keys32_q8_n8<D, false>(qa, qb, kt, kt + C::CODE_BYTES, kr, key0, L, lim, p.qscale, scl,
                                      scl + C::SCALE_SLOT / 4, o, ob, m_run, l_run);
        else
          warp_keys32_q8_n8<D, true>(qa, qb, kt, kt + C::CODE_BYTES, kr, key0, L, lim, p.qscale, scl,
                                     scl + C::SCALE_SLOT / 4, o, ob, m_run, l_run);
      } else {
        if (key0 + 32 <= lim_all)
          warp_keys32_q8<D, false>(qa, qb, kt, kt + C::CODE_BYTES, kr, key0, L, lim, p.qscale, scl,
                                   scl + C::SCALE_SLOT / 4, o, ob, m_run, l_run);
        else
          warp_keys32_q8<D, true>(qa, qb, kt, kt + C::CODE_BYTES, kr, key0, L, lim, p.qscale, scl,
                                  scl + C::SCALE_SLOT / 4, o, ob, m_run, l_run);
      }
    }
    consumed = st + 1;
  }
  if (!ok) {
    const int issued = min(nstages, consumed + NST - 1);
    for (int st = consumed; st < issued; ++st)
      mbar_wait_bounded(smem_u32(&s_bars[(seq + st) % NST]), ((seq + st) / NST) & 1u);
    if (tid == 0) report(p.status, TD_DEV_WAIT_TIMEOUT);
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
  }
  seq += nstages;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if constexpr (NARROW) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
    } else {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
  }
  __syncthreads();  // ring idle: reuse it as the combine area
  float *combine = reinterpret_cast<float *>(smem);
  float *cm = combine;
  float *cl = combine + kWarps * kMmaRows;
  float *ca = combine + 2 * kWarps * kMmaRows;
  if constexpr (NARROW) {
    // rows 2c + e; thread (g, c) holds dims 32i + 2g, +1 and 32i + 16 + 2g, +1
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * tig + e;
      if (gid == 0) {
        cm[warp * kMmaRows + r] = m_run[e];
        cl[warp * kMmaRows + r] = l_run[e];
      }
      const float bias = ob[e];  // 1152 * sum(p) of row r
      float *row = &ca[(warp * kMmaRows + r) * combine_stride<D>()];
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        *reinterpret_cast<float2 *>(&row[32 * i + 2 * gid]) = make_float2(o[2 * i][e] - bias, o[2 * i + 1][e] - bias);
        *reinterpret_cast<float2 *>(&row[32 * i + 16 + 2 * gid]) =
            make_float2(o[2 * i][2 + e] - bias, o[2 * i + 1][2 + e] - bias);
      }
    }
    __syncthreads();
    return ok;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = gid + 8 * h;
    if (tig == 0) {
      cm[warp * kMmaRows + r] = m_run[h];
      cl[warp * kMmaRows + r] = l_run[h];
    }
    const float bias = ob[2 * h];  // 1152 * sum(p) of row r: the code bias in every output
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
      *reinterpret_cast<float4 *>(&ca[(warp * kMmaRows + r) * combine_stride<D>() + 16 * j + 4 * tig]) =
          make_float4(o[2 * j][2 * h] - bias, o[2 * j + 1][2 * h] - bias, o[2 * j][2 * h + 1] - bias,
                      o[2 * j + 1][2 * h + 1] - bias);
  }
  __syncthreads();
  return ok;
}

// Persistent kernel over an int8 cache: the same items, chunks and fused merge as
// split_attn_mma_kernel.
// NARROW: a row block has at most 8 rows and the warps step with warp_keys32_q8_n8.
// EARLY_PLAN: planned before the wait (launched when the plan leaves slots free for the
// previous call's merging CTAs).
template <int D, bool NARROW = false, bool EARLY_PLAN = false>
__global__ void __launch_bounds__(kThreads, 2) split_attn_q8_kernel(const __grid_constant__ Q8Args a) {
  constexpr int NST = kQ8Stages<D>;
  using C = Q8Cfg<D, NST>;
  using E = __nv_bfloat16;
  static_assert((merge_fixed_floats<D, kMmaRows>() + part_block_floats(kMmaRows, D)) * 4 <= C::RING_BYTES,
                "merge stages at least one chunk");
  const SplitParams &p = a.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_len[TD_MAX_BATCH];
  __shared__ int s_prefix[TD_MAX_BATCH + 1];
  __shared__ long long s_red[2 * kWarps];
  __shared__ int s_chunk, s_last;
  __shared__ __align__(8) uint64_t s_merge_bar;
  __shared__ __align__(8) uint64_t s_bars[NST];

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
  if (tid == 0) prefetch_first_item<D, true>(p, prefetch_stages(p), blockIdx.x);
  // EARLY_PLAN: planned before the wait and kept when the lengths read the same after it,
  // as the bf16 decode kernel does. With the slots left free for the previous call's merging
  // CTAs this measured 4k 9.06 -> 8.07 us, 16k 13.05 -> 12.13, 32k 16.78 -> 15.95
  // (3B-style layer, B = 1; either change alone: 9.1 / 12.8 / 16.5 with the spare slots,
  // 8.2 / 14.3 / 17.7 with the early plan)
  if constexpr (EARLY_PLAN) plan_items(p, s_len, s_prefix, &s_chunk, s_red, false);
  griddep_wait();  // inputs may come from the previous kernel in the stream
  griddep_launch_dependents();
  if constexpr (EARLY_PLAN)
    confirm_plan(p, s_len, s_prefix, &s_chunk, s_red);  // ends with __syncthreads
  else
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
    const bool ok = stream_chunk_q8<D, NST, NARROW>(a, smem, s_bars, seq, b, kvh, rb, L, c0, min(c0 + S, L));
    finish_item<E, D, kMmaRows, kWarps, combine_stride<D>()>(p, combine, C::RING_BYTES / 4, &s_merge_bar, merge_phase, b,
                                        kvh, rb, c, NC, &s_last, W <= (int)gridDim.x);
    fence_proxy_async_smem();
    __syncthreads();
    if (!ok) break;
  }
}

}  // namespace td
