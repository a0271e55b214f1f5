// Split-KV attention for bf16 caches on the tensor cores.
//
// Same method and work decomposition as split_attn_kernel ("tinydecode", section "how the
// decode step is put together"; "llm-decode-cuda", split-KV attention section): one CTA
// computes, for one chunk of one (sequence, kv head), the partial softmax of every query row
// reading that kv head, and chunks are merged by log-sum-exp.
//
// The grouped-query rows of a kv head (up to 16 per CTA: G heads x T verify tokens) form
// the M side of mma.sync m16n8k16 tiles, so each K/V tile in shared memory is read once for
// all of them:
//   scores  S[rows x 16 keys] = Q[rows x D] . K^T   (B operand from K rows via ldmatrix)
//   output  O[rows x D]      += P[rows x 16 keys] . V (B operand via ldmatrix.trans)
// with fp32 accumulation; P is rounded to bf16 for the second product while the softmax
// statistics (m, l) stay fp32. A kv head with at most 8 query rows (decode with grouped
// heads) takes the narrow tile instead: keys on the M side and the rows on the 8-wide N side
// (S^T = K Q^T, O^T += V^T P^T; warp_keys16_n8), half the tensor-core tiles per step; a row
// block of 17 to 24 rows (a speculative-verify chunk of a grouped kv head: 4 heads x 6
// tokens) takes the same layout with three 8-wide N tiles (warp_keys16_n24), so each K/V tile
// in shared memory serves all 24 rows once.
//
// K/V stages of 64 rows are fetched by the TMA engine (cp.async.bulk.tensor: one thread
// issues one box of 64 rows x 128 bytes per half-row) through a 3-D tensor map over the
// cache [B*Hkv][Smax][D] with the 128-byte swizzle, so the 8 rows an ldmatrix reads sit in 8
// different bank groups; completion is counted on one mbarrier per stage, waited on with a
// bounded wait. Rows past Smax are zero-filled by the TMA unit; rows past a sequence's
// length inside its last stage are zeroed in shared memory before use. The 4 warps split
// every stage's keys 4 ways and combine at the end of the chunk.
//
// Two kernels share the chunk code: a persistent one (this file: CTAs walk work items and
// merge through the workspace) and a cluster one (td_split_cluster.cuh).
#pragma once

#include <cudaTypedefs.h>

#include "td_mma.cuh"
#include "td_rope.cuh"
#include "td_split_attn.cuh"

namespace td {

constexpr int kMmaRows = 16;  // query rows per CTA: one m16 tile

// Tile of a warp's 16-key step, by the query rows of a row block:
//   kTileN8   at most 8 rows: keys on the m side, the rows on one 8-wide n tile (warp_keys16_n8);
//   kTileM16  9 to 16 rows: the rows on the m side of one 16-row tile, keys on n (warp_keys16);
//   kTileN24  17 to 24 rows: keys on the m side, the rows on three 8-wide n tiles
//             (warp_keys16_n24).
enum : int { kTileM16 = 0, kTileN8 = 1, kTileN24 = 2 };
constexpr int kMaxTileRows = 24;
// Rows of a tile's combine area and partial blocks.
template <int TILE>
__host__ __device__ constexpr int tile_rows() {
  return TILE == kTileN24 ? kMaxTileRows : kMmaRows;
}
// Floats between consecutive rows of the combine area's p @ V sums: D + 4 puts the 32 lanes'
// stores of one fragment (narrow layouts: dims gid (+8) of rows 2 tig (+1)) in 32 different
// banks (4-way conflicts with a stride of D).
template <int D>
__host__ __device__ constexpr int combine_stride() {
  return D + 4;
}
template <int D, int TILE>
__host__ __device__ constexpr int combine_floats() {
  return kWarps * tile_rows<TILE>() * (combine_stride<D>() + 2);
}
// Tile for a row block of R query rows.
__host__ __device__ constexpr int tile_of_rows(int R) { return R <= 8 ? kTileN8 : R <= 16 ? kTileM16 : kTileN24; }

template <int D, int NST_>
struct MmaCfg {
  static constexpr int NST = NST_;            // ring stages
  static constexpr int TK = 64;               // keys per pipeline stage
  static constexpr int TKW = TK / kWarps;     // keys per warp per stage
  static constexpr int ROWB = D * 2;          // bytes per cache row
  static constexpr int NCH = ROWB / 16;       // 16-byte chunks per cache row
  static constexpr int HALVES = D / 64;       // 128-byte column halves (TMA boxes per tile)
  static constexpr int BOX_BYTES = TK * 128;  // one box: 64 rows x 128 bytes
  static constexpr int TILE_BYTES = TK * ROWB;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = NST * STAGE_BYTES;
  static constexpr int NTD = D / 8;           // 8-wide output n tiles
  static constexpr int KSD = D / 16;          // 16-deep score k steps
  static constexpr int COMBINE_FLOATS = kWarps * kMaxTileRows * (D + 6);  // the widest tile's
  static_assert(TKW == 16, "each warp takes one 16-key step per stage");
  static_assert(D % 64 == 0, "whole 128-byte halves");
  static_assert(COMBINE_FLOATS * 4 <= RING_BYTES, "combine area fits in the ring");
  static_assert(kMaxTileRows * D * 2 <= TILE_BYTES, "the query tile fits in one K tile");
};

// Ring depth of the persistent kernel (two CTAs per SM) and of the cluster kernel (one).
template <int D>
constexpr int kPersistentStages = D == 128 ? 3 : 4;
// Units of 64 rows of a CTA's first chunk warmed in L2 before the wait for the previous
// kernel; the host sizes it from the device's L2 (plan_split).
__device__ __forceinline__ int prefetch_stages(const SplitParams &p) { return p.warm_stages; }
template <int D>
constexpr int kClusterStages = D == 128 ? 3 : 6;

// Kernel arguments: tensor maps of the two caches, then the common parameters.
struct MmaArgs {
  CUtensorMap kmap;
  CUtensorMap vmap;
  SplitParams p;
};

// Byte offset of 16-byte chunk `ch` of row `row` in the query tile (row-major, chunks XOR-ed
// with the row's low 3 bits).
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * ROWB + ((ch ^ (row & 7)) << 4));
}

// Byte offset of 16-byte chunk `ch` of row `row` in a K/V tile written by the TMA unit with
// the 128-byte swizzle: the tile is HALVES boxes of [64 rows][128 bytes], each 1024-byte
// aligned, and inside a box chunk c of row r lives at chunk position c ^ (r & 7).
template <int TK>
__device__ __forceinline__ uint32_t tma_swz(int row, int ch) {
  return (uint32_t)((ch >> 3) * (TK * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Fused step: cache rows [L - T, L) of (b, kvh) are this launch's new rows, whose copies in
// global memory are not written yet (or are being written). Where they fall inside the
// stage that holds rows [j0, j0 + valid), they are placed into the landed K/V tiles at
// `stage` from k_new / v_new, the keys rotated to their positions when rope tables are given;
// the CTAs of row block 0 also write them to the cache (each new row lies in exactly one
// chunk, so exactly one CTA writes it). Every thread that writes shared memory fences it
// against the TMA unit's next refill of the stage.
template <int D, int NST>
__device__ void place_new_rows(const SplitParams &p, unsigned char *stage, int b, int kvh, int rb, int L, int j0,
                               int valid) {
  using C = MmaCfg<D, NST>;
  constexpr int NH = C::NCH / 2;
  const int n0 = max(L - p.T, j0), n1 = min(L, j0 + valid);
  if (n0 >= n1) return;
  const bool rope = p.rope_cos != nullptr;
  const int kitems = rope ? NH : C::NCH;  // key work items per row (vector pairs or vectors)
  const int per_row = kitems + C::NCH;
  const size_t hb = (size_t)b * p.Hkv + kvh;
  const uint4 *kn = static_cast<const uint4 *>(p.k_new) + hb * p.T * C::NCH;
  const uint4 *vn = static_cast<const uint4 *>(p.v_new) + hb * p.T * C::NCH;
  // the caches are written only in the fused step, whose caller passes them writable
  uint4 *kc = static_cast<uint4 *>(const_cast<void *>(p.k)) + hb * p.Smax * C::NCH;
  uint4 *vc = static_cast<uint4 *>(const_cast<void *>(p.v)) + hb * p.Smax * C::NCH;
  unsigned char *ktile = stage, *vtile = stage + C::TILE_BYTES;
  const bool writer = rb == 0;
  for (int idx = threadIdx.x; idx < (n1 - n0) * per_row; idx += kThreads) {
    const int j = n0 + idx / per_row, it = idx % per_row;
    const int t = j - (L - p.T), srow = j - j0;
    if (it < kitems) {
      if (rope) {
        uint4 lo = kn[(size_t)t * C::NCH + it], hi = kn[(size_t)t * C::NCH + it + NH];
        const size_t tab = (size_t)j * (D / 2) + it * 8;
        rope_vec16<__nv_bfloat16>(lo, hi, p.rope_cos + tab, p.rope_sin + tab);
        *reinterpret_cast<uint4 *>(ktile + tma_swz<C::TK>(srow, it)) = lo;
        *reinterpret_cast<uint4 *>(ktile + tma_swz<C::TK>(srow, it + NH)) = hi;
        if (writer) {
          kc[(size_t)j * C::NCH + it] = lo;
          kc[(size_t)j * C::NCH + it + NH] = hi;
        }
      } else {
        const uint4 x = kn[(size_t)t * C::NCH + it];
        *reinterpret_cast<uint4 *>(ktile + tma_swz<C::TK>(srow, it)) = x;
        if (writer) kc[(size_t)j * C::NCH + it] = x;
      }
    } else {
      const int ch = it - kitems;
      const uint4 x = vn[(size_t)t * C::NCH + ch];
      *reinterpret_cast<uint4 *>(vtile + tma_swz<C::TK>(srow, ch)) = x;
      if (writer) vc[(size_t)j * C::NCH + ch] = x;
    }
  }
  fence_proxy_async_smem();
}

// Rise (base 2) of a row's scores above its reference maximum before that maximum moves and
// the accumulators are rescaled.
constexpr float kMaxGap = 8.f;

// One warp's step over 16 keys of a landed stage (keys key0 .. key0+15, rows kr .. kr+15 of
// the stage's tiles): S = Q K^T over two 8-key n tiles, masking by the rows' visible-key
// limits `lim`, the online softmax in base 2, then O += P V. kt / vt address bf16 K / V
// tiles in the TMA-swizzled layout.
template <int D>
__device__ __forceinline__ void warp_keys16(const uint32_t (&qa)[D / 16][4], uint32_t kt, uint32_t vt, int kr,
                                            int key0, const int (&lim)[2], float qscale, float (&o)[D / 8][4],
                                            float (&m_run)[2], float (&l_run)[2]) {
  constexpr int TK = 64, KSD = D / 16, NTD = D / 8;
  const int lane = threadIdx.x & 31, tig = lane & 3;
  float sc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < KSD / 2; ++i) {
      uint32_t bk[4];
      ldmatrix_x4(bk, kt + tma_swz<TK>(kr + nt * 8 + (lane & 7), 4 * i + (lane >> 3)));
      mma_bf16_16816(sc[nt], qa[2 * i], bk[0], bk[1]);
      mma_bf16_16816(sc[nt], qa[2 * i + 1], bk[2], bk[3]);
    }
  }
  // scale to base-2 units, mask, online softmax; row half h holds sc[nt][2h], sc[nt][2h+1]
  float alpha[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + nt * 8 + 2 * tig + e;
        const float v = key < lim[h] ? sc[nt][2 * h + e] * qscale : -INFINITY;
        sc[nt][2 * h + e] = v;
        mx = fmaxf(mx, v);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // the reference maximum moves only when the row's scores rise more than kMaxGap above
    // it (a row's first finite scores always move it), so most steps leave the accumulators'
    // scale alone; probabilities stay below 2^kMaxGap. A row with no visible key keeps -inf.
    const bool move = mx > m_run[h] + kMaxGap;
    alpha[h] = move ? exp2_approx(m_run[h] - mx) : 1.f;
    if (move) m_run[h] = mx;
    const float base = m_run[h] == -INFINITY ? 0.f : m_run[h];
    float ps = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pv = exp2_approx(sc[nt][2 * h + e] - base);
        sc[nt][2 * h + e] = pv;
        ps += pv;
      }
    l_run[h] = l_run[h] * alpha[h] + ps;
  }
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < NTD; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
  }
  const uint32_t pa[4] = {pack_bf16x2(sc[0][0], sc[0][1]), pack_bf16x2(sc[0][2], sc[0][3]),
                          pack_bf16x2(sc[1][0], sc[1][1]), pack_bf16x2(sc[1][2], sc[1][3])};
  // O += P V over these 16 keys, two 8-wide output tiles per ldmatrix
#pragma unroll
  for (int i = 0; i < NTD / 2; ++i) {
    uint32_t bv[4];
    ldmatrix_x4_trans(bv, vt + tma_swz<TK>(kr + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * i + (lane >> 4)));
    mma_bf16_16816(o[2 * i], pa, bv[0], bv[1]);
    mma_bf16_16816(o[2 * i + 1], pa, bv[2], bv[3]);
  }
}

// The same step for at most 8 query rows, with the roles of keys and rows swapped so that
// the rows fill the 8-wide n side of the tile instead of 16 rows of the m side:
//   S^T = K Q^T  (m: the 16 keys, n: the 8 rows, k: head dims; K from ldmatrix, Q^T held
//                as B fragments qb),
//   O^T += V^T P^T  (m: 16 head dims per tile, n: the rows, k: the 16 keys; V^T from
//                ldmatrix.trans, P^T from the score accumulators by one movmatrix
//                transpose per 8 keys).
// A thread holds keys gid and gid + 8 of rows 2*tig and 2*tig + 1, so a row's reductions
// run over the 8 lanes of one tig. Half the tensor-core tiles, exponentials and output
// registers of warp_keys16 when a kv head has 8 query rows or fewer (decode with grouped
// heads). o[dt] holds O^T of dims 16*dt + gid (+8) and rows 2*tig (+1).
template <int D>
__device__ __forceinline__ void warp_keys16_n8(const uint32_t (&qb)[D / 16][2], uint32_t kt, uint32_t vt, int kr,
                                               int key0, const int (&lim)[2], float qscale, float (&o)[D / 16][4],
                                               float (&m_run)[2], float (&l_run)[2]) {
  constexpr int TK = 64, KSD = D / 16;
  const int lane = threadIdx.x & 31, gid = lane >> 2;
  // two accumulators (even and odd k steps) halve the dependent chain of tensor-core tiles
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  const int krow = kr + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int j = 0; j < KSD; ++j) {
    uint32_t ak[4];
    ldmatrix_x4(ak, kt + tma_swz<TK>(krow, 2 * j + (lane >> 4)));
    mma_bf16_16816((j & 1) ? sb : sa, ak, qb[j][0], qb[j][1]);
  }
  float sc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sc[i] = sa[i] + sb[i];
  // scale to base-2 units and mask; element i is key gid + 8 * (i >> 1) of row 2*tig + (i & 1)
  float alpha[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int hk = 0; hk < 2; ++hk) {
      const int key = key0 + gid + 8 * hk;
      sc[2 * hk + e] = key < lim[e] ? sc[2 * hk + e] * qscale : -INFINITY;
    }
    float mx = fmaxf(sc[e], sc[2 + e]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    // lazy reference maximum, as in warp_keys16
    const bool move = mx > m_run[e] + kMaxGap;
    alpha[e] = move ? exp2_approx(m_run[e] - mx) : 1.f;
    if (move) m_run[e] = mx;
    const float base = m_run[e] == -INFINITY ? 0.f : m_run[e];
    const float p0 = exp2_approx(sc[e] - base), p1 = exp2_approx(sc[2 + e] - base);
    sc[e] = p0;
    sc[2 + e] = p1;
    l_run[e] = l_run[e] * alpha[e] + (p0 + p1);  // this thread's keys; lanes summed at the end
  }
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int dt = 0; dt < KSD; ++dt) {
      o[dt][0] *= alpha[0];
      o[dt][1] *= alpha[1];
      o[dt][2] *= alpha[0];
      o[dt][3] *= alpha[1];
    }
  }
  // P^T as the B operand: keys 2*tig (+1) (+8) of row gid
  const uint32_t pb0 = movmatrix_trans(pack_bf16x2(sc[0], sc[1]));
  const uint32_t pb1 = movmatrix_trans(pack_bf16x2(sc[2], sc[3]));
  const int vrow = kr + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
  for (int dt = 0; dt < KSD; ++dt) {
    uint32_t av[4];
    ldmatrix_x4_trans(av, vt + tma_swz<TK>(vrow, 2 * dt + ((lane >> 3) & 1)));
    mma_bf16_16816(o[dt], av, pb0, pb1);
  }
}

// The narrow step for 17 to 24 query rows: warp_keys16_n8's layout with three 8-wide n tiles
// (rows 8 nt .. 8 nt + 7 on tile nt), so one K and one V fragment load per 16 keys serve all
// 24 rows. A thread holds keys gid and gid + 8 of rows 8 nt + 2 tig (+1) of each tile, i.e. six
// rows, reduced over the 8 lanes that share a tig. o[nt][dt] holds O^T of dims 16 dt + gid (+8)
// and rows 8 nt + 2 tig (+1); the row limits, maxima and sums are indexed 2 nt + e.
template <int D>
__device__ __forceinline__ void warp_keys16_n24(const uint32_t (&qb)[3][D / 16][2], uint32_t kt, uint32_t vt, int kr,
                                                int key0, const int (&lim)[6], float qscale, float (&o)[3][D / 16][4],
                                                float (&m_run)[6], float (&l_run)[6]) {
  constexpr int TK = 64, KSD = D / 16;
  const int lane = threadIdx.x & 31, gid = lane >> 2;
  // three independent accumulators, one per n tile
  float sc[3][4];
#pragma unroll
  for (int nt = 0; nt < 3; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const int krow = kr + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int j = 0; j < KSD; ++j) {
    uint32_t ak[4];
    ldmatrix_x4(ak, kt + tma_swz<TK>(krow, 2 * j + (lane >> 4)));
#pragma unroll
    for (int nt = 0; nt < 3; ++nt) mma_bf16_16816(sc[nt], ak, qb[nt][j][0], qb[nt][j][1]);
  }
  // scale to base-2 units and mask; element i of tile nt is key gid + 8 (i >> 1) of row
  // 8 nt + 2 tig + (i & 1)
  float alpha[6];
#pragma unroll
  for (int nt = 0; nt < 3; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int ri = 2 * nt + e;
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        const int key = key0 + gid + 8 * hk;
        sc[nt][2 * hk + e] = key < lim[ri] ? sc[nt][2 * hk + e] * qscale : -INFINITY;
      }
      float mx = fmaxf(sc[nt][e], sc[nt][2 + e]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // lazy reference maximum, as in warp_keys16
      const bool move = mx > m_run[ri] + kMaxGap;
      alpha[ri] = move ? exp2_approx(m_run[ri] - mx) : 1.f;
      if (move) m_run[ri] = mx;
      const float base = m_run[ri] == -INFINITY ? 0.f : m_run[ri];
      const float p0 = exp2_approx(sc[nt][e] - base), p1 = exp2_approx(sc[nt][2 + e] - base);
      sc[nt][e] = p0;
      sc[nt][2 + e] = p1;
      l_run[ri] = l_run[ri] * alpha[ri] + (p0 + p1);  // this thread's keys; lanes summed at the end
    }
  }
  bool rescale = false;
#pragma unroll
  for (int ri = 0; ri < 6; ++ri) rescale |= alpha[ri] != 1.f;
  if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
    for (int nt = 0; nt < 3; ++nt)
#pragma unroll
      for (int dt = 0; dt < KSD; ++dt) {
        o[nt][dt][0] *= alpha[2 * nt];
        o[nt][dt][1] *= alpha[2 * nt + 1];
        o[nt][dt][2] *= alpha[2 * nt];
        o[nt][dt][3] *= alpha[2 * nt + 1];
      }
  }
  // P^T of each n tile as B operands: keys 2 tig (+1) (+8) of row 8 nt + gid
  uint32_t pb[3][2];
#pragma unroll
  for (int nt = 0; nt < 3; ++nt) {
    pb[nt][0] = movmatrix_trans(pack_bf16x2(sc[nt][0], sc[nt][1]));
    pb[nt][1] = movmatrix_trans(pack_bf16x2(sc[nt][2], sc[nt][3]));
  }
  const int vrow = kr + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
  for (int dt = 0; dt < KSD; ++dt) {
    uint32_t av[4];
    ldmatrix_x4_trans(av, vt + tma_swz<TK>(vrow, 2 * dt + ((lane >> 3) & 1)));
#pragma unroll
    for (int nt = 0; nt < 3; ++nt) mma_bf16_16816(o[nt][dt], av, pb[nt][0], pb[nt][1]);
  }
}

// Streams keys [c0, c1) of kv head kvh of sequence b (attended length L) for the query rows
// of row block rb through the ring at `smem` (1024-byte aligned; NST stages with barriers
// s_bars; `seq` counts the stages this CTA has consumed, for the barrier parities) and leaves
// the four warps' partial results, in base-2 units, in the combine area at the start of the
// ring, TR = tile_rows<TILE>() rows per warp: cm[4][TR] (row max), cl[4][TR] (row sum),
// ca[4][TR][CAS] (unnormalised p @ V, rows CAS = combine_stride<D>() floats apart). An empty
// range (c0 == c1) leaves empty partials.
// Returns false, CTA-uniformly, if a copy never completed: the status bit is set, the other
// copies in flight have been waited for, and the combine area holds empty partials.
// Ends with a __syncthreads.
template <int D, int NST, int TILE = kTileM16>
__device__ bool stream_chunk(const MmaArgs &a, unsigned char *smem, uint64_t *s_bars, uint32_t &seq, int b, int kvh,
                             int rb, int L, int c0, int c1) {
  using C = MmaCfg<D, NST>;
  constexpr int TR = tile_rows<TILE>();
  constexpr bool KEYS_ON_M = TILE != kTileM16;       // the narrow layouts
  constexpr int NT = TILE == kTileN24 ? 3 : 1;       // n tiles of rows (narrow layouts)
  constexpr int NL = 2 * NT;                         // query rows a thread holds
  const SplitParams &p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t sbase = smem_u32(smem);
  const int GT = p.G * p.T;
  const int nstages = (c1 - c0 + C::TK - 1) / C::TK;
  const int zc = b * p.Hkv + kvh;  // tensor-map coordinate of this (sequence, kv head)
  const uint64_t policy = l2_evict_first_policy();

  // stage sidx goes to ring buffer (seq + sidx) % NST
  auto issue = [&](int sidx) {
    const int buf = (seq + sidx) % NST;
    const uint32_t bar = smem_u32(&s_bars[buf]);
    const uint32_t kdst = sbase + buf * C::STAGE_BYTES;
    const uint32_t vdst = kdst + C::TILE_BYTES;
    const int y = c0 + sidx * C::TK;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
    for (int h = 0; h < C::HALVES; ++h) {
      tma_load_3d(kdst + h * C::BOX_BYTES, &a.kmap, 64 * h, y, zc, bar, policy);
      tma_load_3d(vdst + h * C::BOX_BYTES, &a.vmap, 64 * h, y, zc, bar, policy);
    }
  };
  // the query rows of this row block go to the K tile of the ring buffer the first stage
  // refills last; they are read into registers before that buffer is refilled
  const uint32_t qtile = sbase + ((seq + NST - 1) % NST) * C::STAGE_BYTES;
  if (p.rope_cos == nullptr) {
    for (int idx = tid; idx < TR * C::NCH; idx += kThreads) {
      const int r = idx / C::NCH, ch = idx % C::NCH;
      const int gr = rb * p.R + r;
      const bool valid = r < p.R && gr < GT;
      const int hq = kvh * p.G + (valid ? gr / p.T : 0);
      const int t = valid ? gr % p.T : 0;
      const unsigned char *qrow =
          static_cast<const unsigned char *>(p.q) + (((size_t)b * p.Hq + hq) * p.T + t) * C::ROWB;
      cp_async_16(qtile + swz<C::ROWB>(r, ch), qrow + ch * 16, valid ? 16u : 0u);
    }
  } else {
    // fused step: query row (hq, t) rotated to its position L - T + t on the way in
    constexpr int NH = C::NCH / 2;
    unsigned char *qt = smem + ((seq + NST - 1) % NST) * C::STAGE_BYTES;
    for (int idx = tid; idx < TR * NH; idx += kThreads) {
      const int r = idx / NH, ch = idx % NH;
      const int gr = rb * p.R + r;
      uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
      if (r < p.R && gr < GT) {
        const int hq = kvh * p.G + gr / p.T, t = gr % p.T;
        const uint4 *qrow = static_cast<const uint4 *>(p.q) + (((size_t)b * p.Hq + hq) * p.T + t) * C::NCH;
        lo = qrow[ch];
        hi = qrow[ch + NH];
        const size_t tab = (size_t)(L - p.T + t) * (D / 2) + ch * 8;
        rope_vec16<__nv_bfloat16>(lo, hi, p.rope_cos + tab, p.rope_sin + tab);
      }
      *reinterpret_cast<uint4 *>(qt + swz<C::ROWB>(r, ch)) = lo;
      *reinterpret_cast<uint4 *>(qt + swz<C::ROWB>(r, ch + NH)) = hi;
    }
    fence_proxy_async_smem();  // these writes precede the buffer's refill by the TMA unit
  }
  cp_async_commit();
  if (tid == 0) {
    for (int s2 = 0; s2 < min(NST - 1, nstages); ++s2) issue(s2);
  }

  // keys visible to this thread's rows of the row block: gid and gid + 8 (m16 layout), or
  // 8 nt + 2 tig and 8 nt + 2 tig + 1 of each n tile (narrow layouts)
  int lim[NL];
#pragma unroll
  for (int h = 0; h < NL; ++h) {
    const int r = KEYS_ON_M ? 8 * (h >> 1) + 2 * tig + (h & 1) : gid + 8 * h;
    const int gr = rb * p.R + r;
    const bool valid = r < p.R && gr < GT;
    lim[h] = valid ? min(max(L - p.T + gr % p.T + 1, 0), c1) : 0;
  }
  // query rows as mma A fragments (narrow: B fragments of each n tile), read once the first
  // stage lands
  uint32_t qa[NT][C::KSD][KEYS_ON_M ? 2 : 4];
  constexpr int NO = KEYS_ON_M ? C::KSD : C::NTD;  // output tiles per n tile
  float o[NT][NO][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < NO; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
  float m_run[NL], l_run[NL];
#pragma unroll
  for (int h = 0; h < NL; ++h) m_run[h] = -INFINITY, l_run[h] = 0.f;

  int consumed = 0;
  bool ok = true;
  for (int st = 0; st < nstages; ++st) {
    const int buf = (seq + st) % NST;
    const bool landed = mbar_wait_bounded(smem_u32(&s_bars[buf]), ((seq + st) / NST) & 1u);
    const int j0 = c0 + st * C::TK;
    const int valid = min(C::TK, c1 - j0);
    const uint32_t kt = sbase + buf * C::STAGE_BYTES;
    const uint32_t vt = kt + C::TILE_BYTES;
    if (landed && valid < C::TK) {
      // rows past the sequence's length were fetched (or zero-filled past Smax): zero the
      // V rows so a masked probability never meets a non-finite value
      unsigned char *vrow = smem + buf * C::STAGE_BYTES + C::TILE_BYTES;
      for (int idx = tid; idx < (C::TK - valid) * C::NCH; idx += kThreads) {
        const int r = valid + idx / C::NCH, ch = idx % C::NCH;
        *reinterpret_cast<uint4 *>(vrow + tma_swz<C::TK>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();  // these writes precede the buffer's next refill by the TMA unit
    }
    if (landed && p.k_new != nullptr) place_new_rows<D, NST>(p, smem + buf * C::STAGE_BYTES, b, kvh, rb, L, j0, valid);
    if (st == 0) cp_async_wait<0>();  // this thread's part of the query tile
    // one decision for the whole CTA: a thread whose wait gave up stops every thread
    if (!__syncthreads_and(landed)) {
      ok = false;
      break;
    }
    if (st == 0) {
      if constexpr (KEYS_ON_M) {
        // rows 8 nt .. 8 nt + 7: matrices of 16-byte chunks 4j .. 4j+3 are B words of k steps
        // 2j, 2j+1
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < C::KSD / 2; ++j) {
            uint32_t w[4];
            ldmatrix_x4(w, qtile + swz<C::ROWB>(8 * nt + (lane & 7), 4 * j + (lane >> 3)));
            qa[nt][2 * j][0] = w[0];
            qa[nt][2 * j][1] = w[1];
            qa[nt][2 * j + 1][0] = w[2];
            qa[nt][2 * j + 1][1] = w[3];
          }
      } else {
#pragma unroll
        for (int j = 0; j < C::KSD; ++j)
          ldmatrix_x4(qa[0][j], qtile + swz<C::ROWB>(((lane >> 3) & 1) * 8 + (lane & 7), 2 * j + (lane >> 4)));
      }
      __syncthreads();  // every warp holds its query fragments before that buffer is refilled
    }
    if (tid == 0 && st + NST - 1 < nstages) issue(st + NST - 1);
    const int kr = warp * C::TKW;  // first key row (within the stage) of this warp's step
    const int key0 = j0 + kr;
    if (key0 < c1) {
      if constexpr (TILE == kTileN24)
        warp_keys16_n24<D>(qa, kt, vt, kr, key0, lim, p.qscale, o, m_run, l_run);
      else if constexpr (TILE == kTileN8)
        warp_keys16_n8<D>(qa[0], kt, vt, kr, key0, lim, p.qscale, o[0], m_run, l_run);
      else
        warp_keys16<D>(qa[0], kt, vt, kr, key0, lim, p.qscale, o[0], m_run, l_run);
    }
    consumed = st + 1;
  }
  if (!ok) {
    // a copy never completed: wait (bounded) for this chunk's copies in flight, then drop it
    const int issued = min(nstages, consumed + NST - 1);
    for (int st = consumed; st < issued; ++st)
      mbar_wait_bounded(smem_u32(&s_bars[(seq + st) % NST]), ((seq + st) / NST) & 1u);
    if (tid == 0) report(p.status, TD_DEV_WAIT_TIMEOUT);
#pragma unroll
    for (int h = 0; h < NL; ++h) m_run[h] = -INFINITY, l_run[h] = 0.f;
  }
  cp_async_wait<0>();
  seq += nstages;
#pragma unroll
  for (int h = 0; h < NL; ++h) {
    if constexpr (KEYS_ON_M) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
    } else {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
  }
  __syncthreads();  // ring idle: reuse it as the combine area
  constexpr int CAS = combine_stride<D>();
  float *combine = reinterpret_cast<float *>(smem);
  float *cm = combine;
  float *cl = combine + kWarps * TR;
  float *ca = combine + 2 * kWarps * TR;
  if constexpr (KEYS_ON_M) {
    // rows 8 nt + 2 tig + e (the narrow n8 layout leaves rows 8..15 of its area unused)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 8 * nt + 2 * tig + e;
        if (gid == 0) {
          cm[warp * TR + r] = m_run[2 * nt + e];
          cl[warp * TR + r] = l_run[2 * nt + e];
        }
        float *row = &ca[(warp * TR + r) * CAS];
#pragma unroll
        for (int dt = 0; dt < C::KSD; ++dt) {
          row[16 * dt + gid] = o[nt][dt][e];
          row[16 * dt + gid + 8] = o[nt][dt][2 + e];
        }
      }
    __syncthreads();
    return ok;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = gid + 8 * h;
    if (tig == 0) {
      cm[warp * TR + r] = m_run[h];
      cl[warp * TR + r] = l_run[h];
    }
#pragma unroll
    for (int nt = 0; nt < C::NTD; ++nt) {
      float2 v = make_float2(o[0][nt][2 * h], o[0][nt][2 * h + 1]);
      *reinterpret_cast<float2 *>(&ca[(warp * TR + r) * CAS + nt * 8 + 2 * tig]) = v;
    }
  }
  __syncthreads();
  return ok;
}

// Warms L2 with the first `n` stages (of 64 rows) of K and V of keys [c0, c1) of (b, kvh):
// bf16 rows, or for 8-bit caches (Q8) the code rows and their scales.
template <int D, bool Q8 = false>
__device__ void prefetch_chunk_l2(const SplitParams &p, int b, int kvh, int c0, int c1, int n) {
  constexpr int ROWB = Q8 ? D : D * 2, TK = 64;
  const size_t row0 = ((size_t)b * p.Hkv + kvh) * p.Smax + c0;
  const unsigned char *k = static_cast<const unsigned char *>(p.k) + row0 * ROWB;
  const unsigned char *v = static_cast<const unsigned char *>(p.v) + row0 * ROWB;
  constexpr int kPiece = 65536 / ROWB;  // rows per prefetch instruction (64 KB)
  const int rows = min(c1 - c0, n * TK);
  for (int r = 0; r < rows; r += kPiece) {
    const uint32_t bytes = (uint32_t)min(kPiece, rows - r) * ROWB;
    prefetch_l2_bulk(k + (size_t)r * ROWB, bytes);
    prefetch_l2_bulk(v + (size_t)r * ROWB, bytes);
  }
  if constexpr (Q8) {
    // the whole 16-byte units holding the rows' scales (a sequence's Smax scales are a whole
    // number of 16-byte units, so these stay inside its own)
    const float *sc[2] = {p.k_scales + row0, p.v_scales + row0};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(sc[i]) & ~(uintptr_t)15;
      const uintptr_t a1 = (reinterpret_cast<uintptr_t>(sc[i] + rows) + 15) & ~(uintptr_t)15;
      prefetch_l2_bulk(reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0));
    }
  }
}

// Run by one thread before the wait for the previous kernel in the stream, whose writes
// (seq_lens among them) may not be visible yet: a guess of this CTA's first work item from
// the lengths as they read now, the same arithmetic as plan_items without its overshoot
// check, and an L2 prefetch of that chunk's first `n` stages, so the HBM latency of the
// first stages overlaps the previous kernel's tail. A hint only: a wrong guess wastes a
// prefetch, and the real plan is made after the wait. Batches of up to 8 sequences.
// `item` is the CTA's first work item; a cluster of `parts` CTAs shares each item, this CTA
// taking run `part` of its whole 64-key stages (as split_attn_cc_kernel cuts it).
template <int D, bool Q8 = false>
__device__ void prefetch_first_item(const SplitParams &p, int n, int item, int part = 0, int parts = 1) {
  if (p.B > 8) return;
  long long all = 0;
  int longest = 0, first = 0;
  uint32_t bits = 0;
  for (int b = 0; b < p.B; ++b) {
    const int L = attended_len(p, ld_relaxed(p.seq_lens + b), bits);
    if (b == 0) first = L;
    all += L;
    longest = max(longest, L);
  }
  const int S = first_chunk_size(p, all, longest);
  const int U = p.Hkv * p.RB;
  for (int b = 0; b < p.B; ++b) {
    // (a second read of the later lengths: still a guess)
    const int L = b == 0 ? first : attended_len(p, ld_relaxed(p.seq_lens + b), bits);
    const int NC = (L + S - 1) / S;
    if (item < NC * U) {
      const int c = item % NC, kvh = item / NC / p.RB;
      const int c0 = c * S, c1 = min(c0 + S, L);
      const int per = ((c1 - c0 + parts - 1) / parts + 63) / 64 * 64;
      const int r0 = min(c0 + part * per, c1);
      prefetch_chunk_l2<D, Q8>(p, b, kvh, r0, min(r0 + per, c1), n);
      return;
    }
    item -= NC * U;
  }
}

// Aligns the dynamic shared memory to 1024 bytes (the 128-byte swizzle is a function of the
// address); the allocation carries 1024 bytes of slack for this.
__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Persistent kernel: CTAs walk the work items of plan_items; chunk partials meet in the
// workspace and the CTA that completes a group's last chunk merges them (finish_item).
// EARLY_PLAN (launched when one row block covers a kv head, i.e. decode): the plan is made
// on the lengths as they read before the wait for the previous kernel and kept after it if
// they read the same then (measured on the 3B-style layer: 4k 11.4 -> 10.5 us, 32k 25.7 ->
// 25.5 us). The other instantiation plans after the wait. TILE: the warps' step for the row
// block's rows (tile_of_rows).
template <int D, bool EARLY_PLAN, int TILE = kTileM16>
__global__ void __launch_bounds__(kThreads, 2) split_attn_mma_kernel(const __grid_constant__ MmaArgs a) {
  constexpr int NST = kPersistentStages<D>;
  using C = MmaCfg<D, NST>;
  using E = __nv_bfloat16;
  constexpr int TR = tile_rows<TILE>();
  static_assert((merge_fixed_floats<D, TR>() + part_block_floats(TR, D)) * 4 <= C::RING_BYTES,
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
  if (tid == 0) prefetch_first_item<D>(p, prefetch_stages(p), blockIdx.x);
  if constexpr (EARLY_PLAN) plan_items(p, s_len, s_prefix, &s_chunk, s_red, false);
  griddep_wait();  // inputs may come from the previous kernel in the stream
  griddep_launch_dependents();
  if constexpr (EARLY_PLAN)
    confirm_plan(p, s_len, s_prefix, &s_chunk, s_red);  // ends with __syncthreads
  else
    plan_items(p, s_len, s_prefix, &s_chunk, s_red);  // ends with __syncthreads
  advance_after_reads(p, &s_last);  // fused step: the lengths move on once every CTA has read them
  const int S = s_chunk;
  const int W = s_prefix[p.B];
  const int rows = p.Hq * p.T;

  // sequences with no key get no item: their rows are 0 with lse = -inf
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
    const bool ok = stream_chunk<D, NST, TILE>(a, smem, s_bars, seq, b, kvh, rb, L, c0, min(c0 + S, L));
    finish_item<E, D, TR, kWarps, combine_stride<D>()>(p, combine, C::RING_BYTES / 4, &s_merge_bar, merge_phase, b, kvh,
                                                       rb, c, NC, &s_last, W <= (int)gridDim.x);
    // the combine and merge wrote the ring through the generic proxy; the next item's first
    // stages refill it through the asynchronous proxy
    fence_proxy_async_smem();
    __syncthreads();
    if (!ok) break;  // a copy never completed: stop taking items
  }
}

// Combines the kWarps partial sources left by stream_chunk (base-2 units, TR rows per warp)
// into one partial block at `dst` (generic address, possibly another CTA's shared memory):
// acc[R][D], then m[R] (natural-log units) and l[R], for rows r < nv.
template <int D, int TR>
__device__ void combine_block(const float *combine, float *dst, int R, int nv) {
  constexpr int D4 = D / 4, CAS = combine_stride<D>();
  const float *cm = combine;
  const float *cl = combine + kWarps * TR;
  const float *ca = combine + 2 * kWarps * TR;
  for (int idx = threadIdx.x; idx < nv * D4; idx += kThreads) {
    const int r = idx / D4, d = (idx % D4) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * TR + r]);
    float Ls = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = cm[w * TR + r];
        if (mw != -INFINITY) {
          const float f = exp2f(mw - M);
          Ls = fmaf(cl[w * TR + r], f, Ls);
          const float4 v = *reinterpret_cast<const float4 *>(ca + (w * TR + r) * CAS + d);
          A.x = fmaf(v.x, f, A.x), A.y = fmaf(v.y, f, A.y), A.z = fmaf(v.z, f, A.z), A.w = fmaf(v.w, f, A.w);
        }
      }
    }
    *reinterpret_cast<float4 *>(dst + r * D + d) = A;
    if (d == 0) {
      dst[R * D + r] = Ls > 0.f ? M * kLn2 : -INFINITY;
      dst[R * D + R + r] = Ls;
    }
  }
}

}  // namespace td
