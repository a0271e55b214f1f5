// Split-KV attention for bf16 caches on the tensor cores.
//
// Same method and work decomposition as split_attn_kernel ("tinydecode", section "how the
// decode step is put together"; "llm-decode-cuda", split-KV attention section): one CTA
// per (sequence, kv head, row block, chunk) item computes the chunk's partial softmax for
// every query row reading that kv head, and chunks are merged by log-sum-exp.
//
// The grouped-query rows of a kv head (G heads x T verify tokens, up to 32 per CTA) form
// the M side of mma.sync m16n8k16 tiles, so each K/V tile loaded into shared memory is
// read once for all of them:
//   scores  S[rows x 16 keys] = Q[rows x D] . K^T   (B operand from K rows via ldmatrix)
//   output  O[rows x D]      += P[rows x 16 keys] . V (B operand via ldmatrix.trans)
// with fp32 accumulation; P is rounded to bf16 for the second product while the softmax
// statistics (m, l) stay fp32. K/V stages of 64 rows are copied with 16-byte cp.async
// (zero-filled past the chunk end) into tiles whose 16-byte chunks are XOR-swizzled by
// row, so the 8 rows an ldmatrix reads sit in 8 different bank groups. Warps are arranged
// as (m tile, key slice): with one m tile the 4 warps split every stage's keys 4 ways,
// with two m tiles 2 ways; warps combine at the end of the item.
#pragma once

#include "td_mma.cuh"
#include "td_split_attn.cuh"

namespace td {

template <int D, int MT>
struct MmaCfg {
  static constexpr int KS = kWarps / MT;      // key slices (warps sharing one m tile)
  static constexpr int ROWS = 16 * MT;        // query rows per CTA
  static constexpr int TK = 64;               // keys per pipeline stage
  static constexpr int TKW = TK / KS;         // keys per warp per stage
  static constexpr int NKSTEP = TKW / 16;     // 16-key steps per warp per stage
  static constexpr int ROWB = D * 2;          // bytes per cache row
  static constexpr int NCH = ROWB / 16;       // 16-byte chunks per cache row
  static constexpr int NST = D == 128 ? 3 : 4;
  static constexpr int TILE_BYTES = TK * ROWB;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES;
  static constexpr int NTD = D / 8;           // 8-wide output n tiles
  static constexpr int KSD = D / 16;          // 16-deep score k steps
  static constexpr int COMBINE_FLOATS = KS * ROWS * (D + 2);
  static_assert(TKW % 16 == 0, "each warp takes whole 16-key steps");
  static_assert(COMBINE_FLOATS * 4 <= SMEM_BYTES, "combine area fits in the ring");
  static_assert((merge_fixed_floats<D, ROWS>() + part_block_floats(ROWS, D)) * 4 <= SMEM_BYTES,
                "merge stages at least one chunk");
  static_assert(ROWS * D * 2 <= TILE_BYTES, "the query tile fits in one K tile");
  static constexpr bool kFits = SMEM_BYTES + 8448 <= 227 * 1024;
};

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * ROWB + ((ch ^ (row & 7)) << 4));
}

template <int D, int MT>
__global__ void __launch_bounds__(kThreads, 2) split_attn_mma_kernel(const SplitParams p) {
  using C = MmaCfg<D, MT>;
  using E = __nv_bfloat16;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_len[TD_MAX_BATCH];
  __shared__ int s_prefix[TD_MAX_BATCH + 1];
  __shared__ long long s_red[2 * kWarps];
  __shared__ int s_chunk, s_last;
  __shared__ __align__(8) uint64_t s_merge_bar;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int mt = warp / C::KS, ks = warp % C::KS;
  const uint32_t sbase = smem_u32(smem);
  float *combine = reinterpret_cast<float *>(smem);
  if (tid == 0) {
    mbar_init(smem_u32(&s_merge_bar), 1);
    fence_mbar_init();
  }
  uint32_t merge_phase = 0;
  griddep_wait();  // inputs may come from the previous kernel in the stream
  griddep_launch_dependents();
  plan_items(p, s_len, s_prefix, &s_chunk, s_red);  // ends with __syncthreads
  const int S = s_chunk;
  const int W = s_prefix[p.B];
  const int rows = p.Hq * p.T;
  const int GT = p.G * p.T;

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
    const int c1 = min(c0 + S, L);
    const int nstages = (c1 - c0 + C::TK - 1) / C::TK;
    const size_t head_off = ((size_t)b * p.Hkv + kvh) * (size_t)p.Smax * C::ROWB;
    const unsigned char *kg = static_cast<const unsigned char *>(p.k) + head_off;
    const unsigned char *vg = static_cast<const unsigned char *>(p.v) + head_off;

    auto load_stage = [&](int sidx) {
      const int j0 = c0 + sidx * C::TK;
      const int valid = min(C::TK, c1 - j0);
      const uint32_t kdst = sbase + (sidx % C::NST) * C::STAGE_BYTES;
      const uint32_t vdst = kdst + C::TILE_BYTES;
#pragma unroll 4
      for (int idx = tid; idx < C::TK * C::NCH; idx += kThreads) {
        const int row = idx / C::NCH, ch = idx % C::NCH;
        const bool ok = row < valid;
        const size_t off = (size_t)(j0 + (ok ? row : 0)) * C::ROWB + ch * 16;
        const uint32_t so = swz<C::ROWB>(row, ch);
        cp_async_16(kdst + so, kg + off, ok ? 16u : 0u);
        cp_async_16(vdst + so, vg + off, ok ? 16u : 0u);
      }
    };
    // the query rows of this row block go, swizzled like a K tile, to the K tile of the last
    // ring buffer, which no stage fills before the first stage has been consumed
    const uint32_t qtile = sbase + (C::NST - 1) * C::STAGE_BYTES;
    for (int idx = tid; idx < C::ROWS * C::NCH; idx += kThreads) {
      const int r = idx / C::NCH, ch = idx % C::NCH;
      const int gr = rb * p.R + r;
      const bool valid = r < p.R && gr < GT;
      const int hq = kvh * p.G + (valid ? gr / p.T : 0);
      const int t = valid ? gr % p.T : 0;
      const unsigned char *qrow =
          static_cast<const unsigned char *>(p.q) + (((size_t)b * p.Hq + hq) * p.T + t) * C::ROWB;
      cp_async_16(qtile + swz<C::ROWB>(r, ch), qrow + ch * 16, valid ? 16u : 0u);
    }
#pragma unroll
    for (int s2 = 0; s2 < C::NST - 1; ++s2) {
      if (s2 < nstages) load_stage(s2);
      cp_async_commit();
    }

    // keys visible to rows r0 = 16*mt + gid and r1 = r0 + 8 of this row block
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = mt * 16 + gid + 8 * h;
      const int gr = rb * p.R + r;
      const bool valid = r < p.R && gr < GT;
      lim[h] = valid ? min(max(L - p.T + gr % p.T + 1, 0), c1) : 0;
    }
    uint32_t qa[C::KSD][4];  // query rows as mma A fragments, read once the first group lands

    float o[C::NTD][4];
#pragma unroll
    for (int nt = 0; nt < C::NTD; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int st = 0; st < nstages; ++st) {
      cp_async_wait<C::NST - 2>();
      __syncthreads();
      if (st == 0) {
#pragma unroll
        for (int j = 0; j < C::KSD; ++j)
          ldmatrix_x4(qa[j], qtile + swz<C::ROWB>(mt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * j + (lane >> 4)));
        __syncthreads();  // every warp holds its query fragments before the buffer is refilled
      }
      if (st + C::NST - 1 < nstages) load_stage(st + C::NST - 1);
      cp_async_commit();
      const uint32_t kt = sbase + (st % C::NST) * C::STAGE_BYTES;
      const uint32_t vt = kt + C::TILE_BYTES;
      const int j0 = c0 + st * C::TK;
#pragma unroll
      for (int kk = 0; kk < C::NKSTEP; ++kk) {
        const int kr = ks * C::TKW + kk * 16;  // first key row (within the stage) of this step
        const int key0 = j0 + kr;
        if (key0 >= c1) break;
        // S = Q K^T over 16 keys: two 8-key n tiles
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
          for (int i = 0; i < C::KSD / 2; ++i) {
            uint32_t bk[4];
            ldmatrix_x4(bk, kt + swz<C::ROWB>(kr + nt * 8 + (lane & 7), 4 * i + (lane >> 3)));
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
              const float v = key < lim[h] ? sc[nt][2 * h + e] * p.qscale : -INFINITY;
              sc[nt][2 * h + e] = v;
              mx = fmaxf(mx, v);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float m_new = fmaxf(m_run[h], mx);
          const float base = m_new == -INFINITY ? 0.f : m_new;
          alpha[h] = exp2f(m_run[h] - base);
          m_run[h] = m_new;
          float ps = 0.f;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float pv = exp2f(sc[nt][2 * h + e] - base);
              sc[nt][2 * h + e] = pv;
              ps += pv;
            }
          l_run[h] = l_run[h] * alpha[h] + ps;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int nt = 0; nt < C::NTD; ++nt) {
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
        for (int i = 0; i < C::NTD / 2; ++i) {
          uint32_t bv[4];
          ldmatrix_x4_trans(bv, vt + swz<C::ROWB>(kr + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * i + (lane >> 4)));
          mma_bf16_16816(o[2 * i], pa, bv[0], bv[1]);
          mma_bf16_16816(o[2 * i + 1], pa, bv[2], bv[3]);
        }
      }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    __syncthreads();  // ring idle: reuse it as the combine area
    float *cm = combine;
    float *cl = combine + C::KS * C::ROWS;
    float *ca = combine + 2 * C::KS * C::ROWS;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = mt * 16 + gid + 8 * h;
      if (tig == 0) {
        cm[ks * C::ROWS + r] = m_run[h];
        cl[ks * C::ROWS + r] = l_run[h];
      }
#pragma unroll
      for (int nt = 0; nt < C::NTD; ++nt) {
        float2 v = make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
        *reinterpret_cast<float2 *>(&ca[(ks * C::ROWS + r) * D + nt * 8 + 2 * tig]) = v;
      }
    }
    __syncthreads();
    finish_item<E, D, C::ROWS, C::KS>(p, combine, C::SMEM_BYTES / 4, &s_merge_bar, merge_phase, b, kvh, rb, c, NC,
                                      &s_last);
  }
}

}  // namespace td
