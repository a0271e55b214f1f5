// Tiled causal prefill attention on the fifth-generation tensor cores (tcgen05, TMEM, TMA).
//
// Method ("tinydecode": prefill is the causal attention path over the prompt; "llm-decode-cuda"
// names "a tiled FlashAttention-style kernel" as its next step for prefill): for every query
// row t of a chunk of T tokens on top of the cache (seq_lens[b] = L counting them), the exact
// softmax attention over keys j < L - T + t + 1, the same result td_verify_attn defines,
// computed tile by tile with an online softmax.
//
// GB300 design: one CTA per tile of 128 query rows of one query head, two CTAs per SM. Q, K
// and V tiles cross by TMA with the 128-byte swizzle (K and V double-buffered with their own
// barriers, 64 keys per tile). A fifth warp issues the tensor-core products and a sixth the
// copies (a copy waits for its buffer's previous product, which must not hold up the next
// product's issue); the accumulators live in TMEM (256 columns: S in [0, 64), P buffers in
// [64, 96) and [96, 128), O from column 128):
//   S[128 x 64] = Q K^T     (A = Q, B = K, both K-major in shared memory)  -> S columns
//   O[128 x D] += P V       (A = P in TMEM, B = V MN-major in shared memory) -> O
// Each softmax thread owns one query row (its TMEM lane): it reads its 64 scores once and at
// once releases the S columns (an "S free" barrier, one arrival per warp), so the product S of
// tile kt+1 runs while the four softmax warps work on tile kt. It masks the scores causally
// (only in tiles that reach the diagonal or the sequence's end) and writes P = 2^(s - m) as
// bf16 pairs into P buffer kt % 2 once the P V product of tile kt-2 has read it; the P V
// product reads P as its A operand (lane = row, one column per pair of keys). A softmax warp
// hands its rows over through an mbarrier (one arrival per warp), so the warps do not wait
// for one another within a tile. The reference maximum m moves only when a row's maximum
// rises more than 8 (base 2) above it, and only then are that row's O and l rescaled (after
// the previous P V product is complete); otherwise P stays below 2^8 and O / l, kept against
// the same m, need no correction. Query tiles are launched longest first (causal rows late in
// the prompt see the most keys). Every wait is bounded; a timeout sets TD_DEV_WAIT_TIMEOUT,
// and the CTA waits (bounded) for its copies and products in flight before it frees TMEM.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "td_device.cuh"
#include "td_internal.h"
#include "td_mma.cuh"

namespace td {

namespace {

constexpr int kPfSoftmaxWarps = 4;                         // one query row per thread
constexpr int kPfMmaWarp = kPfSoftmaxWarps;                  // issues the tensor-core products
constexpr int kPfLoadWarp = kPfSoftmaxWarps + 1;             // issues the TMA copies
constexpr int kPfThreads = 32 * (kPfSoftmaxWarps + 2);
constexpr int kPfRows = 128;   // query rows per CTA
constexpr int kPfKeys = 64;    // keys per tile
constexpr int kQRegion = kPfRows * 128;  // bytes of one swizzled [128 rows][64 bf16] region
constexpr int kKRegion = kPfKeys * 128;  // bytes of one swizzled [64 rows][64 bf16] region
constexpr float kRescaleGap = 8.f;       // base-2 rise of a row maximum before m moves

template <int D>
struct PfCfg {
  static constexpr int HALVES = D / 64;                 // 64-column regions per row tile
  static constexpr int Q_TILE = HALVES * kQRegion;
  static constexpr int KV_TILE = HALVES * kKRegion;     // one K or V tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_TILE;                  // two K buffers
  static constexpr int V_OFF = K_OFF + 2 * KV_TILE;     // two V buffers
  static constexpr int SMEM = V_OFF + 2 * KV_TILE + 1024;  // + alignment slack
  static constexpr int TMEM_COLS = 256;                 // S (64), two P buffers (32 each), O (D): a power of two
  static_assert(2 * (SMEM + 1024 + 128) <= 228 * 1024, "two CTAs per SM");
};

struct PfArgs {
  CUtensorMap qmap;  // q [B*Hq][T][D]
  CUtensorMap kmap;  // caches [B*Hkv][Smax][D], boxes of 64 rows
  CUtensorMap vmap;
  const int32_t *seq_lens;
  void *out;         // [B, Hq, T, D] bf16
  float *lse;        // [B, Hq, T] or null
  uint32_t *status;
  int B, Hq, Hkv, T, Smax;
  float qscale;      // scale * log2(e)
};

__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap *m, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(m), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading and stride byte
// offsets (K-major: the stride between 8-row groups; MN-major: leading = the stride between
// 64-column regions, stride = between 8-row groups), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, A K-major, B K- or
// MN-major, M x N.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// The same with A in TMEM (`a_tmem`: lane = row, one 32-bit column per pair of K elements).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 64 consecutive fp32 columns of this thread's TMEM lane: two loads and their wait in one
// statement, so no use of the registers can be placed before the wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&w)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31]) : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
  tmem_st32(taddr, w);
}

// One row's probabilities 2^(s * qscale + nbase) for the 64 scores sv, packed in bf16 pairs
// into pk; MASK: keys from `vis` on get 0. Returns their fp32 sum (in packed pairs, two
// partial sums, so the additions do not form one chain).
template <bool MASK>
__device__ __forceinline__ float p_row(const float (&sv)[kPfKeys], float qscale, float nbase, int vis,
                                       uint32_t (&pk)[kPfKeys / 2]) {
  float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 sc2 = make_float2(qscale, qscale), nb2 = make_float2(nbase, nbase);
#pragma unroll
  for (int i = 0; i < kPfKeys; i += 2) {
    const float2 x = ffma2(make_float2(sv[i], sv[i + 1]), sc2, nb2);
    float2 pr = make_float2(exp2_approx(x.x), exp2_approx(x.y));
    if (MASK) {
      pr.x = i < vis ? pr.x : 0.f;
      pr.y = i + 1 < vis ? pr.y : 0.f;
    }
    l2[(i >> 1) & 1] = fadd2(l2[(i >> 1) & 1], pr);
    pk[i / 2] = pack_bf16x2(pr.x, pr.y);
  }
  const float2 t = fadd2(l2[0], l2[1]);
  return t.x + t.y;
}

// The largest (MIN: smallest) of a row's 64 scores.
template <bool MIN>
__device__ __forceinline__ float row_extreme(const float (&sv)[kPfKeys]) {
  float e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float *v = sv + 8 * j;
    e[j] = MIN ? fmin3f(fmin3f(v[0], v[1], v[2]), fmin3f(v[3], v[4], v[5]), fminf(v[6], v[7]))
               : fmax3f(fmax3f(v[0], v[1], v[2]), fmax3f(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
  }
  return MIN ? fmin3f(fmin3f(e[0], e[1], e[2]), fmin3f(e[3], e[4], e[5]), fminf(e[6], e[7]))
             : fmax3f(fmax3f(e[0], e[1], e[2]), fmax3f(e[3], e[4], e[5]), fmaxf(e[6], e[7]));
}

// Byte offset of 16-byte chunk c of row r in a tile of `rows` rows kept as 128-byte-swizzled
// regions of 64 bf16 columns (the layout TMA writes and the tensor core reads as K-major).
__device__ __forceinline__ uint32_t tile_chunk(int rows, int r, int c) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 2) prefill_kernel(const __grid_constant__ PfArgs a) {
  using C = PfCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_k[2], bar_v[2], bar_s[2], bar_sfree, bar_p[2], bar_vfree[2], bar_o,
      bar_fin;
  __shared__ uint32_t s_taddr;
  __shared__ int s_issued[2], s_seen[3];  // wind-down: K / V tiles issued; K / V tiles, Q seen landed
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  // blocks start in index order, x fastest: every head's tile late in the prompt (most keys)
  // comes before any shorter one
  const int qt = gridDim.y - 1 - blockIdx.y;
  const int hq = blockIdx.x % a.Hq, b = blockIdx.x / a.Hq;
  const int G = a.Hq / a.Hkv, kvh = hq / G;
  const int t0 = qt * kPfRows;

  if (tid == 0) {
    mbar_init(smem_u32(&bar_q), 1);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_k[i]), 1);
      mbar_init(smem_u32(&bar_v[i]), 1);
      mbar_init(smem_u32(&bar_s[i]), 1);
      mbar_init(smem_u32(&bar_p[i]), kPfSoftmaxWarps);
      mbar_init(smem_u32(&bar_vfree[i]), 1);
    }
    s_issued[0] = s_issued[1] = 0;
    s_seen[0] = s_seen[1] = 0;
    s_seen[2] = 1;
    mbar_init(smem_u32(&bar_sfree), kPfSoftmaxWarps);
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_fin), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_taddr)),
                 "n"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_taddr;
  // S of the current tile in columns [0, 64), P of tile kt in P buffer kt % 2 (columns 64 + 32 (kt % 2),
  // bf16 pairs), O in [128, 128 + D)
  const uint32_t tS = tmem, tP = tmem + kPfKeys, tO = tmem + 128;

  griddep_wait();
  griddep_launch_dependents();
  const int32_t raw = a.seq_lens[b];
  const int L = raw < 0 ? 0 : (raw > a.Smax ? a.Smax : raw);
  const int last_t = min(t0 + kPfRows, a.T) - 1;
  const int kend = max(0, min(L, L - a.T + last_t + 1));  // keys any row of the tile sees
  const int kall = max(0, min(L, L - a.T + t0 + 1));      // keys every row of the tile sees
  const int nkt = (kend + kPfKeys - 1) / kPfKeys;
  if (tid == 0 && qt == 0 && hq == 0) {
    uint32_t bits = 0;
    if (raw < 0) bits |= TD_DEV_NEGATIVE_SEQLEN;
    if (raw > a.Smax) bits |= TD_DEV_SEQLEN_CLAMPED;
    if (a.T > 1 && L < a.T) bits |= TD_DEV_VERIFY_SHORT;
    report(a.status, bits);
  }
  const float qscale = a.qscale;
  bool ok = true;
  // copy / tensor-core thread: tiles of K and V issued and seen landed (for the wind-down)
  int kq = 0, kw = 0, vq = 0, vw = 0;
  bool q_seen = false;
  float m_ref = -INFINITY, l = 0.f;  // softmax threads: this row's reference maximum and sum

  if (warp == kPfMmaWarp) {
    if (lane == 0 && nkt > 0) {
      constexpr uint32_t kIdS = mma_idesc(kPfRows, kPfKeys, false);
      constexpr uint32_t kIdO = mma_idesc(kPfRows, D, true);
      // shared-memory descriptors of Q and of K / V buffer 0; any other tile, buffer or k
      // step differs only in its start address (descriptor field in 16-byte units)
      const uint64_t dq = smem_desc(sb + C::Q_OFF, 16, 1024);
      const uint64_t dk = smem_desc(sb + C::K_OFF, 16, 1024);
      const uint64_t dv = smem_desc(sb + C::V_OFF, kKRegion, 1024);
      // S of tile kt into the S columns (K tile kt has landed; its completion is signalled on
      // the barrier of K buffer kt % 2): over D in steps of 16 (32 bytes along a swizzled row;
      // the next 64 columns are the next region)
      auto issue_s = [&](int kt) {
        const uint32_t kb = (uint32_t)(kt & 1) * C::KV_TILE;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k & 3) * 32;
          tc_mma(tS, dq + (((uint32_t)(k >> 2) * kQRegion + off) >> 4),
                 dk + ((kb + (uint32_t)(k >> 2) * kKRegion + off) >> 4), kIdS, k > 0);
        }
        tc_commit(smem_u32(&bar_s[kt & 1]));
      };
      q_seen = mbar_wait_bounded(smem_u32(&bar_q), 0);
      ok = q_seen && mbar_wait_bounded(smem_u32(&bar_k[0]), 0);
      if (ok) {
        kw = 1;
        issue_s(0);
      }
      for (int kt = 0; ok && kt < nkt; ++kt) {
        const int b0 = kt & 1, b1 = b0 ^ 1;
        if (kt + 1 < nkt) {
          // the S columns are free once every softmax warp has read S of kt
          ok = mbar_wait_bounded(smem_u32(&bar_sfree), (uint32_t)kt & 1u);
          ok = ok && mbar_wait_bounded(smem_u32(&bar_k[b1]), (uint32_t)((kt + 1) >> 1) & 1u);
          if (!ok) break;
          kw = kt + 2;
          issue_s(kt + 1);
        }
        // P of kt is in P buffer b0 (all four softmax warps) and V of kt has landed: O += P V
        // over 64 keys in steps of 16 (A: 8 TMEM columns per step; B: MN-major, 16 rows of 128
        // bytes per step, the next 64 columns in the next region)
        ok = mbar_wait_bounded(smem_u32(&bar_p[b0]), (uint32_t)(kt >> 1) & 1u) &&
             mbar_wait_bounded(smem_u32(&bar_v[b0]), (uint32_t)(kt >> 1) & 1u);
        if (!ok) break;
        vw = kt + 1;
        tc_fence_after();
        const uint32_t vb = (uint32_t)b0 * C::KV_TILE;
#pragma unroll
        for (int k = 0; k < kPfKeys / 16; ++k)
          tc_mma_ts(tO, tP + b0 * (kPfKeys / 2) + 8 * k, dv + ((vb + (uint32_t)k * 16 * 128) >> 4), kIdO, kt > 0 || k > 0);
        tc_commit(smem_u32(&bar_o));
        tc_commit(smem_u32(&bar_vfree[b0]));  // V buffer b0 may be refilled, P buffer b0 rewritten
      }
      s_seen[0] = kw;
      s_seen[1] = vw;
      s_seen[2] = q_seen;
    }
    __syncwarp();
  } else if (warp == kPfLoadWarp) {
    if (lane == 0 && nkt > 0) {
      const int zq = b * a.Hq + hq, zk = b * a.Hkv + kvh;
      auto load = [&](bool v, int kt) {  // K or V tile kt into buffer kt % 2
        const int buf = kt & 1;
        const uint32_t bar = smem_u32(v ? &bar_v[buf] : &bar_k[buf]);
        const uint32_t dst = sb + (v ? C::V_OFF : C::K_OFF) + buf * C::KV_TILE;
        mbar_arrive_expect_tx(bar, C::KV_TILE);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) tma3(dst + h * kKRegion, v ? &a.vmap : &a.kmap, 64 * h, kt * kPfKeys, zk, bar);
      };
      {
        const uint32_t bar = smem_u32(&bar_q);
        mbar_arrive_expect_tx(bar, C::Q_TILE);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) tma3(sb + C::Q_OFF + h * kQRegion, &a.qmap, 64 * h, t0, zq, bar);
      }
      for (; kq < min(nkt, 2); ++kq) {
        load(false, kq);
        load(true, kq);
      }
      vq = kq;
      // tile j (j >= 2) goes to buffer j % 2 once its previous user, tile j-2, is done with
      // it: K after the product S of j-2, V after the P V product of j-2. Each buffer's next
      // product needs the copy issued here, so its barrier cannot run a phase ahead.
      for (int j = 2; ok && j < nkt; ++j) {
        const uint32_t ph = (uint32_t)((j - 2) >> 1) & 1u;
        ok = mbar_wait_bounded(smem_u32(&bar_s[j & 1]), ph);
        if (!ok) break;
        load(false, kq++);
        ok = mbar_wait_bounded(smem_u32(&bar_vfree[j & 1]), ph);
        if (!ok) break;
        load(true, vq++);
      }
      s_issued[0] = kq;
      s_issued[1] = vq;
    }
    __syncwarp();
  } else if (nkt > 0) {
    // softmax warps: thread `row` owns query t = t0 + row, which sees keys j < L - T + t + 1
    const int row = tid;
    const int t = t0 + row;
    const int lim = t < a.T ? max(0, min(L, L - a.T + t + 1)) : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int kt = 0; kt < nkt; ++kt) {
      const int b0 = kt & 1;
      const uint32_t ph = (uint32_t)(kt >> 1) & 1u;
      // S of kt is complete (the TMEM accesses below are warp-wide: one decision per warp)
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_s[b0]), ph))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int j0 = kt * kPfKeys;
      const int vrows = min(kPfKeys, L - j0);
      if (vrows < kPfKeys) {
        // V rows at or past the sequence's length, once landed: zeroed (a masked p of 0 must
        // not meet a stale value)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_v[b0]), ph))) {
          ok = false;
          break;
        }
        unsigned char *vt = smem + C::V_OFF + b0 * C::KV_TILE;
        for (int idx = tid; idx < (kPfKeys - vrows) * (D / 8); idx += 32 * kPfSoftmaxWarps) {
          const int r = vrows + idx / (D / 8), c = idx % (D / 8);
          *reinterpret_cast<uint4 *>(vt + tile_chunk(kPfKeys, r, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // read next by the tensor core (asynchronous proxy)
      }
      // this row's 64 scores, read once; then the S columns are released for the next tile
      float sv[kPfKeys];
      tmem_ld64(tS + lane_base, sv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_sfree));
      // tiles short of every row's diagonal and of the sequence's end need no mask; in the
      // others, keys from `vis` on are masked (this row's visible keys of the tile)
      const bool full = j0 + kPfKeys <= kall;
      const int vis = full ? kPfKeys : min(kPfKeys, max(0, lim - j0));
      if (!full) {
#pragma unroll
        for (int i = 0; i < kPfKeys; ++i)
          if (i >= vis) sv[i] = qscale >= 0.f ? -INFINITY : INFINITY;
      }
      // the row maximum, scaled to base 2 (the scale's sign decides which extreme): eight
      // independent chains of three-input steps
      const float ext = qscale >= 0.f ? row_extreme<false>(sv) : row_extreme<true>(sv);
      const float mx = vis > 0 ? ext * qscale : -INFINITY;
      const bool move = mx > m_ref + kRescaleGap || (m_ref == -INFINITY && mx > -INFINITY);
      const float alpha = (move && m_ref != -INFINITY) ? exp2_approx(m_ref - mx) : 1.f;
      if (move) {
        l *= alpha;
        m_ref = mx;
      }
      // a warp rescales its rows of O when any of them must, once the previous P V product
      // is complete (TMEM loads and stores are warp-wide)
      if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_o), (uint32_t)(kt - 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + lane_base + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tO + lane_base + c, o);
        }
      }
      // P = 2^(s - m) as bf16 pairs into P buffer b0, once the P V product of kt-2 has read it
      const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
      uint32_t pk[kPfKeys / 2];
      if (full)
        l += p_row<false>(sv, qscale, nbase, vis, pk);
      else
        l += p_row<true>(sv, qscale, nbase, vis, pk);
      if (kt >= 2) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_vfree[b0]), (uint32_t)((kt - 2) >> 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tP + b0 * (kPfKeys / 2) + lane_base, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_p[b0]));
    }
    // the last P V product is complete before O is read
    if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar_o), (uint32_t)(nkt - 1) & 1u))) ok = false;
  }
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    // before shared memory and TMEM are released: the tensor-core products (one commit
    // tracks them all) and the copies issued but never seen landed
    if (tid == kPfMmaWarp * 32) {
      tc_commit(smem_u32(&bar_fin));
      mbar_wait_bounded(smem_u32(&bar_fin), 0);
    }
    if (tid == kPfLoadWarp * 32) {
      if (nkt > 0 && !s_seen[2]) mbar_wait_bounded(smem_u32(&bar_q), 0);
      for (int kt = s_seen[0]; kt < s_issued[0]; ++kt)
        mbar_wait_bounded(smem_u32(&bar_k[kt & 1]), (uint32_t)(kt >> 1) & 1u);
      for (int kt = s_seen[1]; kt < s_issued[1]; ++kt)
        mbar_wait_bounded(smem_u32(&bar_v[kt & 1]), (uint32_t)(kt >> 1) & 1u);
      report(a.status, TD_DEV_WAIT_TIMEOUT);
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp < kPfSoftmaxWarps) {
    // epilogue: O / l for this row, lse = m + log2(l) (natural-log units); the TMEM loads are
    // warp-wide, so every thread takes part and only the stores depend on the row
    const int row = tid, t = t0 + row;
    const bool row_valid = t < a.T;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
    __nv_bfloat16 *orow =
        static_cast<__nv_bfloat16 *>(a.out) + (((size_t)b * a.Hq + hq) * a.T + (row_valid ? t : 0)) * D;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      float o[32];
      if (nkt > 0) {
        tmem_ld32(tO + lane_base + c, o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (row_valid) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) pk[i / 2] = pack_bf16x2(o[i] * inv, o[i + 1] * inv);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          reinterpret_cast<uint4 *>(orow + c)[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    if (row_valid && a.lse != nullptr)
      a.lse[((size_t)b * a.Hq + hq) * a.T + t] = (ok && l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::TMEM_COLS) : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 pf_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over [planes][rows][D] bf16, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool pf_map(CUtensorMap *m, const void *base, long long planes, int rows, int D, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = pf_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prefill_d(PfArgs &a, const void *q, const void *k, const void *v, cudaStream_t stream) {
  if (!pf_map(&a.qmap, q, (long long)a.B * a.Hq, a.T, D, kPfRows) ||
      !pf_map(&a.kmap, k, (long long)a.B * a.Hkv, a.Smax, D, kPfKeys) ||
      !pf_map(&a.vmap, v, (long long)a.B * a.Hkv, a.Smax, D, kPfKeys))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(reinterpret_cast<const void *>(&prefill_kernel<D>),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::SMEM);
  });
  if (attr != cudaSuccess) return attr;
  const dim3 grid((unsigned)(a.B * a.Hq), (unsigned)((a.T + kPfRows - 1) / kPfRows));
  return launch_pdl(prefill_kernel<D>, grid, dim3(kPfThreads), PfCfg<D>::SMEM, stream, a);
}

}  // namespace

cudaError_t launch_prefill(const void *q, const void *k, const void *v, const int32_t *seq_lens, int B, int Hq, int Hkv,
                           int T, int Smax, int D, float scale, void *out, float *lse, uint32_t *status,
                           cudaStream_t stream) {
  PfArgs a;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.T = T;
  a.Smax = Smax;
  a.qscale = scale * kLog2e;
  return D == 64 ? launch_prefill_d<64>(a, q, k, v, stream) : launch_prefill_d<128>(a, q, k, v, stream);
}

}  // namespace td
