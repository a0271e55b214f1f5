// Split-KV attention for decode and speculative-verify chunks.
//
// Method ("tinydecode", section "how the decode step is put together"; "llm-decode-cuda",
// split-KV attention section): the keys of each sequence are cut into chunks; one CTA
// computes, for one (sequence b, kv head, chunk) and every query row that reads that kv
// head (the whole grouped-query group, times the T tokens of a verify chunk), the partial
// softmax (m, l, acc) of the chunk; the partials are merged with log-sum-exp. Query head hq
// reads kv head hq / G (index math, no copies).
//
// GB300 design:
//  * Work items (b, kv head, row block, chunk) are enumerated on the device from seq_lens,
//    so the grid depends only on the arguments (CUDA-graph capturable) and chunks past a
//    sequence's length are never scheduled. With split = 0 the chunk size is chosen on the
//    device so the items fill the grid (persistent-style, grid-stride over items).
//  * Inside a CTA each warp streams its own slice of the chunk through a private ring of
//    shared-memory stages, filled by bulk asynchronous copies (the TMA engine; one K and one
//    V copy per stage, each a contiguous run of cache rows) and completed on an mbarrier.
//  * Scores: 8 lanes per key, each lane owning D/8 dimensions as 16-byte vectors; the
//    partial dot products of 8 (key, row) pairs are reduced across the 8 lanes with a
//    transposing butterfly, leaving one full score per lane. Online softmax in base 2.
//  * p @ V: each lane owns D/32 dimensions of every row's accumulator; the probabilities are
//    broadcast through a per-warp shared stash.
//  * Warps combine their partials in shared memory; a chunk that is the only one of its
//    sequence writes the output directly, otherwise the partial goes to the workspace and
//    the CTA that completes the last chunk of a (b, kv head, row block) merges (atomic
//    ticket, no spin-wait).
#pragma once

#include "td_device.cuh"
#include "td_merge.cuh"

namespace td {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;

struct SplitParams {
  const void *q;        // [B, Hq, T, D]
  const void *k;        // [B, Hkv, Smax, D]
  const void *v;
  const int32_t *seq_lens;
  void *out;            // [B, Hq, T, D]
  float *lse;           // [B, Hq, T] or null
  float *ws_part;       // [B, Hkv, RB][ns_ws] partial blocks of R rows (see part_row_floats)
  int *counters;        // [B, Hkv, RB] completion tickets, then [B, Hkv, RB] finished slice merges
  uint32_t *status;
  int B, Hq, Hkv, G, T, Smax;
  int R;                // query rows per CTA (<= RP)
  int RB;               // row blocks per kv head: ceil(G*T / R)
  int split;            // fixed chunk size, or 0 = chosen on the device
  int ns_ws;            // partial slots per row in the workspace
  int p_target;         // CTAs the automatic chunk size aims to fill
  int min_chunk;        // smallest automatic chunk (keys)
  int warm_stages;      // 64-row units of its first chunk each CTA warms in L2 before the wait
  float qscale;         // scale * log2(e)
  // Fused step (tensor-core kernels only; k_new == null for plain attention): the T new rows
  // of each (b, kv head) go to cache rows seq_lens[b] .. seq_lens[b]+T-1 in this launch, the
  // query and key rows rotated there first when rope tables are given, and every query row
  // attends over seq_lens[b] + T keys.
  const void *k_new;    // [B, Hkv, T, D]
  const void *v_new;
  const float *rope_cos;   // [Smax, D/2], or null: no rotation
  const float *rope_sin;
  int32_t *advance_lens;   // the seq_lens array, to advance by T once every CTA has read it; or null
  int *done;               // grid-wide count of CTAs that have read the lengths (workspace, zero)
  // 8-bit caches: k and v hold int8 codes, these the fp32 scale of every row [B, Hkv, Smax]
  const float *k_scales;
  const float *v_scales;
};

// Attended length of a sequence whose stored length is `raw`, with the status bits its
// reading raises. Plain attention: raw clamped into [0, Smax]. Fused step: raw + T, or 0
// (nothing attended, nothing written) when the new rows do not fit.
__device__ __forceinline__ int attended_len(const SplitParams &p, int32_t raw, uint32_t &bits) {
  if (p.k_new != nullptr) {
    const bool fits = raw >= 0 && (long long)raw + p.T <= p.Smax;
    if (!fits) bits |= TD_DEV_APPEND_OVERFLOW;
    return fits ? raw + p.T : 0;
  }
  const int L = raw < 0 ? 0 : (raw > p.Smax ? p.Smax : raw);
  if (raw < 0) bits |= TD_DEV_NEGATIVE_SEQLEN;
  if (raw > p.Smax) bits |= TD_DEV_SEQLEN_CLAMPED;
  if (p.T > 1 && L < p.T) bits |= TD_DEV_VERIFY_SHORT;
  return L;
}

// A chunk's partial result for its row block is R rows of part_row_floats(D) floats: acc[D]
// (unnormalised p @ V sums), m (base-2 units) and l, padded to 16 bytes, so a block and any
// run of its rows can be bulk-copied and every acc row is 16-byte aligned.
__host__ __device__ constexpr int part_row_floats(int D) { return D + 4; }
__host__ __device__ constexpr int part_block_floats(int R, int D) { return R * part_row_floats(D); }


template <typename E, int D, int RP>
struct SplitCfg {
  static constexpr int EB = sizeof(E);
  static constexpr int ROW_BYTES = D * EB;
  static constexpr int VE = 16 / EB;             // elements per 16-byte vector
  static constexpr int NV = ROW_BYTES / 16;      // 16-byte vectors per cache row
  static constexpr int QV = NV / 8;              // vectors per lane for scores (8 lanes per key)
  static constexpr int DQ = QV * VE;             // = D / 8 dims per lane for scores
  static constexpr int DV = D / 32;              // dims per lane for p @ V
  static constexpr int KB = 32 / RP;             // keys per batch (one score per lane)
  static constexpr int SLOTS = 8 / RP;           // keys per 8-lane group per batch
  static constexpr int TKW = KB > 16 ? KB : 16;  // keys per warp stage
  static constexpr int TILE_BYTES = TKW * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = kStages * STAGE_BYTES;  // per warp
  static constexpr int STASH_FLOATS = KB * RP + 8;
  static constexpr int COMBINE_FLOATS = kWarps * RP * (D + 2);
  static constexpr int MERGE_FLOATS = 0;
  static constexpr int SMEM_BYTES = kWarps * RING_BYTES + kWarps * STASH_FLOATS * 4 + kWarps * kStages * 8;
  static_assert(NV % 8 == 0, "cache row must hold a multiple of 8 16-byte vectors");
  static_assert(D % 32 == 0, "head dim multiple of 32");
  static_assert(RP == 1 || RP == 2 || RP == 4 || RP == 8, "row padding is a power of two <= 8");
  static_assert(COMBINE_FLOATS * 4 <= kWarps * RING_BYTES, "combine area fits in the rings");
  static_assert(TKW % KB == 0, "stage holds whole batches");
  // fits next to the ~8.3 KB of static shared memory within the 227 KB a CTA may use
  static constexpr bool kFits = SMEM_BYTES + 8448 <= 227 * 1024;
};

// Chunk size before the overshoot check of plan_items: the caller's split, or keys per item
// so the items fill the grid once; then every sequence has at most ceil(p_target / U) chunks,
// which is what the workspace holds (the guard on `longest` only restates that bound).
__device__ __forceinline__ int first_chunk_size(const SplitParams &p, long long all, int longest) {
  if (p.split > 0) return p.split;
  const int U = p.Hkv * p.RB;
  long long want = (all * U + p.p_target - 1) / p.p_target;
  want = (want + 15) / 16 * 16;
  if (want < p.min_chunk) want = p.min_chunk;
  const long long fits = ((long long)longest + p.ns_ws - 1) / p.ns_ws;
  if (want < fits) want = fits;
  int S = (int)(want > p.Smax ? p.Smax : want);
  return S < 1 ? 1 : S;
}

// Exclusive prefix over the per-sequence item counts, computed by the whole CTA.
// s_len[b] receives the clamped length; returns the chunk size through *s_chunk and the
// item total in s_prefix[B]. s_red holds 2 * kWarps values.
static __device__ void plan_items(const SplitParams &p, int *s_len, int *s_prefix, int *s_chunk, long long *s_red,
                                  bool report_bits = true) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int U = p.Hkv * p.RB;
  constexpr int kSeg = (TD_MAX_BATCH + kThreads - 1) / kThreads;
  const int b0 = tid * kSeg;
  long long tot = 0;
  int lmax = 0;
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < kSeg; ++i) {
    const int b = b0 + i;
    if (b < p.B) {
      // before the wait for the previous kernel the lengths may be written meanwhile: read
      // them where that kernel's writes land, not through L1
      const int L = attended_len(p, report_bits ? p.seq_lens[b] : ld_relaxed(p.seq_lens + b), bits);
      s_len[b] = L;
      tot += L;
      lmax = max(lmax, L);
    }
  }
  if (report_bits && blockIdx.x == 0) report(p.status, bits);
  // total keys over the batch
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  if (lane == 0) {
    s_red[warp] = tot;
    s_red[kWarps + warp] = lmax;
  }
  __syncthreads();
  long long all = 0;
  int longest = 0;
  for (int w = 0; w < kWarps; ++w) {
    all += s_red[w];
    longest = max(longest, (int)s_red[kWarps + w]);
  }
  int S = first_chunk_size(p, all, longest);  // the same value in every thread
  // Per-thread segment sums of items, then a CTA-wide exclusive scan. With an automatic
  // chunk size, rounding each sequence's chunk count up can push the items past the grid,
  // leaving a second, mostly idle wave: then S grows, by the overshoot and by at least enough
  // to take one chunk off the longest sequence, and the scan is redone (a few passes at
  // most; it cannot fit once every nonempty sequence is down to one chunk per unit).
  for (int round = 0;; ++round) {
    int seg = 0;
#pragma unroll
    for (int i = 0; i < kSeg; ++i) {
      const int b = b0 + i;
      if (b < p.B) seg += ((s_len[b] + S - 1) / S) * U;
    }
    int incl = seg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();  // s_red reuse
    if (lane == 31) s_red[warp] = incl;
    __syncthreads();
    long long items = 0;
    for (int w = 0; w < kWarps; ++w) items += s_red[w];
    if (p.split == 0 && items > p.p_target && S < longest && round < 4) {
      long long grow = ((long long)S * items + p.p_target - 1) / p.p_target;
      const int n_long = (longest + S - 1) / S;  // >= 2 since S < longest
      const long long drop = ((long long)longest + n_long - 2) / (n_long - 1);
      if (grow < drop) grow = drop;
      grow = (grow + 15) / 16 * 16;
      S = (int)(grow > p.Smax ? p.Smax : grow);
      continue;  // the same decision in every thread
    }
    int before = incl - seg;
    for (int w = 0; w < warp; ++w) before += (int)s_red[w];
#pragma unroll
    for (int i = 0; i < kSeg; ++i) {
      const int b = b0 + i;
      if (b < p.B) {
        s_prefix[b] = before;
        before += ((s_len[b] + S - 1) / S) * U;
      }
    }
    if (tid == 0) {
      s_prefix[p.B] = (int)items;
      *s_chunk = S;
    }
    break;
  }
  __syncthreads();
}

// The plan made before the wait for the previous kernel (from lengths that kernel may still
// have been writing) is kept after the wait if every attended length reads the same now: the
// plan is a function of those lengths alone. Otherwise it is made again. Either way the
// status bits come from the lengths as read after the wait. Ends with a __syncthreads.
static __device__ void confirm_plan(const SplitParams &p, int *s_len, int *s_prefix, int *s_chunk, long long *s_red) {
  constexpr int kSeg = (TD_MAX_BATCH + kThreads - 1) / kThreads;
  const int b0 = threadIdx.x * kSeg;
  uint32_t bits = 0;
  bool same = true;
#pragma unroll
  for (int i = 0; i < kSeg; ++i) {
    const int b = b0 + i;
    if (b < p.B) same = attended_len(p, ld_relaxed(p.seq_lens + b), bits) == s_len[b] && same;
  }
  if (__syncthreads_and(same)) {
    if (blockIdx.x == 0) report(p.status, bits);
    return;
  }
  plan_items(p, s_len, s_prefix, s_chunk, s_red);  // ends with __syncthreads
}

// Fused step with advance: the last CTA of the grid to have read the lengths moves every
// sequence that took its new rows forward by T. Every CTA calls this once, after its last
// read of seq_lens; the count lives in the workspace and is left zero again.
static __device__ void advance_after_reads(const SplitParams &p, int *s_flag) {
  if (p.advance_lens == nullptr) return;
  if (threadIdx.x == 0) {
    const int prev = ticket_acq_rel(p.done);
    if (prev < 0 || prev >= (int)gridDim.x) report(p.status, TD_DEV_WORKSPACE_DIRTY);
    *s_flag = prev == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (*s_flag) {
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
      const int32_t raw = p.advance_lens[b];
      if (raw >= 0 && (long long)raw + p.T <= p.Smax) p.advance_lens[b] = raw + p.T;
    }
    if (threadIdx.x == 0) *p.done = 0;
  }
}

// Shared memory (floats) the fused merge needs besides the staged partial blocks.
template <int D, int ROWS>
__host__ __device__ constexpr int merge_fixed_floats() {
  return ROWS * D + 4 * ROWS + ROWS * 64;
}

// Output row (flattened [B, Hq*T]) of local row r of row block rb of kv head kvh.
__device__ __forceinline__ long long out_row_of(const SplitParams &p, int b, int kvh, int rb, int r) {
  const int gr = rb * p.R + r;
  return (long long)b * p.Hq * p.T + (long long)(kvh * p.G + gr / p.T) * p.T + gr % p.T;
}

// Log-sum-exp merge of the NC chunk partials of (b, kv head, row block), run by the CTA that
// took the last completion ticket; rows r < nv exist. The group's partial blocks are
// contiguous in the workspace, so they cross from L2 in bulk asynchronous copies, as many
// chunks at a time as the free shared memory holds, and are merged online: per row the
// running maximum M, normaliser Lsum and weighted sum are rescaled when a block raises M.
// `smem_f` spans `smem_floats` floats no one else uses now; `bar` is this CTA's merge
// mbarrier and `phase` its current parity (uniform across the CTA).
template <typename E, int D, int ROWS>
__device__ void merge_group(const SplitParams &p, float *smem_f, int smem_floats, uint64_t *bar, uint32_t &phase,
                            int b, int kvh, int rb, int NC, int nv) {
  constexpr int kFB = 64;  // most chunks staged at a time
  constexpr int D4 = D / 4, RF = part_row_floats(D);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.R;
  const int BF = part_block_floats(R, D);
  const long long g = ((long long)b * p.Hkv + kvh) * p.RB + rb;
  const float *src = p.ws_part + g * p.ns_ws * (long long)BF;
  float *acc = smem_f;          // [ROWS][D] running weighted sums (between passes)
  float *st = acc + ROWS * D;   // M[ROWS], Lsum[ROWS], rescale[ROWS], 1 / Lsum[ROWS]
  float *fac = st + 4 * ROWS;   // [ROWS][kFB] factors 2^(m_c - M) of the staged chunks
  float *stage = fac + ROWS * kFB;
  int FB = (smem_floats - merge_fixed_floats<D, ROWS>()) / BF;
  if (FB > kFB) FB = kFB;
  if (tid < nv) {
    st[tid] = -INFINITY;
    st[ROWS + tid] = 0.f;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < NC; c0 += FB) {
    const int nb = min(FB, NC - c0);
    const bool last = c0 + nb >= NC;
    if (tid == 0) {
      fence_proxy_async_global();
      mbar_arrive_expect_tx(smem_u32(bar), (uint32_t)(nb * BF * 4));
      bulk_g2s_plain(smem_u32(stage), src + (long long)c0 * BF, (uint32_t)(nb * BF * 4), smem_u32(bar));
    }
    if (!mbar_wait_bounded(smem_u32(bar), phase)) {
      report(p.status, TD_DEV_WAIT_TIMEOUT);
      mbar_wait_bounded(smem_u32(bar), phase);  // one more bounded wait for the copy in flight
    }
    phase ^= 1u;
    __syncthreads();  // staged blocks and the previous pass's statistics are visible
    // per-row statistics of this block (base 2): a warp per row, lanes over chunks
#pragma unroll 1
    for (int r = warp; r < nv; r += kWarps) {
      float mv[2], lv[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = lane + 32 * k;
        lv[k] = c < nb ? stage[c * BF + r * RF + D + 1] : 0.f;
        mv[k] = lv[k] > 0.f ? stage[c * BF + r * RF + D] : -INFINITY;
      }
      float bm = fmaxf(mv[0], mv[1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
      const float Mo = st[r];
      const float Mn = fmaxf(Mo, bm);
      const float base = Mn == -INFINITY ? 0.f : Mn;
      float ls = 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float f = lv[k] > 0.f ? exp2f(mv[k] - base) : 0.f;
        if (lane + 32 * k < nb) fac[r * kFB + lane + 32 * k] = f;
        ls = fmaf(lv[k], f, ls);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      if (lane == 0) {
        const float alpha = exp2f(Mo - base);
        const float Ls = st[ROWS + r] * alpha + ls;
        st[r] = Mn;
        st[ROWS + r] = Ls;
        st[2 * ROWS + r] = alpha;
        st[3 * ROWS + r] = Ls > 0.f ? 1.f / Ls : 0.f;
        if (last && p.lse != nullptr)
          p.lse[out_row_of(p, b, kvh, rb, r)] = Ls > 0.f ? (Mn + log2f(Ls)) * kLn2 : -INFINITY;
      }
    }
    __syncthreads();
    // weighted sums, four dims per thread, over the staged chunks in four independent
    // accumulators (chunk c into c % 4: a quarter of the dependent chain); in the last pass
    // they are the output
#pragma unroll 1
    for (int idx = tid; idx < nv * D4; idx += kThreads) {
      const int r = idx / D4, d = (idx % D4) * 4;
      const float *a = stage + r * RF + d;
      const float *f = fac + r * kFB;
      float4 xs[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) xs[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 > 0) {
        const float sc = st[2 * ROWS + r];
        xs[0] = *reinterpret_cast<const float4 *>(acc + r * D + d);
        xs[0].x *= sc, xs[0].y *= sc, xs[0].z *= sc, xs[0].w *= sc;
      }
      int c = 0;
#pragma unroll 1
      for (; c + 4 <= nb; c += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = *reinterpret_cast<const float4 *>(a + (c + k) * BF);
          const float w = f[c + k];
          xs[k].x = fmaf(v.x, w, xs[k].x), xs[k].y = fmaf(v.y, w, xs[k].y), xs[k].z = fmaf(v.z, w, xs[k].z),
          xs[k].w = fmaf(v.w, w, xs[k].w);
        }
      }
#pragma unroll 1
      for (; c < nb; ++c) {
        const float4 v = *reinterpret_cast<const float4 *>(a + c * BF);
        const float w = f[c];
        xs[0].x = fmaf(v.x, w, xs[0].x), xs[0].y = fmaf(v.y, w, xs[0].y), xs[0].z = fmaf(v.z, w, xs[0].z),
        xs[0].w = fmaf(v.w, w, xs[0].w);
      }
      float4 x;
      x.x = (xs[0].x + xs[1].x) + (xs[2].x + xs[3].x);
      x.y = (xs[0].y + xs[1].y) + (xs[2].y + xs[3].y);
      x.z = (xs[0].z + xs[1].z) + (xs[2].z + xs[3].z);
      x.w = (xs[0].w + xs[1].w) + (xs[2].w + xs[3].w);
      if (last) {
        const float inv = st[3 * ROWS + r];
        E *o = static_cast<E *>(p.out) + out_row_of(p, b, kvh, rb, r) * D + d;
        store_elem<E>(o + 0, x.x * inv);
        store_elem<E>(o + 1, x.y * inv);
        store_elem<E>(o + 2, x.z * inv);
        store_elem<E>(o + 3, x.w * inv);
      } else {
        *reinterpret_cast<float4 *>(acc + r * D + d) = x;
      }
    }
    __syncthreads();  // the next block overwrites the staging area
  }
}

// Waits, bounded, until the completion counter at `cnt` reads at least `target` (acquire:
// the partials released before those tickets are visible after it). Thread 0 polls; the CTA
// takes one decision. False if the count never arrived (TD_DEV_WAIT_TIMEOUT is set).
__device__ __forceinline__ bool wait_count(const SplitParams &p, const int *cnt, int target) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    int ok = 1;
    if (ld_acquire(cnt) < target) {
      const long long t0 = clock64();
      while (ld_acquire(cnt) < target) {
        if (clock64() - t0 > kWaitLimitCycles) {
          ok = 0;
          report(p.status, TD_DEV_WAIT_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Merges rows [s0, s1) (at most kThreads / (D / 4) of them) of group (b, kv head, row block rb)
// over its NC published partials with direct loads from L2. The threads are (row, column of
// four dims) pairs times CG = kThreads / (rows * D/4) groups of chunks; group j folds chunks
// j, j + CG, ... into a running (M, L, sums) in base 2, kBatch chunks' loads in flight at once,
// and the groups are combined in shared memory `sm` (6 * kThreads floats). Writes out and lse.
template <typename E, int D>
__device__ void merge_rows_direct(const SplitParams &p, float *sm, int b, int kvh, int rb, int NC, int s0, int s1) {
  constexpr int D4 = D / 4, RF = part_row_floats(D), kBatch = 12;
  const int nr = s1 - s0;
  const int cols = nr * D4;
  const int CG = kThreads / cols;
  const int tid = threadIdx.x;
  const int cg = tid / cols, rr = (tid % cols) / D4, col = tid % D4;
  const bool active = cg < CG;
  const long long g = ((long long)b * p.Hkv + kvh) * p.RB + rb;
  const float *row0 = p.ws_part + (g * p.ns_ws * p.R + s0 + rr) * (long long)RF;  // chunk c at + c * R * RF
  const long long cstride = (long long)p.R * RF;
  float M = -INFINITY, Ls = 0.f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active) {
#pragma unroll 1
    for (int c0 = cg; c0 < NC; c0 += CG * kBatch) {
      float mv[kBatch], lv[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int c = c0 + k * CG;
        lv[k] = 0.f;
        mv[k] = -INFINITY;
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < NC) {
          const float *rp = row0 + c * cstride;
          lv[k] = __ldcg(rp + D + 1);
          mv[k] = __ldcg(rp + D);
          v[k] = __ldcg(reinterpret_cast<const float4 *>(rp) + col);
        }
      }
      float bm = M;
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (lv[k] > 0.f) bm = fmaxf(bm, mv[k]);
      const float base = bm == -INFINITY ? 0.f : bm;
      const float alpha = exp2f(M - base);  // 0 while nothing is folded in (M = -inf)
      Ls *= alpha;
      A.x *= alpha, A.y *= alpha, A.z *= alpha, A.w *= alpha;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (lv[k] > 0.f) {
          const float f = exp2f(mv[k] - base);
          Ls = fmaf(lv[k], f, Ls);
          A.x = fmaf(v[k].x, f, A.x), A.y = fmaf(v[k].y, f, A.y), A.z = fmaf(v[k].z, f, A.z),
          A.w = fmaf(v[k].w, f, A.w);
        }
      }
      M = bm;
    }
  }
  float *sM = sm, *sL = sm + kThreads, *sA = sm + 2 * kThreads;  // [CG][nr], [CG][nr], [CG][nr][D]
  if (active) {
    if (col == 0) {
      sM[cg * nr + rr] = M;
      sL[cg * nr + rr] = Ls;
    }
    *reinterpret_cast<float4 *>(sA + (cg * nr + rr) * D + 4 * col) = A;
  }
  __syncthreads();
  if (cg == 0) {
    float Mt = -INFINITY;
    for (int j = 0; j < CG; ++j)
      if (sL[j * nr + rr] > 0.f) Mt = fmaxf(Mt, sM[j * nr + rr]);
    float Lt = 0.f;
    float4 At = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < CG; ++j) {
      const float lj = sL[j * nr + rr];
      if (lj > 0.f) {
        const float f = exp2f(sM[j * nr + rr] - Mt);
        const float4 x = *reinterpret_cast<const float4 *>(sA + (j * nr + rr) * D + 4 * col);
        Lt = fmaf(lj, f, Lt);
        At.x = fmaf(x.x, f, At.x), At.y = fmaf(x.y, f, At.y), At.z = fmaf(x.z, f, At.z), At.w = fmaf(x.w, f, At.w);
      }
    }
    const long long orow = out_row_of(p, b, kvh, rb, s0 + rr);
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    E *o = static_cast<E *>(p.out) + orow * D + 4 * col;
    store_elem<E>(o + 0, At.x * inv);
    store_elem<E>(o + 1, At.y * inv);
    store_elem<E>(o + 2, At.z * inv);
    store_elem<E>(o + 3, At.w * inv);
    if (col == 0 && p.lse != nullptr) p.lse[orow] = Lt > 0.f ? (Mt + log2f(Lt)) * kLn2 : -INFINITY;
  }
  __syncthreads();  // the scratch may be reused
}

// Completes one work item (sequence b, kv head, row block rb, chunk c of NC).
// The item's partial sources (warps or key slices) have written, in base-2 units,
//   cm[NSRC][ROWS] (row max), cl[NSRC][ROWS] (row sum), ca[NSRC][ROWS][CAS] (unnormalised p @ V)
// at the start of the CTA's shared memory (`smem_f`, `smem_floats` floats free after this
// call's combine), and a __syncthreads has made them visible. The sources are combined; a
// chunk that is its sequence's only one writes out/lse; any other publishes its partial block
// to the workspace and takes a completion ticket on its group's counter. The merge then:
//  * blocks of more than 16 rows (a 24-row verify block of four grouped heads) in a one_wave
//    launch (every CTA holds at most one item, and the launch fits the GPU at once): the CTAs
//    holding the last NSL tickets of the group (NSL = min(rows, chunks)) each merge one slice
//    of the rows, the last ticket slice 0 at once, the others after a bounded wait for the
//    group's last ticket (a CTA they wait for is resident or becomes resident as other CTAs
//    of the launch exit: none of them waits for it); the last of them to finish zeroes the
//    group's counters again. One CTA staging every chunk's 24 rows took 28 us where the
//    chunks streamed in 7;
//  * otherwise the CTA holding the last ticket merges every row (merge_group): with a few rows
//    the helpers' waits cost more than they save (their slots are the next call's).
// Ends with a __syncthreads (the shared areas may be reused afterwards).
template <typename E, int D, int ROWS, int NSRC, int CAS = D>
__device__ void finish_item(const SplitParams &p, float *smem_f, int smem_floats, uint64_t *merge_bar,
                            uint32_t &merge_phase, int b, int kvh, int rb, int c, int NC, int *s_last,
                            bool one_wave) {
  constexpr int D4 = D / 4, RF = part_row_floats(D);
  const int tid = threadIdx.x;
  const int GT = p.G * p.T;
  const int R = p.R;
  const float *cm = smem_f;
  const float *cl = smem_f + NSRC * ROWS;
  const float *ca = smem_f + 2 * NSRC * ROWS;
  // Many rows (more than 8): the factor 2^(m_w - M) of each source and row (0 for an empty
  // source), the maximum and the sum are computed once per row first; few rows: each thread
  // computes its row's from the sources itself (no extra barrier).
  float *fac = smem_f + 2 * NSRC * ROWS + NSRC * ROWS * CAS;
  float *rM = fac + NSRC * ROWS;
  float *rL = rM + ROWS;
  const bool single = NC == 1;
  const int nv = min(R, GT - rb * R);  // rows of this block that exist
  const bool rowwise = ROWS > 16 || nv > 8;  // always for 24-row blocks
  const long long g = ((long long)b * p.Hkv + kvh) * p.RB + rb;
  if (rowwise) {
    for (int r = tid; r < nv; r += kThreads) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NSRC; ++w) M = fmaxf(M, cm[w * ROWS + r]);
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < NSRC; ++w) {
        const float mw = cm[w * ROWS + r];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        fac[w * ROWS + r] = f;
        Ls = fmaf(cl[w * ROWS + r], f, Ls);
      }
      rM[r] = M;
      rL[r] = Ls;
    }
    __syncthreads();
  }
  float *blk = p.ws_part + (g * p.ns_ws + c) * (long long)part_block_floats(R, D);
#pragma unroll 1
  for (int idx = tid; idx < nv * D4; idx += kThreads) {
    const int r = idx / D4, d = (idx % D4) * 4;
    float M, Ls = 0.f, f[NSRC];
    if (rowwise) {
      M = rM[r];
      Ls = rL[r];
#pragma unroll
      for (int w = 0; w < NSRC; ++w) f[w] = fac[w * ROWS + r];
    } else {
      M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NSRC; ++w) M = fmaxf(M, cm[w * ROWS + r]);
#pragma unroll
      for (int w = 0; w < NSRC; ++w) {
        const float mw = cm[w * ROWS + r];
        f[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
        Ls = fmaf(cl[w * ROWS + r], f[w], Ls);
      }
    }
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NSRC; ++w) {
      const float4 v = *reinterpret_cast<const float4 *>(ca + (w * ROWS + r) * CAS + d);
      A.x = fmaf(v.x, f[w], A.x), A.y = fmaf(v.y, f[w], A.y), A.z = fmaf(v.z, f[w], A.z), A.w = fmaf(v.w, f[w], A.w);
    }
    if (single) {
      const long long row = out_row_of(p, b, kvh, rb, r);
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      E *o = static_cast<E *>(p.out) + row * D + d;
      store_elem<E>(o + 0, A.x * inv);
      store_elem<E>(o + 1, A.y * inv);
      store_elem<E>(o + 2, A.z * inv);
      store_elem<E>(o + 3, A.w * inv);
      if (d == 0 && p.lse != nullptr) p.lse[row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    } else {
      float *dst = blk + r * RF;
      *reinterpret_cast<float4 *>(dst + d) = A;
      if (d == 0) {
        dst[D] = Ls > 0.f ? M : -INFINITY;
        dst[D + 1] = Ls;
      }
    }
  }
  if (!single) {
    __syncthreads();  // every thread's block writes happen before thread 0's release
    int *cnt = p.counters + g;
    int *fin = p.counters + (long long)p.B * p.Hkv * p.RB + g;
    if (tid == 0) {
      const int before = ticket_acq_rel(cnt);
      if (before < 0 || before >= NC) report(p.status, TD_DEV_WORKSPACE_DIRTY);
      *s_last = before;
    }
    __syncthreads();
    const int t = *s_last;
    if (one_wave && ROWS > 16) {
      const int nsl = min(nv, NC);
      const int s = NC - 1 - t;  // 0 for the last ticket
      if (s >= 0 && s < nsl) {
        const int rs = (nv + nsl - 1) / nsl;
        const int r0 = min(s * rs, nv), r1 = min(r0 + rs, nv);
        // slice 0's CTA holds the last ticket: every partial is visible to it already
        const bool ready = s == 0 || wait_count(p, cnt, NC);
        if (ready) {
          constexpr int kMost = kThreads / D4;  // rows one pass of merge_rows_direct takes
          for (int a = r0; a < r1; a += kMost) merge_rows_direct<E, D>(p, smem_f, b, kvh, rb, NC, a, min(a + kMost, r1));
        }
        if (tid == 0) {
          const int done = atomicAdd(fin, 1);
          if (done == nsl - 1) {  // every slice merged (or given up): the counters go back to zero
            *cnt = 0;
            *fin = 0;
          }
        }
      }
    } else if (t == NC - 1) {
      merge_group<E, D, ROWS>(p, smem_f, smem_floats, merge_bar, merge_phase, b, kvh, rb, NC, nv);
      if (tid == 0) *cnt = 0;  // leave the counter area zero for the next call
    }
  }
  __syncthreads();
}

template <typename E, int D, int RP>
__global__ void __launch_bounds__(kThreads, 2) split_attn_kernel(const SplitParams p) {
  using C = SplitCfg<E, D, RP>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_len[TD_MAX_BATCH];
  __shared__ int s_prefix[TD_MAX_BATCH + 1];
  __shared__ long long s_red[2 * kWarps];
  __shared__ int s_chunk, s_last, s_abort;
  __shared__ __align__(8) uint64_t s_merge_bar;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 3, sub = lane & 7;
  unsigned char *ring = smem + warp * C::RING_BYTES;
  float *stash = reinterpret_cast<float *>(smem + kWarps * C::RING_BYTES) + warp * C::STASH_FLOATS;
  uint64_t *bars =
      reinterpret_cast<uint64_t *>(smem + kWarps * C::RING_BYTES + kWarps * C::STASH_FLOATS * 4) + warp * kStages;
  float *combine = reinterpret_cast<float *>(smem);           // after all rings are idle

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  if (tid == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&s_merge_bar), 1);
    fence_mbar_init();
  }
  uint32_t merge_phase = 0;
  // a plan on the lengths as they read now, kept after the wait if they read the same then
  plan_items(p, s_len, s_prefix, &s_chunk, s_red, false);
  griddep_wait();  // inputs may come from the previous kernel in the stream
  griddep_launch_dependents();
  confirm_plan(p, s_len, s_prefix, &s_chunk, s_red);  // ends with __syncthreads

  const int S = s_chunk;
  const int W = s_prefix[p.B];
  const int U = p.Hkv * p.RB;
  const int rows = p.Hq * p.T;
  const int GT = p.G * p.T;
  const uint64_t policy = l2_evict_first_policy();
  uint32_t seq = 0;  // stages consumed by this warp so far (mbarrier phase bookkeeping)

  // sequences with no key get no item: their rows are 0 with lse = -inf
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (s_len[b] != 0) continue;
    for (int idx = tid; idx < rows * D; idx += kThreads)
      store_elem<E>(static_cast<E *>(p.out) + (long long)b * rows * D + idx, 0.f);
    if (p.lse != nullptr)
      for (int r = tid; r < rows; r += kThreads) p.lse[(long long)b * rows + r] = -INFINITY;
  }

  for (int item = blockIdx.x; item < W; item += gridDim.x) {
    // ---- locate the item: sequence b by binary search over the prefix, then kv head, row block, chunk
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

    // ---- this warp's slice of the chunk, in whole stages
    const int n = c1 - c0;
    const int per = ((n + kWarps - 1) / kWarps + C::TKW - 1) / C::TKW * C::TKW;
    const int w0 = c0 + warp * per;
    const int w1 = min(w0 + per, c1);
    const int ntiles = w0 < w1 ? (w1 - w0 + C::TKW - 1) / C::TKW : 0;
    const size_t head_off = ((size_t)b * p.Hkv + kvh) * (size_t)p.Smax * C::ROW_BYTES;
    const unsigned char *kg = static_cast<const unsigned char *>(p.k) + head_off;
    const unsigned char *vg = static_cast<const unsigned char *>(p.v) + head_off;

    auto issue = [&](int i) {
      const int st = (seq + i) % kStages;
      const int j0 = w0 + i * C::TKW;
      const uint32_t bytes = (uint32_t)min(C::TKW, w1 - j0) * C::ROW_BYTES;
      const uint32_t bar = smem_u32(&bars[st]);
      unsigned char *dst = ring + st * C::STAGE_BYTES;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, 2 * bytes);
      bulk_g2s(smem_u32(dst), kg + (size_t)j0 * C::ROW_BYTES, bytes, bar, policy);
      bulk_g2s(smem_u32(dst + C::TILE_BYTES), vg + (size_t)j0 * C::ROW_BYTES, bytes, bar, policy);
    };
    if (lane == 0) {
      for (int i = 0; i < min(kStages, ntiles); ++i) issue(i);
    }

    // ---- query rows of this CTA: row r is group row rb*R + r = (head in group, token t)
    int nvis[RP];
    float qr[RP][C::DQ];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const int gr = rb * p.R + r;
      const bool valid = r < p.R && gr < GT;
      const int hq = kvh * p.G + gr / p.T;
      const int t = gr % p.T;
      nvis[r] = valid ? max(L - p.T + t + 1, 0) : 0;
      const unsigned char *qrow =
          static_cast<const unsigned char *>(p.q) + (((size_t)b * p.Hq + hq) * p.T + t) * C::ROW_BYTES;
#pragma unroll
      for (int qv = 0; qv < C::QV; ++qv) {
        float f[C::VE];
        if (valid) {
          load_widen<E, C::VE>(qrow + (sub + 8 * qv) * 16, f);
        } else {
#pragma unroll
          for (int e = 0; e < C::VE; ++e) f[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < C::VE; ++e) qr[r][qv * C::VE + e] = f[e] * p.qscale;
      }
    }

    // ---- stream the slice: online softmax in base 2
    const int my_row = sub % RP;  // row of the single score this lane holds after the reduction
    int my_nvis = 0;               // (selected without a runtime index so nvis stays in registers)
#pragma unroll
    for (int r = 0; r < RP; ++r)
      if (r == my_row) my_nvis = nvis[r];
    float m_run = -INFINITY, l_run = 0.f;
    float acc[RP][C::DV];
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int d = 0; d < C::DV; ++d) acc[r][d] = 0.f;

    int consumed = 0;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int st = (seq + i) % kStages;
      const uint32_t parity = ((seq + i) / kStages) & 1u;
      // one decision for the whole warp: the shuffles below need every lane
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[st]), parity))) {
        ok = false;
        break;
      }
      const unsigned char *Ks = ring + st * C::STAGE_BYTES;
      const unsigned char *Vs = Ks + C::TILE_BYTES;
      const int j0 = w0 + i * C::TKW;
      const int nk = min(C::TKW, w1 - j0);
      for (int kb0 = 0; kb0 < nk; kb0 += C::KB) {
        // partial scores: slot s holds key kb0 + 4s + g8, for every row
        float part[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) part[x] = 0.f;
#pragma unroll
        for (int s = 0; s < C::SLOTS; ++s) {
          const unsigned char *krow = Ks + (kb0 + 4 * s + g8) * C::ROW_BYTES;
#pragma unroll
          for (int qv = 0; qv < C::QV; ++qv) {
            float kf[C::VE];
            load_widen<E, C::VE>(krow + (sub + 8 * qv) * 16, kf);
#pragma unroll
            for (int r = 0; r < RP; ++r)
#pragma unroll
              for (int e = 0; e < C::VE; ++e) part[s * RP + r] = fmaf(qr[r][qv * C::VE + e], kf[e], part[s * RP + r]);
          }
        }
        // transposing butterfly over the 8 lanes of a key group: lane `sub` ends with pair `sub`
#pragma unroll
        for (int o = 4, nh = 4; o > 0; o >>= 1, nh >>= 1) {
          const bool up = (sub & o) != 0;
#pragma unroll
          for (int x = 0; x < nh; ++x) {
            const float send = up ? part[x] : part[x + nh];
            const float keep = up ? part[x + nh] : part[x];
            part[x] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        const int kk = kb0 + (sub / RP) * 4 + g8;  // key (within the stage) of this lane's score
        const int j = j0 + kk;
        const bool valid = kk < nk && j < my_nvis;
        const float sc = valid ? part[0] : -INFINITY;
        float bm = sc;
#pragma unroll
        for (int o = RP; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        const float m_new = fmaxf(m_run, bm);
        const float base = m_new == -INFINITY ? 0.f : m_new;
        const float pr = exp2f(sc - base);
        const float alpha = exp2f(m_run - base);
        l_run = l_run * alpha + pr;
        m_run = m_new;
        stash[((sub / RP) * 4 + g8) * RP + my_row] = pr;
        if (lane < RP) stash[C::KB * RP + lane] = alpha;
        __syncwarp();
        // p @ V: rescale, then accumulate this batch's keys
        float al[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) al[r] = stash[C::KB * RP + r];
        bool rescale = false;
#pragma unroll
        for (int r = 0; r < RP; ++r) rescale |= al[r] != 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int d = 0; d < C::DV; ++d) acc[r][d] *= al[r];
        }
        const int nkb = min(C::KB, nk - kb0);
#pragma unroll
        for (int x = 0; x < C::KB; ++x) {
          if (x < nkb) {
            float vf[C::DV];
            load_widen<E, C::DV>(Vs + (kb0 + x) * C::ROW_BYTES + lane * C::DV * C::EB, vf);
#pragma unroll
            for (int r = 0; r < RP; ++r) {
              const float pw = stash[x * RP + r];
#pragma unroll
              for (int d = 0; d < C::DV; ++d) acc[r][d] = fmaf(pw, vf[d], acc[r][d]);
            }
          }
        }
        __syncwarp();
      }
      consumed = i + 1;
      if (lane == 0 && i + kStages < ntiles) issue(i + kStages);
    }
    if (!ok) {
      // a copy never completed: wait (bounded) for this warp's other copies, then drop the slice
      const int issued = min(ntiles, consumed + kStages);
      for (int i = consumed + 1; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&bars[(seq + i) % kStages]), ((seq + i) / kStages) & 1u);
      if (lane == 0) {
        report(p.status, TD_DEV_WAIT_TIMEOUT);
        s_abort = 1;
      }
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int d = 0; d < C::DV; ++d) acc[r][d] = 0.f;
    }
    seq += ntiles;

    // ---- combine the warps' partials (shared memory, rings idle)
    float l_tot = l_run;
#pragma unroll
    for (int o = RP; o < 32; o <<= 1) l_tot += __shfl_xor_sync(0xffffffffu, l_tot, o);
    __syncthreads();
    float *cm = combine;                      // [kWarps][RP]
    float *cl = combine + kWarps * RP;        // [kWarps][RP]
    float *ca = combine + 2 * kWarps * RP;    // [kWarps][RP][D]
    if (lane < RP) {
      cm[warp * RP + lane] = m_run;
      cl[warp * RP + lane] = l_tot;
    }
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int d = 0; d < C::DV; ++d) ca[(warp * RP + r) * D + lane * C::DV + d] = acc[r][d];
    __syncthreads();
    finish_item<E, D, RP, kWarps>(p, combine, kWarps * C::RING_BYTES / 4, &s_merge_bar, merge_phase, b, kvh, rb, c,
                                  NC, &s_last, W <= (int)gridDim.x);
    if (s_abort) break;
  }
}

}  // namespace td
