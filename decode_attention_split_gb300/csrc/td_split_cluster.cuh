// Split-KV attention with the chunk merge done inside a thread-block cluster.
//
// Same method as split_attn_mma_kernel ("tinydecode", section "how the decode step is put
// together"; "llm-decode-cuda", split-KV attention section): the keys of one
// (sequence b, kv head, row block) group are cut into chunks whose partial softmax results
// are merged by log-sum-exp. Here a group is one cluster of CS CTAs: CTA `rank` streams
// chunk `rank`, combines its warps' partials into one block in its own shared memory, and
// after a cluster barrier CTA 0 reads the CS blocks through distributed shared memory and
// writes out and lse. No partials in global memory, no atomics, no second pass over L2; a
// second cluster barrier keeps every CTA's shared memory alive until CTA 0 has read it.
//
// Used when the groups fill the GPU in one wave of clusters at about two CTAs per SM
// (batches of a few sequences); the grid is groups x CS CTAs, fixed by the arguments.
#pragma once

#include "td_internal.h"
#include "td_split_mma.cuh"

namespace td {

// TILE: the warps' step for the group's rows (tile_of_rows).
template <int D, int TILE = kTileM16>
__global__ void __launch_bounds__(kThreads, 1) split_attn_cluster_kernel(const __grid_constant__ MmaArgs a) {
  constexpr int NST = kClusterStages<D>;
  constexpr int D4 = D / 4;
  constexpr int TR = tile_rows<TILE>();
  using C = MmaCfg<D, NST>;
  static_assert((combine_floats<D, TILE>() + TR * (D + 2)) * 4 <= C::RING_BYTES, "local block fits in the ring");
  static_assert(combine_floats<D, TILE>() % 4 == 0, "the local block is 16-byte aligned");
  const SplitParams &p = a.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t s_bars[NST];
  __shared__ float s_w[kMaxCluster][TR];  // CTA 0: merge weight of each block's rows
  __shared__ float s_lse[TR];
  __shared__ int s_flag;

  const int tid = threadIdx.x;
  unsigned char *smem = align1024(smem_raw);
  const uint32_t rank = cluster_ctarank();
  const int CS = (int)cluster_nctarank();
  const int g = (int)cluster_id_x();
  const int rb = g % p.RB;
  const int kvh = (g / p.RB) % p.Hkv;
  const int b = g / (p.RB * p.Hkv);
  const int R = p.R;
  const int nv = min(R, p.G * p.T - rb * R);  // rows of this block that exist
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < NST; ++i) mbar_init(smem_u32(&s_bars[i]), 1);
    fence_mbar_init();
  }
  if (tid == 0) {
    // a guess of this CTA's chunk from the length as it reads before the wait (see
    // prefetch_first_item): warm L2 with its first stages
    uint32_t guess_bits = 0;
    const int Lg = attended_len(p, ld_relaxed(p.seq_lens + b), guess_bits);
    const int Sg = ((Lg + CS - 1) / CS + C::TK - 1) / C::TK * C::TK;
    const int g0 = min((int)rank * Sg, Lg);
    prefetch_chunk_l2<D>(p, b, kvh, g0, min(g0 + Sg, Lg), prefetch_stages(p));
  }
  griddep_wait();  // seq_lens and the cache may come from the previous kernel in the stream
  griddep_launch_dependents();
  uint32_t bits = 0;
  const int L = attended_len(p, p.seq_lens[b], bits);
  if (tid == 0 && rank == 0 && kvh == 0 && rb == 0) report(p.status, bits);
  __syncthreads();  // barrier initialisation is visible before any wait
  advance_after_reads(p, &s_flag);  // fused step: the lengths move on once every CTA has read them
  // chunk of this CTA: whole 64-key stages, the group's keys spread over the cluster
  const int S = ((L + CS - 1) / CS + C::TK - 1) / C::TK * C::TK;
  const int c0 = min((int)rank * S, L);
  const int c1 = min(c0 + S, L);
  uint32_t seq = 0;
  stream_chunk<D, NST, TILE>(a, smem, s_bars, seq, b, kvh, rb, L, c0, c1);
  const float *combine = reinterpret_cast<const float *>(smem);
  float *blk = reinterpret_cast<float *>(smem) + combine_floats<D, TILE>();  // acc[R][D], m[R], l[R]
  combine_block<D, TR>(combine, blk, R, nv);
  cluster_sync_all();  // every CTA's block is written and visible to CTA 0

  if (rank == 0) {
    // merge weights: block s's rows count exp(m_s - M) / sum over blocks of l exp(m - M)
    if (tid < nv) {
      const int r = tid;
      float ms[kMaxCluster], ls[kMaxCluster];
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) {
        ms[s] = -INFINITY;
        ls[s] = 0.f;
        if (s < CS) {
          const float *pb = map_to_rank(static_cast<const float *>(blk), (uint32_t)s);
          ls[s] = pb[R * D + R + r];
          ms[s] = ls[s] > 0.f ? pb[R * D + r] : -INFINITY;
        }
        M = fmaxf(M, ms[s]);
      }
      float Ls = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) {
        ms[s] = ls[s] > 0.f ? expf(ms[s] - M) : 0.f;
        Ls = fmaf(ls[s], ms[s], Ls);
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) s_w[s][r] = ms[s] * inv;
      s_lse[r] = Ls > 0.f ? M + logf(Ls) : -INFINITY;
    }
    __syncthreads();
    for (int idx = tid; idx < nv * D4; idx += kThreads) {
      const int r = idx / D4, d = (idx % D4) * 4;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) {
        if (s < CS) {
          const float w = s_w[s][r];
          const float4 v = *reinterpret_cast<const float4 *>(map_to_rank(static_cast<const float *>(blk), (uint32_t)s) +
                                                              r * D + d);
          A.x = fmaf(v.x, w, A.x), A.y = fmaf(v.y, w, A.y), A.z = fmaf(v.z, w, A.z), A.w = fmaf(v.w, w, A.w);
        }
      }
      const long long orow = out_row_of(p, b, kvh, rb, r);
      *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) + orow * D + d) =
          make_uint2(pack_bf16x2(A.x, A.y), pack_bf16x2(A.z, A.w));
      if (d == 0 && p.lse != nullptr) p.lse[orow] = s_lse[r];
    }
  }
  cluster_sync_all();  // no CTA leaves while CTA 0 may still read its shared memory
}

}  // namespace td
