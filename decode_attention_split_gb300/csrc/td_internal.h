// Host-side interfaces between the td translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "td.h"

namespace td {

struct SplitParams;

// Launch geometry and workspace layout of one split-attention call.
struct SplitPlan {
  bool mma;      // tensor-core kernel (bf16) or CUDA-core kernel
  int RP;        // CUDA-core: padded query rows per CTA (1, 2, 4 or 8); tensor-core: m tiles (1 or 2)
  int R;         // real query rows per CTA
  int RB;        // row blocks per kv head
  int ns_ws;     // partial slots per query row
  int p_target;  // CTAs that fill the GPU once
  bool spare;    // p_target leaves one slot per group for the previous call's merging CTAs
  int grid;      // CTAs launched
  int smem;      // dynamic shared memory per CTA
  int min_chunk; // smallest automatic chunk (keys)
  int warm;      // 64-row units of K and V each CTA warms in L2 before the wait for the previous kernel
  int cluster;   // 0: persistent kernel; else CTAs per cluster of the cluster kernel (grid = groups x cluster)
  int counters_n;  // completion and slice-merge counters before the fused step's read count in the workspace
  bool q8;       // int8 cache (codes + per-row scales): the quantised-cache kernel
  size_t off_part, bytes;  // workspace layout: counters, then partial blocks
};

// Records a failed CUDA call for td_last_cuda_error (and clears the runtime's last-error slot,
// so a later call does not report it as its own); returns TD_ERR_CUDA.
td_status cuda_fail(cudaError_t e);

// Fills *plan for the current device; TD_OK, or an error for unsupported shapes.
// q8: the caches hold int8 codes with per-row scales (q and out are bf16; dtype must be TD_BF16).
td_status plan_split(td_dtype dtype, int B, int Hq, int Hkv, int T, int Smax, int D, int split, SplitPlan *plan,
                     bool q8 = false);

// Per-row int8 quantisation (codes + fp32 scales) of `rows` rows of D elements.
cudaError_t launch_quantize_q8(size_t elem_bytes, const void *x, long long rows, int D, int8_t *codes, float *scales,
                               cudaStream_t stream);
// Quantises new rows [B, Hkv, T, D] into an int8 cache at seq_lens (td_kv_append's rules).
cudaError_t launch_append_q8(size_t elem_bytes, const void *k_new, const void *v_new, int8_t *k_codes,
                             float *k_scales, int8_t *v_codes, float *v_scales, int32_t *seq_lens, int B, int Hkv,
                             int T, int Smax, int D, int advance, uint32_t *dev_status, cudaStream_t stream);

cudaError_t launch_split(td_dtype dtype, int D, const SplitPlan &plan, const SplitParams &p, cudaStream_t stream);

cudaError_t launch_merge(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows,
                         int NS, int D, int split, td_dtype out_dtype, void *out, float *lse, cudaStream_t stream);

cudaError_t launch_append(size_t elem_bytes, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                          uint32_t *dev_status, cudaStream_t stream);

cudaError_t launch_rope_append(size_t elem_bytes, const void *q, void *q_out, int Hq, const void *k_new,
                               const void *v_new, const float *cos_t, const float *sin_t, void *k_cache,
                               void *v_cache, int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                               uint32_t *dev_status, cudaStream_t stream);

// Speculative accept/reject: most draft tokens per step, and the launch.
constexpr int kMaxDraft = 16;
constexpr int kMaxCluster = 16;  // CTAs per cluster, at most
int spec_slices(int V);
size_t spec_workspace_bytes(int B, int G, int V);
cudaError_t launch_spec_accept(const float *target, const float *draft, const int32_t *tokens, const float *uniforms,
                               int B, int G, int V, float temperature, int32_t *n_out, int32_t *tok_out,
                               uint32_t *status, void *workspace, cudaStream_t stream);

// Tiled causal prefill attention on the tensor cores (tcgen05); bf16, D 64 or 128.
cudaError_t launch_prefill(const void *q, const void *k, const void *v, const int32_t *seq_lens, int B, int Hq, int Hkv,
                           int T, int Smax, int D, float scale, void *out, float *lse, uint32_t *status,
                           cudaStream_t stream);

// SM count of the current device (cached per device).
int device_sm_count(int device);

// Launches `kernel` with programmatic dependent launch allowed: its CTAs may be scheduled
// while the previous kernel in the stream drains; every td kernel starts with a
// griddepcontrol.wait, so it still sees all of that kernel's writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace td
