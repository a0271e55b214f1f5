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
  int RP;        // padded query rows per CTA (1, 2, 4 or 8)
  int R;         // real query rows per CTA
  int RB;        // row blocks per kv head
  int ns_ws;     // partial slots per query row
  int p_target;  // CTAs that fill the GPU once
  int grid;      // CTAs launched
  int smem;      // dynamic shared memory per CTA
  size_t off_m, off_l, off_acc, bytes;  // workspace layout
};

// Fills *plan for the current device; TD_OK, or an error for unsupported shapes.
td_status plan_split(td_dtype dtype, int B, int Hq, int Hkv, int T, int Smax, int D, int split, SplitPlan *plan);

cudaError_t launch_split(td_dtype dtype, int D, const SplitPlan &plan, const SplitParams &p, cudaStream_t stream);

cudaError_t launch_merge(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows,
                         int NS, int D, int split, td_dtype out_dtype, void *out, float *lse, cudaStream_t stream);

cudaError_t launch_append(size_t elem_bytes, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                          uint32_t *dev_status, cudaStream_t stream);

// SM count of the current device (cached per device).
int device_sm_count(int device);

}  // namespace td
