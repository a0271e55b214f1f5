// td_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.
//
// td_decode_attn needs a caller-provided workspace (completion counters and per-chunk partial
// results). Some callers have no way to provide one: a plugin or launch hook that is handed
// only the input and output pointers by its host framework, a service loop that must not
// allocate once it is serving (allocation can block on device synchronisation or fail under
// memory pressure), or code running while another runtime owns the whole device heap. For them
// this entry point keeps its scratch in a fixed array compiled into the library, so it needs
// nothing beyond the caller's inputs and outputs and calls no allocator.
//
// The array is kScratchBytes (4 MiB) of device memory that every GPU which loads the library
// holds until the process exits. Calls whose workspace would exceed it are rejected.
#include <mutex>

#include "td_internal.h"
#include "td_split_attn.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; it keeps whatever the last call left in it.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device. In host code the array's name is only a
// host-side handle, so the address is looked up once per device (with that device current)
// and cached.
td_status scratch_address(void **addr) {
  int dev = 0;
  const cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) return td::cuda_fail(ed);
  if (dev < 0 || dev >= kMaxDevices) return TD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return td::cuda_fail(e);
    if (p == nullptr) return td::cuda_fail(cudaErrorInvalidSymbol);
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return TD_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" td_status td_decode_attn_noalloc(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D,
                                            float scale, int split, void *out, float *lse, uint32_t *dev_status,
                                            void *stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr || out == nullptr)
    return TD_ERR_INVALID_ARG;
  if (!isfinite(scale)) return TD_ERR_INVALID_ARG;
  td::SplitPlan plan;
  const td_status st = td::plan_split(dtype, B, Hq, Hkv, 1, Smax, D, split, &plan);
  if (st == TD_ERR_CUDA) return td::cuda_fail(cudaGetLastError());
  if (st != TD_OK) return st;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(seq_lens, 4) || (lse != nullptr && !aligned(lse, 4)) || (dev_status != nullptr && !aligned(dev_status, 4)))
    return TD_ERR_UNSUPPORTED;
  // the shape needs more scratch than the array holds: the same test a caller can make with
  // td_decode_workspace_bytes (the largest layout over the element types), so the documented
  // limit and this check agree
  if (plan.bytes > kScratchBytes || td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, 1, split) > kScratchBytes)
    return TD_ERR_WORKSPACE;
  void *scratch = nullptr;
  const td_status sa = scratch_address(&scratch);
  if (sa != TD_OK) return sa;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the completion counters must start at zero; the previous call (any shape) may have left
  // partial results where this layout keeps its counters
  const cudaError_t em = cudaMemsetAsync(scratch, 0, plan.off_part, s);
  if (em != cudaSuccess) return td::cuda_fail(em);
  unsigned char *ws = static_cast<unsigned char *>(scratch);
  td::SplitParams p = {};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse = lse;
  p.ws_part = reinterpret_cast<float *>(ws + plan.off_part);
  p.counters = reinterpret_cast<int *>(ws);
  p.status = dev_status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.T = 1;
  p.Smax = Smax;
  p.R = plan.R;
  p.RB = plan.RB;
  p.split = split;
  p.ns_ws = plan.ns_ws;
  p.p_target = plan.p_target;
  p.min_chunk = plan.min_chunk;
  p.warm_stages = plan.warm;
  p.qscale = scale * td::kLog2e;
  p.done = p.counters + plan.counters_n;
  const cudaError_t e = td::launch_split(dtype, D, plan, p, s);
  return e == cudaSuccess ? TD_OK : td::cuda_fail(e);
}
