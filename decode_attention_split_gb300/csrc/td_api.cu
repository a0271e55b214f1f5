// The C ABI declared in td.h: host-side argument checks, then one launch per call.
#include <math.h>

#include "td_internal.h"
#include "td_split_attn.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

}  // namespace

namespace td {

td_status cuda_fail(cudaError_t e) {
  cudaGetLastError();  // a launch error is reported once, by the call that met it
  g_last_cuda_error = (int)e;
  return TD_ERR_CUDA;
}

}  // namespace td

namespace {

using td::cuda_fail;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t elem_size(td_dtype d) { return d == TD_F32 ? 4 : 2; }

// Checks shared by the attention calls and fills the launch parameters; TD_OK or an error.
td_status prepare(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                  int B, int Hq, int Hkv, int T, int Smax, int D, float scale, int split, void *out, float *lse,
                  void *workspace, size_t workspace_bytes, uint32_t *dev_status, td::SplitPlan *plan,
                  td::SplitParams *p, bool q8 = false) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr || out == nullptr)
    return TD_ERR_INVALID_ARG;
  if (!isfinite(scale)) return TD_ERR_INVALID_ARG;
  const td_status st = td::plan_split(dtype, B, Hq, Hkv, T, Smax, D, split, plan, q8);
  if (st == TD_ERR_CUDA) return cuda_fail(cudaGetLastError());
  if (st != TD_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned4(seq_lens) ||
      (lse != nullptr && !aligned4(lse)) || (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < plan->bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return TD_ERR_WORKSPACE;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  *p = td::SplitParams{};
  p->q = q;
  p->k = k_cache;
  p->v = v_cache;
  p->seq_lens = seq_lens;
  p->out = out;
  p->lse = lse;
  p->ws_part = reinterpret_cast<float *>(ws + plan->off_part);
  p->counters = reinterpret_cast<int *>(ws);
  p->status = dev_status;
  p->B = B;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->G = Hq / Hkv;
  p->T = T;
  p->Smax = Smax;
  p->R = plan->R;
  p->RB = plan->RB;
  p->split = split;
  p->ns_ws = plan->ns_ws;
  p->p_target = plan->p_target;
  p->min_chunk = plan->min_chunk;
  p->warm_stages = plan->warm;
  p->qscale = scale * td::kLog2e;
  p->done = p->counters + plan->counters_n;
  return TD_OK;
}

td_status attn(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
               int B, int Hq, int Hkv, int T, int Smax, int D, float scale, int split, void *out, float *lse,
               void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream) {
  td::SplitPlan plan;
  td::SplitParams p;
  const td_status st = prepare(dtype, q, k_cache, v_cache, seq_lens, B, Hq, Hkv, T, Smax, D, scale, split, out, lse,
                               workspace, workspace_bytes, dev_status, &plan, &p);
  if (st != TD_OK) return st;
  const cudaError_t e = td::launch_split(dtype, D, plan, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

const char *td_status_string(td_status s) {
  switch (s) {
    case TD_OK: return "ok";
    case TD_ERR_INVALID_ARG: return "invalid argument";
    case TD_ERR_UNSUPPORTED: return "unsupported shape, dtype or alignment";
    case TD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case TD_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char *td_version(void) { return "td 0.1 (sm_103a)"; }

int td_last_cuda_error(void) { return g_last_cuda_error; }

size_t td_decode_workspace_bytes(int B, int Hq, int Hkv, int Smax, int D, int q_len, int split) {
  // the kernel variant (and so the grid and the partial slots) may differ by element type:
  // size for the larger of the two so one workspace serves both
  size_t bytes = 0;
  for (td_dtype dt : {TD_F32, TD_BF16}) {
    td::SplitPlan plan;
    if (td::plan_split(dt, B, Hq, Hkv, q_len, Smax, D, split, &plan) != TD_OK) return 0;
    if (plan.bytes > bytes) bytes = plan.bytes;
  }
  td::SplitPlan plan;  // the 8-bit cache kernel's layout (its grid may differ)
  if (td::plan_split(TD_BF16, B, Hq, Hkv, q_len, Smax, D, split, &plan, true) == TD_OK && plan.bytes > bytes)
    bytes = plan.bytes;
  return bytes;
}

td_status td_split_plan(td_dtype dtype, int B, int Hq, int Hkv, int Smax, int D, int q_len, int split, int *kernel,
                        int *grid, int *cluster, int *rows) {
  td::SplitPlan plan;
  const td_status st = td::plan_split(dtype, B, Hq, Hkv, q_len, Smax, D, split, &plan);
  if (st == TD_ERR_CUDA) return cuda_fail(cudaGetLastError());
  if (st != TD_OK) return st;
  if (kernel != nullptr) *kernel = !plan.mma ? 0 : plan.cluster > 0 ? 2 : 1;
  if (grid != nullptr) *grid = plan.grid;
  if (cluster != nullptr) *cluster = plan.cluster;
  if (rows != nullptr) *rows = plan.R;
  return TD_OK;
}

td_status td_kv_append(td_dtype dtype, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance, uint32_t *dev_status,
                       void *stream) {
  if (dtype != TD_F32 && dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr)
    return TD_ERR_INVALID_ARG;
  if (B < 1 || Hkv < 1 || T < 1 || Smax < 1 || D < 1) return TD_ERR_INVALID_ARG;
  if (B > 65535 || ((size_t)D * elem_size(dtype)) % 16 != 0) return TD_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(seq_lens) ||
      (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_append(elem_size(dtype), k_new, v_new, k_cache, v_cache, seq_lens, B, Hkv, T,
                                          Smax, D, advance, dev_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

td_status td_decode_attn(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D, float scale, int split,
                         void *out, float *lse, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                         void *stream) {
  return attn(dtype, q, k_cache, v_cache, seq_lens, B, Hq, Hkv, 1, Smax, D, scale, split, out, lse, workspace,
              workspace_bytes, dev_status, stream);
}

td_status td_verify_attn(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int T, int Smax, int D, float scale,
                         int split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                         uint32_t *dev_status, void *stream) {
  return attn(dtype, q, k_cache, v_cache, seq_lens, B, Hq, Hkv, T, Smax, D, scale, split, out, lse, workspace,
              workspace_bytes, dev_status, stream);
}

td_status td_lse_merge(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows,
                       int NS, int D, int split, td_dtype out_dtype, void *out, float *lse, void *stream) {
  if (m == nullptr || l == nullptr || acc == nullptr || seq_lens == nullptr || out == nullptr)
    return TD_ERR_INVALID_ARG;
  if (B < 1 || rows < 1 || NS < 1 || D < 1 || split < 1) return TD_ERR_INVALID_ARG;
  if (out_dtype != TD_F32 && out_dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (D % 4 != 0 || D > 1024 || B > 65535) return TD_ERR_UNSUPPORTED;
  if (!aligned4(m) || !aligned4(l) || !aligned4(acc) || !aligned4(seq_lens) ||
      !aligned4(out) || (lse != nullptr && !aligned4(lse)))
    return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_merge(m, l, acc, seq_lens, B, rows, NS, D, split, out_dtype, out, lse,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

}  // extern "C"

extern "C" {

td_status td_rope_kv_append(td_dtype dtype, const void *q, void *q_out, int Hq, const void *k_new, const void *v_new,
                            const float *cos_t, const float *sin_t, void *k_cache, void *v_cache, int32_t *seq_lens,
                            int B, int Hkv, int T, int Smax, int D, int advance, uint32_t *dev_status, void *stream) {
  if (dtype != TD_F32 && dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
      cos_t == nullptr || sin_t == nullptr || (q == nullptr) != (q_out == nullptr))
    return TD_ERR_INVALID_ARG;
  if (B < 1 || Hkv < 1 || T < 1 || Smax < 1 || D < 2 || (q != nullptr && Hq < 1)) return TD_ERR_INVALID_ARG;
  // rows are rotated as pairs of 16-byte vectors (i, i + D/2)
  if (B > 65535 || ((size_t)D * elem_size(dtype)) % 32 != 0) return TD_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(cos_t) ||
      !aligned16(sin_t) || !aligned4(seq_lens) || (q != nullptr && (!aligned16(q) || !aligned16(q_out))) ||
      (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_rope_append(elem_size(dtype), q, q_out, Hq, k_new, v_new, cos_t, sin_t, k_cache,
                                               v_cache, seq_lens, B, Hkv, T, Smax, D, advance, dev_status,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

td_status td_rope_append_attn(td_dtype dtype, const void *q, const void *k_new, const void *v_new, const float *cos_t,
                              const float *sin_t, void *k_cache, void *v_cache, int32_t *seq_lens, int B, int Hq,
                              int Hkv, int T, int Smax, int D, float scale, int split, int advance, void *out,
                              float *lse, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                              void *stream) {
  if (k_new == nullptr || v_new == nullptr || (cos_t == nullptr) != (sin_t == nullptr)) return TD_ERR_INVALID_ARG;
  if (dtype != TD_BF16) return TD_ERR_UNSUPPORTED;  // the tensor-core kernels carry the fused step
  if (!aligned16(k_new) || !aligned16(v_new) || (cos_t != nullptr && (!aligned16(cos_t) || !aligned16(sin_t))))
    return TD_ERR_UNSUPPORTED;
  td::SplitPlan plan;
  td::SplitParams p;
  const td_status st = prepare(dtype, q, k_cache, v_cache, seq_lens, B, Hq, Hkv, T, Smax, D, scale, split, out, lse,
                               workspace, workspace_bytes, dev_status, &plan, &p);
  if (st != TD_OK) return st;
  if (!plan.mma) return TD_ERR_UNSUPPORTED;
  p.k_new = k_new;
  p.v_new = v_new;
  p.rope_cos = cos_t;
  p.rope_sin = sin_t;
  p.advance_lens = advance ? seq_lens : nullptr;
  const cudaError_t e = td::launch_split(dtype, D, plan, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

}  // extern "C"

extern "C" size_t td_spec_workspace_bytes(int B, int G, int V) {
  if (B < 1 || G < 0 || G > td::kMaxDraft || V < 1) return 0;
  return td::spec_workspace_bytes(B, G, V);
}

extern "C" td_status td_spec_accept(const float *target_logits, const float *draft_logits,
                                    const int32_t *draft_tokens, const float *uniforms, int B, int G, int V,
                                    float temperature, int32_t *n_accepted, int32_t *next_token, void *workspace,
                                    size_t workspace_bytes, uint32_t *dev_status, void *stream) {
  const bool greedy = temperature == 0.f;
  if (target_logits == nullptr || n_accepted == nullptr || next_token == nullptr ||
      (G > 0 && draft_tokens == nullptr) || (!greedy && (uniforms == nullptr || (G > 0 && draft_logits == nullptr))))
    return TD_ERR_INVALID_ARG;
  if (B < 1 || G < 0 || V < 1 || !(temperature >= 0.f) || !isfinite(temperature)) return TD_ERR_INVALID_ARG;
  if (G > td::kMaxDraft) return TD_ERR_UNSUPPORTED;
  if ((long long)B * td::spec_slices(V) > 0x7fffffffLL) return TD_ERR_UNSUPPORTED;
  if (!aligned4(target_logits) || (draft_logits != nullptr && !aligned4(draft_logits)) ||
      (draft_tokens != nullptr && !aligned4(draft_tokens)) || (uniforms != nullptr && !aligned4(uniforms)) ||
      !aligned4(n_accepted) || !aligned4(next_token) || (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  // 16-byte loads need 16-byte aligned rows
  if ((V & 3) == 0 && (!aligned16(target_logits) || (!greedy && G > 0 && !aligned16(draft_logits))))
    return TD_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < td::spec_workspace_bytes(B, G, V) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return TD_ERR_WORKSPACE;
  const cudaError_t e = td::launch_spec_accept(target_logits, greedy ? nullptr : draft_logits, draft_tokens,
                                               greedy ? nullptr : uniforms, B, G, V, temperature, n_accepted,
                                               next_token, dev_status, workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

extern "C" {

td_status td_quantize_q8(td_dtype dtype, const void *x, long long rows, int D, int8_t *codes, float *scales,
                         void *stream) {
  if (dtype != TD_F32 && dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (x == nullptr || codes == nullptr || scales == nullptr || rows < 1 || D < 1) return TD_ERR_INVALID_ARG;
  if (!aligned4(scales)) return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_quantize_q8(elem_size(dtype), x, rows, D, codes, scales,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

td_status td_kv_append_q8(td_dtype dtype, const void *k_new, const void *v_new, int8_t *k_codes, float *k_scales,
                          int8_t *v_codes, float *v_scales, int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D,
                          int advance, uint32_t *dev_status, void *stream) {
  if (dtype != TD_F32 && dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (k_new == nullptr || v_new == nullptr || k_codes == nullptr || k_scales == nullptr || v_codes == nullptr ||
      v_scales == nullptr || seq_lens == nullptr)
    return TD_ERR_INVALID_ARG;
  if (B < 1 || Hkv < 1 || T < 1 || Smax < 1 || D < 1) return TD_ERR_INVALID_ARG;
  if (B > 65535 || !aligned4(seq_lens) || !aligned4(k_scales) || !aligned4(v_scales) ||
      (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_append_q8(elem_size(dtype), k_new, v_new, k_codes, k_scales, v_codes, v_scales,
                                             seq_lens, B, Hkv, T, Smax, D, advance, dev_status,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

td_status td_verify_attn_q8(const void *q, const int8_t *k_codes, const float *k_scales, const int8_t *v_codes,
                            const float *v_scales, const int32_t *seq_lens, int B, int Hq, int Hkv, int T, int Smax,
                            int D, float scale, int split, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, uint32_t *dev_status, void *stream) {
  if (k_scales == nullptr || v_scales == nullptr) return TD_ERR_INVALID_ARG;
  // the scale maps step by whole 16-byte units along a sequence
  if (Smax % 4 != 0 || !aligned16(k_scales) || !aligned16(v_scales)) return TD_ERR_UNSUPPORTED;
  td::SplitPlan plan;
  td::SplitParams p;
  const td_status st = prepare(TD_BF16, q, k_codes, v_codes, seq_lens, B, Hq, Hkv, T, Smax, D, scale, split, out,
                               lse, workspace, workspace_bytes, dev_status, &plan, &p, true);
  if (st != TD_OK) return st;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  const cudaError_t e = td::launch_split(TD_BF16, D, plan, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}

td_status td_decode_attn_q8(const void *q, const int8_t *k_codes, const float *k_scales, const int8_t *v_codes,
                            const float *v_scales, const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D,
                            float scale, int split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            uint32_t *dev_status, void *stream) {
  return td_verify_attn_q8(q, k_codes, k_scales, v_codes, v_scales, seq_lens, B, Hq, Hkv, 1, Smax, D, scale, split,
                           out, lse, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"

extern "C" td_status td_prefill_attn(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                                     int B, int Hq, int Hkv, int T, int Smax, int D, float scale, void *out, float *lse,
                                     uint32_t *dev_status, void *stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr || out == nullptr)
    return TD_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || Smax < 1 || Hq % Hkv != 0 || !isfinite(scale)) return TD_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || T > Smax || B > 65535 || Hq > 65535 || (T + 127) / 128 > 65535)
    return TD_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned4(seq_lens) ||
      (lse != nullptr && !aligned4(lse)) || (dev_status != nullptr && !aligned4(dev_status)))
    return TD_ERR_UNSUPPORTED;
  const cudaError_t e = td::launch_prefill(q, k_cache, v_cache, seq_lens, B, Hq, Hkv, T, Smax, D, scale, out, lse,
                                           dev_status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? TD_OK : cuda_fail(e);
}
