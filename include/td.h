/*
 * td.h - split-KV decode attention over a static KV cache, for NVIDIA GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels. Every pointer argument is a device pointer
 * unless stated otherwise; every buffer is allocated and owned by the caller; the library
 * allocates nothing, keeps no state beyond a per-device cache of attribute queries, and
 * may be called from several host threads at once.
 *
 * Operations (sources are web pages, cited by title and section):
 *   td_kv_append   write new key/value rows at position seq_lens[b] of a preallocated
 *                  cache ("tinydecode", "how the decode step is put together": the cache
 *                  write is an index_put_ at seq_lens, which live on the device).
 *   td_decode_attn single-token attention of every query head over its sequence's cache
 *                  rows j < seq_lens[b], split into key chunks whose partial softmax
 *                  (m, l, acc) is merged by log-sum-exp ("tinydecode", same section;
 *                  "llm-decode-cuda", split-KV attention section: one block per kv head
 *                  and chunk serves the whole query-head group).
 *   td_verify_attn the same for a chunk of T new query tokens that are causal among
 *                  themselves ("tinydecode", "speculative decoding": the verify pass over
 *                  k+1 tokens with the head group folded so the cache is read once).
 *   td_lse_merge   the log-sum-exp merge of per-split partials on its own.
 *   td_rope_kv_append    the cache write with the new keys (and optionally the queries)
 *                  rotated to their positions first ("llm-decode-cuda" fuses "RoPE +
 *                  KV-cache write" in its decode step; "tinydecode" lists an in-place rope).
 *   td_rope_append_attn  the whole decode or verify step of one layer in one launch:
 *                  rotation, cache write and split attention.
 *   td_spec_accept the accept/reject step after a verify pass ("tinydecode", "speculative
 *                  decoding"; "FlashSpec", "How it works": Leviathan et al. Algorithm 1).
 *   td_prefill_attn  causal attention of a long chunk of T new tokens (a prompt) over the
 *                  cache: td_verify_attn's result, tiled for the tensor cores (tcgen05)
 *                  ("llm-decode-cuda" names a tiled FlashAttention-style prefill kernel as
 *                  its next step; "tinydecode"'s prefill path is causal over the prompt).
 *   td_*_q8        an 8-bit KV cache: int8 codes with one fp32 scale per row (the per-row
 *                  INT8 scheme "llm-decode-cuda" applies to its weights, for the K/V bytes).
 *
 * Layouts (row-major, contiguous, element type given by td_dtype):
 *   q, out         [B, Hq, D] for decode; [B, Hq, T, D] for verify
 *   k/v cache      [B, Hkv, Smax, D]
 *   seq_lens       int32 [B], on the device
 *   lse            fp32 [B, Hq] (decode) or [B, Hq, T] (verify); nullable
 *   partials       fp32 m, l [B, rows, NS]; acc [B, rows, NS, D]  (rows = Hq*T, row = hq*T + t)
 * Query head hq reads kv head hq / (Hq / Hkv) (contiguous groups, Hq % Hkv == 0).
 * Accumulation and the softmax statistics are fp32. out is written in the cache's dtype,
 * rounded to nearest even.
 *
 * Errors. Arguments are checked on the host before anything is launched: a bad shape,
 * a null or misaligned pointer (q, caches, new rows, out and workspace need 16-byte
 * alignment), an unsupported head dimension or a too-small workspace returns an error
 * code and launches nothing. TD_ERR_CUDA reports a launch failure (cudaGetLastError).
 * Problems in device-resident data never stop a kernel: they are clamped or skipped as
 * described per call and OR a TD_DEV_* bit into *dev_status (a caller-owned device
 * uint32; pass NULL to ignore them). No call synchronises with the host, allocates, or
 * reads seq_lens on the host, so every call can be captured in a CUDA graph.
 *
 * stream: a cudaStream_t passed as void* (NULL = the legacy default stream).
 */
#ifndef TD_H
#define TD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum td_status {
  TD_OK = 0,
  TD_ERR_INVALID_ARG = 1, /* null pointer, bad shape, bad scale */
  TD_ERR_UNSUPPORTED = 2, /* valid but not built: head dim, dtype, alignment, batch size */
  TD_ERR_WORKSPACE = 3,   /* workspace missing or smaller than td_decode_workspace_bytes() */
  TD_ERR_CUDA = 4         /* a CUDA call failed (see td_last_cuda_error) */
} td_status;

typedef enum td_dtype { TD_F32 = 0, TD_BF16 = 1 } td_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define TD_DEV_SEQLEN_CLAMPED 1u   /* seq_lens[b] > Smax in attention: Smax rows attended */
#define TD_DEV_APPEND_OVERFLOW 2u  /* append with seq_lens[b] < 0 or seq_lens[b] + T > Smax: b skipped */
#define TD_DEV_VERIFY_SHORT 4u     /* verify with seq_lens[b] < T: rows that see no key give 0 */
#define TD_DEV_NEGATIVE_SEQLEN 8u  /* seq_lens[b] < 0 in attention: treated as 0 */
#define TD_DEV_WAIT_TIMEOUT 16u    /* a bounded wait for an asynchronous copy gave up: output invalid */
#define TD_DEV_WORKSPACE_DIRTY 32u /* a completion counter was not zero: workspace not zeroed for this
                                      layout; output invalid (zero the workspace and call again) */
#define TD_DEV_BAD_TOKEN 64u       /* speculative accept: a draft token outside [0, V), counted as rejected */

/* Largest batch a call accepts. */
#define TD_MAX_BATCH 1024

const char *td_status_string(td_status s);
const char *td_version(void);
/* Last CUDA error code seen by a call that returned TD_ERR_CUDA on this host thread. */
int td_last_cuda_error(void);

/*
 * Workspace for td_decode_attn / td_verify_attn, in bytes, for the current CUDA device.
 * q_len = T (1 for decode); split as passed to the attention call (0 = automatic).
 * The workspace holds a counter area followed by per-split partials; their layout follows
 * the shape arguments. It must be zero-filled (e.g. cudaMemset) before its first use; every
 * call that runs to completion leaves its counter area zero again, so the workspace can be
 * reused by later calls with the same (B, Hq, Hkv, Smax, D, q_len, split) on one stream.
 * Before using it for other shapes, zero it again (or use another). Calls running
 * concurrently need separate workspaces. Returns 0 for invalid arguments.
 */
size_t td_decode_workspace_bytes(int B, int Hq, int Hkv, int Smax, int D, int q_len, int split);

/*
 * The launch td_decode_attn (q_len = 1) or td_verify_attn (q_len = T) makes for these
 * arguments on the current CUDA device; nothing is launched. Outputs are host pointers,
 * each nullable:
 *   *kernel  0: CUDA-core split kernel (fp32 caches);
 *            1: tensor-core persistent kernel (bf16; CTAs walk (b, kv head, row block, chunk)
 *               items, partials meet in the workspace and the CTA finishing a group's last
 *               chunk merges them; for row blocks of more than 16 rows in a launch where each
 *               CTA holds one item, the CTAs holding the group's last tickets merge one row
 *               each);
 *            2: tensor-core cluster kernel (bf16, split = 0, few groups: one thread-block
 *               cluster per (b, kv head, row block), one chunk per CTA, the merge done in
 *               distributed shared memory; the workspace is not touched);
 *   *grid    CTAs launched;  *cluster  CTAs per cluster (0 unless kernel 2);
 *   *rows    query rows per CTA (bf16: a kv head's rows cut into row blocks of at most 24: up to
 *            8 on the narrow n8 tile, 9 to 16 on the m16 tile, 17 to 24 on the 24-row tile).
 * Returns what the attention call would return for a bad shape, TD_ERR_CUDA without a device.
 */
td_status td_split_plan(td_dtype dtype, int B, int Hq, int Hkv, int Smax, int D, int q_len, int split, int *kernel,
                        int *grid, int *cluster, int *rows);

/*
 * Cache append: for each b with 0 <= L = seq_lens[b] and L + T <= Smax, copies
 * k_new[b, h, t, :] to k_cache[b, h, L + t, :] (and v likewise) bit for bit for all h < Hkv,
 * t < T. With advance != 0, seq_lens[b] += T afterwards (same launch, after every read of
 * seq_lens[b]). A sequence that does not fit is left untouched and sets
 * TD_DEV_APPEND_OVERFLOW. k_new, v_new: [B, Hkv, T, D]; caches [B, Hkv, Smax, D].
 */
td_status td_kv_append(td_dtype dtype, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D, int advance,
                       uint32_t *dev_status, void *stream);

/*
 * Decode attention: out[b, hq, :] = softmax_j(scale * q[b, hq, :] . k[b, kvh, j, :]) v[b, kvh, j, :]
 * over j < L_b = seq_lens[b] (clamped to [0, Smax], see TD_DEV_* bits); L_b = 0 gives
 * out = 0 and lse = -inf. lse[b, hq] = ln sum_j exp(scale * q . k_j) (nullable).
 * split: keys per chunk; 0 lets the library size chunks from the device lengths and the
 * GPU's SM count. The grid depends only on the arguments (never on the lengths), and
 * chunks past a sequence's length do no work. D must be 64 or 128.
 */
td_status td_decode_attn(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D, float scale, int split,
                         void *out, float *lse, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                         void *stream);

/*
 * Verify-chunk attention: query row (hq, t), t < T, attends keys j < L_b - T + t + 1, where
 * L_b = seq_lens[b] already counts the T new tokens (append them first). q/out [B, Hq, T, D],
 * lse [B, Hq, T]. A row that sees no key (L_b < T) gives out = 0, lse = -inf and sets
 * TD_DEV_VERIFY_SHORT. Otherwise as td_decode_attn.
 */
td_status td_verify_attn(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int T, int Smax, int D, float scale,
                         int split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                         uint32_t *dev_status, void *stream);

/*
 * Log-sum-exp merge of per-split partials computed with split size `split` (>= 1).
 * For each (b, row) the active splits are s < min(NS, ceil(max(seq_lens[b], 0) / split));
 * those with l > 0 are merged:
 *   M = max_s m_s,  Lsum = sum_s l_s exp(m_s - M),  out = sum_s acc_s exp(m_s - M) / Lsum,
 *   lse = M + ln Lsum.
 * A row with no such split gets out = 0, lse = -inf. m, l: [B, rows, NS]; acc [B, rows, NS, D]
 * (acc unnormalised); out [B, rows, D] in out_dtype; lse fp32 [B, rows] (nullable).
 * D must be a multiple of 4 and at most 1024.
 */
td_status td_lse_merge(const float *m, const float *l, const float *acc, const int32_t *seq_lens, int B, int rows,
                       int NS, int D, int split, td_dtype out_dtype, void *out, float *lse, void *stream);

/*
 * Rotary position embedding: the pages name the kernel but print no formula; the layout of
 * the llama checkpoints is used. For i < D/2 the pair (x[i], x[i + D/2]) of a row at position
 * P turns by the angle whose cosine and sine are cos_t[P * D/2 + i] and sin_t[P * D/2 + i]:
 *   y[i] = x[i] cos - x[i + D/2] sin,   y[i + D/2] = x[i + D/2] cos + x[i] sin,
 * in fp32, rounded to nearest even into the element type. cos_t, sin_t: fp32 [Smax, D/2]
 * device tables (any angles: the caller chooses the frequencies and any scaling).
 */

/*
 * RoPE + cache append. For each b with 0 <= L = seq_lens[b] and L + T <= Smax, token t sits
 * at position L + t:
 *   k_cache[b, h, L+t, :] = rope(k_new[b, h, t, :], L+t),  v_cache[b, h, L+t, :] = v_new[b, h, t, :],
 *   q_out[b, hq, t, :]    = rope(q[b, hq, t, :], L+t)     (when q is given; q_out may be q),
 * then seq_lens[b] += T if advance (same launch, after the read). A sequence that does not
 * fit is left untouched (its q_out rows too) and sets TD_DEV_APPEND_OVERFLOW.
 * q, q_out: [B, Hq, T, D] or both NULL; k_new, v_new [B, Hkv, T, D]; caches [B, Hkv, Smax, D].
 * D * element size must be a multiple of 32 bytes; tables and row pointers 16-byte aligned.
 */
td_status td_rope_kv_append(td_dtype dtype, const void *q, void *q_out, int Hq, const void *k_new, const void *v_new,
                            const float *cos_t, const float *sin_t, void *k_cache, void *v_cache, int32_t *seq_lens,
                            int B, int Hkv, int T, int Smax, int D, int advance, uint32_t *dev_status, void *stream);

/*
 * One layer's decode (T = 1) or verify (T > 1) step in one launch: for every b whose new rows
 * fit (0 <= L = seq_lens[b], L + T <= Smax), the result of
 *   td_rope_kv_append(q -> rotated q, k_new, v_new at L .. L+T-1)   (no rotation if cos_t is NULL)
 *   td_verify_attn(rotated q, caches, lengths L + T)
 * with out/lse as td_verify_attn defines them, and seq_lens[b] = L + T afterwards if advance.
 * The new rows reach the attention without a round trip through memory, the cache rows are
 * written in the same launch, and the lengths are advanced once every CTA has read them.
 * A sequence whose rows do not fit is left untouched, gives out = 0 and lse = -inf, and sets
 * TD_DEV_APPEND_OVERFLOW. bf16 only (TD_ERR_UNSUPPORTED otherwise), D 64 or 128.
 * q, out [B, Hq, T, D]; lse [B, Hq, T] (nullable); workspace as td_decode_workspace_bytes(q_len = T).
 */
td_status td_rope_append_attn(td_dtype dtype, const void *q, const void *k_new, const void *v_new, const float *cos_t,
                              const float *sin_t, void *k_cache, void *v_cache, int32_t *seq_lens, int B, int Hq,
                              int Hkv, int T, int Smax, int D, float scale, int split, int advance, void *out,
                              float *lse, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                              void *stream);

/*
 * Speculative accept/reject for B sequences, each with G draft tokens (0 <= G <= 16) over a
 * vocabulary of V:
 *   target_logits [B, G+1, V] fp32   row i: the target's next-token logits after the prefix
 *                                     and draft tokens 0..i-1 (row G: the bonus row)
 *   draft_logits  [B, G, V] fp32     row i: the logits draft token i was drawn from
 *   draft_tokens  [B, G] int32
 *   uniforms      [B, G+1] fp32 in [0, 1): entry i < G decides draft token i, entry G draws
 *                                     the extra token (the caller's random numbers)
 * With p = softmax(target / temperature), q = softmax(draft / temperature): draft token i is
 * kept while uniforms[i] < min(1, p_i(x_i) / q_i(x_i)) (tested in log space); n_accepted[b]
 * counts the kept prefix. next_token[b] is drawn by inverse CDF (the smallest id whose
 * running weight exceeds u * total) from max(0, p_n - q_n) when a token was rejected at n,
 * else from p_G; a residual with no weight falls back to p_n. temperature == 0 is greedy:
 * keep while the draft token is the target's argmax (lowest id on ties); next_token is
 * the argmax of row n; draft_logits and uniforms may then be NULL. A draft token outside
 * [0, V) counts as rejected and sets TD_DEV_BAD_TOKEN. All pointers are device pointers,
 * 4-byte aligned (logits 16-byte aligned when V % 4 == 0); n_accepted, next_token int32 [B].
 * workspace: td_spec_workspace_bytes(B, G, V) bytes, 256-byte aligned, zero-filled before its
 * first use; every call leaves it ready for the next on the same stream (any shape up to the
 * size it was sized for). Two launches (the second only when sampling).
 */
size_t td_spec_workspace_bytes(int B, int G, int V);
td_status td_spec_accept(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                         const float *uniforms, int B, int G, int V, float temperature, int32_t *n_accepted,
                         int32_t *next_token, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                         void *stream);

/*
 * 8-bit KV cache. A row x of D elements is stored as int8 codes and one fp32 scale:
 *   scale = max_i |x_i| / 127,  code_i = clamp(rint(x_i / scale), -127, 127) (0 when scale == 0),
 * computed in fp32 with IEEE division and ties to even, and reads back as code_i * scale.
 * Caches: k_codes, v_codes int8 [B, Hkv, Smax, D]; k_scales, v_scales fp32 [B, Hkv, Smax].
 */

/* Quantises `rows` rows of D elements of x (TD_F32 or TD_BF16) into codes [rows, D] and scales [rows]. */
td_status td_quantize_q8(td_dtype dtype, const void *x, long long rows, int D, int8_t *codes, float *scales,
                         void *stream);

/* td_kv_append for an 8-bit cache: the new rows (dtype TD_F32 or TD_BF16) are quantised into
 * rows L_b .. L_b+T-1; the same overflow rule, advance and status bit. */
td_status td_kv_append_q8(td_dtype dtype, const void *k_new, const void *v_new, int8_t *k_codes, float *k_scales,
                          int8_t *v_codes, float *v_scales, int32_t *seq_lens, int B, int Hkv, int T, int Smax, int D,
                          int advance, uint32_t *dev_status, void *stream);

/* td_decode_attn / td_verify_attn over an 8-bit cache: the same results as over the cache
 * the codes stand for (code * scale), q and out bf16, D 64 or 128, Smax a multiple of 4,
 * scales 16-byte aligned. The workspace is td_decode_workspace_bytes' (which covers it). */
td_status td_decode_attn_q8(const void *q, const int8_t *k_codes, const float *k_scales, const int8_t *v_codes,
                            const float *v_scales, const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D,
                            float scale, int split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            uint32_t *dev_status, void *stream);
td_status td_verify_attn_q8(const void *q, const int8_t *k_codes, const float *k_scales, const int8_t *v_codes,
                            const float *v_scales, const int32_t *seq_lens, int B, int Hq, int Hkv, int T, int Smax,
                            int D, float scale, int split, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, uint32_t *dev_status, void *stream);

/*
 * Prefill: query row (hq, t), t < T, attends keys j < L_b - T + t + 1, L_b = seq_lens[b]
 * clamped to [0, Smax] and counting the T new tokens (whose K/V rows must already be in the
 * cache): td_verify_attn's definition, for long chunks. bf16 only; D 64 or 128; T at most
 * 65535 * 128 (TD_ERR_UNSUPPORTED beyond). One CTA per 128 query rows of one query head;
 * no workspace. q, out [B, Hq, T, D]; lse [B, Hq, T] (nullable). Status bits as
 * td_verify_attn; a bounded wait that gives up sets TD_DEV_WAIT_TIMEOUT.
 */
td_status td_prefill_attn(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens, int B,
                          int Hq, int Hkv, int T, int Smax, int D, float scale, void *out, float *lse,
                          uint32_t *dev_status, void *stream);

/*
 * Diagnostic of the bounded wait (the pages describe no such call; it exists so that the
 * failure path every kernel relies on can be exercised without a fault). One CTA waits for
 * the first phase of an mbarrier that nothing arrives on and no copy completes, with the
 * kernels' wait routine and a limit of limit_cycles SM cycles (1 .. 1e9, about half a second
 * at most; TD_ERR_INVALID_ARG outside). The wait gives up, the kernel ORs
 * TD_DEV_WAIT_TIMEOUT into *dev_status (device, required) and returns; nothing is in flight
 * when it gives up. waited_cycles (device, nullable, 8-byte aligned) receives the cycles the
 * wait took. Asynchronous on `stream`.
 */
td_status td_selftest_wait_timeout(long long limit_cycles, uint32_t *dev_status, long long *waited_cycles,
                                   void *stream);

/*
 * Decode attention without a workspace argument: the same computation and arguments as
 * td_decode_attn, minus workspace and workspace_bytes. (The pages describe no such call; it
 * exists for callers of this library that cannot allocate device memory: a plugin or launch
 * hook handed only input and output pointers, a serving loop that must not allocate once
 * running, or code working while another runtime owns the device heap.)
 * Its scratch is a fixed 4 MiB array compiled into the library, which every GPU that loads
 * the library holds until the process exits; the call allocates nothing. A shape whose
 * workspace (td_decode_workspace_bytes with q_len 1) exceeds 4 MiB returns TD_ERR_WORKSPACE.
 * The first call on a device looks up the array's address on that device (make that first
 * call before any stream capture). Every call zeroes the array's counter area on its stream
 * before launching. All calls on a device share the one array, so calls that may overlap on
 * the GPU (different streams without ordering between them) race and must not be issued.
 */
td_status td_decode_attn_noalloc(td_dtype dtype, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *seq_lens, int B, int Hq, int Hkv, int Smax, int D, float scale,
                                 int split, void *out, float *lse, uint32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TD_H */
