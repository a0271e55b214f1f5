"""Python binding of the td C ABI (include/td.h), with the same function names.

Argument marshalling only: shapes and pointers are read off torch tensors, outputs and the
workspace are allocated with torch when the caller does not pass them, and every step of
the computation runs in the CUDA library. Nothing falls back to another implementation:
without the built library, or with tensors off the GPU, the calls raise.

For CUDA-graph capture pass ``out`` (and ``lse``), ``workspace`` and ``stream`` explicitly
and warm the call up once outside the capture.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import threading

import torch

from ._lib import check, lib

TD_F32, TD_BF16 = 0, 1
# bits a call ORs into dev_status (see td.h)
DEV_SEQLEN_CLAMPED = 1
DEV_APPEND_OVERFLOW = 2
DEV_VERIFY_SHORT = 4
DEV_NEGATIVE_SEQLEN = 8
DEV_WAIT_TIMEOUT = 16
DEV_WORKSPACE_DIRTY = 32
DEV_BAD_TOKEN = 64

_ws_lock = threading.Lock()
_ws_cache: dict[tuple[int, int], torch.Tensor] = {}


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TD_F32
    if t.dtype == torch.bfloat16:
        return TD_BF16
    raise TypeError(f"td supports float32 and bfloat16 tensors, got {t.dtype}")


def _cuda(*ts: torch.Tensor | None) -> torch.device:
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("td kernels take CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("td kernels take contiguous tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on one CUDA device")
    return dev


def _on(dev: torch.device):
    """The device guard a launch needs: none when `dev` is already the current device (the
    common case, and a measurable share of a call's host time), else torch's."""
    return contextlib.nullcontext() if torch.cuda.current_device() == dev.index else torch.cuda.device(dev)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def td_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Smax: int, D: int, q_len: int = 1, split: int = 0) -> int:
    """Workspace bytes td_decode_attn / td_verify_attn need on the current device (0 = invalid)."""
    return int(lib().td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, q_len, split))


KERNEL_NAMES = ("cuda_core", "tensor_core_persistent", "tensor_core_cluster")


def td_split_plan(dtype: torch.dtype, B: int, Hq: int, Hkv: int, Smax: int, D: int, q_len: int = 1,
                  split: int = 0) -> dict:
    """Which kernel and launch shape the attention call takes on the current device (td.h)."""
    code = _code(torch.empty(0, dtype=dtype))
    vals = [ctypes.c_int(0) for _ in range(4)]
    check("td_split_plan",
          lib().td_split_plan(code, B, Hq, Hkv, Smax, D, q_len, split, *[ctypes.byref(v) for v in vals]))
    kernel, grid, cluster, rows = (v.value for v in vals)
    return dict(kernel=KERNEL_NAMES[kernel], grid=grid, cluster=cluster, rows=rows)


def make_workspace(B, Hq, Hkv, Smax, D, q_len=1, split=0, device=None) -> torch.Tensor:
    """A zero-filled workspace for a stream of calls with exactly these shape arguments."""
    device = torch.device(device or "cuda")
    with torch.cuda.device(device):
        n = td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, q_len, split)
    if n == 0:
        raise ValueError("invalid shapes for td_decode_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


_WS_CACHE_MAX = 32


def _cached_workspace(nbytes: int, device: torch.device, stream_ptr: int, shape_key: tuple) -> torch.Tensor:
    """A zero-filled workspace per (device, stream, call shape).

    The library leaves the counter area of a workspace zero only for its own layout, and the
    layout follows the call's shape arguments, so a workspace is never shared across shapes."""
    key = (device.index, stream_ptr) + shape_key
    with _ws_lock:
        ws = _ws_cache.pop(key, None)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws  # most recently used last
        while len(_ws_cache) > _WS_CACHE_MAX:
            _ws_cache.pop(next(iter(_ws_cache)))
        return ws


def td_kv_append(k_new, v_new, k_cache, v_cache, seq_lens, advance: bool = True, dev_status=None,
                 stream=None) -> None:
    """Write k_new/v_new [B,Hkv,T,D] into the caches [B,Hkv,Smax,D] at rows seq_lens[b].."""
    dev = _cuda(k_new, v_new, k_cache, v_cache, seq_lens, dev_status)
    B, Hkv, T, D = k_new.shape
    Smax = k_cache.shape[2]
    if v_new.shape != k_new.shape or k_cache.shape != (B, Hkv, Smax, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between new rows and caches")
    if not (k_new.dtype == v_new.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("new rows and caches must share a dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise TypeError("seq_lens must be int32 [B]")
    with _on(dev):
        st = lib().td_kv_append(_code(k_cache), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(seq_lens), B, Hkv, T, Smax, D, int(bool(advance)), _ptr(dev_status),
                                _stream(stream, dev))
    check("td_kv_append", st)


def _attn(name, q4, k_cache, v_cache, seq_lens, scale, split, out, lse, workspace, dev_status, stream):
    dev = _cuda(q4, k_cache, v_cache, seq_lens, out, lse, workspace, dev_status)
    B, Hq, T, D = q4.shape
    _, Hkv, Smax, Dk = k_cache.shape
    if k_cache.shape[0] != B or Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("q and cache shapes disagree")
    if not (q4.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and caches must share a dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise TypeError("seq_lens must be int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on(dev):
        sp = _stream(stream, dev)
        if workspace is None:
            need = td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, T, split)
            workspace = _cached_workspace(need, dev, sp, (B, Hq, Hkv, Smax, D, T, split))
        if workspace.dtype != torch.uint8:
            raise TypeError("workspace must be a uint8 tensor")
        fn = getattr(lib(), name)
        if name == "td_decode_attn":
            st = fn(_code(q4), _ptr(q4), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, Hq, Hkv, Smax, D,
                    float(scale), int(split), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                    _ptr(dev_status), sp)
        else:
            st = fn(_code(q4), _ptr(q4), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, Hq, Hkv, T, Smax, D,
                    float(scale), int(split), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                    _ptr(dev_status), sp)
    check(name, st)


def td_decode_attn(q, k_cache, v_cache, seq_lens, scale: float | None = None, split: int = 0, out=None, lse=None,
                   workspace=None, dev_status=None, stream=None, return_lse: bool = False):
    """Single-token decode attention. q [B,Hq,D] -> out [B,Hq,D] (and lse [B,Hq] fp32)."""
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, Hq)):
        raise TypeError("lse must be float32 [B, Hq]")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise TypeError("out must match q")
    _attn("td_decode_attn", q.view(B, Hq, 1, D), k_cache, v_cache, seq_lens, scale, split, out, lse, workspace,
          dev_status, stream)
    return (out, lse) if (return_lse or lse is not None) else out


def td_verify_attn(q, k_cache, v_cache, seq_lens, scale: float | None = None, split: int = 0, out=None, lse=None,
                   workspace=None, dev_status=None, stream=None, return_lse: bool = False):
    """Verify-chunk attention. q [B,Hq,T,D] (seq_lens count the T new tokens) -> out [B,Hq,T,D]."""
    if q.dim() != 4:
        raise ValueError("q must be [B, Hq, T, D]")
    B, Hq, T, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, Hq, T)):
        raise TypeError("lse must be float32 [B, Hq, T]")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise TypeError("out must match q")
    _attn("td_verify_attn", q, k_cache, v_cache, seq_lens, scale, split, out, lse, workspace, dev_status, stream)
    return (out, lse) if (return_lse or lse is not None) else out


def td_lse_merge(m, l, acc, seq_lens, split: int, out_dtype=torch.float32, out=None, lse=None, stream=None,
                 return_lse: bool = False):
    """Merge per-split partials m,l [B,rows,NS], acc [B,rows,NS,D] -> out [B,rows,D] (+ lse [B,rows])."""
    dev = _cuda(m, l, acc, seq_lens, out, lse)
    B, rows, NS, D = acc.shape
    if m.shape != (B, rows, NS) or l.shape != (B, rows, NS):
        raise ValueError("m and l must be [B, rows, NS]")
    if not (m.dtype == l.dtype == acc.dtype == torch.float32):
        raise TypeError("partials must be float32")
    if out is None:
        out = torch.empty(B, rows, D, dtype=out_dtype, device=acc.device)
    if lse is None and return_lse:
        lse = torch.empty(B, rows, dtype=torch.float32, device=acc.device)
    with _on(dev):
        st = lib().td_lse_merge(_ptr(m), _ptr(l), _ptr(acc), _ptr(seq_lens), B, rows, NS, D, int(split), _code(out),
                                _ptr(out), _ptr(lse), _stream(stream, dev))
    check("td_lse_merge", st)
    return (out, lse) if (return_lse or lse is not None) else out


def _rope_tables(cos_t, sin_t, Smax, D, required):
    if cos_t is None and sin_t is None and not required:
        return None, None
    if cos_t is None or sin_t is None:
        raise ValueError("give both rope tables (cos and sin) or neither")
    for t in (cos_t, sin_t):
        if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != D // 2 or t.shape[0] < Smax:
            raise TypeError("rope tables must be float32 [>= Smax, D/2]")
    return cos_t, sin_t


def td_rope_kv_append(k_new, v_new, k_cache, v_cache, seq_lens, cos_t, sin_t, q=None, q_out=None,
                      advance: bool = True, dev_status=None, stream=None):
    """Rotate k_new [B,Hkv,T,D] to positions seq_lens[b]+t, write it and v_new into the caches;
    with q [B,Hq,T,D], also return q rotated the same way (into q_out, which may be q)."""
    dev = _cuda(k_new, v_new, k_cache, v_cache, seq_lens, cos_t, sin_t, q, q_out, dev_status)
    B, Hkv, T, D = k_new.shape
    Smax = k_cache.shape[2]
    if v_new.shape != k_new.shape or k_cache.shape != (B, Hkv, Smax, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between new rows and caches")
    if not (k_new.dtype == v_new.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("new rows and caches must share a dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise TypeError("seq_lens must be int32 [B]")
    _rope_tables(cos_t, sin_t, Smax, D, required=True)
    Hq = 0
    if q is not None:
        if q.dim() != 4 or q.shape[0] != B or q.shape[2:] != (T, D) or q.dtype != k_new.dtype:
            raise ValueError("q must be [B, Hq, T, D] in the caches' dtype")
        Hq = q.shape[1]
        if q_out is None:
            q_out = torch.empty_like(q)
        if q_out.shape != q.shape or q_out.dtype != q.dtype:
            raise TypeError("q_out must match q")
    with _on(dev):
        st = lib().td_rope_kv_append(_code(k_cache), _ptr(q), _ptr(q_out), Hq, _ptr(k_new), _ptr(v_new), _ptr(cos_t),
                                     _ptr(sin_t), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, Hkv, T, Smax, D,
                                     int(bool(advance)), _ptr(dev_status), _stream(stream, dev))
    check("td_rope_kv_append", st)
    return q_out


def td_rope_append_attn(q, k_new, v_new, k_cache, v_cache, seq_lens, scale: float | None = None, split: int = 0,
                        cos_t=None, sin_t=None, advance: bool = True, out=None, lse=None, workspace=None,
                        dev_status=None, stream=None, return_lse: bool = False):
    """One layer's decode/verify step in one launch: q [B,Hq,T,D] and k_new [B,Hkv,T,D] rotated to
    positions seq_lens[b]+t (when tables are given), k/v rows written into the caches, attention
    over seq_lens[b]+T keys -> out [B,Hq,T,D] (+ lse [B,Hq,T]); seq_lens advanced if asked."""
    if q.dim() != 4:
        raise ValueError("q must be [B, Hq, T, D]")
    dev = _cuda(q, k_new, v_new, k_cache, v_cache, seq_lens, cos_t, sin_t, out, lse, workspace, dev_status)
    B, Hq, T, D = q.shape
    _, Hkv, Smax, Dk = k_cache.shape
    if k_new.shape != (B, Hkv, T, D) or v_new.shape != k_new.shape or Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("q, new rows and cache shapes disagree")
    if not (q.dtype == k_new.dtype == v_new.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, new rows and caches must share a dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise TypeError("seq_lens must be int32 [B]")
    _rope_tables(cos_t, sin_t, Smax, D, required=False)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (B, Hq, T)):
        raise TypeError("lse must be float32 [B, Hq, T]")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise TypeError("out must match q")
    with _on(dev):
        sp = _stream(stream, dev)
        if workspace is None:
            need = td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, T, split)
            workspace = _cached_workspace(need, dev, sp, (B, Hq, Hkv, Smax, D, T, split))
        if workspace.dtype != torch.uint8:
            raise TypeError("workspace must be a uint8 tensor")
        st = lib().td_rope_append_attn(_code(q), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cos_t), _ptr(sin_t),
                                       _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, Hq, Hkv, T, Smax, D,
                                       float(scale), int(split), int(bool(advance)), _ptr(out), _ptr(lse),
                                       _ptr(workspace), workspace.numel(), _ptr(dev_status), sp)
    check("td_rope_append_attn", st)
    return (out, lse) if (return_lse or lse is not None) else out


def td_spec_accept(target_logits, draft_tokens, draft_logits=None, uniforms=None, temperature: float = 1.0,
                   n_accepted=None, next_token=None, workspace=None, dev_status=None, stream=None):
    """Speculative accept/reject (td.h): target_logits fp32 [B, G+1, V], draft_tokens int32
    [B, G], draft_logits fp32 [B, G, V] and uniforms fp32 [B, G+1] (both unused when
    temperature is 0) -> (n_accepted int32 [B], next_token int32 [B])."""
    dev = _cuda(target_logits, draft_tokens, draft_logits, uniforms, n_accepted, next_token, dev_status)
    if target_logits.dim() != 3 or target_logits.dtype != torch.float32:
        raise TypeError("target_logits must be float32 [B, G+1, V]")
    B, G1, V = target_logits.shape
    G = G1 - 1
    if draft_tokens.dtype != torch.int32 or tuple(draft_tokens.shape) != (B, G):
        raise TypeError("draft_tokens must be int32 [B, G]")
    if temperature != 0:
        if draft_logits is None or uniforms is None:
            raise ValueError("sampling needs draft_logits and uniforms")
        if draft_logits.dtype != torch.float32 or tuple(draft_logits.shape) != (B, G, V):
            raise TypeError("draft_logits must be float32 [B, G, V]")
        if uniforms.dtype != torch.float32 or tuple(uniforms.shape) != (B, G + 1):
            raise TypeError("uniforms must be float32 [B, G+1]")
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    with _on(dev):
        sp = _stream(stream, dev)
        if workspace is None:
            need = int(lib().td_spec_workspace_bytes(B, G, V))
            workspace = _cached_workspace(need, dev, sp, ("spec", B, G, V))
        if workspace.dtype != torch.uint8:
            raise TypeError("workspace must be a uint8 tensor")
        st = lib().td_spec_accept(_ptr(target_logits), _ptr(draft_logits if temperature != 0 else None),
                                  _ptr(draft_tokens), _ptr(uniforms if temperature != 0 else None), B, G, V,
                                  float(temperature), _ptr(n_accepted), _ptr(next_token), _ptr(workspace),
                                  workspace.numel(), _ptr(dev_status), sp)
    check("td_spec_accept", st)
    return n_accepted, next_token


def td_quantize_q8(x, codes=None, scales=None, stream=None):
    """Per-row int8 codes and fp32 scales of x [..., D] (float32 or bfloat16), as td.h defines."""
    dev = _cuda(x, codes, scales)
    D = x.shape[-1]
    rows = x.numel() // D
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    with _on(dev):
        st = lib().td_quantize_q8(_code(x), _ptr(x), rows, D, _ptr(codes), _ptr(scales), _stream(stream, dev))
    check("td_quantize_q8", st)
    return codes, scales


def td_kv_append_q8(k_new, v_new, k_codes, k_scales, v_codes, v_scales, seq_lens, advance: bool = True,
                    dev_status=None, stream=None) -> None:
    """Quantise k_new/v_new [B,Hkv,T,D] into an int8 cache at rows seq_lens[b].. (td_kv_append's rules)."""
    dev = _cuda(k_new, v_new, k_codes, k_scales, v_codes, v_scales, seq_lens, dev_status)
    B, Hkv, T, D = k_new.shape
    Smax = k_codes.shape[2]
    if k_codes.dtype != torch.int8 or v_codes.dtype != torch.int8 or k_codes.shape != (B, Hkv, Smax, D):
        raise TypeError("codes must be int8 [B, Hkv, Smax, D]")
    if k_scales.shape != (B, Hkv, Smax) or k_scales.dtype != torch.float32 or v_scales.shape != k_scales.shape:
        raise TypeError("scales must be float32 [B, Hkv, Smax]")
    with _on(dev):
        st = lib().td_kv_append_q8(_code(k_new), _ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(k_scales),
                                   _ptr(v_codes), _ptr(v_scales), _ptr(seq_lens), B, Hkv, T, Smax, D,
                                   int(bool(advance)), _ptr(dev_status), _stream(stream, dev))
    check("td_kv_append_q8", st)


def td_verify_attn_q8(q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale: float | None = None, split: int = 0,
                      out=None, lse=None, workspace=None, dev_status=None, stream=None, return_lse: bool = False):
    """Attention over an int8 cache: q [B,Hq,T,D] or [B,Hq,D] (decode) bf16 -> out like q."""
    decode = q.dim() == 3
    q4 = q.unsqueeze(2) if decode else q
    dev = _cuda(q4, k_codes, k_scales, v_codes, v_scales, seq_lens, out, lse, workspace, dev_status)
    B, Hq, T, D = q4.shape
    _, Hkv, Smax, _ = k_codes.shape
    if q.dtype != torch.bfloat16 or k_codes.dtype != torch.int8 or v_codes.dtype != torch.int8:
        raise TypeError("q must be bfloat16 and the codes int8")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    with _on(dev):
        sp = _stream(stream, dev)
        if workspace is None:
            need = td_decode_workspace_bytes(B, Hq, Hkv, Smax, D, T, split)
            workspace = _cached_workspace(need, dev, sp, ("q8", B, Hq, Hkv, Smax, D, T, split))
        st = lib().td_verify_attn_q8(_ptr(q4), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales),
                                     _ptr(seq_lens), B, Hq, Hkv, T, Smax, D, float(scale), int(split), _ptr(out),
                                     _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(dev_status), sp)
    check("td_verify_attn_q8", st)
    return (out, lse) if (return_lse or lse is not None) else out


def td_decode_attn_q8(q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale: float | None = None, split: int = 0,
                      out=None, lse=None, workspace=None, dev_status=None, stream=None, return_lse: bool = False):
    """Single-token decode over an int8 cache: q [B,Hq,D] bf16 -> out [B,Hq,D]."""
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    return td_verify_attn_q8(q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, split, out, lse, workspace,
                             dev_status, stream, return_lse)


def td_prefill_attn(q, k_cache, v_cache, seq_lens, scale: float | None = None, out=None, lse=None, dev_status=None,
                    stream=None, return_lse: bool = False):
    """Causal prefill over the cache: q [B,Hq,T,D] bf16 (seq_lens count the T tokens, whose K/V
    rows are already written) -> out [B,Hq,T,D] (+ lse [B,Hq,T]); tensor-core tiles."""
    if q.dim() != 4:
        raise ValueError("q must be [B, Hq, T, D]")
    dev = _cuda(q, k_cache, v_cache, seq_lens, out, lse, dev_status)
    B, Hq, T, D = q.shape
    _, Hkv, Smax, Dk = k_cache.shape
    if k_cache.shape[0] != B or Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("q and cache shapes disagree")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16):
        raise TypeError("prefill takes bfloat16 q and caches")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,):
        raise TypeError("seq_lens must be int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    with _on(dev):
        st = lib().td_prefill_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, Hq, Hkv, T, Smax, D,
                                   float(scale), _ptr(out), _ptr(lse), _ptr(dev_status), _stream(stream, dev))
    check("td_prefill_attn", st)
    return (out, lse) if (return_lse or lse is not None) else out
