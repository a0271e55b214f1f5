"""CPU fp64 oracle for split-KV decode attention.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The product (the CUDA library and
its Python binding) never imports it, and it never imports the product: the two share
no code. The arithmetic lives in ``attention.c`` (plain C, fp64, OpenMP over rows);
this module compiles it (and ``speculative.c``, the accept/reject step that follows a verify
pass) with gcc and marshals numpy arrays to it.

Arrays are numpy: float32 or float64 values, or uint16 holding bf16 bit patterns (the
oracle widens them exactly). Layouts are the library's: q/out [B, Hq, T, D], caches
[B, Hkv, Smax, D], seq_lens int32 [B].

Sources: "tinydecode", sections "how the decode step is put together" and "speculative
decoding"; "llm-decode-cuda", the split-KV ("flash-decoding") attention section and the
"RoPE + KV-cache write" step of its decode loop.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attention.c"), os.path.join(_HERE, "speculative.c")]
_BUILD = os.path.join(_HERE, "_build")

# status bits reported for data errors (the CUDA library uses the same meanings)
SEQLEN_CLAMPED = 1
APPEND_OVERFLOW = 2
VERIFY_SHORT = 4
NEGATIVE_SEQLEN = 8
BAD_TOKEN = 64

_DTYPE_CODE = {np.dtype(np.float32): 0, np.dtype(np.uint16): 1, np.dtype(np.float64): 2}
_lock = threading.Lock()
_loaded: dict[int, "Oracle"] = {}


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile attention.c into a shared library and return its path.

    ``mutant`` > 0 builds a copy with one planted mistake (used only by the test that
    shows the oracle's pins catch such mistakes)."""
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    out = os.path.join(_BUILD, name)
    if not force and os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(p) for p in _SRCS):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORC_MUTANT={int(mutant)}", *_SRCS, "-o", tmp, "-lm"]
    try:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
        if r.returncode != 0:  # a compiler without OpenMP still builds the serial oracle
            r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def load(mutant: int = 0) -> "Oracle":
    with _lock:
        if mutant not in _loaded:
            _loaded[mutant] = Oracle(build(mutant))
        return _loaded[mutant]


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _code(a: np.ndarray) -> int:
    try:
        return _DTYPE_CODE[a.dtype]
    except KeyError:
        raise TypeError(f"oracle takes float32, float64 or uint16 (bf16 bits), got {a.dtype}") from None


class Oracle:
    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.orc_attention.argtypes = [i, vp, vp, vp, vp, i, i, i, i, i, i, d, vp, vp]
        lib.orc_attention.restype = ctypes.c_uint
        lib.orc_split_partials.argtypes = [i, vp, vp, vp, vp, i, i, i, i, i, i, d, i, i, vp, vp, vp]
        lib.orc_split_partials.restype = ctypes.c_uint
        lib.orc_lse_merge.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp, vp]
        lib.orc_lse_merge.restype = None
        lib.orc_kv_append.argtypes = [i, vp, vp, vp, vp, vp, i, i, i, i, i, i]
        lib.orc_kv_append.restype = ctypes.c_uint
        lib.orc_rope.argtypes = [i, vp, ctypes.c_int64, i, vp, vp, vp, vp]
        lib.orc_rope.restype = None
        lib.orc_quantize_q8.argtypes = [i, vp, ctypes.c_int64, i, vp, vp]
        lib.orc_quantize_q8.restype = None
        lib.orc_spec_accept.argtypes = [vp, vp, vp, vp, i, i, i, d, vp, vp]
        lib.orc_spec_accept.restype = ctypes.c_uint
        lib.orc_num_threads.restype = i
        lib.orc_set_num_threads.argtypes = [i]
        lib.orc_set_num_threads.restype = None
        lib.orc_mutant.restype = i
        self.lib = lib
        self.mutant = lib.orc_mutant()

    @property
    def num_threads(self) -> int:
        return self.lib.orc_num_threads()

    def set_num_threads(self, n: int) -> None:
        """Threads of later calls (timing only; results do not depend on it)."""
        self.lib.orc_set_num_threads(int(n))

    @staticmethod
    def _shapes(q, k, v, seq_lens):
        if q.ndim == 3:
            q = q[:, :, None, :]
        B, Hq, T, D = q.shape
        Bk, Hkv, Smax, Dk = k.shape
        if k.shape != v.shape or Bk != B or Dk != D or Hq % Hkv != 0 or seq_lens.shape != (B,):
            raise ValueError("inconsistent shapes")
        if not (q.dtype == k.dtype == v.dtype):
            raise TypeError("q, k and v must share a dtype")
        return q, B, Hq, Hkv, T, Smax, D

    def attention(self, q, k, v, seq_lens, scale: float):
        """Exact attention of every query row over its visible keys.

        q [B,Hq,D] (decode) or [B,Hq,T,D] (verify chunk). Returns (out, lse, status):
        out float64 shaped like q, lse float64 [B,Hq] or [B,Hq,T], status bits."""
        squeeze = q.ndim == 3
        q, B, Hq, Hkv, T, Smax, D = self._shapes(q, k, v, seq_lens)
        q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        out = np.empty((B, Hq, T, D), np.float64)
        lse = np.empty((B, Hq, T), np.float64)
        st = self.lib.orc_attention(_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, Hq, Hkv, T, Smax, D,
                                    float(scale), _ptr(out), _ptr(lse))
        if squeeze:
            out, lse = out[:, :, 0], lse[:, :, 0]
        return out, lse, int(st)

    def split_partials(self, q, k, v, seq_lens, scale: float, split: int, num_splits: int | None = None):
        """Per-split (m, l, acc) for split size ``split``; m,l [B, Hq*T, NS], acc [B, Hq*T, NS, D]."""
        q, B, Hq, Hkv, T, Smax, D = self._shapes(q, k, v, seq_lens)
        NS = num_splits if num_splits is not None else -(-Smax // split)
        q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        m = np.empty((B, Hq * T, NS), np.float64)
        l = np.empty((B, Hq * T, NS), np.float64)
        acc = np.empty((B, Hq * T, NS, D), np.float64)
        st = self.lib.orc_split_partials(_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, Hq, Hkv, T, Smax,
                                         D, float(scale), int(split), NS, _ptr(m), _ptr(l), _ptr(acc))
        return m, l, acc, int(st)

    def lse_merge(self, m, l, acc, seq_lens, split: int):
        """Merge per-split partials; returns (out [B, rows, D], lse [B, rows])."""
        m, l, acc = (np.ascontiguousarray(x, dtype=np.float64) for x in (m, l, acc))
        B, rows, NS, D = acc.shape
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        out = np.empty((B, rows, D), np.float64)
        lse = np.empty((B, rows), np.float64)
        self.lib.orc_lse_merge(_ptr(m), _ptr(l), _ptr(acc), _ptr(seq_lens), B, rows, NS, D, int(split), _ptr(out),
                               _ptr(lse))
        return out, lse

    def kv_append(self, k_new, v_new, k_cache, v_cache, seq_lens, advance: bool = True) -> int:
        """In-place cache write of T new rows per (b, kv head) at seq_lens[b]; returns status bits."""
        B, Hkv, T, D = k_new.shape
        Smax = k_cache.shape[2]
        for a in (k_new, v_new, k_cache, v_cache):
            if not a.flags.c_contiguous:
                raise ValueError("kv_append needs contiguous arrays")
        if seq_lens.dtype != np.int32 or not seq_lens.flags.c_contiguous:
            raise TypeError("seq_lens must be a contiguous int32 array")
        return int(self.lib.orc_kv_append(k_new.dtype.itemsize, _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                           _ptr(v_cache), _ptr(seq_lens), B, Hkv, T, Smax, D, int(bool(advance))))

    def rope(self, x, pos, cos_t, sin_t):
        """Rotary embedding of rows x[..., D] at positions pos (shape x.shape[:-1]), rotate-half
        pairs, angles from fp32 tables [positions, D/2]; exact, rounded once to x's type."""
        x = np.ascontiguousarray(x)
        D = x.shape[-1]
        pos = np.ascontiguousarray(np.broadcast_to(pos, x.shape[:-1]), dtype=np.int32)
        cos_t = np.ascontiguousarray(cos_t, dtype=np.float32)
        sin_t = np.ascontiguousarray(sin_t, dtype=np.float32)
        if D % 2 or cos_t.shape != sin_t.shape or cos_t.shape[1] != D // 2:
            raise ValueError("tables must be [positions, D/2]")
        if pos.size and (pos.min() < 0 or pos.max() >= cos_t.shape[0]):
            raise ValueError("position outside the tables")
        y = np.empty_like(x)
        self.lib.orc_rope(_code(x), _ptr(x), pos.size, D, _ptr(pos), _ptr(cos_t), _ptr(sin_t), _ptr(y))
        return y

    def rope_append_attention(self, q, k_new, v_new, k_cache, v_cache, seq_lens, scale: float, cos_t=None,
                              sin_t=None, advance: bool = True):
        """One decode (T = 1) or verify (T > 1) step: token t of sequence b sits at position
        P = seq_lens[b] + t; q and k_new are rotated there (when tables are given), the rotated
        keys and the values are written into the caches, and every query row attends over the
        L_b + T keys it may see. Caches (and seq_lens, with advance) change in place.

        A sequence whose rows do not fit (seq_lens[b] < 0 or seq_lens[b] + T > Smax) is left
        untouched, flagged APPEND_OVERFLOW, and its rows give out = 0, lse = -inf.
        Returns (out float64 [B, Hq, T, D], lse float64 [B, Hq, T], status bits)."""
        B, Hq, T, D = q.shape
        Smax = k_cache.shape[2]
        pre = np.array(seq_lens, dtype=np.int64)
        fits = (pre >= 0) & (pre + T <= Smax)
        pos = np.where(fits, pre, 0)[:, None] + np.arange(T)[None, :]  # [B, T]
        if cos_t is not None:
            q = self.rope(q, np.broadcast_to(pos[:, None, :], (B, Hq, T)), cos_t, sin_t)
            k_new = self.rope(k_new, np.broadcast_to(pos[:, None, :], (B, k_new.shape[1], T)), cos_t, sin_t)
        work = np.ascontiguousarray(seq_lens, dtype=np.int32).copy()
        status = self.kv_append(np.ascontiguousarray(k_new), np.ascontiguousarray(v_new), k_cache, v_cache, work,
                                advance=True)
        out = np.zeros((B, Hq, T, D), np.float64)
        lse = np.full((B, Hq, T), -np.inf)
        idx = np.nonzero(fits)[0]
        if idx.size:
            o, l, st = self.attention(np.ascontiguousarray(q[idx]), np.ascontiguousarray(k_cache[idx]),
                                      np.ascontiguousarray(v_cache[idx]), work[idx], scale)
            out[idx], lse[idx] = o, l
            status |= st
        if advance:
            seq_lens[...] = work
        return out, lse, int(status)

    def spec_accept(self, target_logits, draft_logits, draft_tokens, uniforms, temperature: float):
        """Speculative accept/reject (Leviathan et al. Algorithm 1; greedy at temperature 0).

        target_logits float32 [B, G+1, V], draft_logits float32 [B, G, V] (None when greedy),
        draft_tokens int32 [B, G], uniforms float64 [B, G+1] in [0, 1) (None when greedy).
        Returns (n_accepted int32 [B], next_token int32 [B], status bits)."""
        target_logits = np.ascontiguousarray(target_logits, dtype=np.float32)
        B, G1, V = target_logits.shape
        G = G1 - 1
        draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
        if draft_logits is not None:
            draft_logits = np.ascontiguousarray(draft_logits, dtype=np.float32)
            if draft_logits.shape != (B, G, V):
                raise ValueError("draft logits must be [B, G, V]")
        if uniforms is not None:
            uniforms = np.ascontiguousarray(uniforms, dtype=np.float64)
            if uniforms.shape != (B, G + 1):
                raise ValueError("uniforms must be [B, G+1]")
        if temperature != 0 and (draft_logits is None or uniforms is None):
            raise ValueError("sampling needs the draft logits and the uniforms")
        n = np.empty(B, np.int32)
        nxt = np.empty(B, np.int32)
        st = self.lib.orc_spec_accept(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(uniforms),
                                      B, G, V, float(temperature), _ptr(n), _ptr(nxt))
        return n, nxt, int(st)

    def quantize_q8(self, x):
        """Per-row symmetric int8 codes of rows x[..., D] (bf16 bits or fp32): returns
        (codes int8 shaped like x, scales float32 x.shape[:-1]); decided in fp32."""
        x = np.ascontiguousarray(x)
        D = x.shape[-1]
        rows = x.size // D
        codes = np.empty(x.shape, np.int8)
        scales = np.empty(x.shape[:-1], np.float32)
        self.lib.orc_quantize_q8(_code(x), _ptr(x), rows, D, _ptr(codes), _ptr(scales))
        return codes, scales

    @staticmethod
    def dequantize_q8(codes, scales):
        """The rows the codes stand for, exactly: code * scale in fp64."""
        return codes.astype(np.float64) * scales.astype(np.float64)[..., None]

    def attention_q8(self, q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale: float):
        """Attention over a quantised cache: the exact attention of q (widened) over the
        dequantised rows. Same conventions as attention()."""
        qd = q
        if q.dtype == np.uint16:
            qd = (q.astype(np.uint32) << 16).view(np.float32)
        qd = np.ascontiguousarray(qd, dtype=np.float64)
        return self.attention(qd, np.ascontiguousarray(self.dequantize_q8(k_codes, k_scales)),
                              np.ascontiguousarray(self.dequantize_q8(v_codes, v_scales)), seq_lens, scale)
