"""Tolerances and comparison helpers for CUDA-vs-oracle parity.

Two checks on every bf16 attention output, both against the oracle's fp64 result on the same
rounded inputs:

1. The stated tolerance (pass/fail as specified): fp32 caches max |gpu - ref| <= 1e-5; bf16
   caches |gpu - ref| <= 2e-2 + 1e-2 |ref| elementwise.
2. The value-side bound (bf16 kernels): the error the kernels' own rounding can produce, per
   element. The kernels round the output once to bf16 (at most u |ref|, u = 2^-8 the bf16
   unit roundoff) and round each probability p_j to bf16 before the p @ V product, with the
   normaliser summed from the unrounded p_j. With relative rounding errors d_j (|d_j| <= u,
   modelled as independent and uniform: variance u^2 / 3) the output moves by
   sum_j w_j d_j v_j (or by sum_j w_j d_j (v_j - out) where a normaliser is summed from the
   rounded p_j), whose standard deviation is in either case at most
       (u / sqrt 3) (sqrt(sum_j w_j^2 v_j^2) + |out| sqrt(sum_j w_j^2)),
   w_j the exact softmax weights. The bound allows 6 of those standard deviations, plus
   2e-5 sum_j w_j |v_j| for fp32 effects (score rounding into the exponent, base-2 folding of
   the scale, the fp32 merge) and a floor of 1e-6. For a spread-out softmax over N keys the
   middle term is about 0.013 / sqrt(N), far below the 2e-2 of check 1, so a value row read
   from the wrong place or a chunk of p @ V dropped fails here even where check 1 passes.
   The three sums come from the oracle itself, called on transformed inputs:
       sum_j w_j^2 v_j^2 = out' exp(lse' - 2 lse)   (out', lse': scale 2 scale, values v^2)
       sum_j w_j^2       = exp(lse' - 2 lse)
       sum_j w_j |v_j|   = attention with values |v|.

lse (fp32 on the GPU for both): |gpu - ref| <= 2e-3 + 1e-5 |ref|; the bound covers fp32
accumulation of a D-term dot product with scores up to ~100 (heavy keys).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_attention_split_gb300.workloads import to_numpy

LSE_ATOL, LSE_RTOL = 2e-3, 1e-5

U_BF16 = 2.0 ** -8          # unit roundoff of bf16 (8 significant bits, round to nearest)
VALUE_SIGMAS = 6.0           # standard deviations of the probability-rounding sum allowed
VALUE_FP32_REL = 2e-5        # fp32 effects, relative to sum_j w_j |v_j|
VALUE_FLOOR = 1e-6


def assert_out_close(gpu: torch.Tensor, ref: np.ndarray, dtype: str, what: str = "out"):
    g = gpu.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    if dtype == "f32":
        worst = float(err.max()) if err.size else 0.0
        assert worst <= 1e-5, f"{what}: max abs err {worst:.3e} > 1e-5"
    else:
        bound = 2e-2 + 1e-2 * np.abs(ref)
        bad = err > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside 2e-2+1e-2|ref|; "
                               f"max abs {float(err.max()):.3e}")


def assert_lse_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "lse"):
    g = gpu.detach().double().cpu().numpy().reshape(ref.shape)
    neg = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), neg), f"{what}: -inf pattern differs"
    e = np.abs(g[~neg] - ref[~neg])
    if e.size:
        bad = e > LSE_ATOL + LSE_RTOL * np.abs(ref[~neg])
        assert not bad.any(), f"{what}: max abs err {float(e.max()):.3e}"


def as_f64(a: np.ndarray) -> np.ndarray:
    """An oracle-form array (float32, float64, or uint16 holding bf16 bits) as exact float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def value_stats(q, k, v, seq_lens, scale: float, lse: np.ndarray):
    """Per output element, the sums the value-side bound uses: (sqrt(sum_j w_j^2 v_j^2) [.., D],
    sqrt(sum_j w_j^2) [..], sum_j w_j |v_j| [.., D]). Oracle-form inputs; ``lse`` is the
    oracle's lse for (q, k, v, scale). Rows with no visible key give zeros."""
    orc = oracle.load()
    q64, k64, v64 = as_f64(q), as_f64(k), as_f64(v)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out2, lse2, _ = orc.attention(q64, k64, v64 * v64, sl, 2.0 * scale)
    a, _, _ = orc.attention(q64, k64, np.abs(v64), sl, scale)
    empty = np.isneginf(lse)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.where(empty, 0.0, np.exp(np.where(empty, 0.0, lse2 - 2.0 * lse)))
    return np.sqrt(np.maximum(out2, 0.0) * r[..., None]), np.sqrt(r), a


def value_bound(ref: np.ndarray, stats) -> np.ndarray:
    s1, s2, a = stats
    sig = U_BF16 / np.sqrt(3.0)
    ar = np.abs(ref)
    return U_BF16 * ar + VALUE_SIGMAS * sig * (s1 + ar * s2[..., None]) + VALUE_FP32_REL * a + VALUE_FLOOR


def assert_value_close(gpu, ref: np.ndarray, stats, what: str = "out"):
    """The value-side bound (module docstring, check 2)."""
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    g = g.reshape(ref.shape)
    err = np.abs(g - ref)
    bound = value_bound(ref, stats)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside the value-side bound; worst "
                           f"err/bound {float((err / bound).max()):.2f}, max abs err {float(err.max()):.3e}")


def check_bf16_attention(out, lse, q, k, v, seq_lens, scale: float, what: str = "out"):
    """Both output checks and the lse check of a bf16 attention result against the oracle, on
    oracle-form inputs (numpy; bf16 as uint16 bits). Returns (ref, ref_lse, status)."""
    ref, ref_lse, st = oracle.load().attention(q, k, v, seq_lens, scale)
    assert_out_close(out, ref, "bf16", what=what)
    assert_value_close(out, ref, value_stats(q, k, v, seq_lens, scale, ref_lse), what=what)
    if lse is not None:
        assert_lse_close(lse, ref_lse, what=f"{what} lse")
    return ref, ref_lse, st


def oracle_attention(case, seq_lens=None, k_cache=None, v_cache=None):
    """Oracle result for a workloads.Case (CPU tensors); returns (out, lse, status)."""
    orc = oracle.load()
    sl = case.seq_lens if seq_lens is None else seq_lens
    kc = case.k_cache if k_cache is None else k_cache
    vc = case.v_cache if v_cache is None else v_cache
    return orc.attention(to_numpy(case.q), to_numpy(kc), to_numpy(vc), to_numpy(sl), case.scale)


def case_value_stats(case, ref_lse, seq_lens=None, k_cache=None, v_cache=None):
    """value_stats for a workloads.Case (CPU tensors)."""
    sl = case.seq_lens if seq_lens is None else seq_lens
    kc = case.k_cache if k_cache is None else k_cache
    vc = case.v_cache if v_cache is None else v_cache
    return value_stats(to_numpy(case.q), to_numpy(kc), to_numpy(vc), to_numpy(sl), case.scale, ref_lse)
