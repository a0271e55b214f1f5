"""Tolerances and comparison helpers for CUDA-vs-oracle parity.

Outputs: fp32 caches max |gpu - ref| <= 1e-5; bf16 caches |gpu - ref| <= 2e-2 + 1e-2 |ref|
elementwise (the reference is the oracle's fp64 result on the same rounded inputs).
lse (fp32 on the GPU for both): |gpu - ref| <= 2e-3 + 1e-5 |ref|; the bound covers fp32
accumulation of a D-term dot product with scores up to ~100 (heavy keys), see the design notes.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_attention_split_gb300.workloads import to_numpy

LSE_ATOL, LSE_RTOL = 2e-3, 1e-5


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


def oracle_attention(case, seq_lens=None, k_cache=None, v_cache=None):
    """Oracle result for a workloads.Case (CPU tensors); returns (out, lse, status)."""
    orc = oracle.load()
    sl = case.seq_lens if seq_lens is None else seq_lens
    kc = case.k_cache if k_cache is None else k_cache
    vc = case.v_cache if v_cache is None else v_cache
    return orc.attention(to_numpy(case.q), to_numpy(kc), to_numpy(vc), to_numpy(sl), case.scale)
