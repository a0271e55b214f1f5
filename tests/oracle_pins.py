"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

Each pin takes an oracle handle and raises AssertionError when the oracle disagrees with
a closed form, a library routine (torch's scaled_dot_product_attention and logsumexp,
scipy's logsumexp, all in fp64), or an identity the method fixes: split invariance of
the log-sum-exp merge, grouped-query attention equal to multi-head attention on repeated
kv heads, a verify chunk equal to step-by-step decode, stale rows past seq_len never
read, batch rows independent. The pins are chosen so a plausible mistake anywhere in the
oracle (wrong head mapping, dropped scale, off-by-one mask, lse without its max, merge
without rescale, transposed cache, wrong 16-bit format, append position or advance)
fails at least one of them; the mutant test checks exactly that.

Rotary embedding (a reading: the pages name an in-place rope kernel and a fused
"RoPE + KV-cache write" but print no formula) is pinned to complex multiplication by
e^{i angle} in numpy, to an exact quarter turn, to the identity at angle 0 and to the
relative-position property of the attention scores; the fused step is pinned to its parts.

Sources: "tinydecode", sections "how the decode step is put together" (static cache,
seq_lens mask, split chunks merged by log-sum-exp, q head -> kv head index math) and
"speculative decoding" (verify chunk causal among the new tokens, rollback by seq_lens);
"llm-decode-cuda", split-KV attention section (one block per kv head and chunk serving
the whole query-head group, log-sum-exp merge).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as orc_mod
from decode_attention_split_gb300.workloads import small_case, to_numpy

F64 = np.float64


def _np(t):
    return to_numpy(t)


def _widen(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def _sdpa_reference(case, scale):
    """torch fp64 scaled_dot_product_attention per sequence, GQA by repeating kv heads."""
    q, k, v = _widen(case.q), _widen(case.k_cache), _widen(case.v_cache)
    B, Hq, T, D = q.shape
    g = Hq // k.shape[1]
    outs, lses = [], []
    for b in range(B):
        L = int(case.seq_lens[b])
        kb = k[b, :, :L].repeat_interleave(g, dim=0)  # [Hq, L, D]
        vb = v[b, :, :L].repeat_interleave(g, dim=0)
        # row t sees keys j <= L - T + t
        mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q[b:b + 1], kb[None], vb[None], attn_mask=mask,
                                                             scale=scale)
        s = torch.einsum("htd,hjd->htj", q[b], kb) * scale
        s = s.masked_fill(~mask[None], float("-inf"))
        outs.append(o[0])
        lses.append(torch.logsumexp(s, dim=-1))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


def _run(orc, case, scale=None):
    scale = case.scale if scale is None else scale
    return orc.attention(_np(case.q), _np(case.k_cache), _np(case.v_cache), _np(case.seq_lens), scale)


# --- closed forms ---------------------------------------------------------------------------

def pin_closed_form_two_keys(orc):
    """D=1, keys 0 and ln 2 with q=1, scale 1: weights 1:2, so out = (3 + 2*6)/3 = 5, lse = ln 3."""
    q = np.array([[[[1.0]]]])
    k = np.array([[[[0.0], [math.log(2.0)]]]])
    v = np.array([[[[3.0], [6.0]]]])
    out, lse, st = orc.attention(q, k, v, np.array([2], np.int32), 1.0)
    assert st == 0
    assert abs(out[0, 0, 0, 0] - 5.0) < 1e-12, out
    assert abs(lse[0, 0, 0] - math.log(3.0)) < 1e-12, lse


def pin_closed_form_scaled(orc):
    """D=2, scale 1/2: q.k = (0, 2, 4) gives scores (0, 1, 2); with v = (1,0), (0,1), (1,1)
    out = ((1+e^2)/Z, (e+e^2)/Z) and lse = ln Z, Z = 1 + e + e^2."""
    q = np.array([[[[2.0, 0.0]]]])
    k = np.array([[[[0.0, 1.0], [1.0, 0.0], [2.0, 5.0]]]])
    v = np.array([[[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]]])
    out, lse, _ = orc.attention(q, k, v, np.array([3], np.int32), 0.5)
    e = math.e
    Z = 1 + e + e * e
    assert np.allclose(out[0, 0, 0], [(1 + e * e) / Z, (e + e * e) / Z], rtol=0, atol=1e-12), out
    assert abs(lse[0, 0, 0] - math.log(Z)) < 1e-12


def pin_closed_form_gqa(orc):
    """Hq=4, Hkv=2, D=1: heads 0,1 read kv head 0 (equal keys -> mean of v = 2); heads 2,3 read
    kv head 1 with keys (0, 1): q=0 gives 1/2, q=ln 3 gives weights 1:3 and out 3/4."""
    q = np.array([[[[5.0]], [[-1.0]], [[0.0]], [[math.log(3.0)]]]])
    k = np.array([[[[0.0], [0.0]], [[0.0], [1.0]]]])
    v = np.array([[[[1.0], [3.0]], [[0.0], [1.0]]]])
    out, _, _ = orc.attention(q, k, v, np.array([2], np.int32), 1.0)
    assert np.allclose(out[0, :, 0, 0], [2.0, 2.0, 0.5, 0.75], rtol=0, atol=1e-12), out[0, :, 0, 0]


# --- library routines ---------------------------------------------------------------------

def pin_matches_sdpa_decode(orc):
    """Decode rows against torch fp64 SDPA (bf16 and fp32 inputs, explicit non-default scale)."""
    for dtype, seed in (("bf16", 1), ("f32", 2)):
        case = small_case(dtype=dtype, B=2, Hq=6, Hkv=2, D=16, Smax=40, seq_lens=[17, 40], seed=seed, heavy=0.1)
        out, lse, _ = _run(orc, case, scale=0.3)
        ref, ref_lse = _sdpa_reference(case, 0.3)
        assert np.max(np.abs(out - ref)) < 1e-12, np.max(np.abs(out - ref))
        assert np.max(np.abs(lse - ref_lse)) < 1e-12


def pin_matches_sdpa_verify(orc):
    """A T=3 verify chunk against fp64 SDPA with the causal mask j <= L - T + t."""
    case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=8, Smax=30, T=3, seq_lens=[5, 29], seed=3)
    out, lse, _ = _run(orc, case, scale=0.4)
    ref, ref_lse = _sdpa_reference(case, 0.4)
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-12


def pin_lse_matches_scipy(orc):
    """lse = ln sum_j exp(s_j) via scipy.special.logsumexp on scores from a numpy matmul."""
    from scipy.special import logsumexp
    case = small_case(dtype="f32", B=1, Hq=2, Hkv=1, D=32, Smax=64, seq_lens=[50], seed=4, heavy=0.2)
    _, lse, _ = _run(orc, case, scale=0.7)
    q = case.q.double().numpy()[0, :, 0]
    k = case.k_cache.double().numpy()[0, 0, :50]
    ref = logsumexp(0.7 * (q @ k.T), axis=-1)
    assert np.max(np.abs(lse[0, :, 0] - ref)) < 1e-11


# --- special cases ------------------------------------------------------------------------

def pin_seq_len_one(orc):
    """One visible key has weight 1: out is that value row exactly."""
    case = small_case(dtype="bf16", B=3, Hq=6, Hkv=3, D=32, Smax=9, seq_lens=[1, 1, 1], seed=5)
    out, _, _ = _run(orc, case)
    v0 = case.v_cache.double()[:, :, 0].repeat_interleave(2, dim=1).numpy()  # [B, Hq, D]
    assert np.array_equal(out[:, :, 0], v0)


def pin_identical_keys_and_zero_scale(orc):
    """Equal keys, or scale 0, give equal weights: out is the mean of the visible values."""
    case = small_case(dtype="f32", B=1, Hq=2, Hkv=1, D=16, Smax=20, seq_lens=[13], seed=6)
    mean = case.v_cache.double()[0, 0, :13].mean(0).numpy()
    out0, lse0, _ = _run(orc, case, scale=0.0)
    assert np.max(np.abs(out0[0, :, 0] - mean)) < 1e-13
    assert np.allclose(lse0, math.log(13), atol=1e-13)
    kc = case.k_cache.clone()
    kc[0, 0, :] = kc[0, 0, 5]
    case.k_cache = kc
    out1, _, _ = _run(orc, case)
    assert np.max(np.abs(out1[0, :, 0] - mean)) < 1e-13


def pin_dominant_key(orc):
    """A key whose score exceeds every other by > 60 takes all the weight."""
    case = small_case(dtype="f32", B=1, Hq=1, Hkv=1, D=8, Smax=16, seq_lens=[16], seed=7)
    qv = case.q[0, 0, 0]
    kc = case.k_cache.clone() * 0.01
    kc[0, 0, 11] = qv * (80.0 / float(qv @ qv))  # score 80 at scale 1, others |s| < 1
    case.k_cache = kc
    out, _, _ = _run(orc, case, scale=1.0)
    assert np.max(np.abs(out[0, 0, 0] - case.v_cache.double()[0, 0, 11].numpy())) < 1e-12


def pin_empty_rows(orc):
    """seq_len 0: no visible key, out = 0 and lse = -inf."""
    case = small_case(dtype="bf16", B=2, Hq=2, Hkv=1, D=8, Smax=10, seq_lens=[0, 4], seed=8)
    out, lse, st = _run(orc, case)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1]))
    assert st == 0


# --- invariants -----------------------------------------------------------------------------

def pin_convex_hull(orc):
    """Each output coordinate lies between the smallest and largest visible value coordinate."""
    case = small_case(dtype="bf16", B=2, Hq=8, Hkv=2, D=16, Smax=50, seq_lens=[37, 50], seed=9, heavy=0.05)
    out, _, _ = _run(orc, case)
    v = case.v_cache.double()
    for b, L in enumerate([37, 50]):
        lo = v[b, :, :L].min(1).values.repeat_interleave(4, 0).numpy()
        hi = v[b, :, :L].max(1).values.repeat_interleave(4, 0).numpy()
        assert np.all(out[b, :, 0] >= lo - 1e-12) and np.all(out[b, :, 0] <= hi + 1e-12)


def pin_gqa_equals_repeated_mha(orc):
    """Grouped-query attention equals multi-head attention on kv heads repeated per group."""
    case = small_case(dtype="bf16", B=2, Hq=6, Hkv=3, D=16, Smax=24, seq_lens=[24, 11], seed=10)
    out, lse, _ = _run(orc, case)
    k_rep = case.k_cache.repeat_interleave(2, dim=1)
    v_rep = case.v_cache.repeat_interleave(2, dim=1)
    out2, lse2, _ = orc.attention(_np(case.q), _np(k_rep), _np(v_rep), _np(case.seq_lens), case.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_verify_equals_sequential_decode(orc):
    """Row t of a T-token chunk equals a single-token decode of q_t over L - T + t + 1 keys."""
    T = 4
    case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=16, Smax=40, T=T, seq_lens=[33, 40], seed=11)
    out, lse, _ = _run(orc, case)
    for t in range(T):
        lens = (case.seq_lens - T + t + 1).to(torch.int32)
        o_t, l_t, _ = orc.attention(_np(case.q[:, :, t]), _np(case.k_cache), _np(case.v_cache), _np(lens),
                                    case.scale)
        assert np.array_equal(out[:, :, t], o_t) and np.array_equal(lse[:, :, t], l_t), t


def pin_split_invariance(orc):
    """Per-split partials merged by log-sum-exp equal unsplit attention for any split size."""
    for T, seed in ((1, 12), (3, 13)):
        case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=8, Smax=70, T=T, seq_lens=[70, 23], seed=seed,
                          heavy=0.1)
        out, lse, _ = _run(orc, case)
        B, Hq = 2, 4
        for S in (1, 3, 16, 64, 70):
            m, l, acc, _ = orc.split_partials(_np(case.q), _np(case.k_cache), _np(case.v_cache),
                                              _np(case.seq_lens), case.scale, S)
            mo, ml = orc.lse_merge(m, l, acc, _np(case.seq_lens), S)
            assert np.max(np.abs(mo.reshape(out.shape) - out)) < 1e-12, S
            assert np.max(np.abs(ml.reshape(lse.shape) - lse)) < 1e-12, S


def pin_poison_past_seq_len(orc):
    """Rows at or past seq_len are never read: NaN there leaves the output bit-identical."""
    case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=16, Smax=32, seq_lens=[9, 31], seed=14)
    out, lse, _ = _run(orc, case)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    for b, L in enumerate([9, 31]):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    out2, lse2, _ = orc.attention(_np(case.q), _np(kc), _np(vc), _np(case.seq_lens), case.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_key_permutation(orc):
    """Permuting the visible (key, value) rows together does not change the result."""
    case = small_case(dtype="f32", B=1, Hq=2, Hkv=1, D=16, Smax=16, seq_lens=[16], seed=15)
    out, _, _ = _run(orc, case)
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(0))
    kc, vc = case.k_cache[:, :, perm].contiguous(), case.v_cache[:, :, perm].contiguous()
    out2, _, _ = orc.attention(_np(case.q), _np(kc), _np(vc), _np(case.seq_lens), case.scale)
    assert np.max(np.abs(out - out2)) < 1e-13


def pin_batch_independence(orc):
    """Row b of a batched call equals a batch-of-one call on sequence b."""
    case = small_case(dtype="bf16", B=3, Hq=4, Hkv=2, D=16, Smax=20, seq_lens=[20, 3, 12], seed=16)
    out, lse, _ = _run(orc, case)
    for b in range(3):
        o, l_, _ = orc.attention(_np(case.q[b:b + 1]), _np(case.k_cache[b:b + 1]), _np(case.v_cache[b:b + 1]),
                                 _np(case.seq_lens[b:b + 1]), case.scale)
        assert np.array_equal(out[b:b + 1], o) and np.array_equal(lse[b:b + 1], l_)


def pin_status_bits(orc):
    """Lengths past Smax are clamped and flagged, negative ones count as 0, short verify is flagged."""
    case = small_case(dtype="bf16", B=2, Hq=2, Hkv=1, D=8, Smax=10, seq_lens=[12, -3], seed=17)
    out, lse, st = _run(orc, case)
    assert st == orc_mod.SEQLEN_CLAMPED | orc_mod.NEGATIVE_SEQLEN
    case10 = small_case(dtype="bf16", B=2, Hq=2, Hkv=1, D=8, Smax=10, seq_lens=[10, 0], seed=17)
    out10, _, _ = _run(orc, case10)
    assert np.array_equal(out, out10)
    vcase = small_case(dtype="bf16", B=1, Hq=2, Hkv=1, D=8, Smax=10, T=3, seq_lens=[2], seed=18)
    vout, vlse, vst = _run(orc, vcase)
    assert vst == orc_mod.VERIFY_SHORT
    assert np.all(vout[0, :, 0] == 0) and np.all(np.isneginf(vlse[0, :, 0])) and np.all(np.isfinite(vlse[0, :, 1:]))


# --- cache write ------------------------------------------------------------------------------

def pin_append_bit_exact(orc):
    """New rows land bit for bit at seq_lens..seq_lens+T-1; every other row is untouched."""
    rng = np.random.default_rng(0)
    B, H, T, S, D = 3, 2, 2, 12, 8
    cache_k = rng.integers(0, 2 ** 16, (B, H, S, D), dtype=np.uint16)
    cache_v = rng.integers(0, 2 ** 16, (B, H, S, D), dtype=np.uint16)
    new_k = rng.integers(0, 2 ** 16, (B, H, T, D), dtype=np.uint16)
    new_v = rng.integers(0, 2 ** 16, (B, H, T, D), dtype=np.uint16)
    seq = np.array([0, 5, 10], np.int32)
    k2, v2, s2 = cache_k.copy(), cache_v.copy(), seq.copy()
    st = orc.kv_append(new_k, new_v, k2, v2, s2, advance=True)
    assert st == 0 and np.array_equal(s2, seq + T)
    ek, ev = cache_k.copy(), cache_v.copy()
    for b, L in enumerate(seq):
        ek[b, :, L:L + T] = new_k[b]
        ev[b, :, L:L + T] = new_v[b]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    s3 = seq.copy()
    orc.kv_append(new_k, new_v, cache_k.copy(), cache_v.copy(), s3, advance=False)
    assert np.array_equal(s3, seq)


def pin_append_overflow(orc):
    """A sequence whose new rows would pass Smax (or whose length is negative) is left alone and flagged."""
    B, H, T, S, D = 3, 1, 3, 8, 4
    cache = np.zeros((B, H, S, D), np.float32)
    new = np.ones((B, H, T, D), np.float32)
    seq = np.array([6, 5, -1], np.int32)
    k2, v2 = cache.copy(), cache.copy()
    st = orc.kv_append(new, new, k2, v2, seq, advance=True)
    assert st == orc_mod.APPEND_OVERFLOW
    assert np.array_equal(seq, [6, 8, -1])
    assert k2[0].sum() == 0 and k2[2].sum() == 0 and k2[1, 0, 5:8].sum() == 3 * 4


# --- rotary embedding and the fused step ------------------------------------------------------

def _tables(P, D, base=10000.0):
    """cos/sin tables [P, D/2] of the angles p * base^(-2i/D), computed in fp64, stored fp32."""
    ang = np.arange(P, dtype=F64)[:, None] * base ** (-np.arange(0, D, 2, dtype=F64) / D)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _half_ulp(y, mant_bits):
    """Half a unit in the last place of a float with `mant_bits` stored mantissa bits, at |y|."""
    _, e = np.frexp(np.abs(y))  # |y| in [2^(e-1), 2^e)
    return np.ldexp(1.0, e - 2 - mant_bits)


def pin_rope_quarter_turn(orc):
    """D=2: a quarter turn sends (1, 0) to (0, 1) and (0, 1) to (-1, 0); angle 0 is the identity."""
    x = np.array([[1.0, 0.0], [0.0, 1.0], [0.3, -2.0]], np.float32)
    cos_t = np.array([[1.0], [0.0]], np.float32)
    sin_t = np.array([[0.0], [1.0]], np.float32)
    y = orc.rope(x, np.array([1, 1, 0]), cos_t, sin_t)
    assert np.array_equal(y, np.array([[0.0, 1.0], [-1.0, 0.0], [0.3, -2.0]], np.float32))


def pin_rope_is_complex_multiplication(orc):
    """Pair (x[i], x[i + D/2]) as x[i] + j x[i + D/2], times cos + j sin (numpy complex128):
    the stored result is that product rounded to nearest (within half an ulp), bf16 and fp32."""
    rng = np.random.default_rng(3)
    D, n, P = 16, 40, 64
    cos_t, sin_t = _tables(P, D)
    pos = rng.integers(0, P, n)
    for dtype, mant in (("bf16", 7), ("f32", 23)):
        xt = torch.from_numpy(rng.standard_normal((n, D)).astype(np.float32))
        x = _np(xt.to(torch.bfloat16)) if dtype == "bf16" else xt.numpy()
        xv = (xt.to(torch.bfloat16) if dtype == "bf16" else xt).double().numpy()
        z = (xv[:, :D // 2] + 1j * xv[:, D // 2:]) * (cos_t[pos].astype(F64) + 1j * sin_t[pos].astype(F64))
        ref = np.concatenate([z.real, z.imag], axis=1)
        y = orc.rope(x, pos, cos_t, sin_t)
        yv = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy() if dtype == "bf16" else \
            y.astype(F64)
        assert np.all(np.abs(yv - ref) <= _half_ulp(ref, mant) * (1 + 1e-12)), dtype


def pin_rope_relative_position(orc):
    """With tables of angles p * theta_i, the score of a query at position m and a key at n
    depends only on m - n: <rope(q, m), rope(k, n)> = <rope(q, m - n), k>."""
    rng = np.random.default_rng(4)
    D, P = 32, 200
    cos_t, sin_t = _tables(P, D)
    q = rng.standard_normal((1, D)).astype(np.float32)
    k = rng.standard_normal((1, D)).astype(np.float32)
    for m, n in ((7, 3), (150, 20), (64, 64)):
        lhs = float(orc.rope(q, [m], cos_t, sin_t)[0].astype(F64) @ orc.rope(k, [n], cos_t, sin_t)[0].astype(F64))
        rhs = float(orc.rope(q, [m - n], cos_t, sin_t)[0].astype(F64) @ k[0].astype(F64))
        assert abs(lhs - rhs) <= 1e-4 * (1 + abs(rhs)), (m, n, lhs, rhs)


def pin_fused_step_is_its_parts(orc):
    """rope_append_attention = rotate (pinned above) + cache write + attention, token t of
    sequence b at position seq_lens[b] + t; a sequence that does not fit is untouched,
    flagged, and gives out = 0, lse = -inf."""
    case = small_case(dtype="bf16", B=3, Hq=4, Hkv=2, D=16, Smax=20, T=2, seq_lens=[5, 18, 0], seed=7)
    cos_t, sin_t = _tables(20, 16)
    rng = np.random.default_rng(5)
    k_new = _np(torch.from_numpy(rng.standard_normal((3, 2, 2, 16)).astype(np.float32)).to(torch.bfloat16))
    v_new = _np(torch.from_numpy(rng.standard_normal((3, 2, 2, 16)).astype(np.float32)).to(torch.bfloat16))
    kc, vc, sl = _np(case.k_cache).copy(), _np(case.v_cache).copy(), np.array([5, 19, 0], np.int32)
    out, lse, st = orc.rope_append_attention(_np(case.q), k_new, v_new, kc, vc, sl, 0.25, cos_t, sin_t)
    assert st == orc_mod.APPEND_OVERFLOW and sl.tolist() == [7, 19, 2]
    for b, L in ((0, 5), (2, 0)):
        pos = np.array([L, L + 1])
        assert np.array_equal(kc[b, :, L:L + 2], orc.rope(k_new[b], np.broadcast_to(pos, (2, 2)), cos_t, sin_t))
        assert np.array_equal(vc[b, :, L:L + 2], v_new[b])
        qr = orc.rope(_np(case.q)[b:b + 1], np.broadcast_to(pos, (1, 4, 2)), cos_t, sin_t)
        ref, ref_lse, _ = orc.attention(qr, kc[b:b + 1], vc[b:b + 1], np.array([L + 2], np.int32), 0.25)
        assert np.array_equal(out[b:b + 1], ref) and np.array_equal(lse[b:b + 1], ref_lse)
    assert np.array_equal(kc[1], _np(case.k_cache)[1]) and np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


# --- speculative accept/reject ----------------------------------------------------------------

_CHI2_1PCT_5DOF = 15.086  # chi-square 1% critical value, 5 degrees of freedom


def _softmax(logits, T):
    z = logits.astype(F64) / T
    z = np.exp(z - z.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def _chi2(samples, p):
    counts = np.bincount(samples, minlength=len(p)).astype(F64)
    exp_ = p * len(samples)
    return float(((counts - exp_) ** 2 / exp_).sum())


def _spec_batch(orc, p_logits, q_logits, G, N, T, seed):
    """N independent steps with context-free target/draft rows; drafts drawn from q."""
    rng = np.random.default_rng(seed)
    V = len(p_logits)
    q = _softmax(q_logits, T)
    tokens = np.stack([rng.choice(V, size=N, p=q) for _ in range(G)], axis=1).astype(np.int32)
    target = np.broadcast_to(p_logits.astype(np.float32), (N, G + 1, V)).copy()
    draft = np.broadcast_to(q_logits.astype(np.float32), (N, G, V)).copy()
    u = rng.random((N, G + 1))
    n, nxt, st = orc.spec_accept(target, draft, tokens, u, T)
    return tokens, n, nxt, st


def pin_spec_output_follows_target(orc):
    """The pages' chi-squared check: vocabulary 6, N = 30,000, draft q != target p, gamma 1
    and 4; the first emitted token (and with gamma 4 the second) is distributed as p
    (temperature 0.7 applied to both)."""
    p_logits = np.array([1.2, -0.3, 0.4, 2.0, -1.0, 0.1])
    q_logits = np.array([-0.5, 1.5, 0.3, 0.2, 1.0, -0.2])
    T = 0.7
    p = _softmax(p_logits, T)
    for G, seed in ((1, 11), (4, 12)):
        tokens, n, nxt, st = _spec_batch(orc, p_logits, q_logits, G, 30000, T, seed)
        assert st == 0
        first = np.where(n >= 1, tokens[:, 0], nxt)
        assert _chi2(first, p) < _CHI2_1PCT_5DOF, ("first token", G)
        if G >= 2:
            has2 = n >= 1
            second = np.where(n[has2] >= 2, tokens[has2, 1], nxt[has2])
            assert _chi2(second, p) < _CHI2_1PCT_5DOF, ("second token", G)


def pin_spec_acceptance_rate(orc):
    """P(first draft accepted) = sum_x min(p(x), q(x)) (Leviathan et al.'s alpha), within
    four binomial standard deviations."""
    p_logits = np.array([0.5, 0.0, -1.0, 1.5, 0.2, -0.4])
    q_logits = np.array([0.0, 1.0, 0.5, -0.5, 0.2, 0.3])
    p, q = _softmax(p_logits, 1.0), _softmax(q_logits, 1.0)
    alpha = float(np.minimum(p, q).sum())
    N = 20000
    _, n, _, _ = _spec_batch(orc, p_logits, q_logits, 1, N, 1.0, 13)
    rate = float((n >= 1).mean())
    assert abs(rate - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / N), (rate, alpha)


def pin_spec_residual_distribution(orc):
    """A draft token the target gives probability 0 is always rejected, and the extra token
    then follows max(0, p - q) / ||max(0, p - q)||_1."""
    p_logits = np.array([0.3, -np.inf, 1.0, 0.2, -0.5, 0.8])
    q_logits = np.array([0.0, 2.0, 0.1, 0.4, 0.0, 0.3])
    p, q = _softmax(p_logits, 1.0), _softmax(q_logits, 1.0)
    res = np.maximum(0.0, p - q)
    res /= res.sum()
    N = 30000
    rng = np.random.default_rng(14)
    target = np.broadcast_to(p_logits.astype(np.float32), (N, 2, 6)).copy()
    draft = np.broadcast_to(q_logits.astype(np.float32), (N, 1, 6)).copy()
    tokens = np.full((N, 1), 1, np.int32)
    n, nxt, st = orc.spec_accept(target, draft, tokens, rng.random((N, 2)), 1.0)
    assert st == 0 and np.all(n == 0)
    keep = res > 0
    assert np.all(keep[nxt])  # never a token outside the residual's support
    counts = np.bincount(nxt, minlength=6)[keep].astype(F64)
    exp_ = res[keep] * N
    assert float(((counts - exp_) ** 2 / exp_).sum()) < 13.277  # 1% point, 4 degrees of freedom


def pin_spec_draft_equals_target(orc):
    """q = p: every draft token is accepted and the extra token is the inverse-CDF draw from
    the bonus row (checked against numpy's cumulative sum)."""
    rng = np.random.default_rng(15)
    B, G, V = 64, 3, 50
    logits = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    u = rng.random((B, G + 1))
    n, nxt, st = orc.spec_accept(logits, logits[:, :G].copy(), tokens, u, 1.0)
    assert st == 0 and np.all(n == G)
    cdf = np.cumsum(_softmax(logits[:, G], 1.0), axis=1)
    ref = np.array([int(np.searchsorted(cdf[b], u[b, G] * cdf[b, -1], side="right")) for b in range(B)])
    assert np.array_equal(nxt, ref)


def pin_spec_greedy_prefix(orc):
    """Temperature 0: accept while the draft token is the target's argmax; the extra token is
    the target's argmax after the accepted prefix (ties to the lowest id)."""
    V, G = 8, 3
    target = np.zeros((3, G + 1, V), np.float32)
    arg = np.array([[2, 5, 1, 7], [4, 4, 0, 3], [6, 1, 2, 2]])
    for b in range(3):
        for i in range(G + 1):
            target[b, i, arg[b, i]] = 1.0
    target[2, 3, 0] = 1.0  # a tie at the bonus row: id 0 wins over 2
    draft = np.full((3, G, V), 0.0, np.float32)
    draft[:, :, 3] = 5.0  # the draft's own argmax is 3 everywhere
    tokens = np.array([[2, 5, 0], [4, 4, 0], [6, 1, 2]], np.int32)
    n, nxt, st = orc.spec_accept(target, draft, tokens, None, 0.0)
    assert st == 0 and n.tolist() == [2, 3, 3] and nxt.tolist() == [1, 3, 0]


def pin_spec_bad_token(orc):
    """A draft token outside [0, V) stops acceptance there and raises the status bit."""
    target = np.zeros((1, 3, 4), np.float32)
    draft = np.zeros((1, 2, 4), np.float32)
    n, _, st = orc.spec_accept(target, draft, np.array([[1, 9]], np.int32), np.array([[0.1, 0.1, 0.5]]), 1.0)
    assert st == orc_mod.BAD_TOKEN and n.tolist() == [1]


# --- quantised KV cache ---------------------------------------------------------------------

def pin_q8_round_trip_bound(orc):
    """Every element reads back within half a step of the row's scale; codes are integers in
    [-127, 127] and the largest magnitude of the row takes the full-scale code."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((50, 64)) * rng.uniform(0.01, 100, (50, 1))).astype(np.float32)
    codes, scales = orc.quantize_q8(x)
    back = orc.dequantize_q8(codes, scales)
    assert codes.min() >= -127 and codes.max() <= 127
    assert np.all(np.abs(back - x) <= scales[:, None].astype(F64) * (0.5 + 1e-6))
    top = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(50), top]) == 127)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    cb, sb = orc.quantize_q8(_np(xb))
    assert np.all(np.abs(orc.dequantize_q8(cb, sb) - xb.double().numpy()) <= sb[:, None].astype(F64) * (0.5 + 1e-6))


def pin_q8_ties_to_even_and_symmetry(orc):
    """With amax 127 the scale is exactly 1: halves round to even; negating the row negates the
    codes; doubling it keeps the codes and doubles the scale exactly; a zero row is all zero."""
    x = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.49, -126.6]], np.float32)
    codes, scales = orc.quantize_q8(x)
    assert scales[0] == 1.0 and codes[0].tolist() == [127, 0, 2, 2, 0, -2, 3, -127]
    rng = np.random.default_rng(22)
    y = rng.standard_normal((10, 32)).astype(np.float32)
    c1, s1 = orc.quantize_q8(y)
    c2, s2 = orc.quantize_q8(-y)
    c3, s3 = orc.quantize_q8(2 * y)
    assert np.array_equal(c2, -c1) and np.array_equal(s2, s1)
    assert np.array_equal(c3, c1) and np.array_equal(s3, 2 * s1)
    c0, s0 = orc.quantize_q8(np.zeros((2, 16), np.float32))
    assert not c0.any() and not s0.any()


def pin_q8_attention_reads_the_dequantised_cache(orc):
    """A cache whose rows are small integers with scale 1 quantises to itself, and attention
    over the codes equals attention over the original bf16 cache."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, S, D = 2, 4, 2, 40, 16
    k = rng.integers(-127, 128, (B, Hkv, S, D)).astype(np.float32)
    v = rng.integers(-127, 128, (B, Hkv, S, D)).astype(np.float32)
    k[..., 0] = 127.0  # full-scale element in every row: scale exactly 1
    v[..., 0] = -127.0
    q = rng.standard_normal((B, Hq, D)).astype(np.float32) * 0.01
    kc, ks = orc.quantize_q8(k)
    vc, vs = orc.quantize_q8(v)
    assert np.all(ks == 1.0) and np.all(vs == 1.0) and np.array_equal(kc, k.astype(np.int8))
    sl = np.array([40, 7], np.int32)
    out, lse, _ = orc.attention_q8(q, kc, ks, vc, vs, sl, 0.5)
    ref, ref_lse, _ = orc.attention(q, k, v, sl, 0.5)
    assert np.allclose(out, ref, rtol=0, atol=1e-12) and np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
