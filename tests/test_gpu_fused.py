"""The rotary cache write and the fused decode/verify step against the CPU oracle.

Rotation is checked per element against the oracle's exactly rounded result (the kernel
rotates in fp32, so an element may land one unit in the last place away when the exact
value sits next to a rounding midpoint); every other cache row must be untouched, bit for
bit. The fused step must equal the oracle's rotate + write + attend (within the attention
tolerance) and, bit for bit, the library's own unfused sequence of calls.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_split_gb300.workloads import rope_tables, small_case, to_numpy
from parity import assert_lse_close, assert_out_close, assert_value_close, value_stats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def td():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td
    return td


def _values(a, dtype):
    """numpy values of stored elements (bf16 bit patterns or fp32)."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).double().numpy()
    return np.asarray(a, dtype=np.float64)


def _pair_magnitude(x, dtype):
    """|x[i]| + |x[i + D/2]| at both elements of each rotated pair."""
    v = np.abs(_values(x, dtype))
    h = v.shape[-1] // 2
    m = v[..., :h] + v[..., h:]
    return np.concatenate([m, m], axis=-1)


def assert_rounded_close(gpu, ref, dtype, what, x):
    """Each element is within one unit in the last place of the exactly rounded reference,
    plus the fp32 rounding of the kernel's two operations (about 2^-23 of |x0| + |x1|, which
    matters where the two products cancel); for bf16, under 1% of elements may differ at all
    (those whose exact value sits next to a rounding midpoint). x: the rows before rotation."""
    g, r = _values(gpu, dtype), _values(ref, dtype)
    mant = 7 if dtype == "bf16" else 23
    _, e = np.frexp(np.maximum(np.abs(g), np.abs(r)))
    ulp = np.ldexp(1.0, e - 1 - mant)
    bad = np.abs(g - r) > ulp + np.ldexp(_pair_magnitude(x, dtype), -22)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements more than one ulp from the oracle"
    if dtype == "bf16":
        frac = float(np.mean(g != r))
        assert frac < 0.01, f"{what}: {frac:.3%} of elements differ from the exactly rounded value"


def _new_rows(B, Hkv, T, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.randn(B, Hkv, T, D, generator=g).to(tdt), torch.randn(B, Hkv, T, D, generator=g).to(tdt)


@pytest.mark.parametrize("dtype,D,T,with_q", [("bf16", 128, 1, True), ("bf16", 64, 6, True), ("f32", 64, 3, True),
                                               ("bf16", 128, 2, False)])
def test_rope_kv_append(td, dtype, D, T, with_q):
    B, Hq, Hkv, S = 4, 6, 3, 48
    case = small_case(dtype=dtype, B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=S, T=T, seq_lens=[0, 17, S - T, S - T + 1], seed=D)
    kn, vn = _new_rows(B, Hkv, T, D, dtype, 1)
    cos_t, sin_t = rope_tables(S, D)
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = case.q.cuda() if with_q else None
    q_out = td.td_rope_kv_append(kn.cuda(), vn.cuda(), kc, vc, sl, cos_t.cuda(), sin_t.cuda(), q=q, advance=True,
                                 dev_status=st)
    torch.cuda.synchronize()
    orc = oracle.load()
    pre = case.seq_lens.numpy()
    ek, ev = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy()
    fits = (pre >= 0) & (pre + T <= S)
    pos = np.where(fits, pre, 0)[:, None] + np.arange(T)[None, :]
    kr = orc.rope(to_numpy(kn), np.broadcast_to(pos[:, None, :], (B, Hkv, T)), cos_t.numpy(), sin_t.numpy())
    es = pre.astype(np.int32).copy()
    ost = orc.kv_append(kr, to_numpy(vn), ek, ev, es, advance=True)
    assert int(st.item()) == ost == td.DEV_APPEND_OVERFLOW
    assert sl.cpu().numpy().tolist() == es.tolist()
    gk, gv = to_numpy(kc.cpu()), to_numpy(vc.cpu())
    for b in range(B):
        if not fits[b]:
            assert np.array_equal(gk[b], ek[b]) and np.array_equal(gv[b], ev[b])
            continue
        L = pre[b]
        rows = np.r_[0:L, L + T:S]
        assert np.array_equal(gk[b][:, rows], ek[b][:, rows]) and np.array_equal(gv[b], ev[b])
        assert_rounded_close(gk[b][:, L:L + T], ek[b][:, L:L + T], dtype, f"rotated keys of sequence {b}",
                             to_numpy(kn)[b])
    if with_q:
        qr = orc.rope(to_numpy(case.q), np.broadcast_to(pos[:, None, :], (B, Hq, T)), cos_t.numpy(), sin_t.numpy())
        got = to_numpy(q_out.cpu())
        for b in np.nonzero(fits)[0]:
            assert_rounded_close(got[b], qr[b], dtype, f"rotated queries of sequence {b}", to_numpy(case.q)[b])


def test_rope_kv_append_in_place_query(td):
    case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=64, Smax=32, T=2, seq_lens=[3, 9], seed=2)
    kn, vn = _new_rows(2, 2, 2, 64, "bf16", 3)
    cos_t, sin_t = rope_tables(32, 64)
    args = (kn.cuda(), vn.cuda())
    caches = [(case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()) for _ in range(2)]
    q1 = case.q.cuda()
    sep = td.td_rope_kv_append(*args, *caches[0], cos_t.cuda(), sin_t.cuda(), q=q1)
    q2 = case.q.cuda()
    td.td_rope_kv_append(*args, *caches[1], cos_t.cuda(), sin_t.cuda(), q=q2, q_out=q2)
    torch.cuda.synchronize()
    assert torch.equal(sep, q2)


FUSED = [
    # B, Hq, Hkv, D, Smax, T, lengths before the step, rope, advance
    (1, 24, 8, 128, 4096, 1, [4000], True, True),            # persistent kernel, one sequence
    (1, 24, 8, 128, 300, 1, [0], True, True),                # first token
    (4, 24, 8, 128, 2000, 1, [1999, 1000, 63, 0], True, True),  # cluster kernel (32 groups)
    (2, 32, 8, 128, 700, 6, [600, 100], True, False),        # verify, cluster kernel, no advance
    (1, 32, 8, 128, 700, 6, [600], True, True),              # verify, persistent kernel
    (1, 15, 5, 64, 1000, 1, [999], True, True),              # D = 64
    (3, 8, 2, 128, 256, 3, [250, 254, 40], True, True),      # second sequence overflows
    (1, 24, 8, 128, 4096, 1, [3000], False, True),           # no rotation: append + attention
    # 200 sequences (400 groups): items in several waves; the lengths advance once every CTA read them
    (200, 8, 2, 64, 300, 1, [(13 * i) % 290 for i in range(200)], True, True),
]


def _oracle_step(case, kn, vn, pre, cos_t, sin_t, scale, advance):
    orc = oracle.load()
    ek, ev = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy()
    es = np.array(pre, np.int32)
    out, lse, st = orc.rope_append_attention(to_numpy(case.q), to_numpy(kn), to_numpy(vn), ek, ev, es, scale,
                                             None if cos_t is None else cos_t.numpy(),
                                             None if sin_t is None else sin_t.numpy(), advance=advance)
    return out, lse, st, ek, ev, es


@pytest.mark.parametrize("B,Hq,Hkv,D,Smax,T,pre,rope,advance", FUSED)
def test_fused_step_against_oracle(td, B, Hq, Hkv, D, Smax, T, pre, rope, advance):
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=pre, seed=Smax + T,
                      heavy=0.02)
    kn, vn = _new_rows(B, Hkv, T, D, "bf16", 5)
    cos_t, sin_t = rope_tables(Smax, D) if rope else (None, None)
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), torch.tensor(pre, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = td.td_rope_append_attn(case.q.cuda(), kn.cuda(), vn.cuda(), kc, vc, sl, case.scale, 0,
                                      cos_t=None if cos_t is None else cos_t.cuda(),
                                      sin_t=None if sin_t is None else sin_t.cuda(), advance=advance,
                                      dev_status=st, return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse, ref_st, ek, ev, es = _oracle_step(case, kn, vn, pre, cos_t, sin_t, case.scale, advance)
    assert int(st.item()) == ref_st
    assert sl.cpu().numpy().tolist() == es.tolist()
    assert_out_close(out.cpu(), ref, "bf16")
    if not rope:
        # without rotation the GPU attends exactly the oracle's inputs (with it, a rotated
        # element may differ by one unit in the last place, which the value-side bound does
        # not model; the rotation is checked on its own, and the fused call against the
        # unfused calls bit for bit)
        fits = [b for b, L in enumerate(pre) if 0 <= L and L + T <= Smax]
        es_att = np.array([L + T if b in fits else 0 for b, L in enumerate(pre)], np.int32)
        assert_value_close(out.cpu(), ref, value_stats(to_numpy(case.q), ek, ev, es_att, case.scale, ref_lse))
    assert_lse_close(lse.cpu(), ref_lse)
    gk, gv = to_numpy(kc.cpu()), to_numpy(vc.cpu())
    for b, L in enumerate(pre):
        if not (0 <= L and L + T <= Smax):
            assert np.array_equal(gk[b], ek[b]) and np.array_equal(gv[b], ev[b])
            continue
        rows = np.r_[0:L, L + T:Smax]
        assert np.array_equal(gk[b][:, rows], ek[b][:, rows]) and np.array_equal(gv[b], ev[b])
        if rope:
            assert_rounded_close(gk[b][:, L:L + T], ek[b][:, L:L + T], "bf16", f"rotated keys of sequence {b}",
                                 to_numpy(kn)[b])
        else:
            assert np.array_equal(gk[b], ek[b])


@pytest.mark.parametrize("B,Hq,Hkv,D,Smax,T,pre", [(1, 24, 8, 128, 4096, 1, [4000]), (4, 24, 8, 128, 2000, 1,
                                                     [1999, 1000, 63, 0]), (2, 32, 8, 128, 700, 6, [600, 100])])
def test_fused_step_equals_unfused_calls(td, B, Hq, Hkv, D, Smax, T, pre):
    """One fused launch gives the same bits as rotate + write, then attention."""
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=pre, seed=11)
    kn, vn = _new_rows(B, Hkv, T, D, "bf16", 6)
    cos_t, sin_t = (t.cuda() for t in rope_tables(Smax, D))
    q = case.q.cuda()
    kc1, vc1, sl1 = case.k_cache.cuda(), case.v_cache.cuda(), torch.tensor(pre, dtype=torch.int32, device="cuda")
    kc2, vc2, sl2 = kc1.clone(), vc1.clone(), sl1.clone()
    out1, lse1 = td.td_rope_append_attn(q, kn.cuda(), vn.cuda(), kc1, vc1, sl1, case.scale, 0, cos_t=cos_t,
                                        sin_t=sin_t, return_lse=True)
    qr = td.td_rope_kv_append(kn.cuda(), vn.cuda(), kc2, vc2, sl2, cos_t, sin_t, q=q, advance=True)
    out2, lse2 = td.td_verify_attn(qr, kc2, vc2, sl2, case.scale, 0, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(sl1, sl2) and torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_fused_step_graph_replays_advance(td):
    """Captured once, replayed for successive tokens: each replay writes the next row and moves on."""
    B, Hq, Hkv, D, S = 4, 24, 8, 128, 1024
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=S, seq_lens=[500, 700, 1, 900], seed=12)
    cos_t, sin_t = (t.cuda() for t in rope_tables(S, D))
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    q = torch.zeros(B, Hq, 1, D, dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros(B, Hkv, 1, D, dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    out = torch.empty_like(q)
    ws = td.make_workspace(B, Hq, Hkv, S, D)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):  # warm-up on copies
        td.td_rope_append_attn(q, kn, vn, kc.clone(), vc.clone(), sl.clone(), case.scale, 0, cos_t=cos_t,
                               sin_t=sin_t, out=out, workspace=ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        td.td_rope_append_attn(q, kn, vn, kc, vc, sl, case.scale, 0, cos_t=cos_t, sin_t=sin_t, out=out,
                               workspace=ws, stream=torch.cuda.current_stream())
    gen = torch.Generator().manual_seed(0)
    orc = oracle.load()
    ek, ev, es = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy(), case.seq_lens.numpy().copy()
    for step in range(3):
        qh = torch.randn(B, Hq, 1, D, generator=gen).to(torch.bfloat16)
        knh = torch.randn(B, Hkv, 1, D, generator=gen).to(torch.bfloat16)
        vnh = torch.randn(B, Hkv, 1, D, generator=gen).to(torch.bfloat16)
        q.copy_(qh)
        kn.copy_(knh)
        vn.copy_(vnh)
        g.replay()
        torch.cuda.synchronize()
        ref, _, _ = orc.rope_append_attention(to_numpy(qh), to_numpy(knh), to_numpy(vnh), ek, ev, es, case.scale,
                                              cos_t.cpu().numpy(), sin_t.cpu().numpy())
        assert sl.cpu().numpy().tolist() == es.tolist()
        assert_out_close(out.cpu(), ref, "bf16", what=f"replay {step}")


def test_fused_step_rejects_fp32(td):
    from decode_attention_split_gb300._lib import TDError
    case = small_case(dtype="f32", B=1, Hq=4, Hkv=2, D=64, Smax=64, seq_lens=[10], seed=1)
    kn, vn = _new_rows(1, 2, 1, 64, "f32", 1)
    with pytest.raises(TDError) as e:
        td.td_rope_append_attn(case.q.cuda(), kn.cuda(), vn.cuda(), case.k_cache.cuda(), case.v_cache.cuda(),
                               case.seq_lens.cuda())
    assert e.value.status == 2
