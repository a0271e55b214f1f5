"""The value-side parity bound (tests/parity.py, check 2), pinned on the CPU.

It must be loose enough for the rounding the bf16 kernels really do and tight enough to catch
value-side mistakes that the stated 2e-2 + 1e-2 |ref| tolerance lets through.

* Legitimate rounding: an fp32 emulation of the kernels' arithmetic model (scores in fp32,
  base-2 exponentials against a per-chunk maximum, each probability rounded to bf16 before
  p @ V, the normaliser from the unrounded probabilities, fp32 log-sum-exp merge of chunk
  partials, the output rounded once to bf16) stays inside the bound on the 360M and 3B-style
  layers and on a verify chunk.
* Planted mistakes, computed by the oracle on altered inputs (value rows read one position
  late, everywhere, at stage edges or in one row; value rows of the neighbouring kv head;
  16 value rows read as zero; one 64-key stage's p @ V dropped or counted twice): each one
  fails the bound on the 360M layer at 4096 keys, where the outputs are small (median |out|
  about 0.02). The stated tolerance catches only the wholesale ones and passes every element
  of the others.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_split_gb300.workloads import make_case, small_case, to_numpy
from parity import assert_value_close, value_bound, value_stats

LOG2E = 1.4426950408889634


def emulate_bf16_kernel(case, chunk: int) -> np.ndarray:
    """The kernels' rounding model in fp32 on the CPU (torch), for a workloads.Case."""
    q, k, v = case.q.float(), case.k_cache.float(), case.v_cache.float()
    B, Hq, T, D = q.shape
    G = Hq // k.shape[1]
    qs = torch.tensor(case.scale * LOG2E, dtype=torch.float32)
    out = torch.zeros(B, Hq, T, D)
    for b in range(B):
        L = int(case.seq_lens[b])
        for h in range(Hq):
            K, V = k[b, h // G, :L], v[b, h // G, :L]
            for t in range(T):
                n = L - T + t + 1
                if n <= 0:
                    continue
                s = (K[:n] @ q[b, h, t]) * qs
                ms, ls, accs = [], [], []
                for c0 in range(0, n, chunk):
                    sc = s[c0:c0 + chunk]
                    m = sc.max()
                    p = torch.exp2(sc - m)
                    ms.append(m)
                    ls.append(p.sum())
                    accs.append(p.to(torch.bfloat16).float() @ V[c0:c0 + sc.shape[0]])
                M = torch.stack(ms).max()
                f = torch.exp2(torch.stack(ms) - M)
                acc = (f[:, None] * torch.stack(accs)).sum(0)
                out[b, h, t] = acc / (f * torch.stack(ls)).sum()
    return out.to(torch.bfloat16).double().numpy()


def _ref_and_stats(case, v=None):
    orc = oracle.load()
    vn = to_numpy(case.v_cache) if v is None else v
    ref, lse, _ = orc.attention(to_numpy(case.q), to_numpy(case.k_cache), vn, to_numpy(case.seq_lens), case.scale)
    return ref, lse, value_stats(to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache),
                                 to_numpy(case.seq_lens), case.scale, lse)


@pytest.mark.parametrize("name,L,smax,chunk", [("smollm2_360m", 4096, None, 128), ("smollm2_360m", 1024, None, 64),
                                               ("llama3b", 4096, 4096, 448), ("llama3b", 1024, 1024, 128)])
def test_kernel_rounding_model_inside_the_bound(name, L, smax, chunk):
    case = make_case(name, seq_len=L, smax=smax)
    ref, _, stats = _ref_and_stats(case)
    assert_value_close(emulate_bf16_kernel(case, chunk), ref, stats, what=f"{name} emulated")


def test_kernel_rounding_model_inside_the_bound_verify():
    case = small_case(dtype="bf16", B=2, Hq=32, Hkv=8, D=128, Smax=1200, T=6, seq_lens=[1200, 40], seed=3,
                      heavy=0.01)
    ref, _, stats = _ref_and_stats(case)
    assert_value_close(emulate_bf16_kernel(case, 256), ref, stats, what="verify emulated")


def _mutants(case):
    """Oracle outputs of value-side mistakes a kernel could make, by name: (output, whether the
    stated tolerance already catches it)."""
    orc = oracle.load()
    qn, kn, vn, sl = (to_numpy(x) for x in (case.q, case.k_cache, case.v_cache, case.seq_lens))
    att = lambda v: orc.attention(qn, kn, np.ascontiguousarray(v), sl, case.scale)[0]
    n = vn.shape[2]
    muts = {
        "every value row read one position late": (att(np.roll(vn, -1, axis=2)), True),
        "value rows of the next kv head": (att(np.roll(vn, 1, axis=1)), True),
    }
    edge = vn.copy()
    idx = np.arange(63, n, 64)
    edge[:, :, idx] = vn[:, :, (idx + 1) % n]
    muts["the last key of each 64-key stage reads the next value row"] = (att(edge), False)
    one = vn.copy()
    one[:, :, 2048] = vn[:, :, 2049]
    muts["one value row read one position late"] = (att(one), False)
    zero = vn.copy()
    zero[:, :, 100:116] = 0
    muts["16 value rows read as zero"] = (att(zero), False)
    m, l, acc, _ = orc.split_partials(qn, kn, vn, sl, case.scale, 64)
    for label, factor in (("one 64-key stage of p @ V dropped", 0.0), ("one 64-key stage of p @ V counted twice", 2.0)):
        a2 = acc.copy()
        a2[:, :, 17] *= factor
        muts[label] = (orc.lse_merge(m, l, a2, sl, 64)[0].reshape(case.q.shape), False)
    return muts


def test_value_side_mistakes_fail_the_bound():
    """Every planted value-side mistake fails the bound; the subtle ones (a few rows or one stage)
    pass the stated tolerance on every element."""
    case = make_case("smollm2_360m", seq_len=4096)
    ref, _, stats = _ref_and_stats(case)
    assert float(np.median(np.abs(ref))) < 0.03  # the small outputs that make the stated tolerance weak here
    assert float(np.median(value_bound(ref, stats))) < 0.05 * 2e-2
    for label, (out, coarse) in _mutants(case).items():
        stated_ok = bool(np.all(np.abs(out - ref) <= 2e-2 + 1e-2 * np.abs(ref)))
        assert stated_ok != coarse, label
        with pytest.raises(AssertionError):
            assert_value_close(out, ref, stats, what=label)


def test_value_stats_closed_forms():
    """The sums from the transformed oracle calls against their definitions, by brute force."""
    case = small_case(dtype="bf16", B=1, Hq=4, Hkv=2, D=64, Smax=40, T=2, seq_lens=[37], seed=5)
    q, k, v = (case.q.double().numpy(), case.k_cache.double().numpy(), case.v_cache.double().numpy())
    ref, lse, _ = oracle.load().attention(to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache),
                                          to_numpy(case.seq_lens), case.scale)
    s1, s2, a = value_stats(to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache),
                            to_numpy(case.seq_lens), case.scale, lse)
    for h in range(4):
        for t in range(2):
            n = 37 - 2 + t + 1
            s = case.scale * (k[0, h // 2, :n] @ q[0, h, t])
            w = np.exp(s - s.max())
            w /= w.sum()
            V = v[0, h // 2, :n]
            np.testing.assert_allclose(s1[0, h, t], np.sqrt((w[:, None] ** 2 * V ** 2).sum(0)), rtol=1e-9)
            np.testing.assert_allclose(s2[0, h, t], np.sqrt((w ** 2).sum()), rtol=1e-9)
            np.testing.assert_allclose(a[0, h, t], (w[:, None] * np.abs(V)).sum(0), rtol=1e-9)
