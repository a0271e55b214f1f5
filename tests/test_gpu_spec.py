"""Speculative accept/reject on the GPU against the CPU oracle and the pages' chi-squared test.

The accept decisions and the inverse-CDF draw are decided in fp32 on the GPU and in fp64 in
the oracle, so a row is compared exactly unless its decision sits within a small margin of
the threshold (then either outcome is valid); a drawn token must lie in the fp64 interval of
the cumulative weights that holds u * total (widened by the same margin). Greedy decisions
compare stored fp32 logits only and must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHI2_1PCT_5DOF = 15.086


@pytest.fixture(scope="module")
def td():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td
    return td


def _softmax(x, T):
    z = x.astype(np.float64) / T
    z = np.exp(z - z.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def _run(td, target, draft, tokens, u, T):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, nxt = td.td_spec_accept(torch.from_numpy(target).cuda(), torch.from_numpy(tokens).cuda(),
                               None if draft is None else torch.from_numpy(draft).cuda(),
                               None if u is None else torch.from_numpy(u).cuda(), T, dev_status=st)
    torch.cuda.synchronize()
    return n.cpu().numpy(), nxt.cpu().numpy(), int(st.item())


def _case(B, G, V, seed, T, close=0.5):
    """Random logits; draft tokens drawn from q; the draft's logits a perturbation of the target's."""
    rng = np.random.default_rng(seed)
    target = rng.standard_normal((B, G + 1, V)).astype(np.float32) * 2
    draft = (target[:, :G] + close * rng.standard_normal((B, G, V))).astype(np.float32)
    q = _softmax(draft, T)
    tokens = np.array([[rng.choice(V, p=q[b, i]) for i in range(G)] for b in range(B)], np.int32).reshape(B, G)
    u = rng.random((B, G + 1)).astype(np.float32)
    return target, draft, tokens, u


def _check_against_oracle(td, target, draft, tokens, u, T, margin=1e-4):
    B, G1, V = target.shape
    G = G1 - 1
    n, nxt, st = _run(td, target, draft, tokens, u, T)
    rn, rnxt, rst = oracle.load().spec_accept(target, draft, tokens, u.astype(np.float64), T)
    assert st == rst
    p = _softmax(target, T)
    q = _softmax(draft, T) if G else None
    exact = 0
    for b in range(B):
        if n[b] != rn[b]:
            # the deciding token must sit within the margin of its threshold
            i = min(n[b], rn[b])
            x = tokens[b, i]
            gap = np.log(u[b, i]) - (np.log(p[b, i, x]) - np.log(q[b, i, x]))
            assert abs(gap) < margin, (b, n[b], rn[b], gap)
            continue
        k = int(n[b])
        w = np.maximum(0.0, p[b, k] - q[b, k]) if k < G else p[b, k]
        if not w.sum() > 0:
            w = p[b, k]
        cdf = np.cumsum(w)
        tgt = float(u[b, G]) * cdf[-1]
        lo = cdf[nxt[b] - 1] if nxt[b] > 0 else 0.0
        tol = margin * cdf[-1]
        assert w[nxt[b]] > 0 and lo - tol <= tgt <= cdf[nxt[b]] + tol, (b, nxt[b], rnxt[b], tgt, lo, cdf[nxt[b]])
        exact += int(nxt[b] == rnxt[b])
    assert exact >= 0.98 * B, f"only {exact} of {B} draws equal the oracle's"


@pytest.mark.parametrize("G,V,T", [(4, 6, 1.0), (4, 1000, 0.7), (1, 32000, 1.0), (8, 5000, 1.3), (0, 777, 1.0)])
def test_spec_accept_matches_oracle(td, G, V, T):
    target, draft, tokens, u = _case(64, G, V, seed=V + G, T=T)
    _check_against_oracle(td, target, draft, tokens, u, T)


def test_spec_accept_large_vocabulary_clusters(td):
    """A llama-3 sized vocabulary: 16 CTAs per sequence share it."""
    target, draft, tokens, u = _case(6, 4, 128256, seed=3, T=1.0, close=0.3)
    _check_against_oracle(td, target, draft, tokens, u, 1.0)


@pytest.mark.parametrize("V", [6, 50000])
def test_spec_accept_greedy_exact(td, V):
    rng = np.random.default_rng(V)
    B, G = 40, 5
    target = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    tokens = target[:, :G].argmax(-1).astype(np.int32)
    # break the prefix at a random place in most rows
    cut = rng.integers(0, G + 1, B)
    for b in range(B):
        if cut[b] < G:
            tokens[b, cut[b]] = (tokens[b, cut[b]] + 1) % V
    target[0, 2, :] = 1.0  # an all-equal row: the lowest id wins
    n, nxt, st = _run(td, target, None, tokens, None, 0.0)
    rn, rnxt, rst = oracle.load().spec_accept(target, None, tokens, None, 0.0)
    assert st == rst == 0
    assert np.array_equal(n, rn) and np.array_equal(nxt, rnxt)


@pytest.mark.parametrize("G", [1, 4])
def test_spec_accept_output_follows_target(td, G):
    """The pages' chi-squared check on the kernel: vocabulary 6, N = 30,000, q != p."""
    p_logits = np.array([1.2, -0.3, 0.4, 2.0, -1.0, 0.1])
    q_logits = np.array([-0.5, 1.5, 0.3, 0.2, 1.0, -0.2])
    T, N = 0.7, 30000
    rng = np.random.default_rng(20 + G)
    q = _softmax(q_logits, T)
    p = _softmax(p_logits, T)
    tokens = rng.choice(6, size=(N, G), p=q).astype(np.int32)
    target = np.broadcast_to(p_logits.astype(np.float32), (N, G + 1, 6)).copy()
    draft = np.broadcast_to(q_logits.astype(np.float32), (N, G, 6)).copy()
    u = rng.random((N, G + 1)).astype(np.float32)
    n, nxt, st = _run(td, target, draft, tokens, u, T)
    assert st == 0

    def chi2(s):
        c = np.bincount(s, minlength=6).astype(np.float64)
        e = p * len(s)
        return float(((c - e) ** 2 / e).sum())

    assert chi2(np.where(n >= 1, tokens[:, 0], nxt)) < CHI2_1PCT_5DOF
    if G >= 2:
        has2 = n >= 1
        assert chi2(np.where(n[has2] >= 2, tokens[has2, 1], nxt[has2])) < CHI2_1PCT_5DOF


def test_spec_accept_draft_equals_target_keeps_all(td):
    rng = np.random.default_rng(7)
    B, G, V = 32, 6, 3000
    logits = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    u = rng.random((B, G + 1)).astype(np.float32) * 0.999
    n, nxt, st = _run(td, logits, logits[:, :G].copy(), tokens, u, 1.0)
    assert st == 0 and np.all(n == G)


def test_spec_accept_bad_token_flags(td):
    rng = np.random.default_rng(8)
    target = rng.standard_normal((2, 3, 10)).astype(np.float32)
    draft = target[:, :2].copy()
    tokens = np.array([[3, 10], [-1, 2]], np.int32)
    u = np.full((2, 3), 0.5, np.float32)
    n, _, st = _run(td, target, draft, tokens, u, 1.0)
    assert st == td.DEV_BAD_TOKEN and n.tolist() == [1, 0]


def test_spec_accept_rejects_bad_arguments(td):
    from decode_attention_split_gb300._lib import TDError
    t = torch.zeros(1, 18, 10, device="cuda")
    with pytest.raises(TDError) as e:
        td.td_spec_accept(t, torch.zeros(1, 17, dtype=torch.int32, device="cuda"), torch.zeros(1, 17, 10, device="cuda"),
                          torch.zeros(1, 18, device="cuda"), 1.0)
    assert e.value.status == 2  # more than 16 draft tokens
