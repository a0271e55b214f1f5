"""Tiled causal prefill (tcgen05) against the CPU oracle: td_verify_attn's definition.

Small cases span several 128-row query tiles and 128-key tiles with ragged ends, a prefix
already in the cache, grouped-query heads, both head dims, a chunk longer than its sequence
and stale rows poisoned with NaN past the length. A 4096-token prompt is checked on sampled
rows (each row is a decode over its own visible keys in the oracle).
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_split_gb300.workloads import small_case, to_numpy
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


def _run(td, case, k=None, v=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = td.td_prefill_attn(case.q.cuda(), (case.k_cache if k is None else k).cuda(),
                                  (case.v_cache if v is None else v).cuda(), case.seq_lens.cuda(), case.scale,
                                  dev_status=st, return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), int(st.item())


PREFILL = [
    # B, Hq, Hkv, D, Smax, T, lengths (counting the T new tokens)
    (1, 4, 2, 128, 300, 300, [300]),            # a fresh prompt: 3 query tiles, ragged
    (2, 6, 2, 64, 520, 260, [400, 260]),        # a 140-token prefix in sequence 0; D = 64
    (1, 8, 8, 128, 1000, 129, [1000]),          # 129 tokens on an 871-token prefix
    (1, 4, 1, 128, 64, 64, [64]),
    (3, 12, 4, 128, 700, 200, [700, 200, 455]),
    # more query tiles (heads x tiles) than CTA slots: a second wave of CTAs
    (2, 40, 8, 128, 700, 512, [512, 700]),      # with a 188-token prefix in sequence 1
    (4, 32, 4, 64, 400, 384, [384, 400, 390, 384]),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,Smax,T,lens", PREFILL)
def test_prefill_against_oracle(td, B, Hq, Hkv, D, Smax, T, lens):
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens, seed=T + D,
                      heavy=0.02)
    out, lse, st = _run(td, case)
    args = (to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache), case.seq_lens.numpy(), case.scale)
    ref, ref_lse, ref_st = oracle.load().attention(*args)
    assert st == ref_st
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, value_stats(*args, ref_lse))
    assert_lse_close(lse, ref_lse)


def test_prefill_chunk_longer_than_sequence_flags(td):
    """Rows that see no key give 0 and -inf and the verify-short bit, as td_verify_attn."""
    case = small_case(dtype="bf16", B=1, Hq=2, Hkv=1, D=128, Smax=64, T=40, seq_lens=[30], seed=3)
    out, lse, st = _run(td, case)
    args = (to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache), case.seq_lens.numpy(), case.scale)
    ref, ref_lse, ref_st = oracle.load().attention(*args)
    assert st == ref_st == td.DEV_VERIFY_SHORT
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, value_stats(*args, ref_lse))
    assert_lse_close(lse, ref_lse)


def test_prefill_never_reads_past_the_length(td):
    case = small_case(dtype="bf16", B=1, Hq=4, Hkv=2, D=128, Smax=400, T=150, seq_lens=[333], seed=4)
    k, v = case.k_cache.clone(), case.v_cache.clone()
    k[:, :, 333:] = float("nan")
    v[:, :, 333:] = float("nan")
    out, lse, _ = _run(td, case, k, v)
    args = (to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache), case.seq_lens.numpy(), case.scale)
    ref, ref_lse, _ = oracle.load().attention(*args)
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, value_stats(*args, ref_lse))
    assert_lse_close(lse, ref_lse)


def test_prefill_matches_verify_kernel(td):
    case = small_case(dtype="bf16", B=1, Hq=24, Hkv=8, D=128, Smax=1024, T=512, seq_lens=[1000], seed=5)
    out, _, _ = _run(td, case)
    ver = td.td_verify_attn(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda(),
                            case.scale)
    torch.cuda.synchronize()
    assert_out_close(out, ver.cpu().double().numpy(), "bf16", what="prefill vs verify kernel")


@pytest.mark.parametrize("T", [4096, 8192])
def test_prefill_long_prompt_sampled_rows(td, T):
    """The prompts the bench line times (3B-style layer); 40 sampled (head, row) pairs in the oracle."""
    case = small_case(dtype="bf16", B=1, Hq=24, Hkv=8, D=128, Smax=T, T=T, seq_lens=[T], seed=6, heavy=0.01)
    out, lse, st = _run(td, case)
    assert st == 0
    rng = np.random.default_rng(0)
    orc = oracle.load()
    kn, vn = to_numpy(case.k_cache), to_numpy(case.v_cache)
    picks = [(0, 0), (23, T - 1), (5, T - 64)] + [(int(rng.integers(0, 24)), int(rng.integers(0, T))) for _ in range(37)]
    for hq, t in picks:  # the first row, the last rows of the prompt, then random ones
        kvh = hq // 3
        qrow = to_numpy(case.q[:, hq:hq + 1, t])  # [1, 1, D]
        args = (qrow, kn[:, kvh:kvh + 1], vn[:, kvh:kvh + 1], np.array([t + 1], np.int32), case.scale)
        ref, ref_lse, _ = orc.attention(*args)
        assert_out_close(out[:, hq:hq + 1, t], ref, "bf16", what=f"row ({hq}, {t})")
        assert_value_close(out[:, hq:hq + 1, t], ref, value_stats(*args, ref_lse), what=f"row ({hq}, {t})")
        assert_lse_close(lse[:, hq:hq + 1, t], ref_lse)


@pytest.mark.parametrize("scale", [0.0, -0.05])
def test_prefill_zero_and_negative_scale(td, scale):
    """scale 0: each row is the mean of its visible values; a negative scale turns the row
    minimum into the softmax's reference (both through masked and unmasked tiles)."""
    case = small_case(dtype="bf16", B=1, Hq=4, Hkv=2, D=128, Smax=400, T=300, seq_lens=[390], seed=8)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = td.td_prefill_attn(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda(),
                                  scale, dev_status=st, return_lse=True)
    torch.cuda.synchronize()
    args = (to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache), case.seq_lens.numpy(), scale)
    ref, ref_lse, _ = oracle.load().attention(*args)
    assert_out_close(out.cpu(), ref, "bf16")
    assert_value_close(out.cpu(), ref, value_stats(*args, ref_lse))
    assert_lse_close(lse.cpu(), ref_lse)
