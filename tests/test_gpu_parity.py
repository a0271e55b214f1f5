"""CUDA path against the CPU oracle, element by element, through the C ABI (Python binding).

Small cases span several stages and chunks with ragged tails; the five named workloads run
at their full sizes in the configuration the benchmark times (automatic split), and with
the split sizes the pages discuss. Edge cases: empty and length-1 sequences, lengths past
Smax or negative, short verify chunks, NaN past seq_len, batch independence, graph capture.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_split_gb300.workloads import WORKLOADS, make_case, small_case, to_numpy
from parity import (assert_lse_close, assert_out_close, assert_value_close, case_value_stats, oracle_attention,
                    value_stats)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def td():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td
    return td


def run_attention(td, case, split=0, seq_lens=None, k_cache=None, v_cache=None):
    q = case.q.cuda()
    k = (case.k_cache if k_cache is None else k_cache).cuda()
    v = (case.v_cache if v_cache is None else v_cache).cuda()
    sl = (case.seq_lens if seq_lens is None else seq_lens).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if case.q.shape[2] == 1:
        out, lse = td.td_decode_attn(q[:, :, 0], k, v, sl, case.scale, split, return_lse=True, dev_status=st)
        out = out[:, :, None]
    else:
        out, lse = td.td_verify_attn(q, k, v, sl, case.scale, split, return_lse=True, dev_status=st)
        lse = lse
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu().reshape(case.q.shape[:3]), int(st.item())


def check_case(td, case, split=0, **kw):
    out, lse, st = run_attention(td, case, split=split, **kw)
    ref, ref_lse, ref_st = oracle_attention(case, **kw)
    assert_out_close(out, ref, case.w.dtype)
    if case.w.dtype == "bf16":
        assert_value_close(out, ref, case_value_stats(case, ref_lse, **kw))
    assert_lse_close(lse, ref_lse)
    assert st == ref_st
    return out, lse


# ---------------------------------------------------------------------------------- append

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,advance", [(1, True), (6, True), (3, False)])
def test_append_bit_exact(td, dtype, T, advance):
    B, H, S, D = 5, 3, 40, 64
    g = torch.Generator().manual_seed(T)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kc = torch.randn(B, H, S, D, generator=g).to(tdt)
    vc = torch.randn(B, H, S, D, generator=g).to(tdt)
    kn = torch.randn(B, H, T, D, generator=g).to(tdt)
    vn = torch.randn(B, H, T, D, generator=g).to(tdt)
    seq = torch.tensor([0, 1, 17, S - T, S - T - 1], dtype=torch.int32)
    kc_d, vc_d, sl_d = kc.cuda(), vc.cuda(), seq.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    td.td_kv_append(kn.cuda(), vn.cuda(), kc_d, vc_d, sl_d, advance=advance, dev_status=st)
    torch.cuda.synchronize()
    ek, ev, es = to_numpy(kc).copy(), to_numpy(vc).copy(), seq.numpy().copy()
    ost = oracle.load().kv_append(to_numpy(kn), to_numpy(vn), ek, ev, es, advance=advance)
    assert np.array_equal(to_numpy(kc_d.cpu()), ek) and np.array_equal(to_numpy(vc_d.cpu()), ev)
    assert np.array_equal(sl_d.cpu().numpy(), es)
    assert int(st.item()) == ost == 0


def test_append_overflow_skips_and_flags(td):
    B, H, T, S, D = 3, 2, 4, 16, 128
    kc = torch.zeros(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(B, H, T, D, dtype=torch.bfloat16, device="cuda")
    seq = torch.tensor([13, 12, -2], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    td.td_kv_append(kn, kn, kc, vc, seq, advance=True, dev_status=st)
    torch.cuda.synchronize()
    assert seq.cpu().tolist() == [13, 16, -2]
    assert int(st.item()) == td.DEV_APPEND_OVERFLOW
    assert kc[0].abs().sum().item() == 0 and kc[2].abs().sum().item() == 0
    assert kc[1, :, 12:16].float().sum().item() == H * T * D


# -------------------------------------------------------------------------- small decode cases

SMALL = [
    # dtype, D, Hq, Hkv, Smax, lengths, split
    ("f32", 64, 4, 2, 256, [128], 64),
    ("f32", 64, 4, 4, 300, [300, 1, 77], 0),
    ("f32", 128, 8, 2, 300, [299, 33], 0),
    ("f32", 64, 16, 2, 200, [200, 150], 16),   # 8 rows per kv head
    ("bf16", 64, 15, 5, 300, [300, 64, 1], 0),
    ("bf16", 64, 15, 5, 300, [257, 11], 7),
    ("bf16", 128, 24, 8, 520, [520, 100], 0),
    ("bf16", 128, 24, 8, 520, [519, 16], 1),
    ("bf16", 128, 32, 4, 260, [260, 5], 0),    # 8 heads per kv head: the narrow tile's full 8 rows
    ("bf16", 128, 20, 4, 130, [130], 0),       # 5 heads: ragged row block
    ("bf16", 128, 8, 8, 200, [200, 3, 64], 100),
    ("bf16", 64, 8, 1, 400, [400, 399, 31, 2], 0),
    ("bf16", 128, 4, 2, 1000, [1000], 1000),
]


@pytest.mark.parametrize("dtype,D,Hq,Hkv,Smax,lens,split", SMALL)
def test_decode_small(td, dtype, D, Hq, Hkv, Smax, lens, split):
    case = small_case(dtype=dtype, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, seq_lens=lens, seed=D + Hq + split,
                      heavy=0.02)
    check_case(td, case, split=split)


@pytest.mark.parametrize("split", [0, 1, 16, 64, 128, 256, 1024, 4096, 37])
def test_decode_split_sweep(td, split):
    case = small_case(dtype="bf16", B=2, Hq=24, Hkv=8, D=128, Smax=4096, seq_lens=[4096, 1500], seed=3, heavy=0.01)
    check_case(td, case, split=split)


# Rows per kv head on either side of the narrow tile's limit: 8 or fewer put the keys on the
# m side and the rows on n (warp_keys16_n8), 9 to 16 take one 16-row m tile, more take
# several row blocks; verify rows carry their own causal limits inside a tile.
TILE_EDGES = [
    # D, Hq, Hkv, Smax, T, lengths, split
    (128, 14, 2, 700, 1, [700, 129], 0),   # 7 rows
    (64, 16, 2, 700, 1, [700, 1], 0),      # 8 rows
    (128, 18, 2, 700, 1, [650, 64], 0),    # 9 rows
    (64, 32, 2, 700, 1, [700, 333], 0),    # 16 rows
    (128, 4, 2, 300, 4, [300, 70], 0),     # verify, 8 rows
    (128, 4, 2, 300, 4, [300, 4], 13),     # verify, 8 rows, the whole sequence new
    (64, 6, 2, 300, 3, [300, 5], 19),      # verify, 9 rows
]


@pytest.mark.parametrize("D,Hq,Hkv,Smax,T,lens,split", TILE_EDGES)
def test_narrow_tile_edges(td, D, Hq, Hkv, Smax, T, lens, split):
    case = small_case(dtype="bf16", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens,
                      seed=Hq + T + split, heavy=0.02)
    check_case(td, case, split=split)


# ----------------------------------------------------------------------------------- verify

VERIFY = [
    ("bf16", 128, 32, 8, 200, 6, [200, 70], 0),
    ("bf16", 128, 32, 8, 200, 6, [200, 6], 16),
    ("bf16", 64, 6, 2, 90, 3, [90, 3, 50], 5),
    ("f32", 64, 4, 2, 128, 2, [128, 40], 0),
    ("bf16", 128, 8, 8, 64, 4, [64], 1),
    ("bf16", 128, 4, 1, 300, 8, [300, 9], 0),
]


@pytest.mark.parametrize("dtype,D,Hq,Hkv,Smax,T,lens,split", VERIFY)
def test_verify_small(td, dtype, D, Hq, Hkv, Smax, T, lens, split):
    case = small_case(dtype=dtype, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens, seed=T + split)
    check_case(td, case, split=split)


def test_verify_short_sequence_flags(td):
    case = small_case(dtype="bf16", B=2, Hq=4, Hkv=2, D=128, Smax=64, T=6, seq_lens=[3, 64], seed=1)
    out, lse, st = run_attention(td, case)
    ref, ref_lse, ref_st = oracle_attention(case)
    assert st == ref_st == td.DEV_VERIFY_SHORT
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, case_value_stats(case, ref_lse))
    assert_lse_close(lse, ref_lse)


def test_verify_equals_sequential_decode(td):
    """Row t of the chunk matches a decode of q_t over L - T + t + 1 keys, within the bf16 tolerance.

    (The identity is exact in the oracle; on the GPU a 24-row verify tile and a 4-row decode
    tile split their keys differently across warps, so the fp32 summation order differs.)"""
    T = 6
    case = small_case(dtype="bf16", B=1, Hq=32, Hkv=8, D=128, Smax=700, T=T, seq_lens=[690], seed=9)
    out, _, _ = run_attention(td, case, split=64)
    for t in range(T):
        sub = small_case(dtype="bf16", B=1, Hq=32, Hkv=8, D=128, Smax=700, seq_lens=[690 - T + t + 1], seed=9)
        sub.q = case.q[:, :, t:t + 1].contiguous()
        sub.k_cache, sub.v_cache = case.k_cache, case.v_cache
        o_t, _, _ = run_attention(td, sub, split=64)
        assert_out_close(out[:, :, t], o_t[:, :, 0].double().numpy(), "bf16", what=f"token {t}")


# --------------------------------------------------------------------------- cluster kernel

CLUSTER = [
    # D, Hq, Hkv, Smax, T, lengths: enough (b, kv head, row block) groups for one wave of
    # clusters, automatic split
    (128, 24, 8, 4096, 1, [4096, 4000, 1, 0]),                 # 32 groups: clusters of 8
    (128, 24, 8, 2000, 1, [1999, 1999, 65, 64]),               # ragged last stages
    (128, 24, 8, 300, 1, [65, 1, 0, 300, 299, 128, 64, 3]),    # 64 groups: clusters of 4
    (64, 64, 8, 1000, 1, [1000, 999, 500, 17, 1, 0, 640, 64]),  # 8 heads per kv head
    (64, 32, 8, 700, 1, [700] * 12 + [1, 0, 333, 64]),         # 128 groups: clusters of 2
    (128, 32, 8, 700, 6, [690, 100, 350, 7]),                  # verify: 24 rows on the 24-row tile
    (128, 32, 8, 64, 6, [64, 3, 60, 6]),                       # verify with short sequences
    (128, 24, 8, 1000, 1, [1000, 1000, 999, 1000]),            # Smax not a stage multiple
    # ragged batches: long sequences beside short and empty ones
    (128, 24, 8, 8192, 1, [8192, 64, 8192, 100]),               # long sequences beside short ones
    (128, 32, 8, 4096, 6, [4096, 100, 50, 2000]),               # verify rows on the 24-row tile
    (64, 16, 4, 5000, 1, [5000, 3, 2500, 4999, 1, 0, 4000, 700]),  # D = 64, short and empty ones
    (128, 32, 8, 6000, 1, [5911, 443, 5723, 17, 600, 3000, 1, 4500]),  # pieces beside whole groups
]


@pytest.mark.parametrize("D,Hq,Hkv,Smax,T,lens", CLUSTER)
def test_cluster_kernel_against_oracle_and_persistent(td, D, Hq, Hkv, Smax, T, lens):
    B = len(lens)
    plan = td.td_split_plan(torch.bfloat16, B, Hq, Hkv, Smax, D, T, 0)
    assert plan["kernel"] == "tensor_core_cluster", plan
    assert plan["grid"] % plan["cluster"] == 0 and plan["cluster"] in (2, 4, 8, 16)
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens, seed=Smax + T,
                      heavy=0.02)
    out_c, lse_c = check_case(td, case, split=0)
    # the persistent kernel (fixed chunks) on the same inputs agrees within the same tolerance
    assert td.td_split_plan(torch.bfloat16, B, Hq, Hkv, Smax, D, T, 128)["kernel"] == "tensor_core_persistent"
    out_p, lse_p = check_case(td, case, split=128)
    assert_out_close(out_c, out_p.double().numpy(), "bf16", what="cluster vs persistent")


# ---------------------------------------------------- 24-row tile, merges by row slices

ROW_SLICES = [
    # D, Hq, Hkv, Smax, T, lengths, split: row blocks of 17 to 24 rows on the 24-row tile; in a
    # one-wave plan the CTAs holding a group's last tickets merge one row slice each, in a
    # plan of several waves (a small explicit split) the last CTA merges every row
    (128, 32, 8, 2000, 6, [1990], 0),          # verify: 24 rows, 6 slices
    (128, 16, 4, 700, 6, [690, 100], 0),       # verify, two sequences
    (128, 16, 4, 300, 6, [300, 6, 0], 0),      # a chunk of exactly T keys and an empty sequence
    (128, 160, 8, 900, 1, [900], 0),           # 20 rows: decode on the 24-row tile
    (64, 36, 2, 1000, 1, [1000, 999], 0),      # 18 rows at D = 64: a ragged last slice
    (128, 32, 8, 2000, 6, [1990], 16),         # 125 chunks, several waves: one CTA merges in rounds
    (128, 32, 8, 600, 6, [600, 33], 37),       # a 37-key split: ragged stages in every chunk
    (128, 40, 4, 500, 2, [500], 0),            # 20 rows from 10 heads x 2 tokens
]


@pytest.mark.parametrize("D,Hq,Hkv,Smax,T,lens,split", ROW_SLICES)
def test_row_slice_merges_against_oracle(td, D, Hq, Hkv, Smax, T, lens, split):
    B = len(lens)
    plan = td.td_split_plan(torch.bfloat16, B, Hq, Hkv, Smax, D, T, split)
    assert plan["kernel"] == "tensor_core_persistent" and 16 < plan["rows"] <= 24, plan
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens, seed=Smax + Hq + T,
                      heavy=0.02)
    check_case(td, case, split=split)


def test_row_slice_merges_repeat_calls_bit_identical_and_counters_rezeroed(td):
    case = small_case(dtype="bf16", B=1, Hq=32, Hkv=8, D=128, Smax=5000, T=6, seq_lens=[5000], seed=21)
    q, k, v, sl = case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    ws = td.make_workspace(1, 32, 8, 5000, 128, 6, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1 = td.td_verify_attn(q, k, v, sl, case.scale, 0, workspace=ws, dev_status=st)
    o2 = td.td_verify_attn(q, k, v, sl, case.scale, 0, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and int(st.item()) == 0
    # completion tickets and finished-slice counts of the 8 groups are back to zero
    assert int(ws[:4 * 16].view(torch.int32).abs().sum()) == 0


def test_cluster_ragged_repeat_calls_bit_identical_and_workspace_clean(td):
    """A ragged batch on the cluster kernel: a second call on the same workspace gives the same
    bits, and the workspace's counters are left at zero for the next call."""
    lens = [8000, 100, 7000, 5]
    B, Hq, Hkv, D, Smax = len(lens), 32, 8, 128, 8000
    assert td.td_split_plan(torch.bfloat16, B, Hq, Hkv, Smax, D, 1, 0)["kernel"] == "tensor_core_cluster"
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=1, seq_lens=lens, seed=5)
    q, k, v, sl = case.q.cuda()[:, :, 0], case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    ws = td.make_workspace(B, Hq, Hkv, Smax, D, 1, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1 = td.td_decode_attn(q, k, v, sl, case.scale, 0, workspace=ws, dev_status=st)
    o2 = td.td_decode_attn(q, k, v, sl, case.scale, 0, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and int(st.item()) == 0
    assert int(ws[:4 * 2 * B * Hkv].view(torch.int32).abs().sum()) == 0
    ref, _, _ = oracle.load().attention(to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache),
                                        to_numpy(case.seq_lens), case.scale)
    assert_out_close(o1.cpu()[:, :, None], ref, "bf16")


def test_automatic_split_fills_one_wave(td):
    """Uniform batches whose per-sequence chunk round-up would overshoot the grid still match."""
    for B, L in ((8, 3000), (4, 2900)):
        case = small_case(dtype="bf16", B=B, Hq=32, Hkv=8, D=128, Smax=L, seq_lens=[L] * B, seed=B, heavy=0.01)
        check_case(td, case, split=0)


# ------------------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name", ["tiny_fp32", "smollm2_360m", "llama3b"])
def test_workload_decode_full_size(td, name):
    w = WORKLOADS[name]
    for L in w.seq_lens:
        case = make_case(w, seq_len=L)
        check_case(td, case, split=w.split)


def test_workload_tiny_fp32_named_split(td):
    case = make_case("tiny_fp32")
    check_case(td, case, split=64)


@pytest.mark.parametrize("split", [0, 256])
def test_workload_ragged8_append_then_attend(td, split):
    case = make_case("ragged8")
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens_pre.cuda()
    td.td_kv_append(case.k_new.cuda(), case.v_new.cuda(), kc, vc, sl, advance=True)
    # oracle side: its own append on its own copy
    ek, ev, es = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy(), to_numpy(case.seq_lens_pre).copy()
    oracle.load().kv_append(to_numpy(case.k_new), to_numpy(case.v_new), ek, ev, es, advance=True)
    assert np.array_equal(sl.cpu().numpy(), es) and np.array_equal(es, case.seq_lens.numpy())
    assert np.array_equal(to_numpy(kc.cpu()), ek) and np.array_equal(to_numpy(vc.cpu()), ev)
    out, lse = td.td_decode_attn(case.q.cuda()[:, :, 0], kc, vc, sl, case.scale, split, return_lse=True)
    ref, ref_lse, _ = oracle.load().attention(to_numpy(case.q), ek, ev, es, case.scale)
    assert_out_close(out.cpu()[:, :, None], ref, "bf16")
    assert_value_close(out.cpu()[:, :, None], ref, value_stats(to_numpy(case.q), ek, ev, es, case.scale, ref_lse))
    assert_lse_close(lse.cpu()[:, :, None], ref_lse)


@pytest.mark.parametrize("split", [0, 256])
def test_workload_verify6_append_then_verify(td, split):
    case = make_case("verify6")
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens_pre.cuda()
    td.td_kv_append(case.k_new.cuda(), case.v_new.cuda(), kc, vc, sl, advance=True)
    ek, ev, es = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy(), to_numpy(case.seq_lens_pre).copy()
    oracle.load().kv_append(to_numpy(case.k_new), to_numpy(case.v_new), ek, ev, es, advance=True)
    assert es.tolist() == [16390]
    out, lse = td.td_verify_attn(case.q.cuda(), kc, vc, sl, case.scale, split, return_lse=True)
    ref, ref_lse, _ = oracle.load().attention(to_numpy(case.q), ek, ev, es, case.scale)
    assert_out_close(out.cpu(), ref, "bf16")
    assert_value_close(out.cpu(), ref, value_stats(to_numpy(case.q), ek, ev, es, case.scale, ref_lse))
    assert_lse_close(lse.cpu(), ref_lse)


# ------------------------------------------------------------------------------- merge alone

@pytest.mark.parametrize("out_dtype,T,split", [("f32", 1, 16), ("bf16", 1, 64), ("f32", 3, 7), ("bf16", 6, 128)])
def test_lse_merge_alone(td, out_dtype, T, split):
    dtype = "f32" if out_dtype == "f32" else "bf16"
    case = small_case(dtype=dtype, B=3, Hq=8, Hkv=2, D=128, Smax=400, T=T, seq_lens=[400, 5, 250], seed=split)
    orc = oracle.load()
    m, l, acc, _ = orc.split_partials(to_numpy(case.q), to_numpy(case.k_cache), to_numpy(case.v_cache),
                                      to_numpy(case.seq_lens), case.scale, split)
    # the GPU merges fp32 partials: round them first and give the oracle the same numbers
    m32, l32, a32 = (np.asarray(x, np.float32) for x in (m, l, acc))
    ref, ref_lse = orc.lse_merge(m32.astype(np.float64), l32.astype(np.float64), a32.astype(np.float64),
                                 to_numpy(case.seq_lens), split)
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out, lse = td.td_lse_merge(torch.from_numpy(m32).cuda(), torch.from_numpy(l32).cuda(),
                               torch.from_numpy(a32).cuda(), case.seq_lens.cuda(), split, out_dtype=tdt,
                               return_lse=True)
    assert_out_close(out.cpu(), ref, out_dtype)
    assert_lse_close(lse.cpu(), ref_lse)


# ------------------------------------------------------------------------------ invariants

@pytest.mark.parametrize("split", [0, 32])
def test_poison_past_seq_len_is_never_read(td, split):
    case = small_case(dtype="bf16", B=3, Hq=24, Hkv=8, D=128, Smax=600, seq_lens=[333, 600, 17], seed=5)
    out, lse, _ = run_attention(td, case, split=split)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    for b, L in enumerate(case.seq_lens.tolist()):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    out2, lse2, _ = run_attention(td, case, split=split, k_cache=kc, v_cache=vc)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_batch_rows_independent(td):
    case = small_case(dtype="bf16", B=4, Hq=24, Hkv=8, D=128, Smax=500, seq_lens=[500, 2, 300, 77], seed=6)
    out, _, _ = run_attention(td, case, split=64)
    for b in range(4):
        sub = small_case(dtype="bf16", B=1, Hq=24, Hkv=8, D=128, Smax=500, seq_lens=[int(case.seq_lens[b])], seed=6)
        sub.q, sub.k_cache, sub.v_cache = case.q[b:b + 1], case.k_cache[b:b + 1], case.v_cache[b:b + 1]
        o, _, _ = run_attention(td, sub, split=64)
        assert torch.equal(out[b:b + 1], o), b


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_seq_len_one_returns_first_value_row(td, dtype):
    case = small_case(dtype=dtype, B=2, Hq=8, Hkv=2, D=128, Smax=50, seq_lens=[1, 1], seed=7)
    out, _, _ = run_attention(td, case)
    v0 = case.v_cache[:, :, 0].repeat_interleave(4, dim=1)
    assert torch.equal(out[:, :, 0], v0)


def test_empty_sequence(td):
    case = small_case(dtype="bf16", B=3, Hq=8, Hkv=2, D=128, Smax=50, seq_lens=[0, 9, 0], seed=8)
    out, lse, st = run_attention(td, case)
    assert st == 0
    assert out[0].abs().sum() == 0 and out[2].abs().sum() == 0
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all() and torch.isfinite(lse[1]).all()
    ref, ref_lse, _ = oracle_attention(case)
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, case_value_stats(case, ref_lse))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_largest_batch(td, dtype):
    """1024 sequences (the library's batch limit) of short mixed lengths, some empty: the
    device plan's per-sequence arrays at their size limit, a plan of several waves, and every
    row against the oracle."""
    B = 1024
    g = torch.Generator().manual_seed(11)
    lens = torch.randint(0, 101, (B,), generator=g)
    lens[::97] = 0
    case = small_case(dtype=dtype, B=B, Hq=4, Hkv=2, D=64, Smax=100, seq_lens=lens.tolist(), seed=12)
    check_case(td, case, split=0)


def test_all_empty_batch(td):
    case = small_case(dtype="f32", B=2, Hq=4, Hkv=2, D=64, Smax=32, seq_lens=[0, 0], seed=8)
    out, lse, _ = run_attention(td, case)
    assert out.abs().sum() == 0 and torch.isneginf(lse).all()


def test_lengths_out_of_range_are_clamped_and_flagged(td):
    case = small_case(dtype="bf16", B=2, Hq=8, Hkv=2, D=128, Smax=64, seq_lens=[90, -4], seed=10)
    out, lse, st = run_attention(td, case)
    assert st == td.DEV_SEQLEN_CLAMPED | td.DEV_NEGATIVE_SEQLEN
    ref, ref_lse, ref_st = oracle_attention(case)
    assert ref_st == st
    assert_out_close(out, ref, "bf16")
    assert_value_close(out, ref, case_value_stats(case, ref_lse))
    assert_lse_close(lse, ref_lse)


def test_repeat_calls_bit_identical_and_counters_rezeroed(td):
    case = small_case(dtype="bf16", B=2, Hq=24, Hkv=8, D=128, Smax=3000, seq_lens=[3000, 2500], seed=11)
    q, k, v, sl = case.q.cuda()[:, :, 0], case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    ws = td.make_workspace(2, 24, 8, 3000, 128, 1, 0)
    o1 = td.td_decode_attn(q, k, v, sl, case.scale, 0, workspace=ws)
    o2 = td.td_decode_attn(q, k, v, sl, case.scale, 0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    counters = ws[:2 * 2 * 8 * 4].view(torch.int32)  # tickets and finished-slice counts
    assert int(counters.abs().sum()) == 0


def test_graph_capture_and_replay(td):
    """append + decode captured once, replayed with new inputs written into the static buffers."""
    B, Hq, Hkv, D, S = 2, 24, 8, 128, 2048
    case = small_case(dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, D=D, Smax=S, seq_lens=[1000, 1500], seed=12)
    kc, vc = case.k_cache.cuda(), case.v_cache.cuda()
    sl = case.seq_lens.cuda()
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros(B, Hkv, 1, D, dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    out = torch.empty_like(q)
    ws = td.make_workspace(B, Hq, Hkv, S, D)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        td.td_kv_append(kn, vn, kc.clone(), vc.clone(), sl.clone(), advance=False, stream=stream)  # warm-up
        td.td_decode_attn(q, kc, vc, sl, case.scale, 0, out=out, workspace=ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        td.td_kv_append(kn, vn, kc, vc, sl, advance=True, stream=torch.cuda.current_stream())
        td.td_decode_attn(q, kc, vc, sl, case.scale, 0, out=out, workspace=ws, stream=torch.cuda.current_stream())
    gen = torch.Generator().manual_seed(0)
    ek, ev, es = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy(), to_numpy(case.seq_lens).copy()
    orc = oracle.load()
    for step in range(3):
        qh = torch.randn(B, Hq, D, generator=gen).to(torch.bfloat16)
        knh = torch.randn(B, Hkv, 1, D, generator=gen).to(torch.bfloat16)
        vnh = torch.randn(B, Hkv, 1, D, generator=gen).to(torch.bfloat16)
        q.copy_(qh)
        kn.copy_(knh)
        vn.copy_(vnh)
        g.replay()
        torch.cuda.synchronize()
        orc.kv_append(to_numpy(knh), to_numpy(vnh), ek, ev, es, advance=True)
        ref, ref_lse, _ = orc.attention(to_numpy(qh), ek, ev, es, case.scale)
        assert sl.cpu().numpy().tolist() == es.tolist()
        assert_out_close(out.cpu(), ref, "bf16", what=f"replay {step}")
        assert_value_close(out.cpu(), ref, value_stats(to_numpy(qh), ek, ev, es, case.scale, ref_lse),
                           what=f"replay {step}")


def test_binding_errors(td):
    from decode_attention_split_gb300._lib import TDError
    case = small_case(dtype="bf16", B=1, Hq=8, Hkv=2, D=128, Smax=64, seq_lens=[64], seed=13)
    q, k, v, sl = case.q.cuda()[:, :, 0], case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    with pytest.raises(TDError) as e:
        td.td_decode_attn(q, k, v, sl, case.scale, 0, workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3
    flat = torch.zeros(q.numel() + 1, dtype=torch.bfloat16, device="cuda")
    q_mis = flat[1:].view_as(q)
    with pytest.raises(TDError) as e:
        td.td_decode_attn(q_mis, k, v, sl, case.scale, 0)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        td.td_decode_attn(q.cpu(), k, v, sl)


def test_dirty_workspace_is_reported(td):
    """Counters that were not zeroed are detected and flagged instead of merging early."""
    case = small_case(dtype="bf16", B=1, Hq=8, Hkv=2, D=128, Smax=4096, seq_lens=[4096], seed=14)
    q, k, v, sl = case.q.cuda()[:, :, 0], case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    ws = td.make_workspace(1, 8, 2, 4096, 128)
    ws.fill_(0x7F)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    td.td_decode_attn(q, k, v, sl, case.scale, 64, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & td.DEV_WORKSPACE_DIRTY
