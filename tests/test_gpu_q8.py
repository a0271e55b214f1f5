"""The 8-bit KV cache on the GPU against the CPU oracle.

Codes and scales are integer-valued decisions made in fp32 on both sides: bit-exact.
Attention over the codes must match the oracle's exact attention over code * scale within
the bf16 tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_split_gb300.workloads import make_case, small_case, to_numpy
from parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def td():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td
    return td


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 48)])
def test_quantize_bit_exact(td, dtype, D):
    g = torch.Generator().manual_seed(D)
    x = torch.randn(300, D, generator=g) * torch.rand(300, 1, generator=g) * 10
    x[0] = 0.0                                   # zero row
    x[1, :8] = torch.tensor([127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.5, -126.5])  # scale 1: ties
    x[1, 8:] = 0.0
    x = x.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    codes, scales = td.td_quantize_q8(x.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.load().quantize_q8(to_numpy(x))
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_append_q8_bit_exact(td):
    B, H, T, S, D = 4, 3, 2, 40, 128
    g = torch.Generator().manual_seed(5)
    kc = torch.randint(-127, 128, (B, H, S, D), generator=g, dtype=torch.int8)
    vc = torch.randint(-127, 128, (B, H, S, D), generator=g, dtype=torch.int8)
    ks = torch.rand(B, H, S, generator=g)
    vs = torch.rand(B, H, S, generator=g)
    kn = torch.randn(B, H, T, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, H, T, D, generator=g).to(torch.bfloat16)
    seq = torch.tensor([0, 17, S - T, S - T + 1], dtype=torch.int32)
    d = [t.cuda() for t in (kc, ks, vc, vs, seq)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    td.td_kv_append_q8(kn.cuda(), vn.cuda(), d[0], d[1], d[2], d[3], d[4], advance=True, dev_status=st)
    torch.cuda.synchronize()
    orc = oracle.load()
    qk, sk = orc.quantize_q8(to_numpy(kn))
    qv, sv = orc.quantize_q8(to_numpy(vn))
    ek, eks, ev, evs = kc.numpy().copy(), ks.numpy().copy(), vc.numpy().copy(), vs.numpy().copy()
    for b, L in enumerate(seq.tolist()):
        if L + T <= S:
            ek[b, :, L:L + T], eks[b, :, L:L + T] = qk[b], sk[b]
            ev[b, :, L:L + T], evs[b, :, L:L + T] = qv[b], sv[b]
    assert int(st.item()) == td.DEV_APPEND_OVERFLOW
    assert d[4].cpu().tolist() == [T, 17 + T, S, S - T + 1]
    assert np.array_equal(d[0].cpu().numpy(), ek) and np.array_equal(d[2].cpu().numpy(), ev)
    assert np.array_equal(d[1].cpu().numpy(), eks) and np.array_equal(d[3].cpu().numpy(), evs)


def _q8_case(case):
    orc = oracle.load()
    kc, ks = orc.quantize_q8(to_numpy(case.k_cache))
    vc, vs = orc.quantize_q8(to_numpy(case.v_cache))
    return kc, ks, vc, vs


def _run_q8(td, case, kc, ks, vc, vs, split=0):
    q = case.q.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = [torch.from_numpy(a).cuda() for a in (kc, ks, vc, vs)]
    if case.q.shape[2] == 1:
        out, lse = td.td_decode_attn_q8(q[:, :, 0], *args, case.seq_lens.cuda(), case.scale, split, return_lse=True,
                                        dev_status=st)
        out = out[:, :, None]
    else:
        out, lse = td.td_verify_attn_q8(q, *args, case.seq_lens.cuda(), case.scale, split, return_lse=True,
                                        dev_status=st)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu().reshape(case.q.shape[:3]), int(st.item())


Q8 = [
    # D, Hq, Hkv, Smax, T, lengths, split
    (128, 24, 8, 520, 1, [520, 100], 0),
    (128, 24, 8, 520, 1, [519, 16], 64),
    (64, 15, 5, 300, 1, [300, 64, 1], 0),
    (128, 32, 4, 260, 1, [260, 5], 0),          # two row blocks per kv head
    (128, 32, 8, 200, 6, [200, 70], 0),         # verify
    (64, 8, 1, 400, 1, [400, 399, 31, 2], 37),
    (128, 24, 8, 4096, 1, [4096, 1500, 0], 0),  # several chunks, an empty sequence
    (128, 16, 2, 700, 1, [700, 129], 0),        # 8 rows per kv head: the narrow tile's limit
    (64, 18, 2, 700, 1, [650, 64], 0),          # 9 rows: one 16-row m tile
    (128, 4, 2, 300, 4, [300, 70], 0),          # verify, 8 rows, each with its own causal limit
    # 40 sequences of mixed lengths (one empty): past 1/16 of the slots, the late plan and the full grid
    (128, 24, 8, 600, 1, [(37 * i) % 601 for i in range(40)], 0),
]


@pytest.mark.parametrize("D,Hq,Hkv,Smax,T,lens,split", Q8)
def test_q8_attention_against_oracle(td, D, Hq, Hkv, Smax, T, lens, split):
    case = small_case(dtype="bf16", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, Smax=Smax, T=T, seq_lens=lens,
                      seed=D + Smax + T, heavy=0.02)
    kc, ks, vc, vs = _q8_case(case)
    out, lse, st = _run_q8(td, case, kc, ks, vc, vs, split)
    ref, ref_lse, ref_st = oracle.load().attention_q8(to_numpy(case.q), kc, ks, vc, vs, case.seq_lens.numpy(),
                                                      case.scale)
    assert st == ref_st
    assert_out_close(out, ref, "bf16")
    assert_lse_close(lse, ref_lse)


def test_q8_full_size_3b_layer_32k(td):
    """The 3B-style layer at 32k, the cache quantised on the GPU (bit-exact with the oracle's codes)."""
    case = make_case("llama3b", seq_len=32768)
    k_codes, k_scales = td.td_quantize_q8(case.k_cache.cuda())
    v_codes, v_scales = td.td_quantize_q8(case.v_cache.cuda())
    torch.cuda.synchronize()
    kc, ks, vc, vs = _q8_case(case)
    assert np.array_equal(k_codes.cpu().numpy(), kc) and np.array_equal(v_scales.cpu().numpy(), vs)
    out = td.td_decode_attn_q8(case.q.cuda()[:, :, 0], k_codes, k_scales, v_codes, v_scales, case.seq_lens.cuda(),
                               case.scale)
    torch.cuda.synchronize()
    ref, _, _ = oracle.load().attention_q8(to_numpy(case.q), kc, ks, vc, vs, case.seq_lens.numpy(), case.scale)
    assert_out_close(out.cpu()[:, :, None], ref, "bf16")


def test_q8_rejects_unaligned_smax(td):
    from decode_attention_split_gb300._lib import TDError
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros(1, 2, 30, 128, dtype=torch.int8, device="cuda")
    scales = torch.zeros(1, 2, 32, dtype=torch.float32, device="cuda")[:, :, :30].contiguous()
    with pytest.raises(TDError) as e:
        td.td_decode_attn_q8(q, codes, scales, codes, scales, torch.tensor([30], dtype=torch.int32, device="cuda"))
    assert e.value.status == 2


@pytest.mark.parametrize("T,split", [(1, 0), (1, 100), (5, 0)])
def test_q8_stale_rows_past_the_length_are_never_used(td, T, split):
    """Codes and scales past a sequence's length (stale rows) leave the result unchanged, even
    non-finite scales: a masked key's zero probability never meets its value scale."""
    case = small_case(dtype="bf16", B=2, Hq=24, Hkv=8, D=128, Smax=1024, T=T, seq_lens=[700, 333], seed=11 + T)
    kc, ks, vc, vs = _q8_case(case)
    ref = _run_q8(td, case, kc, ks, vc, vs, split)
    ks2, vs2, vc2 = ks.copy(), vs.copy(), vc.copy()
    for b, L in enumerate(case.seq_lens.tolist()):
        ks2[b, :, L:] = np.nan
        vs2[b, :, L:] = np.inf
        vc2[b, :, L:] = 127
    out, lse, st = _run_q8(td, case, kc, ks2, vc2, vs2, split)
    assert st == ref[2]
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
