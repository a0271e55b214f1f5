"""td_decode_attn_noalloc through the C ABI, against the oracle and against td_decode_attn.

The entry point serves callers that cannot allocate device memory: a plugin or launch hook
that is handed only its input and output pointers, or a serving loop that must not allocate
once it runs. Its scratch is a fixed array inside the library. Four calls in a row on that one
array, with different shapes, element types and split sizes (a bf16 3B-style layer, the
fp32 config with its named split 64, the bf16 360M layer, the 3B-style layer with an explicit
split), so every call after the first runs on scratch an earlier call left behind. Each must
match the oracle (the stated tolerance and, for bf16, the value-side bound) and the workspace
entry point on the same inputs. A ragged batch of four then runs on the cluster kernel's plan
on the same array. A shape beyond the array's size is refused on the host. This
file is collected last so a run stopping at its first failure has already run every other
test.
"""
import ctypes

import pytest
import torch

from decode_attention_split_gb300.workloads import make_case, to_numpy
from parity import assert_lse_close, assert_out_close, check_bf16_attention, oracle_attention

pytestmark = pytest.mark.gpu

_DTYPE = {torch.float32: 0, torch.bfloat16: 1}


def _noalloc(lib, q, kc, vc, sl, scale, split, out, lse, status):
    B, Hq, D = q.shape
    _, Hkv, Smax, _ = kc.shape
    return lib.td_decode_attn_noalloc(_DTYPE[q.dtype], q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), B,
                                      Hq, Hkv, Smax, D, ctypes.c_float(scale), split, out.data_ptr(), lse.data_ptr(),
                                      status.data_ptr(), torch.cuda.current_stream().cuda_stream)


CALLS = [("llama3b", 4096, 0), ("tiny_fp32", 128, 64), ("smollm2_360m", 4096, 0), ("llama3b", 16384, 512)]


def test_noalloc_matches_oracle_and_workspace_entry_point_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import _lib, build
    build.build()
    import decode_attention_split_gb300 as td
    lib = _lib.lib()
    for name, L, split in CALLS:
        case = make_case(name, seq_len=L)
        dt = case.w.dtype
        q = case.q[:, :, 0].contiguous().cuda()
        kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, q, kc, vc, sl, case.scale, split, out, lse, status) == 0, name
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        what = f"{name} L={L} split={split}"
        if dt == "bf16":
            check_bf16_attention(out.cpu(), lse.cpu(), to_numpy(case.q[:, :, 0]), to_numpy(case.k_cache),
                                 to_numpy(case.v_cache), to_numpy(case.seq_lens), case.scale, what=what)
        else:
            ref, ref_lse, _ = oracle_attention(case)
            assert_out_close(out.cpu()[:, :, None], ref, dt, what=what)
            assert_lse_close(lse.cpu()[:, :, None], ref_lse, what=f"{what} lse")
        ws_out, ws_lse = td.td_decode_attn(q, kc, vc, sl, case.scale, split, return_lse=True)
        torch.cuda.synchronize()
        assert_out_close(out.cpu(), ws_out.double().cpu().numpy(), dt, what=f"{what} vs workspace call")
        assert_lse_close(lse.cpu(), ws_lse.double().cpu().numpy(), what=f"{what} lse vs workspace call")


def test_noalloc_batch_on_the_cluster_kernel():
    """A ragged batch of four on the same array: the cluster kernel's plan (no partials in the
    scratch, only its counter area), against the oracle and the workspace entry point."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import _lib, build
    build.build()
    import decode_attention_split_gb300 as td
    from decode_attention_split_gb300.workloads import small_case
    lib = _lib.lib()
    lens = [2048, 1000, 77, 1900]
    assert td.td_split_plan(torch.bfloat16, 4, 24, 8, 2048, 128, 1, 0)["kernel"] == "tensor_core_cluster"
    case = small_case(dtype="bf16", B=4, Hq=24, Hkv=8, D=128, Smax=2048, seq_lens=lens, seed=31, heavy=0.01)
    q = case.q[:, :, 0].contiguous().cuda()
    kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, q, kc, vc, sl, case.scale, 0, out, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_bf16_attention(out.cpu(), lse.cpu(), to_numpy(case.q[:, :, 0]), to_numpy(case.k_cache),
                         to_numpy(case.v_cache), to_numpy(case.seq_lens), case.scale, what="cluster batch")
    ws_out, ws_lse = td.td_decode_attn(q, kc, vc, sl, case.scale, 0, return_lse=True)
    torch.cuda.synchronize()
    assert_out_close(out.cpu(), ws_out.double().cpu().numpy(), "bf16", what="cluster batch vs workspace call")
    assert_lse_close(lse.cpu(), ws_lse.double().cpu().numpy(), what="cluster batch lse vs workspace call")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A batch of 16 sequences of 8192 rows needs more than the 4 MiB array: refused before launch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import _lib, build
    build.build()
    import decode_attention_split_gb300 as td
    lib = _lib.lib()
    assert td.td_decode_workspace_bytes(16, 32, 8, 8192, 128) > 4 << 20
    q = torch.zeros(16, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(16, 8, 8192, 128, dtype=torch.bfloat16, device="cuda")
    sl = torch.full((16,), 8192, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(16, 32, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, q, kc, kc, sl, 0.1, 0, out, lse, status) == 3  # TD_ERR_WORKSPACE
