"""td_decode_attn_noalloc through the C ABI, against td_decode_attn.

The entry point serves callers that cannot allocate device memory (its scratch is a fixed
array inside the library). Two calls in a row, with different shapes, so the second call
runs on the scratch the first left behind; each must match the workspace entry point within
the bf16 tolerance. A shape beyond the array's size is refused on the host. This file is collected last so a run stopping at its first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from decode_attention_split_gb300.workloads import make_case
from parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kc, vc, sl, scale, out, lse, status):
    B, Hq, D = q.shape
    _, Hkv, Smax, _ = kc.shape
    st = lib.td_decode_attn_noalloc(1, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), B, Hq, Hkv, Smax,
                                    D, ctypes.c_float(scale), 0, out.data_ptr(), lse.data_ptr(), status.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import _lib, build
    build.build()
    import decode_attention_split_gb300 as td
    lib = _lib.lib()
    for name, L in (("llama3b", 4096), ("smollm2_360m", 4096)):
        case = make_case(name, seq_len=L)
        q = case.q[:, :, 0].contiguous().cuda()
        kc, vc, sl = case.k_cache.cuda(), case.v_cache.cuda(), case.seq_lens.cuda()
        ref, ref_lse = td.td_decode_attn(q, kc, vc, sl, case.scale, 0, return_lse=True)
        out = torch.full_like(q, float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, q, kc, vc, sl, case.scale, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_out_close(out.cpu(), ref.double().cpu().numpy(), "bf16", what=f"{name} out")
        assert_lse_close(lse.cpu(), ref_lse.double().cpu().numpy(), what=f"{name} lse")


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
    assert _noalloc(lib, q, kc, kc, sl, 0.1, out, lse, status) == 3  # TD_ERR_WORKSPACE
