"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every td kernel waits for its asynchronous copies with a bounded wait that, when it gives
up, sets TD_DEV_WAIT_TIMEOUT in the caller's status word and lets the kernel return instead
of hanging. td_selftest_wait_timeout runs that wait routine on an mbarrier that nothing ever
arrives on (no copy is issued against it, so nothing is in flight): the wait must give up
after its limit, the bit must be set, and the context must stay usable for the next call.
"""
import ctypes

import pytest
import torch

from decode_attention_split_gb300.workloads import small_case, to_numpy
from parity import check_bf16_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def td():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td
    return td


@pytest.mark.parametrize("limit", [1000, 2_000_000])
def test_bounded_wait_gives_up_and_reports(td, limit):
    from decode_attention_split_gb300 import _lib
    lib = _lib.lib()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = lib.td_selftest_wait_timeout(ctypes.c_longlong(limit), status.data_ptr(), waited.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(status.item()) == td.DEV_WAIT_TIMEOUT
    assert limit < int(waited.item()) < limit + 1_000_000  # gave up just after its limit
    # the context is still usable: an attention call right after it runs and is correct
    case = small_case(dtype="bf16", B=1, Hq=24, Hkv=8, D=128, Smax=2048, seq_lens=[2000], seed=2, heavy=0.01)
    dev_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = td.td_decode_attn(case.q.cuda()[:, :, 0], case.k_cache.cuda(), case.v_cache.cuda(),
                                 case.seq_lens.cuda(), case.scale, 0, return_lse=True, dev_status=dev_status)
    torch.cuda.synchronize()
    assert int(dev_status.item()) == 0
    check_bf16_attention(out.cpu(), lse.cpu(), to_numpy(case.q[:, :, 0]), to_numpy(case.k_cache),
                         to_numpy(case.v_cache), to_numpy(case.seq_lens), case.scale)
