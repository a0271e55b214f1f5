"""The C-ABI library without a GPU: it builds, loads, exports what include/td.h declares,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from decode_attention_split_gb300 import build as td_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "td.h")

TD_OK, TD_ERR_INVALID_ARG, TD_ERR_UNSUPPORTED, TD_ERR_WORKSPACE, TD_ERR_CUDA = range(5)


@pytest.fixture(scope="module")
def lib():
    path = td_build.build()
    from decode_attention_split_gb300 import _lib
    assert os.path.samefile(path, _lib.LIB_PATH)
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(td_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("td_kv_append", "td_decode_attn", "td_verify_attn", "td_lse_merge", "td_decode_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from decode_attention_split_gb300 import _lib
    names = declared_functions()
    assert sorted(_lib.SYMBOLS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_no_cuda_runtime_symbols_leak(lib):
    # the static CUDA runtime stays private to the library
    raw = ctypes.CDLL(lib._name)
    with pytest.raises(AttributeError):
        raw.cudaMalloc  # noqa: B018


def test_status_strings(lib):
    assert lib.td_status_string(TD_OK) == b"ok"
    assert b"workspace" in lib.td_status_string(TD_ERR_WORKSPACE)
    assert lib.td_version().startswith(b"td ")


FAKE = 0x10000  # a 16-byte aligned address the host never dereferences


def _decode(lib, **kw):
    a = dict(dtype=1, q=FAKE, k=FAKE, v=FAKE, sl=FAKE, B=1, Hq=4, Hkv=2, Smax=64, D=128, scale=0.1, split=0,
             out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    return lib.td_decode_attn(a["dtype"], a["q"], a["k"], a["v"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["Smax"],
                              a["D"], a["scale"], a["split"], a["out"], a["lse"], a["ws"], a["wsb"], a["st"],
                              a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), TD_ERR_INVALID_ARG),
    (dict(out=None), TD_ERR_INVALID_ARG),
    (dict(sl=None), TD_ERR_INVALID_ARG),
    (dict(Hq=5, Hkv=2), TD_ERR_INVALID_ARG),
    (dict(B=0), TD_ERR_INVALID_ARG),
    (dict(split=-1), TD_ERR_INVALID_ARG),
    (dict(scale=float("nan")), TD_ERR_INVALID_ARG),
    (dict(D=96), TD_ERR_UNSUPPORTED),
    (dict(dtype=7), TD_ERR_UNSUPPORTED),
    (dict(B=1025), TD_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, expect):
    assert _decode(lib, **kw) == expect


def test_verify_rejects_chunk_longer_than_cache(lib):
    st = lib.td_verify_attn(1, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 65, 64, 128, 0.1, 0, FAKE, None, FAKE, 1 << 20, None,
                            None)
    assert st == TD_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,expect", [
    (dict(k_new=None), TD_ERR_INVALID_ARG),
    (dict(T=0), TD_ERR_INVALID_ARG),
    (dict(D=4), TD_ERR_UNSUPPORTED),             # a bf16 row of 8 bytes is not a whole 16-byte vector
    (dict(k_cache=FAKE + 8), TD_ERR_UNSUPPORTED),  # misaligned
    (dict(dtype=3), TD_ERR_UNSUPPORTED),
])
def test_append_rejects_bad_arguments_on_host(lib, kw, expect):
    a = dict(dtype=1, k_new=FAKE, v_new=FAKE, k_cache=FAKE, v_cache=FAKE, sl=FAKE, B=2, Hkv=2, T=1, Smax=16, D=64)
    a.update(kw)
    st = lib.td_kv_append(a["dtype"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["sl"], a["B"],
                          a["Hkv"], a["T"], a["Smax"], a["D"], 1, None, None)
    assert st == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(m=None), TD_ERR_INVALID_ARG),
    (dict(split=0), TD_ERR_INVALID_ARG),
    (dict(D=6), TD_ERR_UNSUPPORTED),
    (dict(D=2048), TD_ERR_UNSUPPORTED),
    (dict(out_dtype=5), TD_ERR_UNSUPPORTED),
])
def test_merge_rejects_bad_arguments_on_host(lib, kw, expect):
    a = dict(m=FAKE, l=FAKE, acc=FAKE, sl=FAKE, B=1, rows=4, NS=3, D=64, split=16, out_dtype=0, out=FAKE)
    a.update(kw)
    st = lib.td_lse_merge(a["m"], a["l"], a["acc"], a["sl"], a["B"], a["rows"], a["NS"], a["D"], a["split"],
                          a["out_dtype"], a["out"], None, None)
    assert st == expect


def test_hot_kernels_have_no_spills(lib):
    """Register gate (ptxas): the instantiations the workloads run keep every value in registers."""
    log = open(td_build.PTXAS_LOG).read()
    entries = re.findall(r"Compiling entry function '(\w+)'.*?\n(?:.*?\n)*?\s+(\d+) bytes stack frame, (\d+) bytes "
                         r"spill stores, (\d+) bytes spill loads", log)
    hot = {"split_attn_mma_kernelILi128ELb1ELi1E", "split_attn_mma_kernelILi128ELb1ELi0E",
           "split_attn_mma_kernelILi128ELb0ELi2E", "split_attn_mma_kernelILi128ELb0ELi0E",
           "split_attn_mma_kernelILi64ELb1ELi1E", "split_attn_mma_kernelILi64ELb1ELi0E",
           "split_attn_mma_kernelILi64ELb0ELi0E", "split_attn_kernelIfLi64ELi2E",
           "split_attn_cluster_kernelILi128ELi0E", "split_attn_cluster_kernelILi128ELi1E",
           "split_attn_cluster_kernelILi128ELi2E", "split_attn_q8_kernelILi128ELb0ELb0E",
           "split_attn_q8_kernelILi128ELb1ELb0E", "split_attn_q8_kernelILi128ELb1ELb1E",
           "prefill_kernelILi128E"}
    seen = set()
    for name, _stack, st, ld in entries:
        for h in hot:
            if h in name:
                seen.add(h)
                assert int(st) == 0 and int(ld) == 0, (name, st, ld)
    assert seen == hot


# ------------------------------------------------------------- the later calls' host checks

NAN = float("nan")


def _call(fn, order, defaults, kw):
    a = dict(defaults)
    a.update(kw)
    return fn(*[a[k] for k in order])


ROPE_APPEND = ("dtype", "q", "q_out", "Hq", "k_new", "v_new", "cos", "sin", "kc", "vc", "sl", "B", "Hkv", "T", "Smax",
               "D", "adv", "st", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=3), TD_ERR_UNSUPPORTED),
    (dict(k_new=None), TD_ERR_INVALID_ARG),
    (dict(q=FAKE), TD_ERR_INVALID_ARG),            # q without q_out
    (dict(q=FAKE, q_out=FAKE, Hq=0), TD_ERR_INVALID_ARG),
    (dict(T=0), TD_ERR_INVALID_ARG),
    (dict(D=8), TD_ERR_UNSUPPORTED),               # a bf16 row of 16 bytes is not two 16-byte halves
    (dict(cos=FAKE + 4), TD_ERR_UNSUPPORTED),      # misaligned table
])
def test_rope_append_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(dtype=1, q=None, q_out=None, Hq=0, k_new=FAKE, v_new=FAKE, cos=FAKE, sin=FAKE, kc=FAKE, vc=FAKE, sl=FAKE,
             B=1, Hkv=2, T=1, Smax=16, D=64, adv=1, st=None, stream=None)
    assert _call(lib.td_rope_kv_append, ROPE_APPEND, d, kw) == expect


FUSED = ("dtype", "q", "k_new", "v_new", "cos", "sin", "kc", "vc", "sl", "B", "Hq", "Hkv", "T", "Smax", "D", "scale",
         "split", "adv", "out", "lse", "ws", "wsb", "st", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(k_new=None), TD_ERR_INVALID_ARG),
    (dict(cos=FAKE), TD_ERR_INVALID_ARG),          # a cosine table without the sine table
    (dict(dtype=0), TD_ERR_UNSUPPORTED),           # the fused step is bf16 only
    (dict(k_new=FAKE + 8), TD_ERR_UNSUPPORTED),
    (dict(q=None), TD_ERR_INVALID_ARG),
    (dict(D=96), TD_ERR_UNSUPPORTED),
    (dict(scale=NAN), TD_ERR_INVALID_ARG),
    (dict(Hq=5), TD_ERR_INVALID_ARG),
])
def test_fused_step_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(dtype=1, q=FAKE, k_new=FAKE, v_new=FAKE, cos=None, sin=None, kc=FAKE, vc=FAKE, sl=FAKE, B=1, Hq=4, Hkv=2,
             T=1, Smax=64, D=128, scale=0.1, split=0, adv=1, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, st=None,
             stream=None)
    assert _call(lib.td_rope_append_attn, FUSED, d, kw) == expect


SPEC = ("target", "draft", "tokens", "u", "B", "G", "V", "temp", "n_acc", "next", "ws", "wsb", "st", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(target=None), TD_ERR_INVALID_ARG),
    (dict(u=None), TD_ERR_INVALID_ARG),            # sampling needs the uniforms
    (dict(draft=None), TD_ERR_INVALID_ARG),        # and the draft rows
    (dict(temp=-1.0), TD_ERR_INVALID_ARG),
    (dict(temp=NAN), TD_ERR_INVALID_ARG),
    (dict(G=17), TD_ERR_UNSUPPORTED),
    (dict(n_acc=FAKE + 2), TD_ERR_UNSUPPORTED),
    (dict(target=FAKE + 4), TD_ERR_UNSUPPORTED),   # V % 4 == 0: rows are read 16 bytes at a time
    (dict(wsb=16), TD_ERR_WORKSPACE),
    (dict(temp=0.0, draft=None, u=None, wsb=16), TD_ERR_WORKSPACE),  # greedy needs neither
])
def test_spec_accept_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(target=FAKE, draft=FAKE, tokens=FAKE, u=FAKE, B=1, G=4, V=1000, temp=1.0, n_acc=FAKE, next=FAKE, ws=FAKE,
             wsb=1 << 26, st=None, stream=None)
    assert _call(lib.td_spec_accept, SPEC, d, kw) == expect


def test_spec_workspace_bytes(lib):
    assert lib.td_spec_workspace_bytes(1, 17, 1000) == 0
    assert lib.td_spec_workspace_bytes(0, 4, 1000) == 0
    n1, n8 = lib.td_spec_workspace_bytes(1, 4, 128256), lib.td_spec_workspace_bytes(8, 4, 128256)
    assert 0 < n1 < n8 and n1 % 256 == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=3), TD_ERR_UNSUPPORTED),
    (dict(x=None), TD_ERR_INVALID_ARG),
    (dict(rows=0), TD_ERR_INVALID_ARG),
    (dict(scales=FAKE + 2), TD_ERR_UNSUPPORTED),
])
def test_quantize_q8_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(dtype=1, x=FAKE, rows=4, D=128, codes=FAKE, scales=FAKE, stream=None)
    assert _call(lib.td_quantize_q8, ("dtype", "x", "rows", "D", "codes", "scales", "stream"), d, kw) == expect


APPEND_Q8 = ("dtype", "k_new", "v_new", "kc", "ks", "vc", "vs", "sl", "B", "Hkv", "T", "Smax", "D", "adv", "st",
             "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=3), TD_ERR_UNSUPPORTED),
    (dict(k_new=None), TD_ERR_INVALID_ARG),
    (dict(vs=None), TD_ERR_INVALID_ARG),
    (dict(T=0), TD_ERR_INVALID_ARG),
    (dict(ks=FAKE + 2), TD_ERR_UNSUPPORTED),
    (dict(B=65536), TD_ERR_UNSUPPORTED),
])
def test_append_q8_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(dtype=1, k_new=FAKE, v_new=FAKE, kc=FAKE, ks=FAKE, vc=FAKE, vs=FAKE, sl=FAKE, B=2, Hkv=2, T=1, Smax=16,
             D=64, adv=1, st=None, stream=None)
    assert _call(lib.td_kv_append_q8, APPEND_Q8, d, kw) == expect


VERIFY_Q8 = ("q", "kc", "ks", "vc", "vs", "sl", "B", "Hq", "Hkv", "T", "Smax", "D", "scale", "split", "out", "lse",
             "ws", "wsb", "st", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(ks=None), TD_ERR_INVALID_ARG),
    (dict(Smax=66), TD_ERR_UNSUPPORTED),           # scale rows step by whole 16-byte units
    (dict(vs=FAKE + 4), TD_ERR_UNSUPPORTED),
    (dict(q=None), TD_ERR_INVALID_ARG),
    (dict(D=96), TD_ERR_UNSUPPORTED),
    (dict(Hq=5), TD_ERR_INVALID_ARG),
    (dict(T=65), TD_ERR_UNSUPPORTED),              # a chunk longer than the cache
    (dict(scale=NAN), TD_ERR_INVALID_ARG),
])
def test_q8_attention_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(q=FAKE, kc=FAKE, ks=FAKE, vc=FAKE, vs=FAKE, sl=FAKE, B=1, Hq=4, Hkv=2, T=1, Smax=64, D=128, scale=0.1,
             split=0, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, st=None, stream=None)
    assert _call(lib.td_verify_attn_q8, VERIFY_Q8, d, kw) == expect
    if "T" not in kw:  # the decode entry point is the verify call with T = 1
        order = tuple(k for k in VERIFY_Q8 if k != "T")
        assert _call(lib.td_decode_attn_q8, order, d, kw) == expect


PREFILL = ("q", "kc", "vc", "sl", "B", "Hq", "Hkv", "T", "Smax", "D", "scale", "out", "lse", "st", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), TD_ERR_INVALID_ARG),
    (dict(Hq=5), TD_ERR_INVALID_ARG),
    (dict(T=0), TD_ERR_INVALID_ARG),
    (dict(scale=NAN), TD_ERR_INVALID_ARG),
    (dict(D=96), TD_ERR_UNSUPPORTED),
    (dict(T=65), TD_ERR_UNSUPPORTED),              # longer than the cache
    (dict(out=FAKE + 8), TD_ERR_UNSUPPORTED),
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(q=FAKE, kc=FAKE, vc=FAKE, sl=FAKE, B=1, Hq=4, Hkv=2, T=64, Smax=64, D=128, scale=0.1, out=FAKE,
             lse=None, st=None, stream=None)
    assert _call(lib.td_prefill_attn, PREFILL, d, kw) == expect


NOALLOC = ("dtype", "q", "kc", "vc", "sl", "B", "Hq", "Hkv", "Smax", "D", "scale", "split", "out", "lse", "st",
           "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), TD_ERR_INVALID_ARG),
    (dict(scale=NAN), TD_ERR_INVALID_ARG),
    (dict(D=96), TD_ERR_UNSUPPORTED),
    (dict(dtype=7), TD_ERR_UNSUPPORTED),
    (dict(Hq=5), TD_ERR_INVALID_ARG),
])
def test_noalloc_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(dtype=1, q=FAKE, kc=FAKE, vc=FAKE, sl=FAKE, B=1, Hq=4, Hkv=2, Smax=64, D=128, scale=0.1, split=0,
             out=FAKE, lse=None, st=None, stream=None)
    assert _call(lib.td_decode_attn_noalloc, NOALLOC, d, kw) == expect


SELFTEST = ("limit", "st", "waited", "stream")


@pytest.mark.parametrize("kw,expect", [
    (dict(limit=0), TD_ERR_INVALID_ARG),
    (dict(limit=-5), TD_ERR_INVALID_ARG),
    (dict(limit=2_000_000_000), TD_ERR_INVALID_ARG),   # past the half-second cap
    (dict(st=None), TD_ERR_INVALID_ARG),
    (dict(st=FAKE + 2), TD_ERR_UNSUPPORTED),
    (dict(waited=FAKE + 4), TD_ERR_UNSUPPORTED),
])
def test_wait_timeout_diagnostic_rejects_bad_arguments_on_host(lib, kw, expect):
    d = dict(limit=1000, st=FAKE, waited=None, stream=None)
    assert _call(lib.td_selftest_wait_timeout, SELFTEST, d, kw) == expect
