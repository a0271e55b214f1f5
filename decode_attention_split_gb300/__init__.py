"""GB300-native split-KV decode attention over a static KV cache.

The computation runs in the CUDA library ``_build/libtd.so`` (hand-written sm_103a kernels
behind the C ABI in ``include/td.h``); this package is its Python binding with the same
function names. Build the library with ``python -m decode_attention_split_gb300.build``.
Importing the package does not load the library; the first call does, and raises if it is
missing.
"""
from .api import (  # noqa: F401
    DEV_APPEND_OVERFLOW,
    DEV_BAD_TOKEN,
    DEV_NEGATIVE_SEQLEN,
    DEV_SEQLEN_CLAMPED,
    DEV_VERIFY_SHORT,
    DEV_WAIT_TIMEOUT,
    DEV_WORKSPACE_DIRTY,
    make_workspace,
    td_decode_attn,
    td_decode_attn_q8,
    td_decode_workspace_bytes,
    td_kv_append,
    td_kv_append_q8,
    td_lse_merge,
    td_prefill_attn,
    td_rope_append_attn,
    td_rope_kv_append,
    td_quantize_q8,
    td_spec_accept,
    td_split_plan,
    td_verify_attn,
    td_verify_attn_q8,
)
