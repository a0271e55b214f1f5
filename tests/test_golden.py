"""Byte accounting pinned to the figures the llm-decode-cuda page prints for its 360M model."""
import json
import os

from decode_attention_split_gb300.workloads import WORKLOADS, kv_bytes_per_token, kv_read_bytes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "smollm2_360m_kv_bytes.json")


def test_kv_bytes_per_token_matches_page():
    g = json.load(open(GOLDEN))
    per_layer = kv_bytes_per_token(g["kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per_layer * g["layers"] == g["kv_kib_per_token_all_layers"] * 1024


def test_roofline_at_4k_matches_page():
    g = json.load(open(GOLDEN))
    per_token = kv_bytes_per_token(g["kv_heads"], g["head_dim"], g["elem_bytes"]) * g["layers"]
    tok_s = g["read_bandwidth_gbs"] * 1e9 / (g["weight_bytes_per_token"] + g["context"] * per_token)
    assert round(tok_s) == g["roofline_tokens_per_s"]


def test_workload_byte_counts():
    # the 360M-layer workload is one layer of that model: 1280 B per token of context
    w = WORKLOADS["smollm2_360m"]
    assert kv_read_bytes(w, 4096) == 4096 * 1280
    w3 = WORKLOADS["llama3b"]
    assert kv_read_bytes(w3, 32768) == 134217728
    w5 = WORKLOADS["verify6"]
    assert kv_read_bytes(w5, 16390) == 67133440
