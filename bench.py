#!/usr/bin/env python
"""Benchmark: split-KV decode attention on one GB300, one JSON line on stdout.

Workload (one layer of a 3B Llama-style model): B=1, Hq=24, Hkv=8, D=128, bf16 KV cache
of Smax=32768 rows, attended length 32768, automatic split. One *call* is the hot path
for one decode token: write the new key/value row into the cache and attend, in one launch
(td_rope_append_attn without rotation tables; the same result as td_kv_append followed by
td_decode_attn, whose timing is reported beside it). One *step* is a batch of R such calls,
each on its own query and new row, rotating over C copies of the cache so that every
call's 134 MB of KV reads come from HBM (C * 134 MB > 4x L2), captured once as a CUDA graph
and replayed.

  value      KV-read GB/s = KV bytes attended / device time, inputs resident in HBM
  e2e        the same through the Python API with host buffers: every call copies its q
             and new rows from pinned host memory and reads its output back
  roofline   the attention kernel timed alone (graph of R attention launches), against the
             measured HBM copy bandwidth
  cpu_baseline  the CPU oracle (fp64, all host cores) on a bounded sample of the workload
  sweep      the other workloads' points (us/call, GB/s), attention kernel only

``--impl reference`` times the CPU oracle as the reference arm instead.
Under torchrun every rank runs the same workload on its own GPU (replicas; no collective
on the data path) and rank 0 prints value = all ranks' bytes / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_split_gb300.workloads import WORKLOADS, kv_read_bytes, make_case, to_numpy  # noqa: E402

METRIC = "decode-attn achieved KV-read GB/s (% of HBM peak) and µs/call, B=1 at 4k–32k ctx"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="td", choices=["td", "reference"])
    ap.add_argument("--calls-per-step", type=int, default=1000)
    ap.add_argument("--workload", default="llama3b")
    ap.add_argument("--seq-len", type=int, default=32768)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="profiling mode: W warm-up calls then this many plain launches, no graphs, no JSON extras")
    ap.add_argument("--profile-row", default=None, choices=["q8", "prefill", "verify6", "ragged8"],
                    help="profiling mode for another kernel instead of the timed step's call: q8 = "
                         "td_decode_attn_q8 on the 3B-style layer at --seq-len with --profile-batch sequences "
                         "(cache quantised on the GPU); prefill = td_prefill_attn on a --seq-len-token prompt; "
                         "verify6 / ragged8 = td_verify_attn / td_decode_attn on those workloads, the launches "
                         "rotating over cache copies that together exceed 4 x L2")
    ap.add_argument("--profile-batch", type=int, default=4)
    return ap.parse_args()


# ------------------------------------------------------------------------------ environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without its comments and blank lines (what the compiler sees)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash() -> str:
    """Hash of the code the timed decode kernel is built from: the translation units that
    define and launch it (td_split_attn.cu, td_api.cu) with every header they include,
    transitively, and td.h, comments and blank lines left out."""
    src = os.path.join(ROOT, "decode_attention_split_gb300", "csrc")
    seen, todo = set(), ["td_split_attn.cu", "td_api.cu"]
    while todo:
        name = todo.pop()
        if name in seen or not os.path.exists(os.path.join(src, name)):
            continue
        seen.add(name)
        with open(os.path.join(src, name)) as f:
            todo += re.findall(r'^#include "([^"]+)"', f.read(), flags=re.M)
    h = hashlib.sha256()
    for name in sorted(seen):
        with open(os.path.join(src, name)) as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    with open(os.path.join(ROOT, "include", "td.h")) as f:
        h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def max_over_ranks(values, device) -> list:
    """Each value's maximum over the ranks of the default process group (the slowest rank's
    time); the values unchanged when there is no group or a single rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_gbs(world: int, calls_per_rank: int, bytes_call: int, ms: float) -> float:
    """GB/s of the whole job: every rank's calls' bytes over the slowest rank's time (ms)."""
    return world * calls_per_rank * bytes_call / (ms * 1e-3) / 1e9


def recorded_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel, {}).get(workload_key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.proc = None
        self.lines = []
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:  # noqa: BLE001
            sel = []
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100", *sel]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, pw, reasons = [], [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples under load: the busiest half by power
        order = sorted(range(len(sm)), key=lambda i: pw[i], reverse=True)
        loaded = [sm[i] for i in order[:max(1, len(order) // 2)]]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


# ---------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    orc = oracle.load()
    w = WORKLOADS[args.workload]
    case = make_case(w, seq_len=args.seq_len)
    qn, kn, vn, sn = (to_numpy(x) for x in (case.q, case.k_cache, case.v_cache, case.seq_lens))
    bytes_call = kv_read_bytes(w, args.seq_len)
    for _ in range(args.warmup):
        orc.attention(qn, kn, vn, sn, case.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.attention(qn, kn, vn, sn, case.scale)
    dt = time.perf_counter() - t0
    gbs = bytes_call * args.steps / dt / 1e9
    cfg = workload_config(w, args.seq_len, None, None)
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": orc.num_threads, "kind": "oracle",
                         "sample": f"{args.steps} full oracle calls (24 heads x {args.seq_len} keys), fp64"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------- our arm

def workload_config(w, L, R, C):
    cfg = {
        "workload": f"{w.name} decode attention: B={w.B} Hq={w.Hq} Hkv={w.Hkv} D={w.D} Smax={w.Smax} "
                    f"seq_len={L} {w.dtype}, split auto",
        "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "Smax": w.Smax, "seq_len": L, "split": "auto",
        "kv_bytes_per_call": kv_read_bytes(w, L),
        "step": "R calls, each kv_append of 1 token + decode attention, one CUDA graph replay",
    }
    if R is not None:
        cfg["calls_per_step"] = R
    if C is not None:
        cfg["l2"] = (f"inputs larger than L2: each call reads {kv_read_bytes(w, L) / 1e6:.1f} MB of KV and "
                     f"calls rotate over {C} cache copies")
    return cfg


def rotating_copies(src: torch.Tensor, n: int) -> torch.Tensor:
    out = torch.empty((n,) + tuple(src.shape), dtype=src.dtype, device=src.device)
    out.copy_(src.unsqueeze(0).expand_as(out))
    return out


def time_graph(graph, stream, reps, warm=2):
    """Replays (which launch on the current stream) and events, all on `stream`; returns ms."""
    with torch.cuda.stream(stream):
        for _ in range(warm):
            graph.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def kernel_label(td, w) -> str:
    """Which split-attention kernel the timed call runs, from the library's own launch plan."""
    plan = td.td_split_plan(w.torch_dtype, w.B, w.Hq, w.Hkv, w.Smax, w.D, w.T, 0)
    # query rows per CTA: 8 or fewer go on one n8 tile, 17 to 24 on three (the narrow tiles)
    r = plan["rows"]
    tile = "narrow n8 tile" if r <= 8 else "m16 tile" if r <= 16 else "narrow 24-row tile"
    names = {
        "tensor_core_persistent": f"split_attn_mma_kernel<{w.D}> (persistent, fused split + workspace merge, "
                                  f"mma.sync bf16 {tile}, TMA)",
        "tensor_core_cluster": f"split_attn_cluster_kernel<{w.D}> (clusters of {plan['cluster']}, on-chip merge, "
                               f"mma.sync bf16 {tile}, TMA)",
        "cuda_core": f"split_attn_kernel<{w.D}> (CUDA cores)",
    }
    return f"{names[plan['kernel']]}, grid {plan['grid']}, timed alone"


def spec_point(td, dev, l2_bytes, peak, B=1, G=4, V=128256, budget_calls=200):
    """The speculative accept/reject step alone (a NEXT row): graph of R launches over rotating
    copies of fp32 logits (a Llama-3-sized vocabulary); algorithmic bytes = every target and
    draft row read once, (2G+1) * V * 4 per sequence."""
    gen = torch.Generator().manual_seed(5)
    bytes_call = B * (2 * G + 1) * V * 4
    C = max(2, math.ceil(4 * l2_bytes / bytes_call))
    target = torch.randn(C, B, G + 1, V, generator=gen).to(dev)
    draft = (target[:, :, :G] + 0.5 * torch.randn(C, B, G, V, generator=gen).to(dev)).contiguous()
    tokens = torch.randint(0, V, (B, G), generator=gen, dtype=torch.int32).to(dev)
    u = torch.rand(B, G + 1, generator=gen).to(dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    R = max(C, budget_calls)
    s = torch.cuda.Stream(dev)

    def calls():
        for i in range(R):
            td.td_spec_accept(target[i % C], tokens, draft[i % C], u, 1.0, n_accepted=n, next_token=nxt, stream=s)

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    ms = statistics.median(time_graph(g, s, 3) for _ in range(5))
    us = ms * 1e3 / (3 * R)
    del target, draft
    torch.cuda.empty_cache()
    gbs = bytes_call / (us * 1e-6) / 1e9
    return {"row": "speculative accept/reject (td_spec_accept)", "B": B, "draft_tokens": G, "vocab": V,
            "temperature": 1.0, "us_per_call": round(us, 3), "logit_gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "bytes_per_call": bytes_call}


def q8_point(td, name, L, dev, l2_bytes, peak, budget_calls=200):
    """Decode over the 8-bit cache (a NEXT row): the workload's cache quantised on the GPU, then
    a graph of R attention launches over rotating copies. Algorithmic bytes: every visible K
    and V row's codes and scale, L * Hkv * 2 * (D + 4) per sequence."""
    w = WORKLOADS[name]
    case = make_case(w, seq_len=L)
    kc, ks = td.td_quantize_q8(case.k_cache.to(dev))
    vc, vs = td.td_quantize_q8(case.v_cache.to(dev))
    bytes_call = sum(case.seq_lens.tolist()) * w.Hkv * 2 * (w.D + 4)
    C = max(2, math.ceil(4 * l2_bytes / bytes_call))
    per_copy = (kc.numel() + ks.numel() * 4) * 2
    C = min(C, max(2, int(24e9 // per_copy)))
    kcs, kss, vcs, vss = (rotating_copies(t, C) for t in (kc, ks, vc, vs))
    q = case.q.to(dev)[:, :, 0]
    sl = case.seq_lens.to(dev)
    out = torch.empty_like(q)
    ws = td.make_workspace(w.B, w.Hq, w.Hkv, w.Smax, w.D, 1, 0, device=dev)
    R = max(C, budget_calls)
    s = torch.cuda.Stream(dev)

    def calls():
        for i in range(R):
            c = i % C
            td.td_decode_attn_q8(q, kcs[c], kss[c], vcs[c], vss[c], sl, case.scale, 0, out=out, workspace=ws,
                                 stream=s)

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    ms = statistics.median(time_graph(g, s, 3) for _ in range(5))
    us = ms * 1e3 / (3 * R)
    del kcs, kss, vcs, vss
    torch.cuda.empty_cache()
    gbs = bytes_call / (us * 1e-6) / 1e9
    bf16_bytes = kv_read_bytes(w, case.seq_lens.tolist())
    return {"row": "int8 KV cache (td_decode_attn_q8)", "workload": name, "seq_len": L, "us_per_call": round(us, 3),
            "kv_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4), "kv_bytes": bytes_call,
            "bf16_equivalent_gbs": round(bf16_bytes / (us * 1e-6) / 1e9, 1)}


def prefill_point(td, dev, T=4096, B=1, Hq=24, Hkv=8, D=128, reps=20):
    """Causal prefill of a T-token prompt on the tensor cores (a NEXT row): a graph of `reps`
    launches; FLOPs = 4 * D * Hq * B * T(T+1)/2 (Q K^T and P V over the visible keys)."""
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).to(dev)
    sl = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        td.td_prefill_attn(q, k, v, sl, out=out, stream=s)
    s.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        for _ in range(reps):
            td.td_prefill_attn(q, k, v, sl, out=out, stream=s)
    ms = statistics.median(time_graph(gr, s, 2) for _ in range(5)) / (2 * reps)
    flops = 4 * D * Hq * B * T * (T + 1) / 2
    tf = flops / (ms * 1e-3) / 1e12
    peaks, kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    return {"row": "tiled causal prefill (td_prefill_attn, tcgen05)", "B": B, "T": T, "Hq": Hq, "Hkv": Hkv, "D": D,
            "us_per_call": round(ms * 1e3, 2), "tflops": round(tf, 1), "peak_bf16_tflops": peak,
            "frac_of_peak": round(tf / peak, 4), "peak_kind": f"bf16_tflops of {kind}"}


def sweep_point(td, name, L, dev, l2_bytes, peak, budget_calls=200, split=0):
    """Attention kernel alone on one workload point: graph of R launches over rotating caches."""
    w = WORKLOADS[name]
    case = make_case(w, seq_len=L if not w.ragged else None)
    bytes_call = kv_read_bytes(w, case.seq_lens.tolist())
    C = max(2, math.ceil(4 * l2_bytes / bytes_call))
    per_copy = case.k_cache.numel() * case.k_cache.element_size() * 2
    C = min(C, max(2, int(48e9 // per_copy)))
    kc = rotating_copies(case.k_cache.to(dev), C)
    vc = rotating_copies(case.v_cache.to(dev), C)
    q = case.q.to(dev)
    sl = case.seq_lens.to(dev)
    R = max(C, budget_calls)
    out = torch.empty_like(q)
    ws = td.make_workspace(w.B, w.Hq, w.Hkv, w.Smax, w.D, w.T, split, device=dev)
    s = torch.cuda.Stream(dev)

    def calls():
        for i in range(R):
            c = i % C
            if w.T == 1:
                td.td_decode_attn(q[:, :, 0], kc[c], vc[c], sl, case.scale, split, out=out[:, :, 0], workspace=ws,
                                  stream=s)
            else:
                td.td_verify_attn(q, kc[c], vc[c], sl, case.scale, split, out=out, workspace=ws, stream=s)

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    ms = statistics.median(time_graph(g, s, 3) for _ in range(5))
    us = ms * 1e3 / (3 * R)
    gbs = bytes_call / (us * 1e-6) / 1e9
    del kc, vc
    torch.cuda.empty_cache()
    return {"workload": name, "seq_len": L if not w.ragged else "ragged", "split": split or "auto",
            "dtype": w.dtype, "us_per_call": round(us, 3), "kv_gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "kv_bytes": bytes_call, "cache_copies": C}


def profile_row(td, args, dev):
    """Plain launches of one NEXT row's kernel (W warm-up, then --profile-launches), no timing."""
    if args.profile_row in ("verify6", "ragged8"):
        w = WORKLOADS[args.profile_row]
        case = make_case(w, seq_len=16390 if w.T > 1 else None)
        nbytes = kv_read_bytes(w, case.seq_lens.tolist())
        C = max(2, math.ceil(4 * torch.cuda.get_device_properties(dev).L2_cache_size / nbytes))
        kc = rotating_copies(case.k_cache.to(dev), C)
        vc = rotating_copies(case.v_cache.to(dev), C)
        q, sl = case.q.to(dev), case.seq_lens.to(dev)
        out = torch.empty_like(q)
        ws = td.make_workspace(w.B, w.Hq, w.Hkv, w.Smax, w.D, w.T, 0, device=dev)
        for i in range(args.warmup + args.profile_launches):
            c = i % C
            if w.T > 1:
                td.td_verify_attn(q, kc[c], vc[c], sl, case.scale, 0, out=out, workspace=ws)
            else:
                td.td_decode_attn(q[:, :, 0], kc[c], vc[c], sl, case.scale, 0, out=out[:, :, 0], workspace=ws)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_row": args.profile_row, "kv_bytes_per_launch": nbytes, "cache_copies": C,
                          "launches": args.warmup + args.profile_launches, "ok": True}))
        return
    g = torch.Generator(device=dev).manual_seed(0)
    w = WORKLOADS["llama3b"]
    L, B = args.seq_len, args.profile_batch
    if args.profile_row == "q8":
        k = torch.randn(B, w.Hkv, L, w.D, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(B, w.Hkv, L, w.D, device=dev, generator=g).to(torch.bfloat16)
        q = torch.randn(B, w.Hq, w.D, device=dev, generator=g).to(torch.bfloat16)
        kc, ks = td.td_quantize_q8(k)
        vc, vs = td.td_quantize_q8(v)
        del k, v
        seq = torch.full((B,), L, dtype=torch.int32, device=dev)
        call = lambda: td.td_decode_attn_q8(q, kc, ks, vc, vs, seq, w.D ** -0.5)  # noqa: E731
    else:
        q = torch.randn(B, w.Hq, L, w.D, device=dev, generator=g).to(torch.bfloat16)
        k = torch.randn(B, w.Hkv, L, w.D, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(B, w.Hkv, L, w.D, device=dev, generator=g).to(torch.bfloat16)
        seq = torch.full((B,), L, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        call = lambda: td.td_prefill_attn(q, k, v, seq, out=out)  # noqa: E731
    for _ in range(args.warmup + args.profile_launches):
        call()
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_row": args.profile_row, "seq_len": L, "batch": B,
                      "launches": args.warmup + args.profile_launches, "ok": True}))


def run_td(args, world, rank, local):
    from decode_attention_split_gb300 import build
    build.build()
    import decode_attention_split_gb300 as td

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.profile_row:
        profile_row(td, args, dev)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = WORKLOADS[args.workload]
    L = args.seq_len
    case = make_case(w, seq_len=L)
    bytes_call = kv_read_bytes(w, L)
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    C = max(2, math.ceil(4 * l2 / bytes_call))
    R = max(args.calls_per_step, C)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    kc = rotating_copies(case.k_cache.to(dev), C)
    vc = rotating_copies(case.v_cache.to(dev), C)
    gen = torch.Generator().manual_seed(1)
    qh = torch.randn(R, w.B, w.Hq, w.D, generator=gen).to(torch.bfloat16)
    knh = torch.randn(R, w.B, w.Hkv, 1, w.D, generator=gen).to(torch.bfloat16)
    vnh = torch.randn(R, w.B, w.Hkv, 1, w.D, generator=gen).to(torch.bfloat16)
    q, kn, vn = qh.to(dev), knh.to(dev), vnh.to(dev)
    out = torch.empty_like(q)
    sl_pre = torch.full((w.B,), L - 1, dtype=torch.int32, device=dev)  # new row goes to position L-1
    sl_post = torch.full((w.B,), L, dtype=torch.int32, device=dev)
    ws = td.make_workspace(w.B, w.Hq, w.Hkv, w.Smax, w.D, 1, 0, device=dev)
    s = torch.cuda.Stream(dev)

    from decode_attention_split_gb300.workloads import rope_tables
    cos_t, sin_t = (t.to(dev) for t in rope_tables(w.Smax, w.D))

    def calls(mode="fused"):
        """fused: one launch per call (cache write + attention); rope: the same with the query and
        key rotated; separate: td_kv_append then td_decode_attn; attn: the attention alone."""
        for i in range(R):
            c = i % C
            if mode in ("fused", "rope"):
                rot = mode == "rope"
                td.td_rope_append_attn(q[i][:, :, None], kn[i], vn[i], kc[c], vc[c], sl_pre, case.scale, 0,
                                       cos_t=cos_t if rot else None, sin_t=sin_t if rot else None, advance=False,
                                       out=out[i][:, :, None], workspace=ws, stream=s)
                continue
            if mode == "separate":
                td.td_kv_append(kn[i], vn[i], kc[c], vc[c], sl_pre, advance=False, stream=s)
            td.td_decode_attn(q[i], kc[c], vc[c], sl_post, case.scale, 0, out=out[i], workspace=ws, stream=s)

    if args.profile_launches:
        # the timed step's call, launched plainly (no graph): W warm-up calls, then the ones to profile
        with torch.cuda.stream(s):
            for i in range(args.warmup + args.profile_launches):
                c = i % C
                td.td_rope_append_attn(q[i % R][:, :, None], kn[i % R], vn[i % R], kc[c], vc[c], sl_pre, case.scale,
                                       0, advance=False, out=out[i % R][:, :, None], workspace=ws, stream=s)
        s.synchronize()
        print(json.dumps({"profile_launches": args.profile_launches, "ok": True}))
        return

    graphs = {}
    for mode in ("separate", "rope", "attn", "fused"):  # the timed step's graph is captured last
        with torch.cuda.stream(s):
            calls(mode)
        s.synchronize()
        graphs[mode] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[mode], stream=s):
            calls(mode)
    g_step, g_attn = graphs["fused"], graphs["attn"]

    with torch.cuda.stream(s):  # graph replays launch on the current stream
        for _ in range(args.warmup):
            g_step.replay()
    s.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(args.steps):
                g_step.replay()
            e1.record(s)
        e1.synchronize()
        torch.cuda.synchronize()
        ms_attn = time_graph(g_attn, s, args.steps, warm=2)
        ms_separate = time_graph(graphs["separate"], s, max(3, args.steps // 4), warm=2) * args.steps / \
            max(3, args.steps // 4)
        ms_rope = time_graph(graphs["rope"], s, max(3, args.steps // 4), warm=2) * args.steps / max(3, args.steps // 4)
    ms = e0.elapsed_time(e1)
    if world > 1:
        ms, ms_attn = max_over_ranks([ms, ms_attn], dev)
        torch.distributed.barrier()

    # correctness of what was timed: one more replay of the step graph, then its call 0 (which
    # wrote its own new row into copy 0 and attended over it) against the oracle
    checked = None
    with torch.cuda.stream(s):
        g_step.replay()
    s.synchronize()
    if rank == 0:
        import numpy as np
        import oracle
        ek = to_numpy(case.k_cache).copy()
        ev = to_numpy(case.v_cache).copy()
        ek[:, :, L - 1] = to_numpy(knh[0])[:, :, 0]
        ev[:, :, L - 1] = to_numpy(vnh[0])[:, :, 0]
        ref, _, _ = oracle.load().attention(to_numpy(qh[0]), ek, ev, np.array([L], np.int32), case.scale)
        got = out[0].double().cpu().numpy()
        checked = bool(np.all(np.abs(got - ref) <= 2e-2 + 1e-2 * np.abs(ref)))

    total_calls = args.steps * R
    value = whole_job_gbs(world, total_calls, bytes_call, ms)
    us_attn = ms_attn * 1e3 / total_calls
    achieved = bytes_call / (us_attn * 1e-6) / 1e9

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(td, args, w, case, kc, vc, C, R, sl_pre, sl_post, ws, dev, bytes_call, world)

    if rank != 0:
        return
    cpu = None if (args.no_cpu or world > 1) else cpu_baseline(case, w, L, args.cpu_seconds)
    ctable = None if (args.no_cpu or args.no_sweep or world > 1) else cpu_table()
    sweep = next_rows = None
    if not args.no_sweep:
        del kc, vc
        torch.cuda.empty_cache()
        sweep = [sweep_point(td, "tiny_fp32", 128, dev, l2, peak, split=WORKLOADS["tiny_fp32"].split)]
        for name in ("smollm2_360m", "llama3b"):
            for Ls in WORKLOADS[name].seq_lens:
                sweep.append(sweep_point(td, name, Ls, dev, l2, peak))
        sweep.append(sweep_point(td, "ragged8", None, dev, l2, peak))
        sweep.append(sweep_point(td, "verify6", 16390, dev, l2, peak))
        next_rows = [spec_point(td, dev, l2, peak), spec_point(td, dev, l2, peak, B=8)]
        next_rows += [q8_point(td, "llama3b", Ls, dev, l2, peak) for Ls in (4096, 16384, 32768)]
        next_rows += [prefill_point(td, dev, T=4096), prefill_point(td, dev, T=8192)]
    traffic = recorded_traffic("split_attn_kernel", f"{w.name}:{L}")
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, 1% keys x8; no model weights)",
        "config": dict(workload_config(w, L, R, C), parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "us_per_call": round(ms * 1e3 / total_calls, 3),
        "frac_of_measured_hbm": round(value / world / peak, 4),
        "checked_against_oracle": checked,
        "clocks": clk.summary(),
        "gpu_launches": total_calls,
        "step_variants_us_per_call": {
            "fused (timed step: one launch, cache write + attention)": round(ms * 1e3 / total_calls, 3),
            "fused with rotary embedding of q and k": round(ms_rope * 1e3 / total_calls, 3),
            "separate launches (td_kv_append, td_decode_attn)": round(ms_separate * 1e3 / total_calls, 3),
            "attention alone": round(us_attn, 3)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_label(td, w),
                     "us_per_launch": round(us_attn, 3), "peak_kind": f"hbm_gbs of {peak_kind}",
                     "algorithmic_bytes_per_launch": bytes_call},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_table": ctable,
        "sweep": sweep,
        "next_rows": next_rows,
        "kernel_source": kernel_source_hash(),
        "device": props.name,
    }
    print(json.dumps(line), flush=True)


def run_e2e(td, args, w, case, kc, vc, C, R, sl_pre, sl_post, ws, dev, bytes_call, world):
    """Through the public Python API with host buffers: each step copies its R calls' inputs (q and
    the new rows, packed in one pinned buffer) to the device in one transfer, makes the R calls,
    and reads all R outputs back in one transfer."""
    steps = max(1, min(args.steps, 10))
    gen = torch.Generator().manual_seed(2)
    nq, nk = w.B * w.Hq * w.D, w.B * w.Hkv * w.D
    per = nq + 2 * nk  # bf16 elements of one call's inputs: q, k_new, v_new
    inh = torch.randn(R, per, generator=gen).to(torch.bfloat16).pin_memory()
    outh = torch.empty(R, nq, dtype=torch.bfloat16).pin_memory()
    ind = torch.empty(R, per, dtype=torch.bfloat16, device=dev)
    outd = torch.empty(R, nq, dtype=torch.bfloat16, device=dev)
    # per-call views of the packed device buffers (contiguous), made once
    views = [(ind[i, :nq].view(w.B, w.Hq, 1, w.D), ind[i, nq:nq + nk].view(w.B, w.Hkv, 1, w.D),
              ind[i, nq + nk:].view(w.B, w.Hkv, 1, w.D), outd[i].view(w.B, w.Hq, 1, w.D)) for i in range(R)]
    s = torch.cuda.Stream(dev)

    def one_step():
        with torch.cuda.stream(s):
            ind.copy_(inh, non_blocking=True)
            for i in range(R):
                q, kn, vn, o = views[i]
                td.td_rope_append_attn(q, kn, vn, kc[i % C], vc[i % C], sl_pre, case.scale, 0, advance=False,
                                       out=o, workspace=ws, stream=s)
            outh.copy_(outd, non_blocking=True)

    one_step()
    s.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    host_s = time.perf_counter() - t0
    e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    if world > 1:
        ms = max_over_ranks([ms], dev)[0]
    return {"value": round(whole_job_gbs(world, steps * R, bytes_call, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": inh.numel() * 2, "d2h_bytes_per_step": outh.numel() * 2,
            "steps": steps, "us_per_call": round(ms * 1e3 / (steps * R), 3),
            "host_us_per_call": round(host_s * 1e6 / (steps * R), 3),
            "path": "python binding td_rope_append_attn (one launch per call); per step, the calls' inputs "
                    "(q and new rows) in one pinned host-to-device copy and their outputs in one copy back"}


def cpu_baseline(case, w, L, seconds):
    import oracle
    orc = oracle.load()
    qn, kn, vn, sn = (to_numpy(x) for x in (case.q, case.k_cache, case.v_cache, case.seq_lens))
    n, t0 = 0, time.perf_counter()
    while n < 3 or time.perf_counter() - t0 < seconds:
        orc.attention(qn, kn, vn, sn, case.scale)
        n += 1
    dt = (time.perf_counter() - t0) / n
    return {"value": round(kv_read_bytes(w, L) / dt / 1e9, 3), "unit": "GB/s", "cores": orc.num_threads,
            "kind": "oracle", "sample": f"{n} full calls (B=1, 24 heads x {L} keys, fp64), {dt * 1e3:.1f} ms each"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the architecture."""
    import platform
    import subprocess
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip() in ("Model name", "Vendor ID") and val.strip() and not name.endswith(val.strip()):
                name = (name + " " + val.strip()).strip()
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    name = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return f"{name or 'unknown'} ({platform.machine()}, {os.cpu_count()} logical CPUs)"


def cpu_table(reps: int = 3):
    """The oracle (fp64) on every workload point, single-threaded and on all host cores: median of
    `reps` full calls each. A reported baseline, not a target."""
    import oracle
    orc = oracle.load()
    cores = os.cpu_count() or 1
    rows = []
    points = [("tiny_fp32", 128)] + [("smollm2_360m", L) for L in WORKLOADS["smollm2_360m"].seq_lens] + \
        [("llama3b", L) for L in WORKLOADS["llama3b"].seq_lens] + [("ragged8", None), ("verify6", 16390)]
    for name, L in points:
        w = WORKLOADS[name]
        case = make_case(w, seq_len=L if not w.ragged else None)
        qn, kn, vn, sn = (to_numpy(x) for x in (case.q, case.k_cache, case.v_cache, case.seq_lens))
        nbytes = kv_read_bytes(w, case.seq_lens.tolist())
        row = {"workload": name, "seq_len": L if L is not None else "ragged", "kv_bytes": nbytes}
        for label, threads in (("single_thread", 1), ("all_cores", cores)):
            orc.set_num_threads(threads)
            times = []
            for _ in range(reps):
                t0 = time.perf_counter()
                orc.attention(qn, kn, vn, sn, case.scale)
                times.append(time.perf_counter() - t0)
            med = sorted(times)[len(times) // 2]
            row[label] = {"threads": threads, "us_per_call": round(med * 1e6, 1),
                          "kv_gbs": round(nbytes / med / 1e9, 4)}
        rows.append(row)
    orc.set_num_threads(cores)
    return {"cpu": cpu_model(), "statistic": f"median of {reps} full calls", "kind": "oracle (fp64 C, OpenMP)",
            "rows": rows}


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_td(args, world, rank, local)


if __name__ == "__main__":
    main()
