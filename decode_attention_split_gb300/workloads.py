"""Seeded synthetic inputs for the decode-attention workloads.

This module only draws numbers and states shapes: it holds none of the attention
arithmetic, so the CUDA path and the CPU oracle can both be fed from it without
sharing any of the method. Everything is drawn on the CPU from
``torch.Generator('cpu').manual_seed(seed)`` in a fixed order:

    q, k cache, v cache (N(0,1) fp32, whole cache through Smax),
    then the heavy-key mask (Bernoulli(p) per (b, kv head, position); keys scaled x8),
    then per-sequence lengths (ragged batch only),
    then the new key/value rows (workloads that append),

and cast to the storage dtype last (bf16: round to nearest even, torch's cast).
``rope_tables`` gives the rotary-embedding cos/sin tables (an input, like a weight).

Workloads (shapes from the pages' models; the data is synthetic, no weights are used):

  tiny_fp32        fp32, B=1 Hq=4 Hkv=2 D=64 Smax=256, seq_len 128, split 64
  smollm2_360m     bf16 layer of a 360M Llama-architecture model: B=1 Hq=15 Hkv=5 D=64
                   Smax=4096, seq_len in {64, 1024, 2048, 4096}
  llama3b          bf16 layer of a 3B Llama-style model: B=1 Hq=24 Hkv=8 D=128 Smax=32768,
                   seq_len in {1024, 4096, 16384, 32768}, 1% of keys scaled x8
  ragged8          bf16 batch of 8: Hq=32 Hkv=8 D=128 Smax=8192; attended lengths L'_b
                   uniform in [1, 8192]; one new token appended at L'_b - 1, then attend L'_b
  verify6          bf16 speculative-verify chunk: B=1 T=6 Hq=32 Hkv=8 D=128 Smax=16400;
                   6 new tokens appended at 16384..16389, then verify over 16390 rows
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str  # "f32" or "bf16"
    B: int
    Hq: int
    Hkv: int
    D: int
    Smax: int
    seq_lens: tuple = ()  # attended lengths swept for B=1 workloads
    T: int = 1  # query rows per sequence (1 = decode, >1 = verify chunk)
    split: int = 0  # split size the workload names (0 = library's choice)
    heavy_key_frac: float = 0.0
    ragged: bool = False
    append: bool = False  # the workload writes its T new rows before attending
    notes: str = ""

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", "f32", 1, 4, 2, 64, 256, seq_lens=(128,), split=64),
        Workload("smollm2_360m", "bf16", 1, 15, 5, 64, 4096, seq_lens=(64, 1024, 2048, 4096)),
        Workload("llama3b", "bf16", 1, 24, 8, 128, 32768, seq_lens=(1024, 4096, 16384, 32768), heavy_key_frac=0.01),
        Workload("ragged8", "bf16", 8, 32, 8, 128, 8192, ragged=True, append=True),
        Workload("verify6", "bf16", 1, 32, 8, 128, 16400, seq_lens=(16390,), T=6, append=True),
    ]
}


def kv_bytes_per_token(Hkv: int, D: int, elem_bytes: int) -> int:
    """Bytes of K plus V one cached token occupies in one layer."""
    return 2 * Hkv * D * elem_bytes


def kv_read_bytes(w: Workload, attended) -> int:
    """Algorithmic KV bytes one attention call reads: every visible key and value row once.

    ``attended`` is an int (B=1) or a sequence of per-sequence attended lengths."""
    lens = [attended] if isinstance(attended, int) else list(attended)
    return sum(int(L) for L in lens) * kv_bytes_per_token(w.Hkv, w.D, w.elem_bytes)


@dataclass
class Case:
    """One seeded problem, all tensors on the CPU in the storage dtype (seq_lens int32)."""

    w: Workload
    q: torch.Tensor  # [B, Hq, T, D]
    k_cache: torch.Tensor  # [B, Hkv, Smax, D]
    v_cache: torch.Tensor
    seq_lens: torch.Tensor  # attended lengths (after any append), int32 [B]
    seq_lens_pre: torch.Tensor  # lengths before the append (== seq_lens when nothing is appended)
    k_new: torch.Tensor | None = None  # [B, Hkv, T, D]
    v_new: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return self.w.scale


def make_case(name_or_w, seq_len: int | None = None, seed: int = 0, smax: int | None = None) -> Case:
    """Draw the seeded inputs of a workload.

    ``seq_len`` picks one attended length of a B=1 sweep (default: the largest).
    ``smax`` shrinks the cache (for quick tests); the recipe is otherwise unchanged."""
    w = WORKLOADS[name_or_w] if isinstance(name_or_w, str) else name_or_w
    Smax = smax or w.Smax
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(w.B, w.Hq, w.T, w.D, generator=g)
    k = torch.randn(w.B, w.Hkv, Smax, w.D, generator=g)
    v = torch.randn(w.B, w.Hkv, Smax, w.D, generator=g)
    if w.heavy_key_frac > 0:
        heavy = torch.rand(w.B, w.Hkv, Smax, generator=g) < w.heavy_key_frac
        k = torch.where(heavy[..., None], k * 8.0, k)
    if w.ragged:
        attended = torch.randint(1, Smax + 1, (w.B,), generator=g, dtype=torch.int64)
    else:
        L = seq_len if seq_len is not None else (max(w.seq_lens) if w.seq_lens else Smax)
        if L > Smax:
            raise ValueError(f"seq_len {L} > Smax {Smax}")
        attended = torch.full((w.B,), L, dtype=torch.int64)
    k_new = v_new = None
    if w.append:
        k_new = torch.randn(w.B, w.Hkv, w.T, w.D, generator=g).to(w.torch_dtype)
        v_new = torch.randn(w.B, w.Hkv, w.T, w.D, generator=g).to(w.torch_dtype)
        pre = attended - w.T
    else:
        pre = attended.clone()
    dt = w.torch_dtype
    return Case(w, q.to(dt), k.to(dt), v.to(dt), attended.to(torch.int32), pre.to(torch.int32), k_new, v_new)


def small_case(dtype="bf16", B=2, Hq=8, Hkv=2, D=128, Smax=300, T=1, seq_lens=None, seed=0, heavy=0.0) -> Case:
    """A small seeded problem with the same recipe (tests at sizes the oracle finishes fast)."""
    w = Workload("small", dtype, B, Hq, Hkv, D, Smax, T=T, heavy_key_frac=heavy)
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, Hq, T, D, generator=g)
    k = torch.randn(B, Hkv, Smax, D, generator=g)
    v = torch.randn(B, Hkv, Smax, D, generator=g)
    if heavy > 0:
        mask = torch.rand(B, Hkv, Smax, generator=g) < heavy
        k = torch.where(mask[..., None], k * 8.0, k)
    if seq_lens is None:
        seq_lens = torch.randint(T, Smax + 1, (B,), generator=g)
    sl = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    dt = w.torch_dtype
    return Case(w, q.to(dt), k.to(dt), v.to(dt), sl, sl.clone())


def to_numpy(t: torch.Tensor):
    """CPU tensor -> numpy array in a form the oracle reads (bf16 as its uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def rope_tables(positions: int, D: int, base: float = 500000.0):
    """Rotary-embedding input tables (cos, sin), fp32 [positions, D/2], of the angles
    p * base^(-2i/D) (the llama frequency ladder; 500000 is Llama 3's base). They are an
    input of the rotation like any weight, computed here in fp64 and stored fp32."""
    inv = base ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    ang = torch.arange(positions, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)
