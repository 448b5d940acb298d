"""Seeded synthetic inputs and the workload shapes they are drawn for.

This module only draws random numbers and names shapes; it holds none of the
attention arithmetic. Both the CUDA path and the fp64 oracle take their inputs
from here, so the two see the same bits.

Every tensor is drawn on the host with a CPU ``torch.Generator``. A tensor
whose first axis is the batch draws each batch row from a generator of its
own, seeded by (workload seed, tensor name, row), so a test can rebuild one
row of a multi-gigabyte cache without drawing the rest.

The shapes follow the model families the attention pages describe: a
Llama-3-8B-shaped layer (32 query heads, 8 key/value heads, head_dim 128,
rope_theta 5e5 with the Llama 3 frequency ramp), a Gemma-2-shaped sliding
window layer (head_dim 256, window 4096, logit softcap 50, q/k RMSNorm), and
long-context decode with partial rotary. Values are iid N(0, 1) fp32; the
q/k norm weights are N(1, 0.1).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    H: int
    Hkv: int
    D: int
    L: int = 0                      # prefill tokens per row (0: decode only)
    decode_steps: int = 0           # single-token steps after the prefill
    rope_dim: int = 0               # 0: the whole head dimension
    theta: float = 10000.0
    scaling: tuple | None = None    # None, ("linear", f), ("llama3", f, lo, hi, orig)
    window: int = 0
    softcap: float = 0.0
    qk_norm: bool = False
    norm_eps: float = 1e-6
    max_positions: int = 8192
    capacity: int = 0               # cache slots per (row, kv head)
    cache_len_range: tuple | None = None   # decode over a random cache: n_b ~ U{lo..hi}
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.D if self.rope_dim == 0 else self.rope_dim

    @property
    def G(self) -> int:
        return self.H // self.Hkv


WORKLOADS = {
    "tiny": Workload(
        name="tiny", seed=0, B=1, H=4, Hkv=2, D=16, L=16, decode_steps=4, theta=1e4,
        capacity=20, notes="16-token prefill then 4 decode steps, positions 0..19"),
    "llama3_8b_prefill": Workload(
        name="llama3_8b_prefill", seed=1, B=4, H=32, Hkv=8, D=128, L=2048, theta=5e5,
        scaling=("llama3", 8.0, 1.0, 4.0, 8192), capacity=2048,
        notes="Llama-3-8B-shaped causal prefill"),
    "batched_decode": Workload(
        name="batched_decode", seed=2, B=64, H=32, Hkv=8, D=128, theta=5e5,
        cache_len_range=(512, 8192), capacity=8193, max_positions=16384,
        notes="64 rows, one new token each, cached lengths iid U{512..8192}"),
    "gemma2_window": Workload(
        name="gemma2_window", seed=3, B=1, H=16, Hkv=8, D=256, L=16384, theta=1e4,
        window=4096, softcap=50.0, qk_norm=True, capacity=4096, max_positions=16384,
        notes="Gemma-2-shaped sliding-window prefill with softcap and q/k RMSNorm"),
    "long_decode": Workload(
        name="long_decode", seed=4, B=8, H=64, Hkv=8, D=128, L=1024, decode_steps=1024,
        rope_dim=64, theta=1e6, capacity=2048,
        notes="1024-token prefill then 1024 single-token steps, partial rotary 64"),
}


def _seed(seed: int, name: str, row: int) -> int:
    return (seed * 1_000_003 + zlib.crc32(name.encode()) * 8191 + row * 131_071) % (2**62)


def normal_row(seed: int, name: str, shape: tuple, row: int, mean: float = 0.0,
               std: float = 1.0) -> torch.Tensor:
    """Batch row ``row`` of the tensor ``normal(seed, name, shape)``: shape[1:] fp32."""
    g = torch.Generator().manual_seed(_seed(seed, name, row))
    x = torch.randn(tuple(shape[1:]), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def normal(seed: int, name: str, shape: tuple, mean: float = 0.0, std: float = 1.0,
           out: torch.Tensor | None = None) -> torch.Tensor:
    """iid N(mean, std^2) fp32 of ``shape``, row by row along axis 0."""
    if out is None:
        out = torch.empty(tuple(shape), dtype=torch.float32)
    for b in range(shape[0]):
        out[b].copy_(normal_row(seed, name, shape, b, mean, std))
    return out


def norm_weight(seed: int, name: str, D: int) -> torch.Tensor:
    """q/k RMSNorm weight [D], N(1, 0.1)."""
    return normal(seed, name, (1, D), mean=1.0, std=0.1)[0]


def cache_lengths(seed: int, B: int, lo: int, hi: int) -> torch.Tensor:
    """Per-row cached token counts, iid uniform on {lo, ..., hi} (int32 [B])."""
    g = torch.Generator().manual_seed(_seed(seed, "cache_len", 0))
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def prefill_inputs(w: Workload, L: int | None = None, B: int | None = None) -> dict:
    """q [B,H,L,D], k and v [B,Hkv,L,D], and the q/k norm weights (or None)."""
    L = w.L if L is None else L
    B = w.B if B is None else B
    d = {
        "q": normal(w.seed, "q", (B, w.H, L, w.D)),
        "k": normal(w.seed, "k", (B, w.Hkv, L, w.D)),
        "v": normal(w.seed, "v", (B, w.Hkv, L, w.D)),
        "q_norm_w": norm_weight(w.seed, "q_norm_w", w.D) if w.qk_norm else None,
        "k_norm_w": norm_weight(w.seed, "k_norm_w", w.D) if w.qk_norm else None,
    }
    return d


def decode_token_inputs(w: Workload, step: int) -> dict:
    """The new token's q [B,H,1,D], k and v [B,Hkv,1,D] for decode step ``step``."""
    tag = f"step{step}"
    return {
        "q": normal(w.seed, "q_" + tag, (w.B, w.H, 1, w.D)),
        "k": normal(w.seed, "k_" + tag, (w.B, w.Hkv, 1, w.D)),
        "v": normal(w.seed, "v_" + tag, (w.B, w.Hkv, 1, w.D)),
    }


def random_cache_row(w: Workload, which: str, row: int) -> torch.Tensor:
    """Row ``row`` of a random cache ('k' or 'v'): [Hkv, capacity, D] fp32."""
    return normal_row(w.seed, "cache_" + which, (w.B, w.Hkv, w.capacity, w.D), row)
