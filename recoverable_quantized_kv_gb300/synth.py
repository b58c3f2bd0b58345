"""Seeded synthetic inputs shaped like the QEvict paper's long-context workloads.

This module only draws numbers.  It holds no part of the method's arithmetic
(no budget, window partition, quantisation, attention or routing); both the
CUDA path and the CPU oracle receive the same tensors produced here.

Workload shapes follow the decoding setups of "QEvict: Recoverable Quantized KV
Eviction for Attention-Drift-Robust Long-Context Decoding" (arXiv 2608.05326):
Llama-3-8B-shaped attention (32 layers, 32 query heads, 8 KV heads, head
dimension 128, §5 Setup), RULER-class 32K contexts under a 20% budget (§5
"Long-range retrieval"), Omega = 8, q = 0.70, INT2 (§5 Setup, App. B.5).  No
dataset is read: the keys carry "planted" windows aligned with drifting query
directions so that window importance changes while decoding, the behaviour the
paper's §3 Observation III describes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "workload", "prompt_inputs", "decode_inputs", "seed_of", "rope_table"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Sizes of one synthetic decoding workload (all per sequence unless noted)."""

    name: str
    batch: int
    n_layers: int
    h_q: int
    h_kv: int
    d_head: int = 128
    n_sink: int = 4
    n_recent: int = 128
    window: int = 32
    bits: int = 2
    omega: int = 8
    q_num: int = 70           # quantised-tier fraction q = q_num / q_den
    q_den: int = 100
    budget_num: int = 20      # B_total = budget_num / budget_den of the full KV bytes
    budget_den: int = 100
    prompt_len: int = 4096
    steps: int = 64
    seed: int = 1
    # input structure
    n_plant: int = 0          # planted key windows per (sequence, layer); 0 = none
    plant_frac_num: int = 0   # alternatively a fraction of the prompt's windows
    plant_frac_den: int = 100
    kappa: float = 0.0        # planted direction gain on keys and queries
    switch_every: int = 16    # decode steps between changes of the active planted window
    query_walk_sigma: float = 0.0   # >0: decode queries follow a Gaussian random walk
    key_lognormal_sigma: float = 0.0  # >0: keys of each window scaled by exp(N(0, sigma^2))
    # routing policy (QEvict App. J / K): ranker 0 cumulative, 1 decayed, 2 p-norm, 3 key norm
    ranker: int = 0
    decay: float = 0.99
    pnorm: float = 3.0
    no_promotion: int = 0
    # rotate-half RoPE base of the keys (0 = keys carry no rotation); see rope_table
    rope_base: float = 0.0

    @property
    def max_len(self) -> int:
        return self.prompt_len + self.steps

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def plant_count(self) -> int:
        full_blocks = max(0, (self.prompt_len - self.n_sink) // self.window)
        if self.n_plant:
            return min(self.n_plant, full_blocks)
        if self.plant_frac_num:
            return max(1, full_blocks * self.plant_frac_num // self.plant_frac_den)
        return 0


WORKLOADS = {
    # single layer, tiny: the case the oracle finishes in seconds
    "tiny_4k": Workload("tiny_4k", batch=1, n_layers=1, h_q=8, h_kv=2, prompt_len=4096, steps=64,
                        budget_num=25, n_plant=16, kappa=8.0, seed=1),
    # Llama-3-8B-shaped, 32K context, batch 1: the headline decode workload
    "llama8b_32k": Workload("llama8b_32k", batch=1, n_layers=32, h_q=32, h_kv=8, prompt_len=32768,
                            steps=256, budget_num=20, plant_frac_num=5, kappa=4.0, seed=2),
    # batched serving: 16 independent sequences of the same shape
    "batched_32k": Workload("batched_32k", batch=16, n_layers=32, h_q=32, h_kv=8, prompt_len=32768,
                            steps=128, budget_num=20, plant_frac_num=5, kappa=4.0, seed=3),
    # long-context sweep point (INT2, 20%, q = 0.7); other points via .replace()
    "long_131k": Workload("long_131k", batch=4, n_layers=32, h_q=32, h_kv=8, prompt_len=131072,
                          steps=128, budget_num=20, key_lognormal_sigma=1.0, seed=4),
    # long-generation drift stress: random-walk queries
    "drift_16k": Workload("drift_16k", batch=8, n_layers=36, h_q=32, h_kv=8, prompt_len=16384,
                          steps=2048, n_recent=256, budget_num=125, budget_den=1000,
                          query_walk_sigma=0.3, seed=5),
}


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.replace(**overrides) if overrides else wl


_KIND = {"q_prompt": 1, "k_prompt": 2, "v_prompt": 3, "dirs": 4, "plants": 5, "q_dec": 6,
         "k_dec": 7, "v_dec": 8, "walk": 9, "lognorm": 10}


def seed_of(*parts: int) -> int:
    """Deterministic 63-bit seed from integer parts (Knuth MMIX LCG mixing)."""
    h = 0x2545F4914F6CDD1D
    for p in parts:
        h = (h * 6364136223846793005 + (int(p) * 2 + 1) * 1442695040888963407) & ((1 << 64) - 1)
    return h & ((1 << 63) - 1)


def _gen(wl: Workload, b: int, layer: int, kind: str, device, extra: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(wl.seed, b, layer, _KIND[kind], extra))
    return g


def _randn(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _plants(wl: Workload, b: int, layer: int, device):
    """Planted window blocks (indices of window-aligned prompt blocks) and their unit directions."""
    n = wl.plant_count()
    if n == 0:
        return None, None
    full_blocks = (wl.prompt_len - wl.n_sink) // wl.window
    g = _gen(wl, b, layer, "plants", "cpu")
    blocks = torch.randperm(full_blocks, generator=g)[:n].sort().values
    dirs = _randn((n, wl.d_head), _gen(wl, b, layer, "dirs", device), device)
    dirs = dirs / dirs.norm(dim=1, keepdim=True)
    return blocks.to(device), dirs


def _rope(x: torch.Tensor, pos0: int, base: float) -> torch.Tensor:
    """The model's own position encoding of its queries and keys: rows of x [S][H][d] sit at positions
    pos0 .. pos0 + S - 1; channel pair (i, i + d/2) is the complex number x_i + j x_{i+d/2}, multiplied
    by exp(j pos base^(-2i/d)) in complex128."""
    d = x.shape[-1]
    theta = base ** (-2.0 * torch.arange(d // 2, dtype=torch.float64, device=x.device) / d)
    ang = torch.arange(pos0, pos0 + x.shape[0], dtype=torch.float64, device=x.device)[:, None] * theta[None, :]
    z = torch.complex(x[..., :d // 2].double(), x[..., d // 2:].double()) * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1).float()


def prompt_inputs(wl: Workload, b: int, layer: int, device="cpu", with_queries: bool = True):
    """Prompt tensors of one (sequence, layer): q [P][H_q][d], k and v [P][H_kv][d], all bf16."""
    P, d = wl.prompt_len, wl.d_head
    k = _randn((P, wl.h_kv, d), _gen(wl, b, layer, "k_prompt", device), device)
    v = _randn((P, wl.h_kv, d), _gen(wl, b, layer, "v_prompt", device), device)
    blocks, dirs = _plants(wl, b, layer, device)
    if blocks is not None:
        for i in range(blocks.numel()):
            s = wl.n_sink + int(blocks[i]) * wl.window
            k[s:s + wl.window] += wl.kappa * dirs[i].view(1, 1, d)
    if wl.key_lognormal_sigma > 0:
        nblk = (P + wl.window - 1) // wl.window
        xi = _randn((nblk,), _gen(wl, b, layer, "lognorm", device), device)
        scale = torch.exp(wl.key_lognormal_sigma * xi).repeat_interleave(wl.window)[:P]
        k = k * scale.view(P, 1, 1)
    if wl.rope_base > 0:
        k = _rope(k, 0, wl.rope_base)
    out = {"k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if with_queries:
        q = _randn((P, wl.h_q, d), _gen(wl, b, layer, "q_prompt", device), device)
        out["q"] = (_rope(q, 0, wl.rope_base) if wl.rope_base > 0 else q).to(torch.bfloat16)
    return out


def decode_inputs(wl: Workload, b: int, layer: int, steps: Optional[int] = None, device="cpu"):
    """Decode-step tensors of one (sequence, layer): q [S][H_q][d], k and v [S][H_kv][d], bf16.

    Step s (1-based) of the planted workloads adds kappa * u_p to every query head,
    where the active planted window p changes every `switch_every` steps.
    """
    S = wl.steps if steps is None else steps
    d = wl.d_head
    q = _randn((S, wl.h_q, d), _gen(wl, b, layer, "q_dec", device), device)
    k = _randn((S, wl.h_kv, d), _gen(wl, b, layer, "k_dec", device), device)
    v = _randn((S, wl.h_kv, d), _gen(wl, b, layer, "v_dec", device), device)
    blocks, dirs = _plants(wl, b, layer, device)
    if blocks is not None:
        n = blocks.numel()
        idx = torch.tensor([(s // wl.switch_every) % n for s in range(S)], device=device)
        q = q + wl.kappa * dirs[idx].view(S, 1, d)
    if wl.query_walk_sigma > 0:
        # q_{s+1} = q_s + sigma * xi_s, starting from a Gaussian q_1
        xi = _randn((S, wl.h_q, d), _gen(wl, b, layer, "walk", device), device)
        xi[0] = 0.0
        q = q[0:1] + wl.query_walk_sigma * torch.cumsum(xi, dim=0)
    if wl.rope_base > 0:   # decode step s sits at position prompt_len + s
        q = _rope(q, wl.prompt_len, wl.rope_base)
        k = _rope(k, wl.prompt_len, wl.rope_base)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}


def describe(wl: Workload) -> str:
    return (f"{wl.name}: B={wl.batch} L={wl.n_layers} H_q={wl.h_q} H_kv={wl.h_kv} d={wl.d_head} "
            f"P={wl.prompt_len}+{wl.steps} sink={wl.n_sink} recent={wl.n_recent} W={wl.window} "
            f"INT{wl.bits} Omega={wl.omega} q={wl.q_num}/{wl.q_den} "
            f"budget={wl.budget_num}/{wl.budget_den} plants={wl.plant_count()} kappa={wl.kappa:g} "
            f"walk={wl.query_walk_sigma:g} lognorm={wl.key_lognormal_sigma:g} "
            f"(context {math.ceil(wl.max_len / 1024)}K)")


def rope_table(rows: int, base: float, d: int = 128) -> np.ndarray:
    """Model input: (cos, sin) of pos * base^(-2i/d) for every position pos < rows and pair
    i < d/2 of a rotate-half RoPE, computed in float64 and stored as float32 [rows][d/2][2]."""
    pos = np.arange(rows, dtype=np.float64)[:, None]
    theta = base ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)
    ang = pos * theta[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
