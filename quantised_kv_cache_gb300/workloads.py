"""Seeded synthetic K/V/q inputs shaped like the pages' setups.

This module draws inputs only: it holds none of the quantisation or attention
arithmetic, so both the CUDA path's tests and the CPU oracle can be fed from it.
No dataset or model weights are involved; the distributions stand in for real
activations:

* i.i.d. N(0, 1) keys, values and queries;
* keys with per-channel log-normal scales and a few fixed outlier channels,
  standing in for the fixed-channel outliers of real key caches
  ("Your KV cache is not a bit problem but a geometry problem", section
  "Keys: outliers live in fixed channels");
* rank-4 keys plus small noise, with queries in the same subspace, and
  Student-t (nu = 3) keys -- the low-rank and heavy-tailed families of
  "Statistical Inference and Quality Measures of KV Cache Quantisations
  Inspired by TurboQuant", technical summary, "Low-rank pathology" and
  "Results".

Every draw comes from a torch.Generator seeded explicitly (data seed
1000 + workload id unless given), on the device asked for.
"""

from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    batch: int
    heads_q: int
    heads_kv: int
    seq: int
    dtype: torch.dtype
    scheme: str                 # "KV" | "KQV" | "QKQV" | "KIVI" | "sweep"
    bits: int = 4
    splits: int = 0             # 0 = library's choice
    key_dist: str = "gauss"
    key_scale_sigma: float = 0.0
    outlier_channels: int = 0
    outlier_factor: float = 1.0
    kivi_layouts: Tuple[Tuple[bool, bool], ...] = field(default_factory=tuple)

    @property
    def d(self) -> int:
        return HEAD_DIM


WORKLOADS = {
    1: Workload(1, "single-head d128 N4096 fp32 KQV n=4", 1, 1, 1, 4096, torch.float32, "KQV", 4),
    2: Workload(2, "Llama-2-7B-shaped decode B16 H32 d128 N8192 bf16 KQV n=4", 16, 32, 32, 8192,
                torch.bfloat16, "KQV", 4, key_scale_sigma=1.0, outlier_channels=4, outlier_factor=10.0),
    3: Workload(3, "scheme sweep B4 H8 d128 N16384 fp32", 4, 8, 8, 16384, torch.float32, "sweep", 4),
    4: Workload(4, "GQA 32q/8kv d128 N131072 B1 bf16 KQV n=3, 64 splits", 1, 32, 8, 131072,
                torch.bfloat16, "KQV", 3, splits=64, key_scale_sigma=0.5),
    5: Workload(5, "KIVI Llama-2-13B-shaped B8 H40 d128 N4096 bf16 2-bit g32 w128", 8, 40, 40, 4096,
                torch.bfloat16, "KIVI", 2, key_scale_sigma=1.0,
                kivi_layouts=((True, True), (False, False), (False, True), (True, False))),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def generate(w: Workload, device="cpu", *, seed: Optional[int] = None, key_dist: Optional[str] = None,
             batch: Optional[int] = None, heads_kv: Optional[int] = None, heads_q: Optional[int] = None,
             seq: Optional[int] = None, dtype: Optional[torch.dtype] = None):
    """Return (q [B,Hq,d], k [B,Hkv,N,d], v [B,Hkv,N,d]) in the workload's dtype.

    Any shape argument overrides the workload's (for small test cases of the
    same family).
    """
    B = batch or w.batch
    Hkv = heads_kv or w.heads_kv
    Hq = heads_q or (w.heads_q if heads_kv is None else Hkv * (w.heads_q // w.heads_kv))
    N = seq or w.seq
    d = w.d
    dt = dtype or w.dtype
    dist = key_dist or w.key_dist
    g = _gen(device, 1000 + w.wid if seed is None else seed)
    f32 = torch.float32

    v = torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=f32)
    if dist == "gauss":
        k = torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=f32)
        q = torch.randn((B, Hq, d), generator=g, device=device, dtype=f32)
    elif dist == "lowrank":
        a = torch.randn((B, Hkv, N, 4), generator=g, device=device, dtype=f32)
        basis = torch.randn((B, Hkv, d, 4), generator=g, device=device, dtype=f32)
        k = a @ basis.transpose(-1, -2) / 2 + 0.01 * torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=f32)
        coef = torch.randn((B, Hq, 4, 1), generator=g, device=device, dtype=f32)
        G = Hq // Hkv
        q = (basis.repeat_interleave(G, dim=1) @ coef).squeeze(-1) / 2
    elif dist == "student3":
        z = torch.randn((B, Hkv, N, d), generator=g, device=device, dtype=f32)
        chi = torch.randn((3, B, Hkv, N, d), generator=g, device=device, dtype=f32).pow(2).sum(0)
        k = z / torch.sqrt(chi / 3.0)
        q = torch.randn((B, Hq, d), generator=g, device=device, dtype=f32)
    else:
        raise ValueError(dist)

    scale = key_channel_scales(w, Hkv, device, 1000 + w.wid if seed is None else seed)
    if scale is not None:
        k = k * scale
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def key_channel_scales(w: Workload, heads_kv: int, device, seed: int):
    """Per-(head, channel) key scales [1, heads_kv, 1, d]: exp(sigma N(0, 1)), with
    `outlier_channels` seeded channels per head multiplied by `outlier_factor`; None when
    the workload has no channel scales. Drawn from a generator of their own (seeded by the
    data seed), so the cache's keys and every decode step's new key share them."""
    if w.key_scale_sigma <= 0:
        return None
    g = _gen(device, seed + 7_919)
    d = w.d
    scale = torch.exp(w.key_scale_sigma * torch.randn((1, heads_kv, 1, d), generator=g, device=device,
                                                      dtype=torch.float32))
    if w.outlier_channels:
        for h in range(heads_kv):
            ch = torch.randperm(d, generator=g, device=device)[: w.outlier_channels]
            scale[0, h, 0, ch] *= w.outlier_factor
    return scale


def step_token(w: Workload, step: int, device="cpu", *, data_seed: Optional[int] = None, batch=None,
               heads_kv=None, heads_q=None, dtype=None):
    """One decode step's new K/V token per sequence and its query (seeded by step).

    The new keys follow the cache's key distribution: N(0, 1) times the per-channel
    scales (and outlier channels) that `generate` drew with the same data seed
    (default 1000 + workload id)."""
    B = batch or w.batch
    Hkv = heads_kv or w.heads_kv
    Hq = heads_q or (w.heads_q if heads_kv is None else Hkv * (w.heads_q // w.heads_kv))
    dt = dtype or w.dtype
    g = _gen(device, 50_000 + 100 * w.wid + step)
    k = torch.randn((B, Hkv, 1, w.d), generator=g, device=device)
    v = torch.randn((B, Hkv, 1, w.d), generator=g, device=device)
    q = torch.randn((B, Hq, w.d), generator=g, device=device)
    scale = key_channel_scales(w, Hkv, device, 1000 + w.wid if data_seed is None else data_seed)
    if scale is not None:
        k = k * scale
    return q.to(dt), k.to(dt), v.to(dt)
