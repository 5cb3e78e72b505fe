"""Seeded synthetic inputs for the LowRAM decode path -- random draws only.

This module holds none of the method's arithmetic: it draws Gaussian tensors, eviction position
sets and placeholder residual lists with fixed seeds, and describes the workload shapes.  Tests
and the benchmark compose the derived inputs (pre-RoPE keys, true values) from these draws with
whatever they are allowed to use; both the CUDA library and the oracle consume the same stored
tensors.

Recipe (all draws are float32 from ``torch.Generator`` on the CPU, then rounded to the storage
dtype with round-to-nearest-even by torch):
  latent coefficients C ~ N(0, 1)            [B, T, r]
  layer basis         W_l ~ N(0, 1/r)        [H_kv*d, r]   (row h*d+i: coefficients of key feature (h, i))
  predictor weights   W1 ~ N(0, 1/d)         [H_kv, m, d];   W2 ~ N(0, 1/m)   [H_kv, d, m]
  query               q ~ N(0, 1/d)          [B, H_q, d]
  value noise         N(0, 0.3^2)            [B, T, H_kv, d]  (true values = predictor(keys) + noise)
  eviction            64 sink + 2048 recent + seeded uniform draws without replacement, to T_nominal/4
Each tensor has its own sub-seed, a hash of (seed, workload, group, layer, tensor name), so any layer
can be drawn alone.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, replace

import torch

__all__ = ["Workload", "WORKLOADS", "sub_seed", "gaussian", "draw_group", "draw_query", "eviction_positions",
           "placeholder_residuals", "n_res_for"]


@dataclass(frozen=True)
class Workload:
    """Shapes of one decode workload.  T is the number of stored tokens per sequence (after eviction)."""
    name: str
    B: int
    T: int
    L: int
    G: int
    H_q: int
    H_kv: int
    d: int
    r: int
    m: int
    theta: float
    rho: float
    S: int
    act: str = "bf16"        # q, basis, predictor weights
    coef_fmt: str = "bf16"   # 'f32' | 'bf16' | 'int4'
    res_fmt: str = "bf16"    # 'f32' | 'bf16' | 'int8'
    T_nominal: int = 0       # > T when eviction is on
    seed: int = 0

    @property
    def n_res(self) -> int:
        return n_res_for(self.rho, self.T)

    @property
    def S_eff(self) -> int:
        return min(self.S, self.T)

    @property
    def groups(self) -> int:
        return self.L // self.G

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def n_res_for(rho: float, T: int) -> int:
    import math
    return max(0, min(T, int(math.ceil(rho * T - 1e-9))))


WORKLOADS = {
    # tiny fp32 case: one group of two layers, selection is a no-op (S = T)
    "tiny": Workload("tiny", B=1, T=256, L=2, G=2, H_q=4, H_kv=2, d=64, r=32, m=64, theta=1e4, rho=0.25, S=256,
                     act="f32", coef_fmt="f32", res_fmt="f32"),
    # Llama-3-8B-shaped decode (the headline workload)
    "llama8b": Workload("llama8b", B=8, T=8192, L=32, G=4, H_q=32, H_kv=8, d=128, r=512, m=128, theta=5e5,
                        rho=0.10, S=1024),
    # long context, B=2, T up to 32768
    "long": Workload("long", B=2, T=32768, L=32, G=4, H_q=32, H_kv=8, d=128, r=640, m=256, theta=1e6, rho=0.10,
                     S=2048),
    # peak decode throughput: batch sweep at T=4096
    "peak": Workload("peak", B=16, T=4096, L=28, G=4, H_q=28, H_kv=4, d=128, r=384, m=128, theta=5e5, rho=0.10,
                     S=512),
    # composed with quantisation and eviction: 65536 nominal tokens, 16384 kept
    "evict_quant": Workload("evict_quant", B=4, T=16384, L=32, G=4, H_q=32, H_kv=8, d=128, r=512, m=128,
                            theta=5e5, rho=0.05, S=1024, coef_fmt="int4", res_fmt="int8", T_nominal=65536),
}


def sub_seed(*parts) -> int:
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "f64": torch.float64}


def gaussian(shape, std: float, *parts, dtype: str = "f32", chunk: int = 1 << 24) -> torch.Tensor:
    """N(0, std^2) of the given shape, seeded by ``parts``; drawn in float32 chunks, then cast."""
    g = torch.Generator().manual_seed(sub_seed(*parts))
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=_DT[dtype])
    for i in range(0, n, chunk):
        k = min(chunk, n - i)
        out[i:i + k] = (torch.randn(k, generator=g, dtype=torch.float32) * std).to(out.dtype)
    return out.view(*shape)


def draw_group(w: Workload, group: int, *, with_noise: bool = True) -> dict:
    """Raw draws of one layer group: coefficients, and per layer basis, predictor weights, value noise.

    Coefficients are returned in float32 (the value before storage) and the rest in the activation
    dtype (noise in float32).
    """
    key = (w.seed, w.name, group)
    out = {
        "coef": gaussian((w.B, w.T, w.r), 1.0, *key, "coef", dtype="f32"),
        "basis": [], "w1": [], "w2": [], "noise": [],
    }
    for li in range(w.G):
        lk = key + (li,)
        out["basis"].append(gaussian((w.H_kv * w.d, w.r), w.r ** -0.5, *lk, "basis", dtype=w.act))
        out["w1"].append(gaussian((w.H_kv, w.m, w.d), w.d ** -0.5, *lk, "w1", dtype=w.act))
        out["w2"].append(gaussian((w.H_kv, w.d, w.m), w.m ** -0.5, *lk, "w2", dtype=w.act))
        if with_noise:
            out["noise"].append(gaussian((w.B, w.T, w.H_kv, w.d), 0.3, *lk, "noise", dtype="f32"))
    return out


def draw_query(w: Workload, layer: int, step: int = 0) -> torch.Tensor:
    return gaussian((w.B, w.H_q, w.d), w.d ** -0.5, w.seed, w.name, "q", layer, step, dtype=w.act)


def eviction_positions(w: Workload, n_sink: int = 64, n_recent: int = 2048) -> torch.Tensor:
    """Kept positions [B, T] (int32, ascending): sinks, the most recent tokens, and seeded uniform picks
    without replacement from the middle, to w.T kept out of w.T_nominal."""
    Tn, T = w.T_nominal, w.T
    assert Tn >= T >= n_sink + n_recent
    rows = []
    for b in range(w.B):
        g = torch.Generator().manual_seed(sub_seed(w.seed, w.name, "evict", b))
        mid = torch.randperm(Tn - n_recent - n_sink, generator=g)[: T - n_sink - n_recent] + n_sink
        keep = torch.cat([torch.arange(n_sink), mid, torch.arange(Tn - n_recent, Tn)])
        rows.append(torch.sort(keep).values)
    return torch.stack(rows).to(torch.int32).contiguous()


def placeholder_residuals(w: Workload, layer: int, scale: float = 0.3):
    """A valid residual list not produced by any compression: n_res distinct ascending token indices per
    (sequence, kv-head), drawn uniformly, with N(0, scale^2) rows.  For decode-only tests."""
    n = w.n_res
    idx = torch.empty((w.B, w.H_kv, n), dtype=torch.int32)
    for b in range(w.B):
        for h in range(w.H_kv):
            g = torch.Generator().manual_seed(sub_seed(w.seed, w.name, "resplace", layer, b, h))
            idx[b, h] = torch.sort(torch.randperm(w.T, generator=g)[:n]).values.to(torch.int32)
    val = gaussian((w.B, w.H_kv, n, w.d), scale, w.seed, w.name, "resval", layer, dtype="f32")
    return idx, val
