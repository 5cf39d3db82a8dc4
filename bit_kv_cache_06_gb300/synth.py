"""Seeded synthetic workloads shaped like the pages' Llama-style attention layers.

This module holds workload shapes and random-number recipes only -- none of
the quantisation or attention arithmetic.  The tests and the benchmark feed
the same tensors from here to both the CUDA library and the CPU oracle.

Shapes: "KV Cache Quantization (KIVI & FP4)", section 1 (Llama-3-70B: 8 KV
heads, head_dim 128, GQA 8:1) and "09 -- KV Cache Quantization", "The number
that motivates everything" (Llama-3-8B: 32 layers, 8 KV heads, head_dim 128).
Outlier structure: "09 -- KV Cache Quantization", "The structural fact that
makes KV quant work" (a few key channels 50-100x larger, consistently across
tokens; value tokens 100-1000x larger than the median).

Recipe: K, V, q ~ N(0, 1) in fp32, outliers multiplied in, then rounded to
fp16.  Seed = 1000 * config_index + layer; outlier positions come from a
second generator seeded with seed + 500000.  The pages' own evaluations use
real models on public suites; these tensors stand in for them.
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                  # config index (seed base)
    B: int
    Hq: int
    Hkv: int
    d: int
    T: int                      # tokens handed to the prefill quantiser
    bits: int
    G: int
    R: int
    steps: int = 1              # decode steps (append + attention) after prefill
    layers: int = 1
    # key outliers: either a count of channels per kv head or a fraction of d
    k_outlier_count: Optional[int] = None
    k_outlier_frac: float = 0.0
    k_outlier_mult: float = 1.0
    # value outliers: a count of tokens per pair, a Bernoulli rate per
    # (batch, head, token), and/or the first (sink) token
    v_outlier_count: int = 0
    v_outlier_prob: float = 0.0
    v_outlier_mult: float = 1.0
    v_sink_mult: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def pairs(self) -> int:
        return self.B * self.Hkv

    def capacity(self) -> int:
        """Quantised-token capacity needed for the prefill plus all steps."""
        n = self.T + self.steps
        cap = ((n + self.R - 1) // self.R) * self.R
        return max(cap, self.R)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


C1 = Workload("tiny-2bit", 1, B=1, Hq=4, Hkv=1, d=128, T=288, bits=2, G=32, R=32,
              k_outlier_count=4, k_outlier_mult=50.0,
              v_outlier_count=2, v_outlier_mult=100.0)
C2 = Workload("llama3-8b-layer-32k-2bit", 2, B=8, Hq=32, Hkv=8, d=128, T=32768, bits=2,
              G=32, R=128, k_outlier_frac=0.02, k_outlier_mult=50.0,
              v_outlier_prob=0.005, v_outlier_mult=200.0)
C3 = Workload("streaming-4bit-8k", 3, B=32, Hq=32, Hkv=8, d=128, T=8192, bits=4, G=64,
              R=128, steps=256, k_outlier_frac=0.02, k_outlier_mult=50.0,
              v_outlier_prob=0.005, v_outlier_mult=200.0)
C4 = Workload("llama3-70b-layer-1m-2bit", 4, B=1, Hq=64, Hkv=8, d=128, T=1048576, bits=2,
              G=32, R=128, k_outlier_count=1, k_outlier_mult=100.0, v_sink_mult=1000.0)
C5 = Workload("llama3-8b-32layer-sweep", 5, B=1, Hq=32, Hkv=8, d=128, T=4096, bits=2, G=32,
              R=128, layers=32, k_outlier_frac=0.02, k_outlier_mult=50.0,
              v_outlier_prob=0.005, v_outlier_mult=200.0)
C5_BATCHES = (1, 16, 64)
C5_CONTEXTS = (4096, 32768, 131072)
C5_BITS = (2, 4)

CONFIGS = {"c1": C1, "c2": C2, "c3": C3, "c4": C4, "c5": C5}


def _gens(w: Workload, layer: int, device) -> Tuple[torch.Generator, torch.Generator]:
    seed = 1000 * w.index + layer
    dev = torch.device(device)
    g_val = torch.Generator(device=dev)
    g_val.manual_seed(seed)
    g_pos = torch.Generator(device="cpu")   # outlier positions: always host-side
    g_pos.manual_seed(seed + 500000)
    return g_val, g_pos


def k_outlier_channels(w: Workload, layer: int = 0) -> torch.Tensor:
    """[Hkv, n] channel indices scaled by k_outlier_mult (fixed per kv head)."""
    _, g_pos = _gens(w, layer, "cpu")
    n = w.k_outlier_count if w.k_outlier_count is not None else round(w.k_outlier_frac * w.d)
    if n <= 0:
        return torch.zeros((w.Hkv, 0), dtype=torch.long)
    return torch.stack([torch.randperm(w.d, generator=g_pos)[:n] for _ in range(w.Hkv)])


def _channel_mult(w: Workload, layer: int, device) -> torch.Tensor:
    mult = torch.ones((w.Hkv, w.d), dtype=torch.float32)
    ch = k_outlier_channels(w, layer)
    for h in range(w.Hkv):
        mult[h, ch[h]] = w.k_outlier_mult
    return mult.to(device)


def make_kv(w: Workload, layer: int = 0, device="cpu", T: Optional[int] = None):
    """Prefill K, V: fp16 [B, Hkv, T, d] with the workload's outliers."""
    T = w.T if T is None else T
    g_val, g_pos = _gens(w, layer, device)
    kmult = _channel_mult(w, layer, device)
    K = torch.empty((w.B, w.Hkv, T, w.d), dtype=torch.float16, device=device)
    V = torch.empty_like(K)
    # generate in slices of pairs to bound fp32 temporaries (<= 2^27 elements)
    chunk_pairs = max(1, (1 << 27) // max(1, T * w.d))
    flatK = K.view(w.pairs, T, w.d)
    flatV = V.view(w.pairs, T, w.d)
    for p0 in range(0, w.pairs, chunk_pairs):
        p1 = min(w.pairs, p0 + chunk_pairs)
        k = torch.randn((p1 - p0, T, w.d), generator=g_val, device=device)
        heads = torch.arange(p0, p1, device=device) % w.Hkv
        k.mul_(kmult[heads].unsqueeze(1))
        flatK[p0:p1].copy_(k)
        del k
        v = torch.randn((p1 - p0, T, w.d), generator=g_val, device=device)
        flatV[p0:p1].copy_(v)
        del v
    # value outliers
    if w.v_outlier_count > 0:
        for p in range(w.pairs):
            toks = torch.randperm(T, generator=g_pos)[: w.v_outlier_count]
            flatV[p, toks.to(device)] = (flatV[p, toks.to(device)].float()
                                         * w.v_outlier_mult).half()
    if w.v_outlier_prob > 0:
        for p in range(w.pairs):
            sel = torch.rand(T, generator=g_pos) < w.v_outlier_prob
            idx = sel.nonzero().flatten().to(device)
            if idx.numel():
                flatV[p, idx] = (flatV[p, idx].float() * w.v_outlier_mult).half()
    if w.v_sink_mult:
        flatV[:, 0] = (flatV[:, 0].float() * w.v_sink_mult).half()
    return K, V


def make_q(w: Workload, step: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """Decode query: fp16 [B, Hq, d] ~ N(0, 1)."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(1000 * w.index + layer + 7919 * (step + 1))
    return torch.randn((w.B, w.Hq, w.d), generator=g, device=device).half()


def make_token(w: Workload, step: int, layer: int = 0, device="cpu"):
    """One streamed decode token: k, v fp16 [B, Hkv, d] with the same key
    outlier channels as the prefill and the same value-outlier rate."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(1000 * w.index + layer + 104729 * (step + 1))
    k = torch.randn((w.B, w.Hkv, w.d), generator=g, device=device)
    k.mul_(_channel_mult(w, layer, device).unsqueeze(0))
    v = torch.randn((w.B, w.Hkv, w.d), generator=g, device=device)
    if w.v_outlier_prob > 0:
        gp = torch.Generator(device="cpu")
        gp.manual_seed(1000 * w.index + layer + 104729 * (step + 1) + 500000)
        sel = (torch.rand((w.B, w.Hkv), generator=gp) < w.v_outlier_prob).to(device)
        v[sel] *= w.v_outlier_mult
    return k.half(), v.half()


def to_bthd(x: torch.Tensor) -> torch.Tensor:
    """[B, Hkv, T, d] -> contiguous [B, T, Hkv, d]."""
    return x.transpose(1, 2).contiguous()
