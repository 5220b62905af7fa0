"""Seeded synthetic inputs for the five workloads.

This module draws random numbers only: it holds none of the compression or
attention arithmetic.  Both the CUDA path and the CPU oracle are fed from here
(the oracle through host copies of the same tensors).  Model names describe
tensor shapes only; no model, weights or data set is involved.

Workloads (shapes and value laws):
  1  one layer, B=1, 8 KV heads x 128, 1024 tokens, N(0,1) with 4 outlier
     channels per head scaled x10; keys 4-bit, values 4-bit; 32 query heads.
  2  Llama-3-8B-shaped KV: 32 layers x 8 heads x 128, 32 query heads, B=1,
     context 16384; N(0,1) times a per-channel log-normal(0,1) scale drawn per
     (layer, head, channel) separately for K and V; keys 8-bit, values 3-bit;
     128 fp16 sink tokens; 64-token chunked compression; then decode steps.
  3  Qwen3-8B-shaped (36 layers x 8 x 128, 32 query heads), B=1, context 131072,
     tiers by age (fp16 / K4V4 / K3V2 / K2V1); N(0,1) with 1% of the (layer,
     head, channel) triples scaled x8.
  4  32 layers x 8 x 128, B=16, context 32768; per-(layer, head) bit widths drawn
     from {6-8: 20%, 3-4: 50%, 1-2: 30%} (uniform inside each band), the same
     width for K and V; QJL on heads with <= 2 bits; N(0,1).
  5  Mistral-Nemo-12B-shaped (40 layers x 8 x 128, 32 query heads), uniform
     K3/V3, 128 fp16 sinks, B in {1, 8, 32} x context in {4096, 16384, 65536};
     N(0,1) with 4 outlier channels per head x10.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
KV_HEADS = 8
Q_HEADS = 32
ROTATION_SEED = 42          # layer l uses ROTATION_SEED + l
QJL_SEED = 42 + 1000
BITS_SEED = 42 + 2000


@dataclass
class Workload:
    name: str
    layers: int
    batch: int
    context: int
    kv_heads: int = KV_HEADS
    q_heads: int = Q_HEADS
    head_dim: int = HEAD_DIM
    kbits: int | None = None        # uniform bits (None: per-head draw or tiers)
    vbits: int | None = None
    sinks: int = 0
    chunk: int = 0                  # chunked compression granularity (0: one shot)
    tiers: bool = False
    per_head_bits: bool = False
    qjl_max_bits: int = 0           # QJL on heads with kbits <= this (0: none)
    law: str = "outliers"           # value law, see kv_block()
    outlier_channels: int = 4
    outlier_scale: float = 10.0
    outlier_fraction: float = 0.0
    decode_steps: int = 1
    notes: dict = field(default_factory=dict)


WORKLOADS = {
    "w1": Workload("w1_single_layer_k4v4", layers=1, batch=1, context=1024, kbits=4, vbits=4,
                   law="outliers"),
    "w2": Workload("w2_llama3_8b_k8v3_sinks_chunked", layers=32, batch=1, context=16384,
                   kbits=8, vbits=3, sinks=128, chunk=64, law="lognormal_channels",
                   decode_steps=256),
    "w3": Workload("w3_qwen3_8b_tiers_131k", layers=36, batch=1, context=131072, tiers=True,
                   law="fraction_outliers", outlier_fraction=0.01, outlier_scale=8.0),
    "w4": Workload("w4_mixed_bits_qjl_b16", layers=32, batch=16, context=32768,
                   per_head_bits=True, qjl_max_bits=2, law="normal"),
    "w5": Workload("w5_mistral_nemo_12b_k3v3", layers=40, batch=32, context=65536, kbits=3,
                   vbits=3, sinks=128, law="outliers"),
}


def draw_head_bits(layers: int, heads: int, seed: int = BITS_SEED) -> np.ndarray:
    """Per-(layer, head) bit widths: band 6-8 w.p. 0.2, 3-4 w.p. 0.5, 1-2 w.p. 0.3,
    then uniform inside the band.  int [layers][heads]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    band = rng.choice(3, size=(layers, heads), p=[0.2, 0.5, 0.3])
    lo = np.array([6, 3, 1])[band]
    hi = np.array([8, 4, 2])[band]
    return (lo + np.floor(rng.random((layers, heads)) * (hi - lo + 1))).astype(np.int64)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def kv_block(w: Workload, layer: int, batch: int, tokens: int, seed: int,
             device="cpu", token_offset: int = 0):
    """fp16 K, V of shape [batch][kv_heads][tokens][head_dim] for one layer.

    The per-channel structure (outlier channels, log-normal scales) is drawn from
    a generator keyed by (seed, layer) only, so blocks of the same layer drawn at
    different token offsets share it; the N(0,1) body is keyed by the offset too."""
    H, d = w.kv_heads, w.head_dim
    body = _gen(seed * 1_000_003 + layer * 7919 + token_offset, device)
    K = torch.randn(batch, H, tokens, d, generator=body, device=device, dtype=torch.float32)
    V = torch.randn(batch, H, tokens, d, generator=body, device=device, dtype=torch.float32)
    chan = _gen(seed * 999_983 + layer, "cpu")
    if w.law == "outliers":
        for X in (K, V):
            scale = torch.ones(H, d)
            for h in range(H):
                idx = torch.randperm(d, generator=chan)[: w.outlier_channels]
                scale[h, idx] = w.outlier_scale
            X.mul_(scale.to(device)[None, :, None, :])
    elif w.law == "lognormal_channels":
        for X in (K, V):
            z = torch.randn(H, d, generator=chan)
            X.mul_(torch.exp(z).to(device)[None, :, None, :])
    elif w.law == "fraction_outliers":
        # round(fraction * layers * H * d) (layer, head, channel) triples overall,
        # drawn once for the whole model from the seed; this layer's share is applied.
        allg = _gen(seed * 131 + 17, "cpu")
        n = int(round(w.outlier_fraction * w.layers * H * d))
        pick = torch.randperm(w.layers * H * d, generator=allg)[:n]
        scale = torch.ones(w.layers * H * d)
        scale[pick] = w.outlier_scale
        scale = scale.view(w.layers, H, d)[layer]
        for X in (K, V):
            X.mul_(scale.to(device)[None, :, None, :])
    elif w.law == "normal":
        pass
    else:
        raise ValueError(w.law)
    return K.to(torch.float16), V.to(torch.float16)


def queries(w: Workload, layer: int, batch: int, seed: int, device="cpu", step: int = 0):
    """fp16 decode queries [batch][q_heads][head_dim], N(0,1)."""
    g = _gen(seed * 524_287 + layer * 31 + step * 1_000_033, device)
    return torch.randn(batch, w.q_heads, w.head_dim, generator=g, device=device).to(torch.float16)


def query_pool(w: Workload, steps: int, batch: int, seed: int, device="cpu"):
    """fp16 decode queries for `steps` steps of every layer: [steps][layers][batch][q_heads][head_dim]."""
    g = _gen(seed * 524_287 + 99, device)
    return torch.randn(steps, w.layers, batch, w.q_heads, w.head_dim, generator=g, device=device).to(
        torch.float16)


def tier_bits(tier: int):
    """(kbits, vbits) of the age tiers: 0 fp16, 1 K4V4, 2 K3V2, 3 K2V1."""
    return [(16, 16), (4, 4), (3, 2), (2, 1)][tier]
