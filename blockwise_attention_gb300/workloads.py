"""Seeded synthetic workloads shaped like the pages' attention settings.

This module only DRAWS inputs: shapes, value distributions, padding lengths and
the boolean masks that describe which (query, key) pairs a workload forbids.
It holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle may import it.

Recipe (every workload):
  * ``g = torch.Generator(device).manual_seed(1000 + index)``;
  * draw Q, K, V in that order with ``torch.randn`` (float32) times ``std``,
    then round to the workload dtype (RNE, torch's float32 -> bfloat16 cast);
  * then draw the per-batch valid lengths with ``torch.randint`` (inclusive
    range) when the workload pads keys; key j of batch b is padded iff
    ``j >= len_b`` (key_padding_mask, 1 = excluded);
  * the banded encoder mask forbids pairs with ``|i - j| > band`` unless the
    row or the column is the CLS position 0 (attn_mask, 1 = excluded).

Large workloads are drawn on the GPU with torch's device generator (the CPU
generator needs minutes for 3 x 268M values); the oracle then reads the very
same tensors back on the host.  Values therefore depend on the device the
generator runs on, never on the attention code.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int               # seed offset: seed = 1000 + index
    B: int
    H: int
    T: int
    d: int
    dtype: str               # "f32" or "bf16"
    std: float               # Q, K, V ~ N(0, 1) * std
    causal: bool
    P: int                   # emulated context-parallel ranks
    partition: str           # "contiguous" or "zigzag"
    rope_base: Optional[float] = None
    pad_len: Optional[tuple] = None   # (lo, hi) inclusive valid-length range
    band: Optional[int] = None        # |i-j| > band forbidden except CLS row/col 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the pages' settings (ring check, padded causal MHA with
# RoPE, zigzag prefill at 8K and 64K, banded bidirectional encoder).
WORKLOADS = {
    "tiny_ring_f32": Workload("tiny_ring_f32", 0, 1, 2, 8, 16, "f32", 1.0, False, 4,
                              "contiguous"),
    "causal_pad_rope_1k": Workload("causal_pad_rope_1k", 1, 2, 8, 1024, 64, "bf16", 1.0, True,
                                   4, "contiguous", rope_base=10000.0, pad_len=(512, 1024)),
    "zigzag_prefill_8k": Workload("zigzag_prefill_8k", 2, 4, 16, 8192, 128, "bf16", 0.5, True,
                                  8, "zigzag"),
    "zigzag_prefill_64k_rope": Workload("zigzag_prefill_64k_rope", 3, 1, 32, 65536, 128, "bf16",
                                        0.5, True, 16, "zigzag", rope_base=10000.0),
    "encoder_pad_band_512": Workload("encoder_pad_band_512", 4, 32, 16, 512, 64, "bf16", 1.0,
                                     False, 2, "contiguous", pad_len=(128, 512), band=64),
}


@dataclass
class Inputs:
    q: torch.Tensor                      # (B, H, T, d) in the workload dtype
    k: torch.Tensor
    v: torch.Tensor
    lengths: Optional[torch.Tensor]      # (B,) int64 valid key lengths, or None
    kpm: Optional[torch.Tensor]          # (B, T) uint8, 1 = padded key (excluded)
    am: Optional[torch.Tensor]           # (T, T) uint8, 1 = forbidden pair


def band_cls_mask(T: int, band: int, device="cpu") -> torch.Tensor:
    """(T, T) uint8: 1 where |i-j| > band and neither i nor j is position 0."""
    i = torch.arange(T, device=device).view(-1, 1)
    j = torch.arange(T, device=device).view(1, -1)
    m = ((i - j).abs() > band) & (i != 0) & (j != 0)
    return m.to(torch.uint8)


def padding_mask(lengths: torch.Tensor, T: int) -> torch.Tensor:
    """(B, T) uint8: 1 where key position j >= lengths[b]."""
    j = torch.arange(T, device=lengths.device).view(1, -1)
    return (j >= lengths.view(-1, 1)).to(torch.uint8)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> Inputs:
    """Draw the seeded inputs of workload ``w`` on ``device``."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(1000 + w.index if seed is None else seed)
    shape = (w.B, w.H, w.T, w.d)
    out = []
    for _ in range(3):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if w.std != 1.0:
            x.mul_(w.std)
        out.append(x.to(w.torch_dtype))
    q, k, v = out
    lengths = kpm = am = None
    if w.pad_len is not None:
        lo, hi = w.pad_len
        lengths = torch.randint(lo, hi + 1, (w.B,), generator=g, device=device)
        kpm = padding_mask(lengths, w.T)
    if w.band is not None:
        am = band_cls_mask(w.T, w.band, device=device)
    return Inputs(q, k, v, lengths, kpm, am)


@dataclass
class DecodeInputs:
    q: torch.Tensor          # (B, H, 1, d)
    k: torch.Tensor          # (B, H, S, d) cache
    v: torch.Tensor
    lengths: torch.Tensor    # int32 (B), valid cache lengths


# Decode workload (one query token per sequence against a long KV cache):
# B=8 sequences, H=32 heads, d=128, bf16, a 65536-slot cache per (b, h) whose
# valid length is drawn uniformly in [32768, 65536] per sequence.
DECODE = dict(B=8, H=32, S=65536, d=128, len_lo=32768, len_hi=65536, std=0.5, seed=2100)


def make_decode_inputs(device="cpu", seed: Optional[int] = None, **over) -> DecodeInputs:
    """Draw the seeded decode inputs (q, then the K cache, the V cache, then lengths)."""
    cfg = dict(DECODE, **over)
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] if seed is None else seed)
    B, H, S, d = cfg["B"], cfg["H"], cfg["S"], cfg["d"]
    q = (torch.randn((B, H, 1, d), generator=g, device=device) * cfg["std"]).to(torch.bfloat16)
    k = (torch.randn((B, H, S, d), generator=g, device=device) * cfg["std"]).to(torch.bfloat16)
    v = torch.randn((B, H, S, d), generator=g, device=device).to(torch.bfloat16)
    lengths = torch.randint(cfg["len_lo"], cfg["len_hi"] + 1, (B,), generator=g, device=device).to(torch.int32)
    return DecodeInputs(q, k, v, lengths)
