"""Seeded synthetic inputs for scaled dot-product attention workloads.

This module only draws random numbers and shapes them. It computes nothing
of attention itself, so both the float64 oracle (through the tests) and the
CUDA path (through the tests and the benchmark) can take their inputs from
here without sharing any of the method's arithmetic.

Recipe (the same for every workload):
  * one CPU ``torch.Generator`` seeded with ``seed`` (default 0);
  * draw order: Q, K, V, dO, then (masked workload only) the per-batch
    valid lengths, the N(0, 0.5) bias, the 10 % Bernoulli blocks and the
    fully masked rows;
  * values are drawn in float32 N(0, 1) and, for bf16 workloads, rounded to
    bfloat16 (round to nearest even), so the oracle and the GPU see the
    very same numbers;
  * the additive mask is float32, ``-inf`` where blocked.

Workload shapes follow the five benchmark configurations of this project
(tiny fp32, MHA causal E=64, GQA causal E=128, padded + additive mask,
GQA decode), plus two that use padding lengths and a diagonal band instead of
a mask: the padded workload's shapes and lengths as seq_len_q = seq_len_kv
(no mask tensor), and the GQA causal workload with a sliding window.  Their
lengths are drawn at the padded workload's place in the draw order (after
Q, K, V, dO) with the same distribution.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "make_band", "make_padded_bias_mask"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    S: int
    E: int
    Ev: int
    dtype: str              # "f32" or "bf16"
    is_causal: bool
    enable_gqa: bool
    scale: Optional[float]  # None: the library default 1/sqrt(E)
    mask: str               # "none" or "padded_bias"
    phases: tuple           # ("fwd", "bwd") or ("fwd",)
    description: str = ""
    band: str = "none"      # "none", "seqlen" (lengths U{256..S} as seq_len_q = seq_len_kv) or "window"
    window: int = 0         # left bound of the "window" band (causal about the top-left diagonal)
    dropout: float = 0.0    # attention dropout probability (seed 0, offset 0)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def flops(self, phase: str) -> float:
        """Nominal FLOPs: 4*B*Hq*L*S*E forward, 10*B*Hq*L*S*E backward, halved when causal."""
        base = self.B * self.Hq * self.L * self.S * self.E
        f = {"fwd": 4.0, "bwd": 10.0}[phase] * base
        return f / 2.0 if self.is_causal else f

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", B=2, Hq=2, Hkv=2, L=64, S=64, E=16, Ev=16, dtype="f32",
        is_causal=False, enable_gqa=False, scale=1.0 / math.sqrt(16), mask="none",
        phases=("fwd", "bwd"),
        description="tiny fp32 forward+backward, no mask"),
    "tiny_f32_causal": Workload(
        "tiny_f32_causal", B=2, Hq=2, Hkv=2, L=64, S=64, E=16, Ev=16, dtype="f32",
        is_causal=True, enable_gqa=False, scale=1.0 / math.sqrt(16), mask="none",
        phases=("fwd", "bwd"),
        description="tiny fp32 forward+backward, causal"),
    "mha_causal_e64": Workload(
        "mha_causal_e64", B=4, Hq=16, Hkv=16, L=1024, S=1024, E=64, Ev=64, dtype="bf16",
        is_causal=True, enable_gqa=False, scale=1.0 / 8.0, mask="none",
        phases=("fwd", "bwd"),
        description="MHA causal bf16 training step"),
    "gqa_causal_e128": Workload(
        "gqa_causal_e128", B=2, Hq=32, Hkv=8, L=4096, S=4096, E=128, Ev=128, dtype="bf16",
        is_causal=True, enable_gqa=True, scale=1.0 / math.sqrt(128), mask="none",
        phases=("fwd", "bwd"),
        description="LLaMA-style GQA causal bf16 forward+backward"),
    "padded_mask_e128": Workload(
        "padded_mask_e128", B=8, Hq=16, Hkv=16, L=2048, S=2048, E=128, Ev=128, dtype="bf16",
        is_causal=False, enable_gqa=False, scale=None, mask="padded_bias",
        phases=("fwd", "bwd"),
        description="padded variable-length with an additive fp32 mask"),
    "padded_seqlen_e128": Workload(
        "padded_seqlen_e128", B=8, Hq=16, Hkv=16, L=2048, S=2048, E=128, Ev=128, dtype="bf16",
        is_causal=False, enable_gqa=False, scale=None, mask="none", phases=("fwd", "bwd"),
        description="padded variable-length batch given as seq_len_q / seq_len_kv (no mask tensor)",
        band="seqlen"),
    "gqa_swa_e128": Workload(
        "gqa_swa_e128", B=2, Hq=32, Hkv=8, L=4096, S=4096, E=128, Ev=128, dtype="bf16",
        is_causal=False, enable_gqa=True, scale=1.0 / math.sqrt(128), mask="none", phases=("fwd", "bwd"),
        description="GQA causal bf16 with a sliding window of 1024 keys", band="window", window=1024),
    "gqa_causal_dropout_e128": Workload(
        "gqa_causal_dropout_e128", B=2, Hq=32, Hkv=8, L=4096, S=4096, E=128, Ev=128, dtype="bf16",
        is_causal=True, enable_gqa=True, scale=1.0 / math.sqrt(128), mask="none", phases=("fwd", "bwd"),
        description="the GQA causal workload with attention dropout p = 0.1", dropout=0.1),
    "gqa_decode_s32k": Workload(
        "gqa_decode_s32k", B=16, Hq=32, Hkv=8, L=1, S=32768, E=128, Ev=128, dtype="bf16",
        is_causal=False, enable_gqa=True, scale=1.0 / math.sqrt(128), mask="none",
        phases=("fwd",),
        description="GQA decode, one query token against a 32k KV cache"),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _randn(gen: torch.Generator, shape, dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    return x.to(dtype)


def make_padded_bias_mask(gen: torch.Generator, B: int, L: int, S: int,
                          min_len: int = 256, p_block: float = 0.10,
                          frac_rows: float = 0.01):
    """Additive float32 mask [B, 1, L, S] of the padded workload.

    * valid key length len_b ~ U{min_len, ..., S} per batch; keys j >= len_b are -inf;
    * a N(0, 0.5) bias (0.5 is the standard deviation) everywhere else;
    * each (b, i, j) element independently blocked (-inf) with probability p_block;
    * floor(frac_rows * L) query rows per batch, drawn without replacement,
      blocked entirely (every key -inf).
    Query rows past len_b are not masked: they attend to the valid keys.
    Returns (mask, lengths).
    """
    lengths = torch.randint(min_len, S + 1, (B,), generator=gen)
    bias = torch.randn(B, 1, L, S, generator=gen, dtype=torch.float32) * 0.5
    blocked = torch.rand(B, 1, L, S, generator=gen) < p_block
    n_rows = int(math.floor(frac_rows * L))
    ninf = float("-inf")
    bias[blocked] = ninf
    for b in range(B):
        bias[b, :, :, int(lengths[b]):] = ninf
        rows = torch.randperm(L, generator=gen)[:n_rows]
        bias[b, :, rows, :] = ninf
    return bias, lengths


def make_band(w: Workload, seed: int = 0):
    """The workload's padding lengths and band as a dict (None when it has none).

    Lengths are drawn with the generator advanced past Q, K, V and dO, exactly
    where the padded workload draws its lengths, from the same U{256, ..., S}.
    """
    if w.band == "none":
        return None
    if w.band == "window":
        return {"seq_len_q": None, "seq_len_kv": None, "alignment": "top_left", "right_bound": 0,
                "left_bound": w.window}
    gen = torch.Generator().manual_seed(seed)
    for shape in ((w.B, w.Hq, w.L, w.E), (w.B, w.Hkv, w.S, w.E), (w.B, w.Hkv, w.S, w.Ev), (w.B, w.Hq, w.L, w.Ev)):
        torch.randn(*shape, generator=gen)
    lengths = [int(x) for x in torch.randint(256, w.S + 1, (w.B,), generator=gen)]
    return {"seq_len_q": lengths, "seq_len_kv": lengths, "alignment": "top_left", "right_bound": None,
            "left_bound": None}


def make_inputs(w: Workload, seed: int = 0, with_grad: bool = True):
    """Draw (q, k, v, dO, mask) on the CPU for workload ``w``.

    q [B,Hq,L,E], k [B,Hkv,S,E], v [B,Hkv,S,Ev], dO [B,Hq,L,Ev] in the
    workload dtype (contiguous BHSD); mask float32 [B,1,L,S] or None.
    """
    gen = torch.Generator().manual_seed(seed)
    dt = w.torch_dtype
    q = _randn(gen, (w.B, w.Hq, w.L, w.E), dt)
    k = _randn(gen, (w.B, w.Hkv, w.S, w.E), dt)
    v = _randn(gen, (w.B, w.Hkv, w.S, w.Ev), dt)
    dO = _randn(gen, (w.B, w.Hq, w.L, w.Ev), dt) if with_grad else None
    mask = None
    if w.mask == "padded_bias":
        mask, _ = make_padded_bias_mask(gen, w.B, w.L, w.S)
    return q, k, v, dO, mask


def random_inputs(B, Hq, Hkv, L, S, E, Ev, dtype=torch.float32, seed=0,
                  mask_shape=None, mask_kind="none", p_block=0.25,
                  full_rows=0, scale_q=1.0):
    """Small seeded cases for tests: same draw rules, free shapes.

    mask_kind: "none"; "bias" (N(0,0.5) plus Bernoulli(p_block) -inf);
    "block" (0 or -inf only). ``full_rows`` query rows of the mask (for every
    broadcast index) are set to -inf entirely. ``scale_q`` multiplies Q
    before rounding (large scores for overflow tests).
    """
    gen = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, Hq, L, E, generator=gen) * scale_q).to(dtype)
    k = torch.randn(B, Hkv, S, E, generator=gen).to(dtype)
    v = torch.randn(B, Hkv, S, Ev, generator=gen).to(dtype)
    dO = torch.randn(B, Hq, L, Ev, generator=gen).to(dtype)
    mask = None
    if mask_kind != "none":
        mb, mh = mask_shape if mask_shape is not None else (B, 1)
        if mask_kind == "bias":
            mask = torch.randn(mb, mh, L, S, generator=gen) * 0.5
        else:
            mask = torch.zeros(mb, mh, L, S)
        blocked = torch.rand(mb, mh, L, S, generator=gen) < p_block
        mask[blocked] = float("-inf")
        if full_rows:
            rows = torch.randperm(L, generator=gen)[:full_rows]
            mask[:, :, rows, :] = float("-inf")
    return q, k, v, dO, mask
