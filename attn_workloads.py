"""Seeded synthetic workloads for streaming attention: shapes and input generators only.

This module holds no attention arithmetic.  It is the one module that both the CUDA
path's tests/benchmark and the fp64 oracle's checks take their inputs from, so that both
sides see the same bytes.

All values are drawn on the CPU with an explicit torch.Generator (fp32 standard normal),
then cast to the stored dtype (bf16 with round-to-nearest-even, or kept fp32).  The
workload shapes follow the Llama3-70B dimensions (Hq = 64, Hkv = 8, G = 8, d = 128) that
"ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)" section 0 takes as its reference
model.  The pages use no public dataset; these synthetic tensors stand in for post-RoPE
Q/K/V.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: str           # "bf16" or "fp32"
    Sq: int = 1          # prefill query length (decode: 1)
    Skv: int = 0         # prefill key length; decode: the cache capacity Lmax
    causal: bool = False
    q_scale: float = 1.0  # Q multiplied by this after drawing (sharpens the softmax)
    num_splits: int = 0   # decode: fixed split count, 0 = automatic per length
    len_lo: int = 0       # decode: kv lengths uniform in [len_lo, len_hi] (equal: fixed)
    len_hi: int = 0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five reference workloads (seed = 1000 + index).
WORKLOADS = {
    1: Workload("tiny-fp32-noncausal", "prefill", B=1, Hq=2, Hkv=1, d=64, dtype="fp32",
                Sq=128, Skv=128, causal=False, seed=1001),
    2: Workload("causal-gqa-prefill-b2-h8-s2048", "prefill", B=2, Hq=8, Hkv=2, d=128,
                dtype="bf16", Sq=2048, Skv=2048, causal=True, seed=1002),
    3: Workload("llama3-70b-causal-prefill-s8192", "prefill", B=1, Hq=64, Hkv=8, d=128,
                dtype="bf16", Sq=8192, Skv=8192, causal=True, q_scale=2.0, seed=1003),
    4: Workload("llama3-70b-decode-b4-l32768-splits16", "decode", B=4, Hq=64, Hkv=8, d=128,
                dtype="bf16", Skv=32768, num_splits=16, len_lo=32768, len_hi=32768,
                seed=1004),
    5: Workload("ragged-decode-b16-l1024-131072-auto", "decode", B=16, Hq=64, Hkv=8, d=128,
                dtype="bf16", Skv=131072, num_splits=0, len_lo=1024, len_hi=131072,
                seed=1005),
}


# Beyond the five reference workloads: chunked prefill of a Llama3-70B-shaped context
# (a 2048-token chunk at the end of a 16384-token context held in a 32768-row cache), and
# multi-token decode.
EXTRA_WORKLOADS = {
    6: Workload("llama3-70b-chunked-prefill-q2048-ctx16384", "chunk", B=1, Hq=64, Hkv=8, d=128,
                dtype="bf16", Sq=2048, Skv=32768, causal=True, len_lo=16384, len_hi=16384,
                seed=1006),
    # speculative decode: 4 new tokens per sequence against a 32768-key cache
    7: Workload("llama3-70b-multitoken-decode-b4-tq4-l32768", "multitoken", B=4, Hq=64, Hkv=8,
                d=128, dtype="bf16", Sq=4, Skv=32768, num_splits=16, len_lo=32768,
                len_hi=32768, seed=1007),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "fp32":
        return x.to(torch.float32)
    raise ValueError(dtype)


def prefill_inputs(w: Workload):
    """Q [B,Hq,Sq,d], K and V [B,Hkv,Skv,d] (contiguous BHSD) as CPU tensors."""
    g = _gen(w.seed)
    q = torch.randn((w.B, w.Hq, w.Sq, w.d), generator=g, dtype=torch.float32)
    if w.q_scale != 1.0:
        q.mul_(w.q_scale)
    k = torch.randn((w.B, w.Hkv, w.Skv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Skv, w.d), generator=g, dtype=torch.float32)
    return _cast(q, w.dtype), _cast(k, w.dtype), _cast(v, w.dtype)


def decode_lengths(w: Workload) -> torch.Tensor:
    """Per-sequence KV lengths (int32 [B]): fixed, or uniform in [len_lo, len_hi]."""
    g = _gen(w.seed)
    if w.len_lo == w.len_hi:
        return torch.full((w.B,), w.len_hi, dtype=torch.int32)
    return torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=g, dtype=torch.int64).to(
        torch.int32)


def decode_inputs(w: Workload, pad_value: float = float("nan")):
    """Q [B,Hq,1,d], K/V caches [B,Hkv,Lmax,d], kv_lens int32 [B] as CPU tensors.

    Only the first kv_lens[b] rows of each cache are drawn; the rows past them are filled
    with `pad_value` (NaN by default, so that a kernel that reads past a sequence's
    length corrupts its output)."""
    lens = decode_lengths(w)
    g = _gen(w.seed + 7919)
    q = _cast(torch.randn((w.B, w.Hq, 1, w.d), generator=g, dtype=torch.float32), w.dtype)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    kc = torch.empty((w.B, w.Hkv, w.Skv, w.d), dtype=tdt)
    vc = torch.empty((w.B, w.Hkv, w.Skv, w.d), dtype=tdt)
    for b in range(w.B):
        n = int(lens[b])
        kc[b, :, :n] = _cast(torch.randn((w.Hkv, n, w.d), generator=g), w.dtype)
        vc[b, :, :n] = _cast(torch.randn((w.Hkv, n, w.d), generator=g), w.dtype)
        if n < w.Skv:
            kc[b, :, n:] = pad_value
            vc[b, :, n:] = pad_value
    return q, kc, vc, lens


def chunk_inputs(w: Workload, pad_value: float = float("nan")):
    """Chunked prefill: Q [B,Hq,Sq,d] and caches [B,Hkv,Lmax,d] (Lmax = w.Skv) whose first
    w.len_hi rows are drawn; the rest hold `pad_value` (NaN: any read of them shows)."""
    ctx = w.len_hi
    g = _gen(w.seed)
    q = _cast(torch.randn((w.B, w.Hq, w.Sq, w.d), generator=g, dtype=torch.float32), w.dtype)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    kc = torch.full((w.B, w.Hkv, w.Skv, w.d), pad_value, dtype=tdt)
    vc = torch.full((w.B, w.Hkv, w.Skv, w.d), pad_value, dtype=tdt)
    kc[:, :, :ctx] = _cast(torch.randn((w.B, w.Hkv, ctx, w.d), generator=g), w.dtype)
    vc[:, :, :ctx] = _cast(torch.randn((w.B, w.Hkv, ctx, w.d), generator=g), w.dtype)
    return q, kc, vc, ctx


def multitoken_inputs(w: Workload, pad_value: float = float("nan")):
    """Multi-token decode: Q [B,Hq,Tq,d] (Tq = w.Sq), caches [B,Hkv,Lmax,d], kv_lens [B]."""
    lens = decode_lengths(w)
    g = _gen(w.seed + 7919)
    q = _cast(torch.randn((w.B, w.Hq, w.Sq, w.d), generator=g, dtype=torch.float32), w.dtype)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    kc = torch.empty((w.B, w.Hkv, w.Skv, w.d), dtype=tdt)
    vc = torch.empty((w.B, w.Hkv, w.Skv, w.d), dtype=tdt)
    for b in range(w.B):
        n = int(lens[b])
        kc[b, :, :n] = _cast(torch.randn((w.Hkv, n, w.d), generator=g), w.dtype)
        vc[b, :, :n] = _cast(torch.randn((w.Hkv, n, w.d), generator=g), w.dtype)
        if n < w.Skv:
            kc[b, :, n:] = pad_value
            vc[b, :, n:] = pad_value
    return q, kc, vc, lens


def to_oracle(x: torch.Tensor) -> np.ndarray:
    """The stored bytes as the oracle takes them: fp32 as float32, bf16 as uint16 bits."""
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    if x.dtype == torch.float32:
        return x.numpy()
    raise TypeError(x.dtype)
