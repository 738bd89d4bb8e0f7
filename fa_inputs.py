"""Seeded synthetic inputs for attention forward: Q, K, V as bf16 bit patterns.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``.
It draws random numbers, rounds them to bf16 and builds ``cu_seqlens``; it holds
none of the attention arithmetic, so both the CUDA path and the oracle can take
their inputs from here without sharing any of the method's code.

Recipe (the same bytes go to the GPU and to the oracle):

* one ``numpy.random.Generator(PCG64(seed))`` per workload; Q, K, V are drawn in
  that order as float32 ``standard_normal`` and rounded to bf16 with
  round-to-nearest-even;
* "spiky" inputs (the long causal workload that exercises the delayed rescale):
  Q is multiplied by 4 after rounding, and in every (batch, head) ceil(1% of N)
  key rows, drawn without replacement, are multiplied by 8. Both factors are
  powers of two, so the scaled values are still exact bf16 numbers;
* varlen: sequence lengths are uniform integers in [lo, hi] (inclusive) drawn
  before Q, K, V from the same generator, packed as [T, H, d].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # For every non-NaN float32 the sum below stays under 2**32.
    t = u >> np.uint32(16)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    out = t.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class Workload:
    """One attention forward problem, described by its shapes and input recipe."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    spiky: bool = False
    varlen_seqs: int = 0          # >0 selects the packed variable-length layout
    varlen_lo: int = 0
    varlen_hi: int = 0
    scale: float = field(default=float("nan"))

    def __post_init__(self):
        if math.isnan(self.scale):
            self.scale = 1.0 / math.sqrt(self.d)

    @property
    def varlen(self) -> bool:
        return self.varlen_seqs > 0


# The five workloads of the hot-path contract (seed 20260 + k for workload k).
WORKLOADS = {
    "c1_b1h1n256d64": Workload("c1_b1h1n256d64", B=1, H=1, N=256, d=64, causal=False, seed=20261),
    "c2_b2h8n1024d128": Workload("c2_b2h8n1024d128", B=2, H=8, N=1024, d=128, causal=False, seed=20262),
    "c3_b4h16n4096d128_causal": Workload("c3_b4h16n4096d128_causal", B=4, H=16, N=4096, d=128,
                                         causal=True, seed=20263),
    "c4_b1h32n16384d128_causal_spiky": Workload("c4_b1h32n16384d128_causal_spiky", B=1, H=32, N=16384,
                                                d=128, causal=True, seed=20264, spiky=True),
    "c5_varlen8_h16d128_causal": Workload("c5_varlen8_h16d128_causal", B=1, H=16, N=0, d=128, causal=True,
                                          seed=20265, varlen_seqs=8, varlen_lo=512, varlen_hi=8192),
}


def make_qkv(B: int, N: int, H: int, d: int, seed: int, spiky: bool = False,
             Nkv: int | None = None):
    """Q [B,N,H,d], K and V [B,Nkv,H,d] as bf16 bit patterns (uint16)."""
    Nkv = N if Nkv is None else Nkv
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (B, N, H, d))
    k = _normal_bf16(rng, (B, Nkv, H, d))
    v = _normal_bf16(rng, (B, Nkv, H, d))
    if spiky:
        q = f32_to_bf16_bits(bf16_bits_to_f32(q) * np.float32(4.0))
        kf = bf16_bits_to_f32(k)
        n_spike = int(math.ceil(0.01 * Nkv))
        for b in range(B):
            for h in range(H):
                rows = rng.choice(Nkv, size=n_spike, replace=False)
                kf[b, rows, h, :] *= np.float32(8.0)
        k = f32_to_bf16_bits(kf)
    return q, k, v


def make_varlen(num_seqs: int, lo: int, hi: int, H: int, d: int, seed: int):
    """Packed variable-length batch: (lengths, cu_seqlens int32 [S+1], q, k, v [T,H,d])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int64)
    return _pack_varlen(rng, lengths, H, d)


def make_varlen_from_lengths(lengths, H: int, d: int, seed: int):
    """Packed batch with the given sequence lengths (zero-length sequences allowed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _pack_varlen(rng, np.asarray(lengths, dtype=np.int64), H, d)


def _pack_varlen(rng, lengths, H, d):
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    q = _normal_bf16(rng, (T, H, d))
    k = _normal_bf16(rng, (T, H, d))
    v = _normal_bf16(rng, (T, H, d))
    return lengths, cu, q, k, v


def make_workload(w: Workload):
    """Inputs of a named workload: dict with q, k, v (and lengths, cu_seqlens for varlen)."""
    if w.varlen:
        lengths, cu, q, k, v = make_varlen(w.varlen_seqs, w.varlen_lo, w.varlen_hi, w.H, w.d, w.seed)
        return {"q": q, "k": k, "v": v, "lengths": lengths, "cu_seqlens": cu}
    q, k, v = make_qkv(w.B, w.N, w.H, w.d, w.seed, spiky=w.spiky)
    return {"q": q, "k": k, "v": v}


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Conventional forward FLOP count: 4*B*H*N^2*d, halved for causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def varlen_flops(lengths, H: int, d: int, causal: bool) -> float:
    return sum(attention_flops(1, H, int(L), d, causal) for L in lengths)
