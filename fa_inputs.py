"""Seeded synthetic inputs for attention forward: Q, K, V as bf16 or fp16 bit patterns.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``.
It draws random numbers, rounds them to bf16 or fp16 and builds ``cu_seqlens``; it holds
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
  before Q, K, V from the same generator, packed as [T, H, d];
* grouped-query attention: K and V have H_kv heads (H a multiple of H_kv); the
  draws are the same with the K/V shapes changed;
* fp16 inputs: the same float32 draws rounded to IEEE binary16 (numpy's
  correctly rounded float32 -> float16 conversion, ties to even).
* tiled tensors (the maximum-size tests, whose tensors of 2^31 elements are too large
  to draw on the host): a table of ``TILE_ROWS`` (a prime) rows drawn as above from
  one seed; row r of the tensor, r the flat index over its leading dimensions in
  order, is table row (r * ``TILE_MULT``) mod ``TILE_ROWS``. The device copy is
  built by gathering table rows on the GPU, and any row can be rebuilt on the host.
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


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE fp16 (round to nearest, ties to even); return uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen fp16 bit patterns (uint16) to float32 exactly."""
    return np.ascontiguousarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    return f16_bits_to_f32(b) if dtype == "f16" else bf16_bits_to_f32(b)


def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_f16_bits(x) if dtype == "f16" else f32_to_bf16_bits(x)


def _normal(rng: np.random.Generator, shape, dtype: str = "bf16") -> np.ndarray:
    return f32_to_bits(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return _normal(rng, shape, "bf16")


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
    Hkv: int = 0                  # K/V heads (0: the same as H)
    dtype: str = "bf16"           # element type of Q, K, V and O: "bf16" or "f16"
    Nk: int = 0                   # key rows per sequence (0: the same as N)
    splits: int = 1               # key ranges per task passed to the library (0: its choice)

    def __post_init__(self):
        if math.isnan(self.scale):
            self.scale = 1.0 / math.sqrt(self.d)
        if self.Hkv == 0:
            self.Hkv = self.H
        if self.Nk == 0:
            self.Nk = self.N

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

# Grouped-query attention and fp16 inputs ("Flash Attention 4", sections "GQA 支持"
# and "编译与验证": 32 query heads over 8 K/V heads, fp16, non-causal, N = 1024), and
# the same grouping at the size of the long causal workloads.
WORKLOADS.update({
    "g1_gqa_b1h32kv8n1024d128_f16": Workload("g1_gqa_b1h32kv8n1024d128_f16", B=1, H=32, N=1024, d=128,
                                             causal=False, seed=20266, Hkv=8, dtype="f16"),
    "g2_gqa_b4h32kv8n4096d128_causal": Workload("g2_gqa_b4h32kv8n4096d128_causal", B=4, H=32, N=4096, d=128,
                                                causal=True, seed=20267, Hkv=8),
    "g3_gqa_varlen8_h32kv4d128_causal_f16": Workload("g3_gqa_varlen8_h32kv4d128_causal_f16", B=1, H=32, N=0,
                                                     d=128, causal=True, seed=20268, varlen_seqs=8,
                                                     varlen_lo=512, varlen_hi=8192, Hkv=4, dtype="f16"),
})

# Decoding against a long key/value cache: one new query row per sequence,
# grouped heads; the rows are few, so the keys are split into ranges that are
# merged through their LSE.
WORKLOADS.update({
    "d1_decode_b8h32kv8nq1nk32768d128": Workload("d1_decode_b8h32kv8nq1nk32768d128", B=8, H=32, N=1, d=128,
                                                 causal=True, seed=20269, Hkv=8, Nk=32768, splits=0),
})


def make_qkv(B: int, N: int, H: int, d: int, seed: int, spiky: bool = False,
             Nkv: int | None = None, Hkv: int | None = None, dtype: str = "bf16"):
    """Q [B,N,H,d], K and V [B,Nkv,Hkv,d] as bf16 or fp16 bit patterns (uint16)."""
    Nkv = N if Nkv is None else Nkv
    Hkv = H if Hkv is None else Hkv
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal(rng, (B, N, H, d), dtype)
    k = _normal(rng, (B, Nkv, Hkv, d), dtype)
    v = _normal(rng, (B, Nkv, Hkv, d), dtype)
    if spiky:
        q = f32_to_bits(bits_to_f32(q, dtype) * np.float32(4.0), dtype)
        kf = bits_to_f32(k, dtype)
        n_spike = int(math.ceil(0.01 * Nkv))
        for b in range(B):
            for h in range(Hkv):
                rows = rng.choice(Nkv, size=n_spike, replace=False)
                kf[b, rows, h, :] *= np.float32(8.0)
        k = f32_to_bits(kf, dtype)
    return q, k, v


def make_varlen(num_seqs: int, lo: int, hi: int, H: int, d: int, seed: int, Hkv: int | None = None,
                dtype: str = "bf16"):
    """Packed variable-length batch: (lengths, cu_seqlens int32 [S+1], q [T,H,d], k, v [T,Hkv,d])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int64)
    return _pack_varlen(rng, lengths, H, d, Hkv, dtype)


def make_varlen_from_lengths(lengths, H: int, d: int, seed: int, Hkv: int | None = None,
                             dtype: str = "bf16"):
    """Packed batch with the given sequence lengths (zero-length sequences allowed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _pack_varlen(rng, np.asarray(lengths, dtype=np.int64), H, d, Hkv, dtype)


def _pack_varlen(rng, lengths, H, d, Hkv=None, dtype="bf16"):
    Hkv = H if Hkv is None else Hkv
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    q = _normal(rng, (T, H, d), dtype)
    k = _normal(rng, (T, Hkv, d), dtype)
    v = _normal(rng, (T, Hkv, d), dtype)
    return lengths, cu, q, k, v


TILE_ROWS = 4099      # a prime, so the multiplier below visits every table row
TILE_MULT = 40503


def make_row_table(d: int, seed: int, dtype: str = "bf16") -> np.ndarray:
    """The table [TILE_ROWS, d] (16-bit bit patterns) that a tiled tensor's rows come from."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _normal(rng, (TILE_ROWS, d), dtype)


def tiled_row_ids(r) -> np.ndarray:
    """Table row of each flat row index r of a tiled tensor."""
    return (np.asarray(r, dtype=np.int64) * TILE_MULT) % TILE_ROWS


def tiled_rows(table: np.ndarray, r) -> np.ndarray:
    """Rows r of the tiled tensor built from table (host copy, 16-bit bit patterns)."""
    return table[tiled_row_ids(r)]


def tiled_tensor_cuda(table: np.ndarray, shape, dtype: str = "bf16"):
    """The whole tiled tensor of the given shape (its last dimension the table's width),
    gathered on the current CUDA device as a torch tensor of the 16-bit type."""
    import torch
    rows = math.prod(shape[:-1])
    t = torch.from_numpy(np.ascontiguousarray(table).view(np.int16)).cuda()
    ids = (torch.arange(rows, dtype=torch.int64, device=t.device) * TILE_MULT) % TILE_ROWS
    out = t[ids].view(*shape)
    del ids
    return out.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def make_workload(w: Workload):
    """Inputs of a named workload: dict with q, k, v (and lengths, cu_seqlens for varlen)."""
    if w.varlen:
        lengths, cu, q, k, v = make_varlen(w.varlen_seqs, w.varlen_lo, w.varlen_hi, w.H, w.d, w.seed,
                                           Hkv=w.Hkv, dtype=w.dtype)
        return {"q": q, "k": k, "v": v, "lengths": lengths, "cu_seqlens": cu}
    q, k, v = make_qkv(w.B, w.N, w.H, w.d, w.seed, spiky=w.spiky, Nkv=w.Nk, Hkv=w.Hkv, dtype=w.dtype)
    return {"q": q, "k": k, "v": v}


def attention_flops(B: int, H: int, N: int, d: int, causal: bool, Nk: int | None = None) -> float:
    """Conventional forward FLOP count: 4*B*H*N^2*d, halved for causal. With N_k keys
    (N_k != N), 4*d per visible (query, key) pair; bottom-right causal: query i sees
    min(i + N_k - N + 1, N_k) keys (at least 0)."""
    if Nk is None or Nk == N:
        f = 4.0 * B * H * N * N * d
        return f / 2 if causal else f
    if not causal:
        return 4.0 * B * H * N * Nk * d
    i = np.arange(N, dtype=np.float64)
    pairs = np.clip(i + (Nk - N) + 1, 0, Nk).sum()
    return 4.0 * B * H * d * float(pairs)


def varlen_flops(lengths, H: int, d: int, causal: bool) -> float:
    return sum(attention_flops(1, H, int(L), d, causal) for L in lengths)
