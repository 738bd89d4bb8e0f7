"""A slow NumPy model of the blocked forward with delayed (conditional) rescaling.

Test infrastructure, like the rest of ``oracle/``. It is NOT the oracle's
definition of the result (that is the two-pass fp64 code in ``attn_oracle.c``);
it replays the per-row update the pages describe so that tests can

* check the update against the pages' hand-worked numbers (the two-round
  example of "FlashAttention：一次前向计算" and exercise 1 of "Flash Attention 4"),
* show that the final O and LSE do not depend on the threshold tau, and
* attribute a GPU difference to the algorithm, to bf16 rounding of P, or to
  the exponential.

The update follows "Flash Attention 4", section "算法结构" (algorithm
structure), pseudo-code for one query block, with the -inf-safe reference of
the softmax code in section "QKᵀ MMA 与 PV MMA":

    candidate = max(row_max, rowmax(S))          (raw, unscaled scores)
    first block:  ref = candidate, acc_scale = 1
    otherwise:    delta = (row_max - safe(candidate)) * scale_log2   (<= 0)
                  delta >= -tau -> ref = row_max,   acc_scale = 1
                  delta <  -tau -> ref = candidate, acc_scale = exp2(delta)
    P       = exp2((S - safe(ref)) * scale_log2)      safe(x) = 0 if x == -inf else x
    row_sum = row_sum * acc_scale + rowsum(P)         (P before any rounding)
    O       = O * acc_scale + P @ V_block             (O = P @ V_block on the first block)

and the final step O / row_sum (0 where row_sum == 0) with
LSE = ln(row_sum) + ref * scale_log2 * ln(2)  (section "重缩放与结果写回").
tau = 0 is the standard online softmax of "FlashAttention：一次前向计算",
section "将刚才的过程写成通用更新" (rescale on every increase of the max).
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)
LOG2E = 1.0 / LN2


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), computed in float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 keeps 8 significant bits: scale the mantissa to an integer in [128, 256)
    r = np.round(m * 256.0) / 256.0   # numpy rounds half to even
    return np.ldexp(r, e)


def online_softmax_rows(q, k, v, *, scale_log2: float, block_n: int, tau: float = 8.0,
                        causal: bool = False, row0: int = 0, off: int = 0,
                        reverse: bool = True, dtype=np.float64, p_round: str | None = None,
                        exp2=None, init=None, trace: bool = False):
    """Run the blocked update for query rows q [M,d] against k, v [Nkv,d].

    Query row m has position row0 + m; with ``causal`` it sees keys j <= row0 + m + off.
    ``init`` = (row_max [M], row_sum [M], O [M,d]) starts from an existing state
    (then no block is treated as the first one). ``p_round='bf16'`` rounds P to
    bf16 before the P @ V product (row_sum still uses the unrounded P).
    Returns (O [M,d], LSE [M]) or, with ``trace``, (O, LSE, states) where states
    holds per block the reference, acc_scale, row_sum and the unnormalised O.
    """
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    M, d = q.shape
    nkv = k.shape[0]
    sl2 = dtype(scale_log2)
    ex2 = exp2 if exp2 is not None else (lambda x: np.exp2(x))
    n_blocks = (nkv + block_n - 1) // block_n
    if causal:
        last_key = row0 + (M - 1) + off           # largest key any row may see
        n_blocks = min(n_blocks, max(0, (last_key + block_n) // block_n))
    order = range(n_blocks - 1, -1, -1) if reverse else range(n_blocks)

    if init is not None:
        row_max = np.array(init[0], dtype=dtype).reshape(M)
        row_sum = np.array(init[1], dtype=dtype).reshape(M)
        O = np.array(init[2], dtype=dtype).reshape(M, d)
        first = False
    else:
        row_max = np.full(M, -np.inf, dtype=dtype)
        row_sum = np.zeros(M, dtype=dtype)
        O = np.zeros((M, d), dtype=dtype)
        first = True
    states = []
    qpos = row0 + np.arange(M)
    for j in order:
        k0 = j * block_n
        kb = k[k0:k0 + block_n]
        vb = v[k0:k0 + block_n]
        S = q @ kb.T
        kpos = k0 + np.arange(kb.shape[0])
        if causal:
            S = np.where(kpos[None, :] <= (qpos[:, None] + off), S, -np.inf)
        blk_max = S.max(axis=1) if S.shape[1] else np.full(M, -np.inf, dtype=dtype)
        cand = np.maximum(row_max, blk_max) if not first else blk_max
        if first:
            ref = cand
            acc = np.ones(M, dtype=dtype)
        else:
            cand_safe = np.where(cand == -np.inf, dtype(0), cand)
            with np.errstate(invalid="ignore"):
                delta = (row_max - cand_safe) * sl2
            keep = delta >= -dtype(tau)
            ref = np.where(keep, row_max, cand)
            acc = np.where(keep, dtype(1), ex2(np.where(keep, dtype(0), delta)).astype(dtype))
        ref_safe = np.where(ref == -np.inf, dtype(0), ref)
        P = ex2(S * sl2 - (ref_safe * sl2)[:, None]).astype(dtype)
        row_sum = row_sum * acc + P.sum(axis=1)
        Pm = _round_bf16(P).astype(dtype) if p_round == "bf16" else P
        if first:
            O = Pm @ vb
        else:
            O = O * acc[:, None] + Pm @ vb
        row_max = ref
        first = False
        if trace:
            states.append({"block": j, "ref": row_max.copy(), "acc_scale": acc.copy(),
                           "row_sum": row_sum.copy(), "O": O.copy()})
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(row_sum[:, None] != 0, O / np.where(row_sum == 0, 1, row_sum)[:, None], 0)
        lse = np.where(row_sum != 0,
                       np.log(np.where(row_sum == 0, 1, row_sum)) + row_max * sl2 * dtype(LN2),
                       -np.inf)
    if trace:
        return out, lse, states
    return out, lse
