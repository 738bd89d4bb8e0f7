"""Oracle merge of partial attention results over disjoint key sets (fp64, NumPy).

Test infrastructure only (see the package docstring).

If the keys of a row are split into parts s, and part s alone gives the
normalised output O_s and LSE_s = ln sum_{j in s} exp(t_j), then the attention
over all the keys is

    LSE = ln sum_s exp(LSE_s)
    O   = sum_s exp(LSE_s - LSE) * O_s

Parts with LSE_s = -inf (no valid key) contribute nothing; a row whose parts
are all -inf has O = 0 and LSE = -inf.

Sources: "FlashAttention：一次前向计算" (qingsen), the two-round example
(figs. 7-10): the results of two key blocks are merged by bringing both to a
common reference (the numerators and denominators of both rounds rescaled by
the same factor) and dividing once by the total denominator; with normalised
parts the common reference is the LSE, since exp(LSE_s) * O_s is part s's
numerator and exp(LSE_s) its denominator relative to reference 0. "Flash
Attention 4", section "重缩放与结果写回": LSE = ln(row_sum) + reference *
scale, -inf for a row without a valid key.

The evaluation subtracts the largest LSE_s before exponentiating (only to stay
in range; it changes no value) and is otherwise the formula above.
"""
from __future__ import annotations

import numpy as np


def lse_combine(o_parts, lse_parts):
    """o_parts [P, R, d], lse_parts [P, R] -> (o [R, d], lse [R]), all float64.

    O of a part whose LSE is -inf is never read (it may hold anything)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    if o_parts.ndim != 3 or lse_parts.shape != o_parts.shape[:2]:
        raise ValueError("o_parts must be [P, R, d] and lse_parts [P, R]")
    if np.isnan(lse_parts).any() or np.isposinf(lse_parts).any():
        raise ValueError("a part's LSE must be finite or -inf")
    m = lse_parts.max(axis=0)                               # [R]
    seen = np.isfinite(m)                                   # rows with at least one key
    m_ref = np.where(seen, m, 0.0)
    used = np.isfinite(lse_parts)                           # [P, R]
    w = np.where(used, np.exp(np.where(used, lse_parts, 0.0) - m_ref), 0.0)
    total = w.sum(axis=0)                                   # [R]
    num = np.einsum("pr,prd->rd", w, np.where(used[:, :, None], o_parts, 0.0))
    o = np.where(seen[:, None], num / np.where(seen, total, 1.0)[:, None], 0.0)
    lse = np.where(seen, m_ref + np.log(np.where(seen, total, 1.0)), -np.inf)
    return o, lse
