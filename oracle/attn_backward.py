"""Oracle for the attention backward pass (fp64, NumPy).

Test infrastructure only (see the package docstring).

For the forward O = softmax(s * Q K^T, masked) V with an upstream gradient dO,
the gradients follow from the chain rule through the row softmax:

    S  = s * Q K^T                    (masked entries are -inf)
    P  = softmax_row(S)               (a row with no valid key: P = 0)
    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - rowsum(P * dP))    (elementwise; the softmax Jacobian)
    dQ = s * dS K
    dK = s * dS^T Q

With grouped heads (H query heads over H_kv K/V heads, G = H / H_kv), query
head h reads K/V head h / G, so dK and dV of a K/V head are the sums of the
contributions of its G query heads.

Sources: "FlashAttention-4（下）" (argus lesson 7), section 1 (the backward
recomputes S and P and runs the products for dV, dP, dQ and dK, with the
elementwise softmax gradient between them); "Flash Attention 4", section
"算法结构" (the forward definition P = softmax(s * S) and O = P V that these
derivatives differentiate), and section "GQA 支持" (the head mapping). The
mask is the forward's bottom-right causal mask ("Causal Mask").

No blocking, no recomputation from the LSE, no reordering: every matrix is
formed in full for one head at a time. ``attention_forward`` is the matching
fp64 forward on float inputs, used to pin the gradients by finite differences.
"""
from __future__ import annotations

import numpy as np


def _widen(x, dtype):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        from fa_inputs import bits_to_f32
        return bits_to_f32(x, dtype).astype(np.float64)
    return x.astype(np.float64)


def _mask(nq, nk, causal):
    """valid[i, j]: query i sees key j (bottom-right alignment, off = nk - nq)."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    off = nk - nq
    return np.arange(nk)[None, :] <= np.arange(nq)[:, None] + off


def _softmax_rows(S, valid):
    S = np.where(valid, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    seen = np.isfinite(m)
    E = np.where(valid, np.exp(S - np.where(seen, m, 0.0)), 0.0)
    den = E.sum(axis=1, keepdims=True)
    return np.where(seen, E / np.where(seen, den, 1.0), 0.0)


def attention_forward(q, k, v, scale: float, causal: bool, dtype: str = "bf16"):
    """O [B, Nq, H, d] (fp64) for q [B, Nq, H, d], k/v [B, Nk, Hkv, d] (bit patterns or floats)."""
    q, k, v = (_widen(x, dtype) for x in (q, k, v))
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = H // Hkv
    valid = _mask(Nq, Nk, causal)
    o = np.zeros((B, Nq, H, d))
    for b in range(B):
        for h in range(H):
            P = _softmax_rows(scale * q[b, :, h] @ k[b, :, h // G].T, valid)
            o[b, :, h] = P @ v[b, :, h // G]
    return o


def attention_backward(q, k, v, do, scale: float, causal: bool, dtype: str = "bf16"):
    """Gradients (dq [B, Nq, H, d], dk [B, Nk, Hkv, d], dv [B, Nk, Hkv, d]), fp64.

    q [B, Nq, H, d], k and v [B, Nk, Hkv, d], do [B, Nq, H, d]: bit patterns of
    ``dtype`` (uint16) or float arrays."""
    q, k, v, do = (_widen(x, dtype) for x in (q, k, v, do))
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if H % Hkv or k.shape != (B, Nk, Hkv, d) or v.shape != k.shape or do.shape != q.shape:
        raise ValueError("shape mismatch")
    G = H // Hkv
    valid = _mask(Nq, Nk, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            Q, K, V, dO = q[b, :, h], k[b, :, h // G], v[b, :, h // G], do[b, :, h]
            P = _softmax_rows(scale * Q @ K.T, valid)
            dv[b, :, h // G] += P.T @ dO
            dP = dO @ V.T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dq[b, :, h] = scale * dS @ K
            dk[b, :, h // G] += scale * dS.T @ Q
    return dq, dk, dv


def attention_backward_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool,
                              dtype: str = "bf16"):
    """Packed variable-length gradients: q, do [T, H, d]; k, v [T_kv, H_kv, d]; sequence s
    has query rows [cu_q[s], cu_q[s+1]) and key rows [cu_k[s], cu_k[s+1]), with its own
    bottom-right causal diagonal. Each sequence is ``attention_backward`` of its own
    slices (a sequence without keys: dQ = 0; without queries: dK = dV = 0)."""
    q, k, v, do = (_widen(x, dtype) for x in (q, k, v, do))
    cu_q = np.asarray(cu_seqlens_q, dtype=np.int64)
    cu_k = np.asarray(cu_seqlens_k, dtype=np.int64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cu_q) - 1):
        a, b = cu_q[s], cu_q[s + 1]
        c, e = cu_k[s], cu_k[s + 1]
        if b == a or e == c:
            continue
        g = attention_backward(q[None, a:b], k[None, c:e], v[None, c:e], do[None, a:b], scale, causal)
        dq[a:b], dk[c:e], dv[c:e] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv
