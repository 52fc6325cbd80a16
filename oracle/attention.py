"""Plain double-precision CPU oracle for attention forward and backward.

TEST INFRASTRUCTURE ONLY. This module is the yardstick the CUDA library is
checked against. It is imported by ``tests/``, by the package's ``smoke()``
self-check and by the CPU-baseline leg of ``bench.py`` — never by the product
path, which fails loudly when its CUDA library is missing instead of falling
back to anything here. It shares no code with the CUDA side: no kernels,
headers, tables or helpers; the only thing both sides consume is the seeded
input generator, which holds none of the method's arithmetic.

What is computed (one head at a time, every value widened to float64; the
N x N probability matrix is materialised, which is exactly what the CUDA
kernels avoid):

* Forward, "FlashAttention backward" §What the forward left behind and
  "Lecture 7 — Backward Pass and Validation" §The math:
  S = scale * Q K^T, masked entries set to -inf; L_i = m_i + log sum_j
  exp(S_ij - m_i) (natural log, computed before dropout); P = exp(S - L);
  O = (P o Z / (1 - p)) V with Z the dropout keep-mask.
* Backward, "FlashAttention backward" §The gradients, and the one scalar that
  makes them local; "Lecture 7" §The math; "Implementing Flash Attention's
  Backward Pass in Raw CUDA" §Deriving the gradients, with dropout folded in
  by the chain rule:
  dV = (P o Z/(1-p))^T dO; dP = (dO V^T) o Z/(1-p); D_i = sum_k dO_ik O_ik;
  dS = P o (dP - D); dQ = scale * dS K; dK = scale * dS^T Q.
* Masks, "Lecture 7" §Mask behaviour: causal keeps j <= i (top-left aligned,
  square), a window W > 0 keeps j > i - W; both may be on at once.
* ALiBi ("Lecture 7" §Use it in the real stack names it among the cases a
  complete harness covers; the pages give no formula): the usual linear
  position bias, S_ij = scale * q_i.k_j - m * |i - j| with one slope m per
  head (or per batch and head), added after the scale and before the mask. The
  slopes are constants, so the gradient formulas above are unchanged.
* attn_bias ("Lecture 7" §Mask behaviour: custom masks enter as an additive
  bias and need their own test path): a given [B or 1, H or 1, N, N] tensor
  added to the scaled scores, S_ij = scale * q_i.k_j + bias_ij, before the
  mask; -inf entries mask pairs out. A constant: no gradient is taken for it.
  A row with no allowed key has L = -inf, P = 0, O = 0 and zero gradients.

Parity pins (tests that fix this oracle to something other than itself) live
in ``tests/test_oracle_pins.py``: central finite differences, the D identity,
zero row sums of dS, closed forms, exact zero flow across mask boundaries, and
cross-checks against torch's float64 autograd and SDPA. The dropout generator
is pinned against cuRAND's device Philox on a GPU.
"""
from __future__ import annotations

import numpy as np

from .philox import keep_mask

# Largest probability panel (rows x N, float64) held at once: 256 MiB.
_PANEL_BYTES = 1 << 28


def allowed(rows, N: int, causal: bool, window: int):
    """Boolean matrix of (query row i, key j) pairs the mask lets through."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    ok = np.ones((i.shape[0], N), dtype=bool)
    if causal:
        ok &= j <= i
    if window > 0:
        ok &= j > i - window
    return ok


def alibi_bias(alibi, b: int, h: int, rows, cols):
    """-m * |i - j| for the given query rows and key columns (0 without ALiBi).

    ``alibi`` holds the slopes m, shaped [H] (shared over the batch) or [B, H].
    """
    if alibi is None:
        return 0.0
    sl = np.asarray(alibi, dtype=np.float64)
    m = sl[h] if sl.ndim == 1 else sl[b, h]
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    return -m * np.abs(i - j).astype(np.float64)


def tensor_bias(bias, b: int, h: int, rows, cols):
    """bias[b, h, rows, cols] of a [B or 1, H or 1, N, N] array (size-1 dims
    broadcast); 0 without one."""
    if bias is None:
        return 0.0
    t = np.asarray(bias)
    bb = b if t.shape[0] > 1 else 0
    hh = h if t.shape[1] > 1 else 0
    return t[bb, hh][np.ix_(np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64))].astype(np.float64)


def _panels(N: int):
    rows = max(1, min(N, _PANEL_BYTES // (8 * max(N, 1))))
    for r0 in range(0, N, rows):
        yield r0, min(N, r0 + rows)


def _f64(x):
    return np.asarray(x).astype(np.float64)


def _dropout_scale(b, h, H, N, rows, seed, offset, p):
    """Z / (1 - p) as float64 (1 everywhere when p == 0)."""
    if p == 0.0:
        return None
    z = keep_mask(b, h, H, N, rows, seed, offset, p)
    return z.astype(np.float64) / (1.0 - p)


def forward(q, k, v, scale, causal=False, window=0, dropout_p=0.0, seed=0, offset=0, alibi=None, bias=None):
    """Attention forward; returns (O [B,N,H,d] float64, L [B,H,N] float64).

    q, k, v are [B, N, H, d] arrays of any float dtype (widened exactly).
    ``scale`` is taken as the float32 value the CUDA side receives, widened.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    scale = float(np.float32(scale))
    O = np.zeros((B, N, H, d))
    L = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
            for r0, r1 in _panels(N):
                rows = np.arange(r0, r1)
                ok = allowed(rows, N, causal, window)
                S = np.where(ok, scale * (Q[r0:r1] @ K.T) + alibi_bias(alibi, b, h, rows, np.arange(N))
                             + tensor_bias(bias, b, h, rows, np.arange(N)), -np.inf)
                m = S.max(axis=1)
                live = np.isfinite(m)
                ms = np.where(live, m, 0.0)
                E = np.where(ok, np.exp(S - ms[:, None]), 0.0)
                lse = np.where(live, ms + np.log(np.where(live, E.sum(axis=1), 1.0)), -np.inf)
                P = np.where(ok, np.exp(S - np.where(live, lse, 0.0)[:, None]), 0.0)
                zs = _dropout_scale(b, h, H, N, rows, seed, offset, dropout_p)
                Pt = P if zs is None else P * zs
                O[b, r0:r1, h, :] = Pt @ V
                L[b, h, r0:r1] = lse
    return O, L


def preprocess_D(o, do):
    """D_i = rowsum(dO o O) per (b, h, i) in float64, returned as [B, H, N].

    "FlashAttention backward" §The gradients, and the one scalar that makes
    them local; "Implementing Flash Attention's Backward Pass" §Deriving the
    gradients (D[i] = dot(dO[i], O[i])).
    """
    return np.einsum("bnhd,bnhd->bhn", _f64(do), _f64(o))


def backward(q, k, v, o, do, lse, scale, causal=False, window=0, dropout_p=0.0,
             seed=0, offset=0, alibi=None, bias=None):
    """Attention backward from the saved state (O, L); returns (dQ, dK, dV, D).

    Gradients are [B, N, H, d] float64, D is [B, H, N] float64. ``o`` and
    ``lse`` are used exactly as given (function mode): pass the O and L a
    forward produced to check a backward fed by that forward, or the float64
    ones from :func:`forward` for the exact gradient.
    """
    q, k, v, o, do = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do)
    lse = _f64(lse)
    B, N, H, d = q.shape
    scale = float(np.float32(scale))
    D = preprocess_D(o, do)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            Q, K, V, dO = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], do[b, :, h, :]
            for r0, r1 in _panels(N):
                rows = np.arange(r0, r1)
                ok = allowed(rows, N, causal, window)
                Lr = lse[b, h, r0:r1]
                live = np.isfinite(Lr)
                S = (scale * (Q[r0:r1] @ K.T) + alibi_bias(alibi, b, h, rows, np.arange(N))
                     + tensor_bias(bias, b, h, rows, np.arange(N)))
                # P_ij = exp(S_ij - L_i) on allowed pairs of rows that have any.
                P = np.where(ok & live[:, None],
                             np.exp(np.where(ok, S, 0.0) - np.where(live, Lr, 0.0)[:, None]), 0.0)
                zs = _dropout_scale(b, h, H, N, rows, seed, offset, dropout_p)
                Pt = P if zs is None else P * zs
                dV[b, :, h, :] += Pt.T @ dO[r0:r1]
                dP = dO[r0:r1] @ V.T
                if zs is not None:
                    dP = dP * zs
                dS = P * (dP - D[b, h, r0:r1][:, None])
                dQ[b, r0:r1, h, :] = scale * (dS @ K)
                dK[b, :, h, :] += scale * (dS.T @ Q[r0:r1])
    return dQ, dK, dV, D


def forward_rows(q, k, v, b, h, rows, scale, causal=False, window=0, dropout_p=0.0, seed=0, offset=0,
                 alibi=None, bias=None):
    """O[b, rows, h, :] and L[b, h, rows] of one head: the same definitions as
    :func:`forward`, evaluated for the listed query rows only (rows are independent)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    scale = float(np.float32(scale))
    rows = np.asarray(rows, dtype=np.int64)
    ok = allowed(rows, N, causal, window)
    S = np.where(ok, scale * (q[b, rows, h, :] @ k[b, :, h, :].T) + alibi_bias(alibi, b, h, rows, np.arange(N))
                 + tensor_bias(bias, b, h, rows, np.arange(N)), -np.inf)
    m = S.max(axis=1)
    live = np.isfinite(m)
    ms = np.where(live, m, 0.0)
    E = np.where(ok, np.exp(S - ms[:, None]), 0.0)
    lse = np.where(live, ms + np.log(np.where(live, E.sum(axis=1), 1.0)), -np.inf)
    P = np.where(ok, np.exp(S - np.where(live, lse, 0.0)[:, None]), 0.0)
    zs = _dropout_scale(b, h, H, N, rows, seed, offset, dropout_p)
    Pt = P if zs is None else P * zs
    return Pt @ v[b, :, h, :], lse


def backward_rows(q, k, v, o, do, lse, b, h, rows, scale, causal=False, window=0, dropout_p=0.0, seed=0,
                  offset=0, alibi=None, bias=None):
    """dQ[b, rows, h, :] of one head from the given O and L (function mode), by the
    definitions of :func:`backward` restricted to the listed query rows."""
    q, k, v, o, do = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do)
    lse = _f64(lse)
    B, N, H, d = q.shape
    scale = float(np.float32(scale))
    rows = np.asarray(rows, dtype=np.int64)
    ok = allowed(rows, N, causal, window)
    Lr = lse[b, h, rows]
    live = np.isfinite(Lr)
    S = (scale * (q[b, rows, h, :] @ k[b, :, h, :].T) + alibi_bias(alibi, b, h, rows, np.arange(N))
         + tensor_bias(bias, b, h, rows, np.arange(N)))
    P = np.where(ok & live[:, None], np.exp(np.where(ok, S, 0.0) - np.where(live, Lr, 0.0)[:, None]), 0.0)
    D = np.einsum("rd,rd->r", do[b, rows, h, :], o[b, rows, h, :])
    dP = do[b, rows, h, :] @ v[b, :, h, :].T
    zs = _dropout_scale(b, h, H, N, rows, seed, offset, dropout_p)
    if zs is not None:
        dP = dP * zs
    dS = P * (dP - D[:, None])
    return scale * (dS @ k[b, :, h, :])


def backward_cols(q, k, v, o, do, lse, b, h, cols, scale, causal=False, window=0, dropout_p=0.0, seed=0,
                  offset=0, alibi=None, bias=None):
    """(dK, dV)[b, cols, h, :] of one head from the given O and L (function mode):
    the definitions of :func:`backward` restricted to the listed key rows, which
    need the column slice P[:, cols] over all query rows."""
    q, k, v, o, do = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do)
    lse = _f64(lse)
    B, N, H, d = q.shape
    scale = float(np.float32(scale))
    cols = np.asarray(cols, dtype=np.int64)
    rows = np.arange(N)
    ok = allowed(rows, N, causal, window)[:, cols]
    Lr = lse[b, h, :]
    live = np.isfinite(Lr)
    S = (scale * (q[b, :, h, :] @ k[b, cols, h, :].T) + alibi_bias(alibi, b, h, rows, cols)
         + tensor_bias(bias, b, h, rows, cols))
    P = np.where(ok & live[:, None], np.exp(np.where(ok, S, 0.0) - np.where(live, Lr, 0.0)[:, None]), 0.0)
    D = np.einsum("nd,nd->n", do[b, :, h, :], o[b, :, h, :])
    zs = _dropout_scale(b, h, H, N, rows, seed, offset, dropout_p)
    if zs is not None:
        zs = zs[:, cols]
    Pt = P if zs is None else P * zs
    dP = do[b, :, h, :] @ v[b, cols, h, :].T
    if zs is not None:
        dP = dP * zs
    dS = P * (dP - D[:, None])
    return scale * (dS.T @ q[b, :, h, :]), Pt.T @ do[b, :, h, :]


def reference_grads(q, k, v, do, scale, causal=False, window=0, dropout_p=0.0, seed=0, offset=0, alibi=None,
                    bias=None):
    """Exact mode: forward in float64, then backward from that O and L."""
    O, L = forward(q, k, v, scale, causal, window, dropout_p, seed, offset, alibi, bias)
    dQ, dK, dV, D = backward(q, k, v, O, do, L, scale, causal, window, dropout_p, seed, offset, alibi, bias)
    return O, L, dQ, dK, dV, D


__all__ = ["allowed", "alibi_bias", "tensor_bias", "forward", "backward", "preprocess_D", "reference_grads", "forward_rows",
           "backward_rows", "backward_cols", "varlen_forward", "varlen_backward"]


def _seq_slopes(alibi, sq: int):
    """Slopes of sequence sq: [H] shared by every sequence, or row sq of [nseq, H]."""
    if alibi is None:
        return None
    sl = np.asarray(alibi, dtype=np.float64)
    return sl if sl.ndim == 1 else sl[sq]


def _segments(cu_seqlens):
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    return list(zip(cu[:-1], cu[1:]))


def varlen_forward(q, k, v, cu_seqlens, scale, causal=False, window=0, alibi=None):
    """Packed variable-length forward; returns (O [total,H,d], L [H,total]) float64.

    q, k, v are [total, H, d]; sequence s is rows cu_seqlens[s]:cu_seqlens[s+1]
    and attends only within itself, with mask positions local to it. This is
    :func:`forward` applied to each sequence as a batch of one ("Lecture 7 —
    Backward Pass and Validation" §Use it in the real stack names packed
    variable-length batches among the cases to cover; the attention of each
    sequence is unchanged by its neighbours).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, H, d = q.shape
    O = np.zeros((total, H, d))
    L = np.full((H, total), -np.inf)
    for sq, (s0, s1) in enumerate(_segments(cu_seqlens)):
        if s1 <= s0:
            continue
        o, lse = forward(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], scale, causal, window,
                         alibi=_seq_slopes(alibi, sq))
        O[s0:s1] = o[0]
        L[:, s0:s1] = lse[0]
    return O, L


def varlen_backward(q, k, v, o, do, lse, cu_seqlens, scale, causal=False, window=0, alibi=None):
    """Packed variable-length backward from (O, L [H,total]); returns (dQ, dK, dV) [total,H,d] float64.

    :func:`backward` applied to each sequence of the pack on its own.
    """
    q, k, v, o, do, lse = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do), _f64(lse)
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for sq, (s0, s1) in enumerate(_segments(cu_seqlens)):
        if s1 <= s0:
            continue
        g = backward(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], o[None, s0:s1], do[None, s0:s1],
                     lse[None, :, s0:s1], scale, causal, window, alibi=_seq_slopes(alibi, sq))
        dQ[s0:s1], dK[s0:s1], dV[s0:s1] = g[0][0], g[1][0], g[2][0]
    return dQ, dK, dV
