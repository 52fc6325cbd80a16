"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test fixes the oracle to a fact the mathematics or the pages fix, chosen
so that a plausible slip (a dropped -D term, a wrong sign, a transposed
operand, a misplaced mask bound, a missing 1/(1-p)) fails at least one:

* central finite differences of a random linear loss sum(R o O) against the
  analytic gradients ("Lecture 7 — Backward Pass and Validation" §The math);
* the identity D_i = sum_j P_ij dP_ij = rowsum(dO o O) ("FlashAttention
  backward" §The gradients, and the one scalar that makes them local);
* zero row sums of dS, hence sum_j dK_j = 0, and sum_j dV_j = sum_i dO_i;
* exact zero gradient across causal and window boundaries ("Lecture 7"
  §Mask behaviour; "FlashAttention backward" §The traps, causal row);
* closed forms (N = 1, identical keys, Q = 0 under causal, key shift);
* torch float64 autograd and SDPA as independent library routines.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.attention import allowed

RNG_SHAPES = [
    # N, d, causal, window, p
    (1, 1, False, 0, 0.0),
    (2, 2, False, 0, 0.0),
    (3, 4, True, 0, 0.0),
    (5, 2, True, 2, 0.0),
    (8, 4, False, 3, 0.0),
    (5, 4, True, 0, 0.3),
    (8, 2, True, 3, 0.25),
    (8, 4, False, 0, 0.5),
]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("N,d,causal,window,p", RNG_SHAPES)
def test_central_finite_differences(N, d, causal, window, p):
    B, H = 1, 2
    q, k, v, R = (_rand((B, N, H, d), 100 + t) for t in range(4))
    scale = 0.7
    kw = dict(causal=causal, window=window, dropout_p=p, seed=77, offset=3)
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, R, scale, **kw)

    def loss(qq, kk, vv):
        O, _ = oracle.forward(qq, kk, vv, scale, **kw)
        return float((R * O).sum())

    h = 1e-5
    for which, grad in ((0, dQ), (1, dK), (2, dV)):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            dn = loss(*args)
            fd[idx] = (up - dn) / (2 * h)
        err = np.abs(fd - grad).max()
        assert err <= 1e-6 * max(1.0, np.abs(grad).max()), (which, err)


@pytest.mark.parametrize("causal,window,p", [(False, 0, 0.0), (True, 0, 0.0), (True, 7, 0.2), (False, 5, 0.4)])
def test_D_identity(causal, window, p):
    """D_i = sum_j P~_ij dP~_ij = rowsum(dO o O), with or without dropout."""
    B, N, H, d = 2, 19, 3, 8
    q, k, v, do = (_rand((B, N, H, d), 200 + t) for t in range(4))
    scale = 0.375  # exactly representable in float32, as the oracle takes it
    O, L = oracle.forward(q, k, v, scale, causal, window, p, seed=5, offset=9)
    D = oracle.preprocess_D(O, do)
    for b in range(B):
        for hh in range(H):
            rows = np.arange(N)
            ok = allowed(rows, N, causal, window)
            S = scale * q[b, :, hh] @ k[b, :, hh].T
            P = np.where(ok, np.exp(np.where(ok, S, 0) - L[b, hh][:, None]), 0.0)
            Z = oracle.keep_mask(b, hh, H, N, rows, 5, 9, p) / (1 - p)
            Pt = P * Z
            dPt = do[b, :, hh] @ v[b, :, hh].T
            lhs = (Pt * dPt).sum(axis=1)
            np.testing.assert_allclose(lhs, D[b, hh], rtol=0, atol=1e-12 * max(1, np.abs(D).max()))


@pytest.mark.parametrize("causal,window,p", [(False, 0, 0.0), (True, 0, 0.0), (True, 4, 0.3), (False, 3, 0.0)])
def test_row_sums(causal, window, p):
    """sum_j dS_ij = 0 makes sum_j dK_j = 0; with p = 0, sum_j dV_j = sum_i dO_i."""
    B, N, H, d = 2, 13, 2, 5
    q, k, v, do = (_rand((B, N, H, d), 300 + t) for t in range(4))
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.45, causal, window, p, 11, 0)
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, atol=1e-12)
    if p == 0.0:
        np.testing.assert_allclose(dV.sum(axis=1), do.sum(axis=1), atol=1e-12)


def test_zero_flow_causal():
    """dO zero on rows >= r under causal: keys >= r and those query rows get exactly 0."""
    B, N, H, d, r = 1, 16, 2, 4, 9
    q, k, v, do = (_rand((B, N, H, d), 400 + t) for t in range(4))
    do[:, r:] = 0.0
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.5, causal=True)
    assert np.all(dK[:, r:] == 0.0) and np.all(dV[:, r:] == 0.0) and np.all(dQ[:, r:] == 0.0)
    assert np.abs(dK[:, :r]).min() > 0 and np.abs(dV[:, :r]).min() > 0


@pytest.mark.parametrize("causal", [True, False])
def test_zero_flow_window(causal):
    """dO nonzero only in row r under window W: only keys in (r-W, r] (causal) get gradient."""
    B, N, H, d, r, W = 1, 20, 1, 4, 12, 5
    q, k, v, do = (_rand((B, N, H, d), 500 + t) for t in range(4))
    mask = np.zeros(N, bool)
    mask[r] = True
    do[:, ~mask] = 0.0
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.5, causal=causal, window=W)
    j = np.arange(N)
    inside = (j > r - W) & ((j <= r) if causal else True)
    assert np.all(dK[:, ~inside] == 0.0) and np.all(dV[:, ~inside] == 0.0)
    assert np.all(np.abs(dV[:, inside]).sum(axis=-1) > 0)
    assert np.all(dQ[:, j != r] == 0.0)


def test_closed_form_single_key():
    """N = 1: P = 1, so O = V, L = S, dV = dO and dQ = dK = 0."""
    q, k, v, do = (_rand((2, 1, 3, 6), 600 + t) for t in range(4))
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.25)
    np.testing.assert_allclose(O, v, atol=1e-15)
    np.testing.assert_allclose(L, 0.25 * np.einsum("bnhd,bnhd->bhn", q, k), atol=1e-14)
    np.testing.assert_array_equal(dV, do)
    # dS = 1 * (dO.V - dO.O) with O = V: zero up to the rounding of two dot products
    np.testing.assert_allclose(dQ, 0.0, atol=1e-14)
    np.testing.assert_allclose(dK, 0.0, atol=1e-14)


def test_closed_form_identical_keys():
    """All keys equal, no mask: P = 1/N, dQ = 0, dV_j = mean_i dO_i, L = s + log N."""
    B, N, H, d = 1, 7, 2, 3
    q, v, do = (_rand((B, N, H, d), 700 + t) for t in range(3))
    k = np.broadcast_to(_rand((B, 1, H, d), 710), (B, N, H, d)).copy()
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.75)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-13)
    np.testing.assert_allclose(dV, np.broadcast_to(do.mean(axis=1, keepdims=True), dV.shape), atol=1e-14)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape), atol=1e-14)
    s = 0.75 * np.einsum("bnhd,bhd->bhn", q, k[:, 0])
    np.testing.assert_allclose(L, s + np.log(N), atol=1e-13)


def test_closed_form_zero_queries_causal():
    """Q = 0 under causal: P_ij = 1/(i+1), dK = 0, dV_j = sum_{i>=j} dO_i/(i+1)."""
    B, N, H, d = 1, 9, 2, 4
    k, v, do = (_rand((B, N, H, d), 800 + t) for t in range(3))
    q = np.zeros_like(k)
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.6, causal=True)
    assert np.all(dK == 0)
    w = 1.0 / (np.arange(N) + 1.0)
    expect = np.zeros_like(dV)
    for j in range(N):
        expect[:, j] = (do[:, j:] * w[j:, None, None]).sum(axis=1)
    np.testing.assert_allclose(dV, expect, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.log(np.arange(N) + 1.0), atol=1e-14)


def test_key_shift_invariance():
    """Adding one vector c to every key adds q_i.c to a whole row of S: nothing changes."""
    B, N, H, d = 1, 11, 2, 5
    q, k, v, do = (_rand((B, N, H, d), 900 + t) for t in range(4))
    c = _rand((1, 1, H, d), 950)
    for causal, W in ((False, 0), (True, 0), (True, 4)):
        a = oracle.reference_grads(q, k, v, do, 0.4, causal, W)
        b = oracle.reference_grads(q, k + c, v, do, 0.4, causal, W)
        for x, y in zip((a[0], a[2], a[3], a[4]), (b[0], b[2], b[3], b[4])):
            np.testing.assert_allclose(x, y, atol=1e-12)


def _torch_attention(q, k, v, scale, ok, zs):
    s = torch.einsum("bnhd,bmhd->bhnm", q, k) * scale
    s = s.masked_fill(~ok, float("-inf"))
    p = torch.softmax(s, dim=-1)
    if zs is not None:
        p = p * zs
    return torch.einsum("bhnm,bmhd->bnhd", p, v)


@pytest.mark.parametrize("N,d,causal,window,p", [(64, 16, False, 0, 0.0), (128, 32, True, 0, 0.0),
                                                 (97, 8, True, 20, 0.0), (256, 64, False, 0, 0.0),
                                                 (50, 8, True, 9, 0.15), (33, 4, False, 6, 0.0)])
def test_torch_float64_autograd(N, d, causal, window, p):
    B, H = 2, 2
    q, k, v, do = (_rand((B, N, H, d), 1000 + t) for t in range(4))
    scale = float(np.float32(1.0 / np.sqrt(d)))
    seed, off = 42, 7
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, scale, causal, window, p, seed, off)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ok = torch.tensor(allowed(np.arange(N), N, causal, window))[None, None]
    zs = None
    if p > 0:
        zs = torch.tensor(np.stack([np.stack([oracle.keep_mask(b, h, H, N, np.arange(N), seed, off, p)
                                              for h in range(H)]) for b in range(B)]) / (1 - p))
    out = _torch_attention(tq, tk, tv, scale, ok, zs)
    out.backward(torch.tensor(do))
    for a, t in ((O, out.detach()), (dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        t = t.numpy()
        assert np.linalg.norm(a - t) <= 1e-12 * max(1e-300, np.linalg.norm(t)) + 1e-15
    s = torch.einsum("bnhd,bmhd->bhnm", tq.detach(), tk.detach()) * scale
    lse = torch.logsumexp(s.masked_fill(~ok, float("-inf")), dim=-1).numpy()
    np.testing.assert_allclose(L, lse, rtol=1e-13, atol=1e-13)


def test_torch_sdpa_forward():
    """Forward O against torch's scaled_dot_product_attention in float64 (causal and windowed)."""
    B, N, H, d = 1, 70, 3, 16
    q, k, v = (_rand((B, N, H, d), 1100 + t) for t in range(3))
    F = torch.nn.functional
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3) for x in (q, k, v))
    for causal, W in ((False, 0), (True, 0), (True, 10), (False, 10)):
        O, _ = oracle.forward(q, k, v, 0.25, causal, W)
        ok = torch.tensor(allowed(np.arange(N), N, causal, W))
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=ok, scale=0.25).permute(0, 2, 1, 3)
        np.testing.assert_allclose(O, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_row_panels_match_whole_matrix(monkeypatch):
    """Row panels (used for long sequences) reproduce the single-panel result."""
    import oracle.attention as oa
    B, N, H, d = 1, 37, 2, 8
    q, k, v, do = (_rand((B, N, H, d), 1200 + t) for t in range(4))
    whole = oa.reference_grads(q, k, v, do, 0.3, True, 9, 0.2, 3, 1)
    monkeypatch.setattr(oa, "_PANEL_BYTES", 8 * N * 5)  # 5-row panels
    parts = oa.reference_grads(q, k, v, do, 0.3, True, 9, 0.2, 3, 1)
    for a, b in zip(whole, parts):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal,window,p", [(True, 0, 0.0), (False, 0, 0.0), (True, 6, 0.3)])
def test_sampled_rows_and_columns_match_whole_head(causal, window, p):
    """The row / column restrictions used for full-size checks reproduce the whole-head results."""
    B, N, H, d = 2, 29, 3, 8
    q, k, v, do = (_rand((B, N, H, d), 1300 + t) for t in range(4))
    O, L = oracle.forward(q, k, v, 0.3, causal, window, p, 9, 2)
    dQ, dK, dV, _ = oracle.backward(q, k, v, O, do, L, 0.3, causal, window, p, 9, 2)
    rows = [0, 3, 17, 28]
    for b in range(B):
        for h in range(H):
            o_r, l_r = oracle.forward_rows(q, k, v, b, h, rows, 0.3, causal, window, p, 9, 2)
            np.testing.assert_allclose(o_r, O[b, rows, h], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(l_r, L[b, h, rows], rtol=1e-13, atol=1e-14)
            dq_r = oracle.backward_rows(q, k, v, O, do, L, b, h, rows, 0.3, causal, window, p, 9, 2)
            np.testing.assert_allclose(dq_r, dQ[b, rows, h], rtol=1e-12, atol=1e-13)
            dk_c, dv_c = oracle.backward_cols(q, k, v, O, do, L, b, h, rows, 0.3, causal, window, p, 9, 2)
            np.testing.assert_allclose(dk_c, dK[b, rows, h], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(dv_c, dV[b, rows, h], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5), (False, 4)])
def test_varlen_matches_block_diagonal_dense(causal, window):
    """Packed sequences against one dense attention over the whole pack whose
    mask keeps only pairs inside one sequence (positions counted from each
    sequence's start), differentiated by torch float64 autograd. An off-by-one
    in the segment bounds or a mask taken on packed instead of local
    positions fails this."""
    cu = np.array([0, 7, 8, 8, 29, 40])  # lengths 7, 1, 0 (empty), 21, 11
    total, H, d = int(cu[-1]), 2, 8
    q, k, v, do = (_rand((total, H, d), 1200 + t) for t in range(4))
    scale = float(np.float32(0.3))  # the oracle takes the float32 value the kernels receive
    O, L = oracle.varlen_forward(q, k, v, cu, scale, causal, window)
    dQ, dK, dV = oracle.varlen_backward(q, k, v, O, do, L, cu, scale, causal, window)
    seg = np.searchsorted(cu, np.arange(total), side="right") - 1
    pos = np.arange(total) - cu[seg]
    ok = seg[:, None] == seg[None, :]
    if causal:
        ok &= pos[None, :] <= pos[:, None]
    if window > 0:
        ok &= pos[None, :] > pos[:, None] - window
    tq, tk, tv = (torch.tensor(x[None], requires_grad=True) for x in (q, k, v))
    out = _torch_attention(tq, tk, tv, scale, torch.tensor(ok)[None, None], None)
    out.backward(torch.tensor(do[None]))
    for a, t in ((O, out.detach()[0]), (dQ, tq.grad[0]), (dK, tk.grad[0]), (dV, tv.grad[0])):
        t = t.numpy()
        assert np.linalg.norm(a - t) <= 1e-12 * np.linalg.norm(t)
    s = torch.einsum("nhd,mhd->hnm", torch.tensor(q), torch.tensor(k)) * scale
    np.testing.assert_allclose(L, torch.logsumexp(s.masked_fill(~torch.tensor(ok), float("-inf")), -1).numpy(),
                               rtol=1e-13, atol=1e-13)


# ------------------------------- ALiBi ---------------------------------------
@pytest.mark.parametrize("N,d,causal,window,p", [(6, 3, True, 0, 0.0), (7, 2, False, 0, 0.0), (8, 2, True, 3, 0.25)])
def test_alibi_central_finite_differences(N, d, causal, window, p):
    """Gradients with the position bias on, against central differences of the biased forward."""
    B, H = 2, 2
    q, k, v, R = (_rand((B, N, H, d), 300 + t) for t in range(4))
    slopes = np.array([[0.5, 0.125], [0.25, 1.0]])  # [B, H]
    kw = dict(causal=causal, window=window, dropout_p=p, seed=5, offset=1, alibi=slopes)
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, R, 0.6, **kw)

    def loss(qq, kk, vv):
        return float((R * oracle.forward(qq, kk, vv, 0.6, **kw)[0]).sum())

    h = 1e-5
    for which, grad in ((0, dQ), (1, dK), (2, dV)):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            fd[idx] = (up - loss(*args)) / (2 * h)
        assert np.abs(fd - grad).max() <= 1e-6 * max(1.0, np.abs(grad).max()), which


@pytest.mark.parametrize("causal,window,per_batch", [(True, 0, False), (False, 0, True), (True, 9, True)])
def test_alibi_torch_float64_autograd(causal, window, per_batch):
    """Against torch autograd of softmax(scale QK^T + B) V with the bias matrix
    B_ij = -m |i - j| built by torch from broadcast position vectors."""
    B, N, H, d = 2, 37, 3, 8
    q, k, v, do = (_rand((B, N, H, d), 400 + t) for t in range(4))
    slopes = np.array([0.5, 0.0625, 2.0 ** -0.5]) if not per_batch else np.array([[0.5, 0.25, 0.1], [1.0, 0.0, 0.3]])
    scale = float(np.float32(0.35))
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, scale, causal, window, alibi=slopes)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    pos = torch.arange(N, dtype=torch.float64)
    dist = (pos[:, None] - pos[None, :]).abs()                      # [N, N]
    m = torch.tensor(slopes if per_batch else np.broadcast_to(slopes, (B, H)).copy())  # [B, H]
    bias = -m[:, :, None, None] * dist[None, None]                  # [B, H, N, N]
    s = torch.einsum("bnhd,bmhd->bhnm", tq, tk) * scale + bias
    ok = torch.tensor(allowed(np.arange(N), N, causal, window))[None, None]
    s = s.masked_fill(~ok, float("-inf"))
    out = torch.einsum("bhnm,bmhd->bnhd", torch.softmax(s, dim=-1), tv)
    out.backward(torch.tensor(do))
    for a, t in ((O, out.detach()), (dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        t = t.numpy()
        assert np.linalg.norm(a - t) <= 1e-12 * np.linalg.norm(t)
    np.testing.assert_allclose(L, torch.logsumexp(s.detach(), dim=-1).numpy(), rtol=1e-13, atol=1e-13)


def test_alibi_closed_form_zero_queries_causal():
    """Q = 0 under a causal mask leaves only the bias: P_ij = r^(i-j) (1 - r) / (1 - r^(i+1))
    with r = exp(-m), and L_i = log((1 - r^(i+1)) / (1 - r))."""
    N, d, m = 12, 3, 0.7
    q = np.zeros((1, N, 1, d))
    k, v = _rand((1, N, 1, d), 500), _rand((1, N, 1, d), 501)
    O, L = oracle.forward(q, k, v, 1.0, causal=True, alibi=np.array([m]))
    r = np.exp(-m)
    for i in range(N):
        j = np.arange(i + 1)
        P = r ** (i - j) * (1 - r) / (1 - r ** (i + 1))
        np.testing.assert_allclose(O[0, i, 0], P @ v[0, : i + 1, 0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(L[0, 0, i], np.log((1 - r ** (i + 1)) / (1 - r)), rtol=1e-12)


def test_alibi_zero_slope_is_plain_attention_and_sign_matters():
    B, N, H, d = 1, 20, 2, 4
    q, k, v, do = (_rand((B, N, H, d), 600 + t) for t in range(4))
    a = oracle.reference_grads(q, k, v, do, 0.5, True)
    b = oracle.reference_grads(q, k, v, do, 0.5, True, alibi=np.zeros(H))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # a positive slope pulls probability toward the diagonal: row i's weight on
    # key i grows against the unbiased softmax
    O1, L1 = oracle.forward(q, k, v, 0.5, True)
    O2, L2 = oracle.forward(q, k, v, 0.5, True, alibi=np.full(H, 0.8))
    s = 0.5 * np.einsum("bnhd,bnhd->bhn", q, k)  # diagonal scores (bias 0 there)
    assert np.all(s[:, :, 1:] - L2[:, :, 1:] > s[:, :, 1:] - L1[:, :, 1:])


# ------------------------------ attn_bias -------------------------------------
def _bias(shape, seed, neg_inf_frac=0.0, keep_diag=True):
    r = np.random.default_rng(seed)
    b = r.standard_normal(shape) * 2.0
    if neg_inf_frac:
        mask = r.random(shape) < neg_inf_frac
        if keep_diag:
            n = shape[-1]
            mask[..., np.arange(n), np.arange(n)] = False
        b[mask] = -np.inf
    return b


@pytest.mark.parametrize("bshape,causal,window", [((1, 3, 29, 29), True, 0), ((2, 1, 29, 29), False, 0),
                                                   ((2, 3, 29, 29), True, 7), ((1, 1, 29, 29), False, 5)])
def test_bias_torch_float64_autograd(bshape, causal, window):
    """Against torch autograd of softmax(scale QK^T + bias) V, broadcast bias shapes,
    with a fifth of the entries -inf (masked) off the diagonal."""
    B, N, H, d = 2, 29, 3, 8
    q, k, v, do = (_rand((B, N, H, d), 700 + t) for t in range(4))
    bias = _bias(bshape, 710, neg_inf_frac=0.2)
    scale = float(np.float32(0.3))
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, scale, causal, window, bias=bias)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = torch.einsum("bnhd,bmhd->bhnm", tq, tk) * scale + torch.tensor(bias)
    ok = torch.tensor(allowed(np.arange(N), N, causal, window))[None, None]
    s = s.masked_fill(~ok, float("-inf"))
    out = torch.einsum("bhnm,bmhd->bnhd", torch.softmax(s, dim=-1), tv)
    out.backward(torch.tensor(do))
    for a, t in ((O, out.detach()), (dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        t = t.numpy()
        assert np.linalg.norm(a - t) <= 1e-12 * np.linalg.norm(t)
    np.testing.assert_allclose(L, torch.logsumexp(s.detach(), dim=-1).numpy(), rtol=1e-13, atol=1e-13)


def test_bias_central_finite_differences():
    B, N, H, d = 1, 7, 2, 3
    q, k, v, R = (_rand((B, N, H, d), 720 + t) for t in range(4))
    bias = _bias((1, H, N, N), 730, neg_inf_frac=0.25)
    kw = dict(causal=True, window=0, dropout_p=0.2, seed=4, offset=2, bias=bias)
    _, _, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, R, 0.5, **kw)

    def loss(qq, kk, vv):
        return float((R * oracle.forward(qq, kk, vv, 0.5, **kw)[0]).sum())

    h = 1e-5
    for which, grad in ((0, dQ), (1, dK), (2, dV)):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            fd[idx] = (up - loss(*args)) / (2 * h)
        assert np.abs(fd - grad).max() <= 1e-6 * max(1.0, np.abs(grad).max()), which


def test_bias_special_cases():
    """A -inf upper triangle is the causal mask; a row of -inf is a dead row
    (O = 0, L = -inf, no gradient through it); the ALiBi matrix as a bias is ALiBi."""
    B, N, H, d = 1, 16, 2, 4
    q, k, v, do = (_rand((B, N, H, d), 740 + t) for t in range(4))
    tri = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, 0.0)[None, None]
    a = oracle.reference_grads(q, k, v, do, 0.5, bias=tri)
    b = oracle.reference_grads(q, k, v, do, 0.5, causal=True)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-15)
    dead = np.zeros((1, 1, N, N))
    dead[0, 0, 5, :] = -np.inf
    O, L, dQ, dK, dV, _ = oracle.reference_grads(q, k, v, do, 0.5, bias=dead)
    assert np.all(O[0, 5] == 0) and np.all(np.isneginf(L[0, :, 5])) and np.all(dQ[0, 5] == 0)
    slopes = np.array([0.3, 0.05])
    pos = np.arange(N)
    ab = (-slopes[:, None, None] * np.abs(pos[:, None] - pos[None, :]))[None]
    a = oracle.reference_grads(q, k, v, do, 0.5, True, bias=ab)
    b = oracle.reference_grads(q, k, v, do, 0.5, True, alibi=slopes)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
