"""Pins for the float64 oracle: checks against what the attention pages and the
mathematics fix, independent of the oracle's own code.

Each test names the property it pins and where it comes from.  Together they
are chosen so that a plausible slip in the oracle (a dropped scale, a
transposed operand, a wrong sign in dS, an off-by-one causal mask, a wrong
log base for LSE) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_derived_tiny.json")


def _val(x):
    if isinstance(x, str):
        env = {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln4": math.log(4.0), "ln10": math.log(10.0)}
        return float(eval(x, {"__builtins__": {}}, env))
    return float(x)


def _arr(a):
    return np.array([[_val(x) for x in row] if isinstance(row, list) else _val(row) for row in a])


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden/hand_derived_tiny.json)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_golden_hand_derived(causal):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        N, D, scale = c["N"], c["D"], c["scale"]
        q = _arr(c["q"]).reshape(1, 1, N, D)
        k = _arr(c["k"]).reshape(1, 1, N, D)
        v = _arr(c["v"]).reshape(1, 1, N, D)
        dO = _arr(c["dO"]).reshape(1, 1, N, D)
        exp = c["causal" if causal else "noncausal"]
        o, lse = oracle.forward(q, k, v, scale, causal)
        np.testing.assert_allclose(o[0, 0], _arr(exp["o"]).reshape(N, D), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], _arr(exp["lse"]).reshape(N), rtol=0, atol=1e-13)
        g = oracle.backward(q, k, v, dO, scale, causal)
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(g[name][0, 0], _arr(exp[name]).reshape(N, D), rtol=0, atol=1e-13,
                                       err_msg=f"{c['name']} {name}")
        np.testing.assert_allclose(g["lse"][0, 0], _arr(exp["lse"]).reshape(N), rtol=0, atol=1e-13)
        np.testing.assert_allclose(g["delta"][0, 0], _arr(exp["delta"]).reshape(N), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_rows_return_v_and_zero_dq_dk(causal):
    """All value rows equal v  =>  O_i = v for every row; and since
    dP_ij = <dO_i, v> = D_i, dS = 0 so dQ = dK = 0 while dV = P^T dO."""
    B, H, N, D = 1, 2, 13, 8
    q, k, dO = _rand((B, H, N, D), 1), _rand((B, H, N, D), 2), _rand((B, H, N, D), 3)
    vrow = _rand((D,), 4)
    v = np.broadcast_to(vrow, (B, H, N, D)).copy()
    o, _ = oracle.forward(q, k, v, 0.37, causal)
    np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), atol=1e-13)
    g = oracle.backward(q, k, v, dO, 0.37, causal)
    assert np.abs(g["dq"]).max() < 1e-12
    assert np.abs(g["dk"]).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_v(causal):
    """Q = 0  =>  every visible score is 0, P is uniform: O_i = mean of the
    visible V rows and LSE_i = ln(#visible)."""
    B, H, N, D = 2, 1, 11, 5
    q = np.zeros((B, H, N, D))
    k, v = _rand((B, H, N, D), 5), _rand((B, H, N, D), 6)
    o, lse = oracle.forward(q, k, v, 0.25, causal)
    for i in range(N):
        nvis = i + 1 if causal else N
        np.testing.assert_allclose(o[:, :, i], v[:, :, :nvis].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(nvis), atol=1e-13)


def test_single_key():
    """N = 1  =>  O_0 = v_0 and LSE_0 = scale <q_0, k_0>."""
    q, k, v = _rand((1, 3, 1, 7), 7), _rand((1, 3, 1, 7), 8), _rand((1, 3, 1, 7), 9)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.5, causal)
        np.testing.assert_allclose(o, v, atol=1e-14)
        np.testing.assert_allclose(lse[..., 0], 0.5 * (q * k).sum(-1)[..., 0], atol=1e-13)


def test_causal_row_zero_returns_v0():
    q, k, v = _rand((2, 2, 9, 4), 10), _rand((2, 2, 9, 4), 11), _rand((2, 2, 9, 4), 12)
    o, lse = oracle.forward(q, k, v, 0.9, True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.9 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-13)


# ---------------------------------------------------------------------------
# P itself: with V = identity (D = N), O = P.  Rows sum to 1 and equal the
# library softmax of the scaled scores (scipy), zero above the diagonal when causal.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_rows_sum_to_one_and_match_library_softmax(causal):
    from scipy.special import softmax
    N = 10
    q, k = _rand((1, 1, N, N), 13), _rand((1, 1, N, N), 14)
    v = np.eye(N).reshape(1, 1, N, N)
    scale = 0.7
    p, lse = oracle.forward(q, k, v, scale, causal)
    p = p[0, 0]
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    s = scale * q[0, 0] @ k[0, 0].T
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    np.testing.assert_allclose(p, softmax(s, axis=1), atol=1e-14)
    from scipy.special import logsumexp
    np.testing.assert_allclose(lse[0, 0], logsumexp(s, axis=1), atol=1e-13)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    """sum_j dS_ij = 0 for each row  =>  column sum of dK is 0;
    rows of P sum to 1  =>  sum_j dV_j = sum_i dO_i;  D_i = <dO_i, O_i>."""
    B, H, N, D = 1, 2, 17, 6
    q, k, v, dO = (_rand((B, H, N, D), s) for s in (20, 21, 22, 23))
    g = oracle.backward(q, k, v, dO, 0.41, causal)
    np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dv"].sum(axis=2), dO.sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(g["delta"], (dO * g["o"]).sum(-1), atol=1e-12)


def test_key_shift_invariance():
    """K <- K + 1 u^T adds scale <q_i, u> to every score of row i: O unchanged,
    LSE_i shifted by scale <q_i, u> (softmax is shift invariant per row)."""
    B, H, N, D = 1, 1, 12, 4
    q, k, v = _rand((B, H, N, D), 30), _rand((B, H, N, D), 31), _rand((B, H, N, D), 32)
    u = _rand((D,), 33)
    for causal in (False, True):
        o1, l1 = oracle.forward(q, k, v, 0.6, causal)
        o2, l2 = oracle.forward(q, k + u, v, 0.6, causal)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, 0.6 * (q @ u), atol=1e-12)


def test_permutation_equivariance_noncausal():
    """Non-causal: permuting K and V rows jointly leaves O and LSE unchanged;
    permuting Q rows permutes O and LSE the same way."""
    B, H, N, D = 1, 1, 9, 3
    q, k, v = _rand((B, H, N, D), 40), _rand((B, H, N, D), 41), _rand((B, H, N, D), 42)
    perm = np.random.default_rng(43).permutation(N)
    o, l = oracle.forward(q, k, v, 1.1, False)
    o2, l2 = oracle.forward(q, k[:, :, perm], v[:, :, perm], 1.1, False)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(l2, l, atol=1e-13)
    o3, l3 = oracle.forward(q[:, :, perm], k, v, 1.1, False)
    np.testing.assert_allclose(o3, o[:, :, perm], atol=1e-13)
    np.testing.assert_allclose(l3, l[:, :, perm], atol=1e-13)


def test_hard_attention_limit():
    """A large scale with a unique maximum score per row drives P to the
    indicator of the argmax: O_i -> v_{argmax_j s_ij}."""
    B, H, N, D = 1, 1, 8, 4
    q, k, v = _rand((B, H, N, D), 50), _rand((B, H, N, D), 51), _rand((B, H, N, D), 52)
    o, _ = oracle.forward(q, k, v, 1e4, False)
    arg = (q[0, 0] @ k[0, 0].T).argmax(axis=1)
    np.testing.assert_allclose(o[0, 0], v[0, 0][arg], atol=1e-9)


# ---------------------------------------------------------------------------
# Gradients against central finite differences of f = sum(O * dO)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,D", [(1, 2), (2, 4), (3, 2), (5, 8), (8, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(N, D, causal):
    B, H = 1, 1
    scale = 1.0 / math.sqrt(D)
    q, k, v, dO = (_rand((B, H, N, D), 60 + s) for s in range(4))
    g = oracle.backward(q, k, v, dO, scale, causal)

    def f(qq, kk, vv):
        o, _ = oracle.forward(qq, kk, vv, scale, causal, threads=1)
        return float((o * dO).sum())

    h = 1e-6
    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        fd = np.zeros((N, D))
        for i in range(N):
            for d in range(D):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[idx][0, 0, i, d] += h
                args_m[idx][0, 0, i, d] -= h
                fd[i, d] = (f(*args_p) - f(*args_m)) / (2 * h)
        np.testing.assert_allclose(g[name][0, 0], fd, rtol=1e-6, atol=1e-8, err_msg=name)


# ---------------------------------------------------------------------------
# Library special case: torch float64 CPU attention with autograd
# (a textbook routine that shares nothing with either side)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_float64_sdpa(causal):
    B, H, N, D = 2, 3, 37, 16
    scale = 1.0 / math.sqrt(D)
    q, k, v, dO = (_rand((B, H, N, D), 70 + s) for s in range(4))
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(dO))
    g = oracle.backward(q, k, v, dO, scale, causal)
    np.testing.assert_allclose(g["o"], to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(g["dq"], tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dk"], tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dv"], tv.grad.numpy(), atol=1e-11)


# ---------------------------------------------------------------------------
# The row-sampled entry points agree with the full-head ones
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_row_variants_agree_with_full(causal):
    B, H, N, D = 2, 2, 29, 8
    scale = 0.3
    q, k, v, dO = (_rand((B, H, N, D), 80 + s) for s in range(4))
    g = oracle.backward(q, k, v, dO, scale, causal)
    o_full, lse_full = oracle.forward(q, k, v, scale, causal)
    np.testing.assert_allclose(o_full, g["o"], atol=1e-13)
    np.testing.assert_allclose(lse_full, g["lse"], atol=1e-13)
    rows = [(0, 0, 0), (0, 1, 5), (1, 0, 28), (1, 1, 13), (0, 0, 27)]
    o, lse = oracle.forward_rows(q, k, v, scale, causal, rows)
    dq, delta = oracle.backward_dq_rows(q, k, v, dO, scale, causal, rows)
    dk, dv = oracle.backward_dkdv_rows(q, k, v, dO, scale, causal, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(o[n], g["o"][b, h, i], atol=1e-13)
        np.testing.assert_allclose(lse[n], g["lse"][b, h, i], atol=1e-13)
        np.testing.assert_allclose(dq[n], g["dq"][b, h, i], atol=1e-12)
        np.testing.assert_allclose(delta[n], g["delta"][b, h, i], atol=1e-12)
        np.testing.assert_allclose(dk[n], g["dk"][b, h, i], atol=1e-12)
        np.testing.assert_allclose(dv[n], g["dv"][b, h, i], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_row_ranges_sum_to_full_backward(causal):
    """The row-range form: rows [0, a) plus rows [a, N) give the full-head gradients."""
    B, H, N, D = 1, 2, 23, 4
    q, k, v, dO = (_rand((B, H, N, D), 90 + s) for s in range(4))
    g = oracle.backward(q, k, v, dO, 0.7, causal)
    heads = [(0, 0), (0, 1)]
    lo = oracle.backward_row_range(q, k, v, dO, 0.7, causal, heads, 0, 9)
    hi = oracle.backward_row_range(q, k, v, dO, 0.7, causal, heads, 9, N)
    for b, h in heads:
        np.testing.assert_allclose(lo[(b, h)]["dk"] + hi[(b, h)]["dk"], g["dk"][b, h], atol=1e-12)
        np.testing.assert_allclose(lo[(b, h)]["dv"] + hi[(b, h)]["dv"], g["dv"][b, h], atol=1e-12)
        np.testing.assert_allclose(np.concatenate([lo[(b, h)]["dq"], hi[(b, h)]["dq"]]), g["dq"][b, h],
                                   atol=1e-12)
        np.testing.assert_allclose(hi[(b, h)]["o"], g["o"][b, h, 9:], atol=1e-13)


# ---------------------------------------------------------------------------
# Decode form (n_q query rows that are the last n_q positions, against N_k keys)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_decode_form_equals_self_attention_rows(causal):
    """The last n_q rows of self-attention over N_k positions are exactly the decode form."""
    B, H, N, D, nq = 1, 2, 19, 8, 5
    q, k, v = (_rand((B, H, N, D), 100 + s) for s in range(3))
    o_full, l_full = oracle.forward(q, k, v, 0.45, causal)
    o, l = oracle.forward_kv(q[:, :, N - nq:], k, v, 0.45, causal)
    np.testing.assert_allclose(o, o_full[:, :, N - nq:], atol=1e-13)
    np.testing.assert_allclose(l, l_full[:, :, N - nq:], atol=1e-13)


def test_decode_form_closed_forms_and_library():
    """Q = 0 gives the mean of the visible V rows (causal: the first N_k - n_q + i + 1);
    general inputs match torch float64 SDPA with an explicit end-aligned causal mask."""
    B, H, N, D, nq = 2, 1, 23, 6, 4
    k, v = _rand((B, H, N, D), 110), _rand((B, H, N, D), 111)
    o, lse = oracle.forward_kv(np.zeros((B, H, nq, D)), k, v, 0.3, True)
    for i in range(nq):
        nvis = N - nq + i + 1
        np.testing.assert_allclose(o[:, :, i], v[:, :, :nvis].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(nvis), atol=1e-13)
    q = _rand((B, H, nq, D), 112)
    mask = torch.tensor(np.arange(N)[None, :] <= (N - nq + np.arange(nq))[:, None])
    for causal in (False, True):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q), torch.tensor(k), torch.tensor(v), attn_mask=mask if causal else None, scale=0.3)
        o, _ = oracle.forward_kv(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        oracle.forward_rows(q, q, q, 1.0, False, [(0, 0, 4)])
