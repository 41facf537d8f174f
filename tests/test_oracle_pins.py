"""Pins of the fp64 oracle to facts other than itself.

Each check targets a plausible mistake: a wrong branch or alpha in phi, a
dropped diagonal, a read-before-update in decode, a transposed state (D != M
everywhere), a wrong sign or a prefix/suffix swap in the backward.  The pins
are hand-derived values (tests/golden), closed forms, library routines
(numpy cumsum/einsum, torch autograd), two independent algorithms agreeing,
finite differences and invariants of the definition.
"""
import ast
import json
import math
import operator
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
E = math.e


def _eval_expr(s: str) -> float:
    """Evaluates a golden expression: numbers, e, + - * / and parentheses only."""
    ops = {ast.Add: operator.add, ast.Sub: operator.sub, ast.Mult: operator.mul,
           ast.Div: operator.truediv, ast.USub: operator.neg, ast.UAdd: operator.pos}

    def ev(n):
        if isinstance(n, ast.Expression):
            return ev(n.body)
        if isinstance(n, ast.Constant) and isinstance(n.value, (int, float)):
            return float(n.value)
        if isinstance(n, ast.Name) and n.id == "e":
            return E
        if isinstance(n, ast.BinOp) and type(n.op) in ops:
            return ops[type(n.op)](ev(n.left), ev(n.right))
        if isinstance(n, ast.UnaryOp) and type(n.op) in ops:
            return ops[type(n.op)](ev(n.operand))
        raise ValueError(f"disallowed expression: {s}")

    return ev(ast.parse(s, mode="eval"))


def _arr(x):
    return np.vectorize(_eval_expr, otypes=[float])(np.array(x, dtype=object))


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _phi_np(x):
    # numpy restatement used only to build independent library-routine checks;
    # phi itself is pinned by test_phi_closed_form.
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


# ------------------------------------------------------------------ phi

def test_phi_closed_form():
    assert oracle.phi(0.0) == 1.0
    assert oracle.phi(1.0) == 2.0
    assert oracle.phi(2.5) == 3.5
    assert oracle.phi(-1.0) == pytest.approx(1.0 / E, rel=1e-15)
    assert oracle.phi(-3.0) == pytest.approx(math.exp(-3.0), rel=1e-14)
    # continuous at 0 and strictly positive
    assert oracle.phi(1e-12) == pytest.approx(1.0, abs=1e-11)
    assert oracle.phi(-1e-12) == pytest.approx(1.0, abs=1e-11)
    assert oracle.phi(-700.0) > 0.0
    # derivative: 1 for x > 0, e^x for x <= 0 (alpha = 1, so C^1 at 0)
    assert oracle.dphi(1.0) == 1.0
    assert oracle.dphi(0.0) == 1.0
    assert oracle.dphi(-2.0) == pytest.approx(math.exp(-2.0), rel=1e-15)


def test_dphi_matches_central_difference():
    for x in (-3.0, -0.7, -1e-3, 0.4, 2.0):
        h = 1e-6
        fd = (oracle.phi(x + h) - oracle.phi(x - h)) / (2 * h)
        assert oracle.dphi(x) == pytest.approx(fd, rel=1e-8)


# ----------------------------------------------------- golden hand examples

def test_golden_forward_causal_both_forms():
    g = _golden()["forward_3x2x2"]
    Q, K, V = (np.array(g[k], float) for k in ("Q", "K", "V"))
    want = _arr(g["causal_O"])
    np.testing.assert_allclose(oracle.causal_forward_quadratic(Q, K, V), want, rtol=1e-14)
    O, S, Z, den = oracle.causal_forward_recurrent(Q, K, V, return_den=True)
    np.testing.assert_allclose(O, want, rtol=1e-14)
    np.testing.assert_allclose(S, _arr(g["S_total"]), rtol=1e-14)
    np.testing.assert_allclose(Z, _arr(g["Z_total"]), rtol=1e-14)
    np.testing.assert_allclose(den, _arr(g["causal_den"]), rtol=1e-14)
    # the state after two tokens
    _, S2, Z2 = oracle.causal_forward_recurrent(Q[:2], K[:2], V[:2])
    np.testing.assert_allclose(S2, _arr(g["S_after_2"]), rtol=1e-14)
    np.testing.assert_allclose(Z2, _arr(g["Z_after_2"]), rtol=1e-14)


def test_golden_forward_noncausal_both_forms():
    g = _golden()["forward_3x2x2"]
    Q, K, V = (np.array(g[k], float) for k in ("Q", "K", "V"))
    want = _arr(g["noncausal_O"])
    np.testing.assert_allclose(oracle.noncausal_forward_quadratic(Q, K, V), want, rtol=1e-14)
    O, S, Z = oracle.noncausal_forward_assoc(Q, K, V)
    np.testing.assert_allclose(O, want, rtol=1e-14)
    np.testing.assert_allclose(S, _arr(g["S_total"]), rtol=1e-14)
    np.testing.assert_allclose(Z, _arr(g["Z_total"]), rtol=1e-14)


def test_golden_decode_updates_then_reads():
    g = _golden()["forward_3x2x2"]
    Q, K, V = (np.array(g[k], float) for k in ("Q", "K", "V"))
    S2, Z2 = _arr(g["S_after_2"]), _arr(g["Z_after_2"])
    out, S3, Z3 = oracle.decode_step(Q[2], K[2], V[2], S2, Z2)
    np.testing.assert_allclose(out, _arr(g["decode_out_step3"]), rtol=1e-14)
    np.testing.assert_allclose(S3, _arr(g["S_total"]), rtol=1e-14)
    np.testing.assert_allclose(Z3, _arr(g["Z_total"]), rtol=1e-14)


@pytest.mark.parametrize("case", ["backward_2x1x1", "backward_2x2x1"])
def test_golden_backward_both_forms(case):
    g = _golden()[case]
    Q, K, V, G = (np.array(g[k], float) for k in ("Q", "K", "V", "G"))
    want = [_arr(g[k]) for k in ("dQ", "dK", "dV")]
    for got in (oracle.causal_backward_cumsum(Q, K, V, G), oracle.causal_backward_quadratic(Q, K, V, G)):
        for a, b in zip(got, want):
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------ forward pins

SHAPES = [(1, 1, 3, 2), (2, 7, 3, 5), (3, 33, 4, 2), (1, 64, 8, 16), (2, 17, 16, 8)]


@pytest.mark.parametrize("nh,N,D,M", SHAPES)
def test_causal_quadratic_equals_recurrent(nh, N, D, M):
    Q, K, V = _rand((nh, N, D), 1), _rand((nh, N, D), 2), _rand((nh, N, M), 3)
    a = oracle.causal_forward_quadratic(Q, K, V)
    b, _, _ = oracle.causal_forward_recurrent(Q, K, V)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_first_row_is_v1_and_threads_do_not_matter():
    Q, K, V = _rand((5, 40, 6), 4), _rand((5, 40, 6), 5), _rand((5, 40, 3), 6)
    O1, S1, Z1 = oracle.causal_forward_recurrent(Q, K, V, nthreads=1)
    O4, S4, Z4 = oracle.causal_forward_recurrent(Q, K, V, nthreads=4)
    np.testing.assert_allclose(O1[:, 0], V[:, 0], rtol=1e-14)
    assert np.array_equal(O1, O4) and np.array_equal(S1, S4) and np.array_equal(Z1, Z4)


def test_equal_keys_give_prefix_mean():
    nh, N, D, M = 2, 25, 4, 3
    Q, V = _rand((nh, N, D), 7), _rand((nh, N, M), 8)
    K = np.broadcast_to(_rand((nh, 1, D), 9), (nh, N, D)).copy()
    want = np.cumsum(V, axis=1) / np.arange(1, N + 1)[None, :, None]
    for O in (oracle.causal_forward_quadratic(Q, K, V), oracle.causal_forward_recurrent(Q, K, V)[0]):
        np.testing.assert_allclose(O, want, rtol=1e-12, atol=1e-13)
    # non-causal: every row is the mean of all V
    On = oracle.noncausal_forward_assoc(Q, K, V)[0]
    np.testing.assert_allclose(On, np.broadcast_to(V.mean(axis=1, keepdims=True), On.shape),
                               rtol=1e-12, atol=1e-13)


def test_d1_is_weighted_prefix_mean():
    # With D = 1 the query factor cancels: O_i = sum_{j<=i} phi(k_j) V_j / sum_{j<=i} phi(k_j).
    N, M = 30, 4
    Q, K, V = _rand((1, N, 1), 10), _rand((1, N, 1), 11), _rand((1, N, M), 12)
    w = _phi_np(K[0, :, 0])
    want = np.cumsum(w[:, None] * V[0], axis=0) / np.cumsum(w)[:, None]
    np.testing.assert_allclose(oracle.causal_forward_recurrent(Q, K, V)[0][0], want, rtol=1e-12)


def test_convex_hull_and_translation():
    nh, N, D, M = 3, 50, 5, 4
    Q, K, V = _rand((nh, N, D), 13), _rand((nh, N, D), 14), _rand((nh, N, M), 15)
    O = oracle.causal_forward_recurrent(Q, K, V)[0]
    lo = np.minimum.accumulate(V, axis=1)
    hi = np.maximum.accumulate(V, axis=1)
    assert np.all(O >= lo - 1e-12) and np.all(O <= hi + 1e-12)
    c = _rand((1, 1, M), 16)
    O2 = oracle.causal_forward_recurrent(Q, K, V + c)[0]
    np.testing.assert_allclose(O2, O + c, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("nh,N,D,M", SHAPES)
def test_noncausal_forms_and_states(nh, N, D, M):
    Q, K, V = _rand((nh, N, D), 17), _rand((nh, N, D), 18), _rand((nh, N, M), 19)
    a = oracle.noncausal_forward_quadratic(Q, K, V)
    b, S, Z = oracle.noncausal_forward_assoc(Q, K, V)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
    # states equal the library contraction phi(K)^T V and the column sums of phi(K)
    fk = _phi_np(K)
    np.testing.assert_allclose(S, np.einsum("hnd,hne->hde", fk, V), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Z, fk.sum(axis=1), rtol=1e-13)
    # causal last row == non-causal row; recurrent final state == total state
    Oc, Sc, Zc = oracle.causal_forward_recurrent(Q, K, V)
    np.testing.assert_allclose(Oc[:, -1], a[:, -1], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Zc, Z, rtol=1e-13)


def test_recurrent_carry_in_state_splits_sequence():
    nh, N, D, M, cut = 2, 40, 6, 3, 17
    Q, K, V = _rand((nh, N, D), 20), _rand((nh, N, D), 21), _rand((nh, N, M), 22)
    O, S, Z = oracle.causal_forward_recurrent(Q, K, V)
    Oa, Sa, Za = oracle.causal_forward_recurrent(Q[:, :cut], K[:, :cut], V[:, :cut])
    Ob, Sb, Zb = oracle.causal_forward_recurrent(Q[:, cut:], K[:, cut:], V[:, cut:], Sa, Za)
    np.testing.assert_allclose(np.concatenate([Oa, Ob], 1), O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Zb, Z, rtol=1e-13)


def test_decode_continues_the_causal_forward():
    nh, N0, T, D, M = 3, 12, 9, 4, 5
    Q, K, V = _rand((nh, N0 + T, D), 23), _rand((nh, N0 + T, D), 24), _rand((nh, N0 + T, M), 25)
    O_full, S_full, Z_full = oracle.causal_forward_recurrent(Q, K, V)
    _, S, Z = oracle.causal_forward_recurrent(Q[:, :N0], K[:, :N0], V[:, :N0])
    for t in range(T):
        out, S, Z = oracle.decode_step(Q[:, N0 + t], K[:, N0 + t], V[:, N0 + t], S, Z)
        np.testing.assert_allclose(out, O_full[:, N0 + t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, S_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Z, Z_full, rtol=1e-13)


# ----------------------------------------------------------- backward pins

@pytest.mark.parametrize("nh,N,D,M", SHAPES)
def test_backward_cumsum_equals_quadratic(nh, N, D, M):
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 26), (D, 27), (M, 28), (M, 29)))
    a = oracle.causal_backward_cumsum(Q, K, V, G)
    b = oracle.causal_backward_quadratic(Q, K, V, G)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-11)


def test_backward_finite_differences():
    nh, N, D, M = 1, 7, 3, 2
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 30), (D, 31), (M, 32), (M, 33)))
    dQ, dK, dV = oracle.causal_backward_cumsum(Q, K, V, G)

    def loss(q, k, v):
        return float(np.sum(G * oracle.causal_forward_recurrent(q, k, v)[0]))

    h = 1e-6
    for X, dX, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            xp, xm = X.copy(), X.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(dX, fd, rtol=1e-6, atol=1e-8)


def test_backward_matches_torch_autograd():
    nh, N, D, M = 2, 19, 5, 3
    arrays = [_rand((nh, N, x), s) for x, s in ((D, 34), (D, 35), (M, 36), (M, 37))]
    Q, K, V, G = (torch.tensor(a, dtype=torch.float64) for a in arrays)
    Q.requires_grad_(True)
    K.requires_grad_(True)
    V.requires_grad_(True)
    fq = torch.nn.functional.elu(Q, alpha=1.0) + 1.0
    fk = torch.nn.functional.elu(K, alpha=1.0) + 1.0
    w = torch.tril(fq @ fk.transpose(-1, -2))
    O = (w @ V) / w.sum(-1, keepdim=True)
    (O * G).sum().backward()
    got = oracle.causal_backward_cumsum(*arrays)
    for a, b in zip(got, (Q.grad, K.grad, V.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(oracle.causal_forward_recurrent(*arrays[:3])[0],
                               O.detach().numpy(), rtol=1e-11, atol=1e-12)


def test_backward_invariants():
    nh, N, D, M = 3, 45, 6, 4
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 38), (D, 39), (M, 40), (M, 41)))
    dQ, dK, dV = oracle.causal_backward_cumsum(Q, K, V, G)
    # translation equivariance of O in V: sum_j dV_j = sum_i G_i
    np.testing.assert_allclose(dV.sum(axis=1), G.sum(axis=1), rtol=1e-10, atol=1e-11)
    # O_i is invariant to scaling phi(Q_i), and to scaling every phi(K_j) of a head
    fq, fk = _phi_np(Q), _phi_np(K)
    dfq = dQ / np.where(Q > 0, 1.0, np.exp(np.minimum(Q, 0.0)))
    dfk = dK / np.where(K > 0, 1.0, np.exp(np.minimum(K, 0.0)))
    np.testing.assert_allclose((fq * dfq).sum(-1), 0.0, atol=1e-10)
    np.testing.assert_allclose((fk * dfk).sum(axis=(1, 2)), 0.0, atol=1e-9)
    # row 1 of the causal output depends on V_1 only: its query gets no gradient
    np.testing.assert_allclose(dQ[:, 0], 0.0, atol=1e-13)


# ------------------------------------------------ non-causal backward pins

@pytest.mark.parametrize("case", ["noncausal_backward_2x1x1", "noncausal_backward_2x2x1"])
def test_golden_noncausal_backward_both_forms(case):
    g = _golden()[case]
    Q, K, V, G = (np.array(g[k], float) for k in ("Q", "K", "V", "G"))
    np.testing.assert_allclose(oracle.noncausal_forward_assoc(Q, K, V)[0], _arr(g["O"]), rtol=1e-14)
    want = [_arr(g[k]) for k in ("dQ", "dK", "dV")]
    for got in (oracle.noncausal_backward_assoc(Q, K, V, G), oracle.noncausal_backward_quadratic(Q, K, V, G)):
        for a, b in zip(got, want):
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("nh,N,D,M", SHAPES)
def test_noncausal_backward_state_equals_quadratic(nh, N, D, M):
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 70), (D, 71), (M, 72), (M, 73)))
    a = oracle.noncausal_backward_assoc(Q, K, V, G)
    b = oracle.noncausal_backward_quadratic(Q, K, V, G)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-11)


def test_noncausal_backward_finite_differences():
    nh, N, D, M = 1, 6, 3, 2
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 74), (D, 75), (M, 76), (M, 77)))
    grads = oracle.noncausal_backward_assoc(Q, K, V, G)

    def loss(q, k, v):
        return float(np.sum(G * oracle.noncausal_forward_assoc(q, k, v)[0]))

    h = 1e-6
    for which, (X, dX) in enumerate(zip((Q, K, V), grads)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            xp, xm = X.copy(), X.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p, args_m = [Q, K, V], [Q, K, V]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(dX, fd, rtol=1e-6, atol=1e-8)


def test_noncausal_backward_matches_torch_autograd():
    nh, N, D, M = 2, 23, 5, 3
    arrays = [_rand((nh, N, x), s) for x, s in ((D, 78), (D, 79), (M, 80), (M, 81))]
    Q, K, V, G = (torch.tensor(a, dtype=torch.float64) for a in arrays)
    for t in (Q, K, V):
        t.requires_grad_(True)
    fq = torch.nn.functional.elu(Q, alpha=1.0) + 1.0
    fk = torch.nn.functional.elu(K, alpha=1.0) + 1.0
    w = fq @ fk.transpose(-1, -2)
    O = (w @ V) / w.sum(-1, keepdim=True)
    (O * G).sum().backward()
    got = oracle.noncausal_backward_assoc(*arrays)
    for a, b in zip(got, (Q.grad, K.grad, V.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-12)


def test_noncausal_backward_invariants():
    nh, N, D, M = 3, 41, 6, 4
    Q, K, V, G = (_rand((nh, N, x), s) for x, s in ((D, 82), (D, 83), (M, 84), (M, 85)))
    dQ, dK, dV = oracle.noncausal_backward_assoc(Q, K, V, G)
    np.testing.assert_allclose(dV.sum(axis=1), G.sum(axis=1), rtol=1e-10, atol=1e-11)
    fq, fk = _phi_np(Q), _phi_np(K)
    dfq = dQ / np.where(Q > 0, 1.0, np.exp(np.minimum(Q, 0.0)))
    dfk = dK / np.where(K > 0, 1.0, np.exp(np.minimum(K, 0.0)))
    np.testing.assert_allclose((fq * dfq).sum(-1), 0.0, atol=1e-10)
    np.testing.assert_allclose((fk * dfk).sum(axis=(1, 2)), 0.0, atol=1e-9)
    # one token: the non-causal and causal gradients coincide (O_1 = V_1, so dQ = dK = 0, dV = G)
    a = oracle.noncausal_backward_assoc(Q[:, :1], K[:, :1], V[:, :1], G[:, :1])
    np.testing.assert_allclose(a[2], G[:, :1], rtol=1e-14)
    np.testing.assert_allclose(a[0], 0.0, atol=1e-14)


# --------------------------------------------- softmax KV-cache decode pins

@pytest.mark.parametrize("case", ["a", "b"])
def test_golden_softmax_decode(case):
    g = _golden()["softmax_decode_T1"][case]
    q, k, v, Kc, Vc = (np.array(g[n], float) for n in ("q", "k", "v", "Kc", "Vc"))
    out = oracle.softmax_decode_step(q[None], k[None], v[None], Kc[None], Vc[None])[0]
    np.testing.assert_allclose(out, _arr(g["out"]), rtol=1e-14)


def test_softmax_decode_matches_library_softmax_and_special_cases():
    nh, T, D, M = 3, 37, 8, 5
    q, k, v = _rand((nh, D), 90), _rand((nh, D), 91), _rand((nh, M), 92)
    Kc, Vc = _rand((nh, T, D), 93), _rand((nh, T, M), 94)
    out = oracle.softmax_decode_step(q, k, v, Kc, Vc)
    Kt = torch.tensor(np.concatenate([Kc, k[:, None]], 1))
    Vt = torch.tensor(np.concatenate([Vc, v[:, None]], 1))
    w = torch.softmax(torch.einsum("hd,htd->ht", torch.tensor(q), Kt) / math.sqrt(D), dim=-1)
    np.testing.assert_allclose(out, torch.einsum("ht,htm->hm", w, Vt).numpy(), rtol=1e-12, atol=1e-13)
    # empty cache: the only position is the new one
    np.testing.assert_allclose(oracle.softmax_decode_step(q, k, v, Kc[:, :0], Vc[:, :0]), v, rtol=1e-15)
    # every key equal: the mean of the values
    Ke = np.broadcast_to(k[:, None], (nh, T, D)).copy()
    np.testing.assert_allclose(oracle.softmax_decode_step(q, k, v, Ke, Vc),
                               np.concatenate([Vc, v[:, None]], 1).mean(axis=1), rtol=1e-12)
    # a common shift of every key moves every score equally: the output is unchanged
    c = _rand((nh, 1, D), 95)
    np.testing.assert_allclose(oracle.softmax_decode_step(q, k + c[:, 0], v, Kc + c, Vc), out,
                               rtol=1e-11, atol=1e-12)


# ------------------------------------------------------- retention pins

def _ret_case(name):
    g = _golden()[name]
    q, k, v = (np.array(g[n], float) for n in ("q", "k", "v"))
    if q.ndim == 1:
        q, k, v = q[:, None], k[:, None], v[:, None]
    return g, q[None, None], k[None, None], v[None, None]


def test_golden_retention_scalar():
    g, Q, K, V = _ret_case("retention_3x1x1")
    gam = np.array([_eval_expr(g["gamma"])])
    gates = _arr(g["gates"])[None, None]
    for kw, want in (({}, "y_decay1"), ({"gamma_head": gam}, "y_retnet"), ({"gates": gates}, "y_gated")):
        w = _arr(g[want])
        np.testing.assert_allclose(oracle.retention_forward_recurrent(Q, K, V, **kw)[0][0, 0, :, 0], w,
                                   rtol=1e-14)
        np.testing.assert_allclose(oracle.retention_forward_quadratic(Q, K, V, **kw)[0, 0, :, 0], w,
                                   rtol=1e-14)


def test_golden_retention_orientation():
    g, Q, K, V = _ret_case("retention_2x2x2")
    O, S = oracle.retention_forward_recurrent(Q, K, V)
    np.testing.assert_allclose(O[0, 0], _arr(g["y_decay1"]), rtol=1e-14)
    np.testing.assert_allclose(S[0, 0], _arr(g["S_decay1"]), rtol=1e-14)
    O, S = oracle.retention_forward_recurrent(Q, K, V, gamma_head=np.array([0.5]))
    np.testing.assert_allclose(O[0, 0], _arr(g["y_half"]), rtol=1e-14)
    np.testing.assert_allclose(S[0, 0], _arr(g["S_half"]), rtol=1e-14)
    # decode continues: the second token as a decode step after the first
    _, S1 = oracle.retention_forward_recurrent(Q[:, :, :1], K[:, :, :1], V[:, :, :1])
    out, S2 = oracle.retention_decode_step(Q[0, 0, 1], K[0, 0, 1], V[0, 0, 1], np.array(0.5), S1[0, 0])
    np.testing.assert_allclose(out, _arr(g["y_half"])[1], rtol=1e-14)
    np.testing.assert_allclose(S2, _arr(g["S_half"]), rtol=1e-14)


def test_retention_against_library_masks():
    B, H, N, D, M = 2, 3, 29, 5, 4
    Q, K, V = _rand((B, H, N, D), 110), _rand((B, H, N, D), 111), _rand((B, H, N, M), 112)
    A = np.einsum("bhid,bhjd->bhij", Q, K)
    # decay 1: y = tril(Q K^T) V
    np.testing.assert_allclose(oracle.retention_forward_recurrent(Q, K, V)[0],
                               np.tril(A) @ V, rtol=1e-11, atol=1e-12)
    # RetNet: y = (tril(Q K^T) * gamma^(i-j)) V, one gamma per head
    gam = np.array([0.9, 0.5, 0.99])
    i = np.arange(N)
    Gm = np.where(i[:, None] >= i[None, :], gam[:, None, None] ** np.maximum(i[:, None] - i[None, :], 0), 0.0)
    want = (A * Gm[None]) @ V
    np.testing.assert_allclose(oracle.retention_forward_recurrent(Q, K, V, gamma_head=gam)[0], want,
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(oracle.retention_forward_quadratic(Q, K, V, gamma_head=gam), want,
                               rtol=1e-10, atol=1e-12)


def test_retention_gated_forms_and_special_cases():
    B, H, N, D, M = 2, 2, 33, 4, 3
    Q, K, V = _rand((B, H, N, D), 113), _rand((B, H, N, D), 114), _rand((B, H, N, M), 115)
    gates = np.random.default_rng(116).uniform(0.5, 1.0, (B, H, N))
    a = oracle.retention_forward_recurrent(Q, K, V, gates=gates)[0]
    np.testing.assert_allclose(a, oracle.retention_forward_quadratic(Q, K, V, gates=gates), rtol=1e-10,
                               atol=1e-12)
    # gates equal to a per-head constant are RetNet
    gam = np.array([0.8, 0.95])
    np.testing.assert_allclose(
        oracle.retention_forward_recurrent(Q, K, V, gates=np.broadcast_to(gam[None, :, None], (B, H, N)))[0],
        oracle.retention_forward_recurrent(Q, K, V, gamma_head=gam)[0], rtol=1e-13)
    # zero decay forgets everything: y_t = (q_t . k_t) v_t
    y0 = oracle.retention_forward_recurrent(Q, K, V, gates=np.zeros((B, H, N)))[0]
    np.testing.assert_allclose(y0, np.einsum("bhnd,bhnd->bhn", Q, K)[..., None] * V, rtol=1e-12)
    # a carried-in state splits the sequence
    cut = 14
    O, S = oracle.retention_forward_recurrent(Q, K, V, gates=gates)
    Oa, Sa = oracle.retention_forward_recurrent(Q[:, :, :cut], K[:, :, :cut], V[:, :, :cut], gates=gates[:, :, :cut])
    Ob, Sb = oracle.retention_forward_recurrent(Q[:, :, cut:], K[:, :, cut:], V[:, :, cut:],
                                                gates=gates[:, :, cut:], S0=Sa)
    np.testing.assert_allclose(np.concatenate([Oa, Ob], 2), O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-13)
    # decode steps continue the forward
    _, Sd = oracle.retention_forward_recurrent(Q[:, :, :cut], K[:, :, :cut], V[:, :, :cut], gates=gates[:, :, :cut])
    for t in range(cut, N):
        out, Sd = oracle.retention_decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], gates[:, :, t], Sd)
        np.testing.assert_allclose(out, O[:, :, t], rtol=1e-11, atol=1e-12)


# ------------------------------------------- degree-2 polynomial kernel pins

def test_golden_poly_both_forms():
    g = _golden()["poly_2x2x1"]
    Q, K, V = (np.array(g[k], float) for k in ("Q", "K", "V"))
    for causal, key in ((True, "causal_O"), (False, "noncausal_O")):
        want = _arr(g[key])
        np.testing.assert_allclose(oracle.poly_forward_quadratic(Q, K, V, causal), want, rtol=1e-14)
        np.testing.assert_allclose(oracle.poly_forward_state(Q, K, V, causal), want, rtol=1e-14)


@pytest.mark.parametrize("nh,N,D,M", [(1, 9, 2, 3), (2, 30, 4, 5), (3, 17, 8, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_poly_forms_agree_and_match_library(nh, N, D, M, causal):
    Q, K, V = _rand((nh, N, D), 130), _rand((nh, N, D), 131), _rand((nh, N, M), 132)
    a = oracle.poly_forward_quadratic(Q, K, V, causal)
    b = oracle.poly_forward_state(Q, K, V, causal)
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)
    W = np.einsum("hid,hjd->hij", Q, K) ** 2
    if causal:
        W = np.tril(W)
    np.testing.assert_allclose(a, (W @ V) / W.sum(-1, keepdims=True), rtol=1e-11, atol=1e-12)


def test_poly_invariants():
    nh, N, D, M = 2, 40, 4, 3
    Q, K, V = _rand((nh, N, D), 133), _rand((nh, N, D), 134), _rand((nh, N, M), 135)
    O = oracle.poly_forward_state(Q, K, V)
    np.testing.assert_allclose(O[:, 0], V[:, 0], rtol=1e-13)       # row 1 sees only V_1
    sgn = np.where(np.random.default_rng(136).random((nh, N, 1)) < 0.5, -1.0, 1.0)
    np.testing.assert_allclose(oracle.poly_forward_state(Q * sgn, -K, V), O, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(oracle.poly_forward_state(3.0 * Q, 0.5 * K, V), O, rtol=1e-11, atol=1e-12)
    lo, hi = np.minimum.accumulate(V, axis=1), np.maximum.accumulate(V, axis=1)
    assert np.all(O >= lo - 1e-12) and np.all(O <= hi + 1e-12)
    Ke = np.broadcast_to(K[:, :1], K.shape).copy()
    np.testing.assert_allclose(oracle.poly_forward_quadratic(Q, Ke, V),
                               np.cumsum(V, 1) / np.arange(1, N + 1)[None, :, None], rtol=1e-12)
