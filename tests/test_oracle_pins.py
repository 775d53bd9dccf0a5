"""Pins of the fp64 oracle against things other than itself (CPU only).

Every check here ties the oracle to the mathematics of the pages
("ops(8)：self-attention 的 CUDA 实现及优化 (下) - 深度分析", §2.1 forward and
backward formulas, §2.2 CPU reference loop, Appendix A.1-A.3): central finite
differences of the scalar loss L = sum(O * dO), invariants of the softmax
Jacobian, closed forms on degenerate inputs, a hand-derived two-token example,
and an independent route (PyTorch CPU fp64 autograd).
"""
import math

import numpy as np
import pytest
import torch

from tests._common import rel_err, to_problems

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _small(n=2, T=16, d=8, dv=None, seed=0, Tk=None):
    dv = d if dv is None else dv
    Tk = T if Tk is None else Tk
    return (_rand((n, T, d), seed), _rand((n, Tk, d), seed + 1),
            _rand((n, Tk, dv), seed + 2), _rand((n, T, dv), seed + 3))


def _fd_grad(oracle, q, k, v, dO, causal, scale, which, idx, h=1e-6, lib=None, window=None):
    """Central difference of L = sum(O * dO) w.r.t. one entry of q, k or v."""
    args = {"q": q, "k": k, "v": v}
    plus = {kk: vv.copy() for kk, vv in args.items()}
    minus = {kk: vv.copy() for kk, vv in args.items()}
    plus[which][idx] += h
    minus[which][idx] -= h
    Op, _, _ = oracle.forward(plus["q"], plus["k"], plus["v"], causal, scale, lib=lib,
                              window=window)
    Om, _, _ = oracle.forward(minus["q"], minus["k"], minus["v"], causal, scale, lib=lib,
                              window=window)
    return float(((np.asarray(Op) - np.asarray(Om)) * dO).sum() / (2 * h))


def _torch_reference(q, k, v, dO, causal, scale, window=None, block_mask=None, block=None):
    """PyTorch CPU fp64 autograd of softmax(s Q K^T + mask) V (independent route).

    block_mask: [nqb][nkb] array expanded to an element mask with a Kronecker
    product (every block entry becomes a block x block square)."""
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    S = scale * qt @ kt.transpose(-1, -2)
    Tq, Tk = S.shape[-2:]
    off = Tk - Tq
    keep = torch.ones(Tq, Tk, dtype=torch.bool)
    if causal:
        # query i is position Tk - Tq + i of the key sequence (bottom-right
        # alignment; top-left when Tq == Tk): keys after it are masked
        keep &= torch.ones(Tq, Tk, dtype=torch.bool).tril(off)
    if window is not None:
        # local window: keys i+off-left .. i+off+right (a negative bound is open)
        left, right = window
        if right >= 0:
            keep &= torch.ones(Tq, Tk, dtype=torch.bool).tril(off + right)
        if left >= 0:
            keep &= torch.ones(Tq, Tk, dtype=torch.bool).triu(off - left)
    if block_mask is not None:
        bm = torch.tensor(np.asarray(block_mask) != 0, dtype=torch.float64)
        dense = torch.kron(bm, torch.ones(block, block, dtype=torch.float64)) > 0
        keep &= dense[:Tq, :Tk]
    if not bool(keep.all()):
        S = S.masked_fill(~keep, float("-inf"))
    P = torch.softmax(S, dim=-1)
    O = P @ vt
    lse = torch.logsumexp(S, dim=-1)
    O.backward(torch.tensor(dO, dtype=torch.float64))
    return {"O": O.detach().numpy(), "LSE": lse.detach().numpy(),
            "dQ": qt.grad.numpy(), "dK": kt.grad.numpy(), "dV": vt.grad.numpy()}


# --------------------------------------------------------------------------
# finite differences
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_every_entry(oracle_mod, causal):
    """Every entry of dQ, dK, dV at T=16, d=8, H=2 against central differences."""
    q, k, v, dO = _small(n=2, T=16, d=8)
    scale = 0.35
    g = oracle_mod.backward(q, k, v, dO, causal, scale)
    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            fd[idx] = _fd_grad(oracle_mod, q, k, v, dO, causal, scale, which, idx)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err <= 1e-7, (which, err)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_tiny_config_sampled(oracle_mod, causal):
    """256 seeded entries per tensor on the tiny workload (bf16 inputs, d=64)."""
    from attention_backward_flashattention_gb300 import synthetic as syn
    w = syn.TINY[1] if causal else syn.TINY[0]
    x = syn.make_inputs(w)
    q, k, v, dO = (to_problems(x[n]) for n in ("q", "k", "v", "dO"))
    g = oracle_mod.backward(q, k, v, dO, causal, w.scale)
    rng = np.random.default_rng(7)
    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        flat = rng.choice(grad.size, size=256, replace=False)
        scale_ref = np.max(np.abs(grad))
        worst = 0.0
        for f in flat:
            idx = np.unravel_index(f, grad.shape)
            fd = _fd_grad(oracle_mod, q, k, v, dO, causal, w.scale, which, idx)
            worst = max(worst, abs(fd - grad[idx]) / scale_ref)
        assert worst <= 1e-7, (which, worst)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_invariants(oracle_mod, causal):
    q, k, v, dO = _small(n=3, T=24, d=16, dv=8, seed=11)
    s = 0.25
    r = oracle_mod.backward(q, k, v, dO, causal, s, mode="E", want_matrices=True)
    P, dS = r["P"], r["dS"]
    # rows of P sum to one; rows of dS sum to zero (J 1 = 0)
    assert np.max(np.abs(P.sum(-1) - 1.0)) <= 1e-13
    assert np.max(np.abs(dS.sum(-1))) <= 1e-12 * np.linalg.norm(dS)
    # D = rowsum(dO * O) = rowsum(P * dP)
    dP = dO @ v.transpose(0, 2, 1)
    D_def = (P * dP).sum(-1)
    D_io = (dO * r["O"]).sum(-1)
    assert rel_err(r["D"], D_def) <= 1e-12
    assert rel_err(D_io, D_def) <= 1e-12
    # dV = P^T dO from the explicitly formed P; dQ, dK from the explicit dS
    assert rel_err(r["dV"], P.transpose(0, 2, 1) @ dO) <= 1e-12
    assert rel_err(r["dQ"], s * dS @ k) <= 1e-12
    assert rel_err(r["dK"], s * dS.transpose(0, 2, 1) @ q) <= 1e-12
    # O = P V and LSE from the explicit P
    assert rel_err(r["O"], P @ v) <= 1e-12
    if causal:
        upper = np.triu(np.ones(P.shape[-2:], dtype=bool), 1)
        assert np.all(P[:, upper] == 0.0) and np.all(dS[:, upper] == 0.0)


def test_causal_masking_properties(oracle_mod):
    q, k, v, dO = _small(n=2, T=20, d=8, seed=21)
    s = 0.4
    T = q.shape[1]
    r = oracle_mod.backward(q, k, v, dO, True, s, mode="E", want_matrices=True)
    # the last key is seen by the last query only
    P, dS = r["P"], r["dS"]
    assert rel_err(r["dV"][:, -1], P[:, -1, -1, None] * dO[:, -1]) <= 1e-13
    assert rel_err(r["dK"][:, -1], s * dS[:, -1, -1, None] * q[:, -1]) <= 1e-13
    # perturbing keys / values above the diagonal leaves earlier rows unchanged
    O0, L0, _ = oracle_mod.forward(q, k, v, True, s)
    for i in (0, 5, 13):
        k2, v2 = k.copy(), v.copy()
        k2[:, i + 1:] += _rand(k2[:, i + 1:].shape, 99)
        v2[:, i + 1:] += _rand(v2[:, i + 1:].shape, 98)
        O1, L1, _ = oracle_mod.forward(q, k2, v2, True, s)
        assert np.array_equal(O1[:, :i + 1], O0[:, :i + 1])
        assert np.array_equal(L1[:, :i + 1], L0[:, :i + 1])
    # the last query row sees every key: causal and non-causal agree there
    Onc, Lnc, _ = oracle_mod.forward(q, k, v, False, s)
    assert rel_err(O0[:, T - 1], Onc[:, T - 1]) <= 1e-14
    assert rel_err(L0[:, T - 1], Lnc[:, T - 1]) <= 1e-14
    # gradients only flow to keys at or before the query
    rows = [np.array([7]), np.array([7])]
    rr = oracle_mod.backward(q, k, v, dO, True, s, rows=rows)
    assert np.all(rr["dK"][:, 8:] == 0.0) and np.all(rr["dV"][:, 8:] == 0.0)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_single_token(oracle_mod):
    """T=1: O=V, LSE=s q.k, dV=dO, dQ=dK=0 (softmax of one score is 1)."""
    q, k, v, dO = _small(n=4, T=1, d=8, dv=5, seed=3)
    s = 0.7
    for causal in (False, True):
        r = oracle_mod.backward(q, k, v, dO, causal, s)
        assert np.allclose(r["O"], v, rtol=0, atol=1e-15)
        assert np.allclose(r["LSE"][:, 0], s * (q[:, 0] * k[:, 0]).sum(-1), rtol=1e-15, atol=0)
        assert np.allclose(r["dV"], dO, rtol=0, atol=1e-15)
        assert np.max(np.abs(r["dQ"])) <= 1e-15 and np.max(np.abs(r["dK"])) <= 1e-15


def test_uniform_attention(oracle_mod):
    """Q = 0, non-causal: every score is 0, so P = 1/T."""
    _, k, v, dO = _small(n=2, T=12, d=6, dv=4, seed=5)
    q = np.zeros_like(k)
    T = k.shape[1]
    r = oracle_mod.backward(q, k, v, dO, False, 0.5)
    assert rel_err(r["O"], np.broadcast_to(v.mean(1, keepdims=True), r["O"].shape)) <= 1e-14
    assert np.allclose(r["LSE"], math.log(T), rtol=1e-15, atol=0)
    assert rel_err(r["dV"], np.broadcast_to(dO.sum(1, keepdims=True) / T, r["dV"].shape)) <= 1e-14
    # dK = s dS^T Q = 0 when Q = 0
    assert np.max(np.abs(r["dK"])) == 0.0


def test_causal_first_row(oracle_mod):
    """Causal row 0 sees key 0 only: O_0 = V_0, LSE_0 = s q_0.k_0, dQ_0 = 0."""
    q, k, v, dO = _small(n=2, T=9, d=8, seed=8)
    s = 0.3
    r = oracle_mod.backward(q, k, v, dO, True, s)
    assert np.allclose(r["O"][:, 0], v[:, 0], rtol=0, atol=1e-15)
    assert np.allclose(r["LSE"][:, 0], s * (q[:, 0] * k[:, 0]).sum(-1), rtol=1e-15, atol=0)
    assert np.max(np.abs(r["dQ"][:, 0])) <= 1e-15


def _golden_value(expr):
    """Evaluate a fixture entry such as '3*ln3/16' (ln2/ln3/ln4 and rationals only)."""
    env = {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln4": math.log(4.0)}
    return float(eval(expr, {"__builtins__": {}}, env))


def _golden(name):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    with open(path) as f:
        return json.load(f)


def test_hand_derived_two_token_example(oracle_mod):
    """Two tokens, d=1, s=1, worked by hand (tests/golden/two_token_example.json)."""
    g = _golden("two_token_example.json")
    ev = lambda a: np.vectorize(_golden_value, otypes=[float])(np.array(a))
    inp = g["inputs"]
    q, k, v, dO = (ev(inp[n]).reshape(1, 2, 1) for n in ("q", "k", "v", "dO"))
    exp = {key: ev(val) for key, val in g["expected"].items()}
    for mode in ("R", "E"):
        r = oracle_mod.backward(q, k, v, dO, inp["causal"], inp["scale"], mode=mode,
                                want_matrices=True)
        np.testing.assert_allclose(r["O"][0, :, 0], exp["O"], rtol=1e-15)
        np.testing.assert_allclose(r["LSE"][0], exp["LSE"], rtol=1e-15)
        np.testing.assert_allclose(r["D"][0], exp["D"], rtol=1e-15)
        np.testing.assert_allclose(r["dS"][0], exp["dS"], rtol=1e-14)
        np.testing.assert_allclose(r["dQ"][0, :, 0], exp["dQ"], rtol=1e-14)
        np.testing.assert_allclose(r["dK"][0, :, 0], exp["dK"], rtol=1e-14)
        np.testing.assert_allclose(r["dV"][0, :, 0], exp["dV"], rtol=1e-15)


# --------------------------------------------------------------------------
# two backward forms and an independent route
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_jacobian_and_rowjvp_agree_tiny(oracle_mod, causal):
    from attention_backward_flashattention_gb300 import synthetic as syn
    w = syn.TINY[1] if causal else syn.TINY[0]
    x = syn.make_inputs(w)
    q, k, v, dO = (to_problems(x[n]) for n in ("q", "k", "v", "dO"))
    rE = oracle_mod.backward(q, k, v, dO, causal, w.scale, mode="E")
    rR = oracle_mod.backward(q, k, v, dO, causal, w.scale, mode="R")
    for key in ("dQ", "dK", "dV"):
        assert rel_err(rR[key], rE[key]) <= 1e-12, key


@pytest.mark.parametrize("causal", [False, True])
def test_torch_autograd_route_tiny(oracle_mod, causal):
    from attention_backward_flashattention_gb300 import synthetic as syn
    w = syn.TINY[1] if causal else syn.TINY[0]
    x = syn.make_inputs(w)
    q, k, v, dO = (to_problems(x[n]) for n in ("q", "k", "v", "dO"))
    r = oracle_mod.backward(q, k, v, dO, causal, w.scale)
    t = _torch_reference(q, k, v, dO, causal, w.scale)
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(r[key], t[key]) <= 1e-10, key
    assert np.max(np.abs(r["LSE"] - t["LSE"])) <= 1e-12


def test_gpt2_shaped_heads_against_autograd_and_jacobian(oracle_mod):
    """A seeded subset of (batch, head) problems of the GPT-2-shaped layer."""
    from attention_backward_flashattention_gb300 import synthetic as syn
    w = syn.GPT2
    x = syn.make_inputs(w)
    q, k, v, dO = (to_problems(x[n]) for n in ("q", "k", "v", "dO"))
    pick = np.random.default_rng(1).choice(q.shape[0], size=3, replace=False)
    q, k, v, dO = q[pick], k[pick], v[pick], dO[pick]
    r = oracle_mod.backward(q, k, v, dO, True, w.scale)
    t = _torch_reference(q, k, v, dO, True, w.scale)
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(r[key], t[key]) <= 1e-10, key
    assert np.max(np.abs(r["LSE"] - t["LSE"])) <= 1e-11
    rE = oracle_mod.backward(q[:1], k[:1], v[:1], dO[:1], True, w.scale, mode="E")
    for key in ("dQ", "dK", "dV"):
        assert rel_err(r[key][:1], rE[key]) <= 1e-12, key


# --------------------------------------------------------------------------
# the sampled entry points used at full sizes agree with the full oracle
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_row_and_column_sampling_matches_full(oracle_mod, causal):
    q, k, v, dO = _small(n=2, T=40, d=16, dv=8, seed=31)
    s = 0.25
    full = oracle_mod.backward(q, k, v, dO, causal, s)
    rows = [np.array([0, 3, 39]), np.array([17, 39])]
    part = oracle_mod.backward(q, k, v, dO, causal, s, rows=rows)
    for p, rr in enumerate(rows):
        for key in ("dQ", "O", "LSE", "D"):
            np.testing.assert_allclose(part[key][p][rr], full[key][p][rr], rtol=1e-14, atol=1e-15)
    O, lse, D = oracle_mod.forward(q, k, v, causal, s, dO=dO)
    np.testing.assert_allclose(D, full["D"], rtol=1e-13, atol=1e-15)
    keys = np.array([0, 1, 20, 39])
    for p in range(2):
        dk, dvv = oracle_mod.kv_rows(q[p], k[p], v[p], dO[p], lse[p], D[p], keys, causal, s)
        np.testing.assert_allclose(dk, full["dK"][p][keys], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dvv, full["dV"][p][keys], rtol=1e-11, atol=1e-13)
    # the row-sampled dK/dV contributions of all rows add up to the full gradient
    halves = [[np.arange(0, 20), np.arange(0, 20)], [np.arange(20, 40), np.arange(20, 40)]]
    a = oracle_mod.backward(q, k, v, dO, causal, s, rows=halves[0])
    b = oracle_mod.backward(q, k, v, dO, causal, s, rows=halves[1])
    assert rel_err(a["dK"] + b["dK"], full["dK"]) <= 1e-13
    assert rel_err(a["dV"] + b["dV"], full["dV"]) <= 1e-13


def test_unequal_lengths_are_independent_problems(oracle_mod):
    lens = [5, 17, 1, 9]
    parts = [_small(n=1, T=L, d=8, seed=40 + i) for i, L in enumerate(lens)]
    q = [p[0][0] for p in parts]
    k = [p[1][0] for p in parts]
    v = [p[2][0] for p in parts]
    dO = [p[3][0] for p in parts]
    r = oracle_mod.backward(q, k, v, dO, True, 0.3)
    for i in range(len(lens)):
        ri = oracle_mod.backward(q[i][None], k[i][None], v[i][None], dO[i][None], True, 0.3)
        for key in ("dQ", "dK", "dV", "O", "LSE"):
            np.testing.assert_array_equal(r[key][i], ri[key][0])


def test_noncausal_rectangular(oracle_mod):
    """Tq != Tk is defined for the non-causal case; FD on a few entries."""
    q, k, v, dO = _small(n=1, T=7, d=4, seed=50, Tk=11)
    s = 0.6
    g = oracle_mod.backward(q, k, v, dO, False, s)
    t = _torch_reference(q, k, v, dO, False, s)
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(g[key], t[key]) <= 1e-12
    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        idx = (0, 2, 1)
        assert abs(_fd_grad(oracle_mod, q, k, v, dO, False, s, which, idx) - grad[idx]) <= 1e-8


def test_rejects_causal_with_more_queries_than_keys(oracle_mod):
    """Bottom-right causal with Tq > Tk would leave query rows that see no key."""
    q, k, v, dO = _small(n=1, T=11, d=4, seed=50, Tk=7)
    with pytest.raises(ValueError):
        oracle_mod.backward(q, k, v, dO, True, 0.5)


def test_causal_rectangular_against_autograd_and_fd(oracle_mod):
    """Causal with fewer queries than keys (bottom-right): the autograd route
    with the shifted triangular mask, and central differences of every entry."""
    q, k, v, dO = _small(n=2, T=6, d=3, seed=51, Tk=10)
    s = 0.7
    g = oracle_mod.backward(q, k, v, dO, True, s)
    t = _torch_reference(q, k, v, dO, True, s)
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(g[key], t[key]) <= 1e-12, key
    assert float(np.max(np.abs(g["LSE"] - t["LSE"]))) <= 1e-12
    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        scale_ref = max(np.max(np.abs(grad)), 1e-30)
        for idx in np.ndindex(*grad.shape):
            fd = _fd_grad(oracle_mod, q, k, v, dO, True, s, which, idx)
            assert abs(fd - grad[idx]) <= 1e-7 * scale_ref, (which, idx)


def test_causal_rectangular_is_the_tail_of_a_square_problem(oracle_mod):
    """The Tq queries of a bottom-right causal problem behave exactly like the
    last Tq queries of the square causal problem over the same keys (whose
    other queries have dO = 0, so they add nothing to dK or dV)."""
    Tq, Tk, d = 5, 12, 4
    q, k, v, dO = _small(n=1, T=Tq, d=d, seed=52, Tk=Tk)
    pre_q, _, _, _ = _small(n=1, T=Tk - Tq, d=d, seed=53)
    qs = np.concatenate([pre_q, q], axis=1)
    dOs = np.concatenate([np.zeros((1, Tk - Tq, d)), dO], axis=1)
    s = 0.45
    rect = oracle_mod.backward(q, k, v, dO, True, s)
    sq = oracle_mod.backward(qs, k, v, dOs, True, s)
    for key in ("O", "LSE", "dQ"):
        np.testing.assert_allclose(rect[key][0], sq[key][0][Tk - Tq:], rtol=1e-13, atol=1e-15)
    for key in ("dK", "dV"):
        np.testing.assert_allclose(rect[key], sq[key], rtol=1e-12, atol=1e-15)


def test_causal_single_query_sees_every_key(oracle_mod):
    """Tq = 1 (one decoding step): bottom-right causal equals non-causal."""
    q, k, v, dO = _small(n=2, T=1, d=5, seed=54, Tk=9)
    a = oracle_mod.backward(q, k, v, dO, True, 0.4)
    b = oracle_mod.backward(q, k, v, dO, False, 0.4)
    for key in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(a[key], b[key])


# --------------------------------------------------------------------------
# local (sliding-window) attention
# --------------------------------------------------------------------------
WINDOWS = [((2, 1), False), ((3, 0), False), ((4, -1), False), ((-1, 2), False),
           ((2, -1), True), ((0, 0), False)]


@pytest.mark.parametrize("window,causal", WINDOWS)
def test_window_against_autograd_and_fd(oracle_mod, window, causal):
    """Local attention: the autograd route with banded masks, and central
    differences of every entry (Tq < Tk, so the band is shifted by Tk - Tq)."""
    q, k, v, dO = _small(n=1, T=7, d=3, seed=70, Tk=10)
    s = 0.6
    g = oracle_mod.backward(q, k, v, dO, causal, s, window=window)
    t = _torch_reference(q, k, v, dO, causal, s, window=window)
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(g[key], t[key]) <= 1e-12, key
    assert float(np.max(np.abs(g["LSE"] - t["LSE"]))) <= 1e-12
    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        ref = max(np.max(np.abs(grad)), 1e-30)
        for idx in np.ndindex(*grad.shape):
            fd = _fd_grad(oracle_mod, q, k, v, dO, causal, s, which, idx, window=window)
            assert abs(fd - grad[idx]) <= 1e-7 * ref, (which, idx)


def test_window_special_cases(oracle_mod):
    q, k, v, dO = _small(n=2, T=9, d=4, seed=71)
    s = 0.5
    full = oracle_mod.backward(q, k, v, dO, False, s)
    causal = oracle_mod.backward(q, k, v, dO, True, s)
    wide = oracle_mod.backward(q, k, v, dO, False, s, window=(50, 50))
    open_right = oracle_mod.backward(q, k, v, dO, False, s, window=(-1, 0))
    for key in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(wide[key], full[key])          # band wider than T
        np.testing.assert_array_equal(open_right[key], causal[key])  # (open, 0) = causal
    # (0, 0): each query sees only its own key: O = V, dQ = dK = 0, dV = dO
    diag = oracle_mod.backward(q, k, v, dO, False, s, window=(0, 0))
    np.testing.assert_allclose(diag["O"], v, rtol=1e-14)
    np.testing.assert_allclose(diag["LSE"], s * np.einsum("ntd,ntd->nt", q, k), rtol=1e-13)
    assert np.max(np.abs(diag["dQ"])) == 0 and np.max(np.abs(diag["dK"])) == 0
    np.testing.assert_allclose(diag["dV"], dO, rtol=1e-14)


def test_window_masks_exactly_the_band(oracle_mod):
    """P and dS vanish outside the band and rows of P sum to one inside it."""
    Tq, Tk, (wl, wr) = 6, 11, (2, 3)
    q, k, v, dO = _small(n=1, T=Tq, d=3, seed=72, Tk=Tk)
    r = oracle_mod.backward(q, k, v, dO, False, 0.7, mode="E", want_matrices=True,
                            window=(wl, wr))
    off = Tk - Tq
    for i in range(Tq):
        for j in range(Tk):
            inside = i + off - wl <= j <= i + off + wr
            assert (r["P"][0, i, j] > 0) == inside, (i, j)
            if not inside:
                assert r["dS"][0, i, j] == 0
    np.testing.assert_allclose(r["P"][0].sum(-1), 1.0, rtol=1e-14)


def test_window_key_rows_match_full(oracle_mod):
    q, k, v, dO = _small(n=1, T=8, d=4, seed=73, Tk=12)
    w = (3, 1)
    g = oracle_mod.backward(q, k, v, dO, True, 0.4, window=w)
    _, lse, D = oracle_mod.forward(q, k, v, True, 0.4, dO=dO, window=w)
    keys = np.arange(12)
    dk, dv = oracle_mod.kv_rows(q[0], k[0], v[0], dO[0], np.asarray(lse)[0], np.asarray(D)[0],
                                keys, True, 0.4, window=w)
    np.testing.assert_allclose(dk, g["dK"][0], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dv, g["dV"][0], rtol=1e-12, atol=1e-15)


def test_window_rejects_more_queries_than_keys(oracle_mod):
    q, k, v, dO = _small(n=1, T=9, d=3, seed=74, Tk=5)
    with pytest.raises(ValueError):
        oracle_mod.backward(q, k, v, dO, False, 0.5, window=(2, 2))


# --------------------------------------------------------------------------
# block-sparse masks: key j visible to query i only where the block pair
# (i // block, j // block) is marked, intersected with the band
# --------------------------------------------------------------------------
BLOCK_CASES = [
    # (Tq, Tk, block, causal, window, mask)  -- every row sees some key
    (10, 13, 4, False, None, [[1, 0, 0, 1], [0, 1, 1, 0], [1, 1, 0, 0]]),
    (12, 12, 4, True, None, [[1, 0, 0], [0, 1, 0], [1, 0, 1]]),
    (9, 12, 3, False, (3, 1), [[0, 1, 1, 0], [1, 0, 1, 1], [0, 1, 0, 1]]),
]


@pytest.mark.parametrize("Tq,Tk,block,causal,window,mask", BLOCK_CASES)
def test_block_mask_against_autograd_and_fd(oracle_mod, Tq, Tk, block, causal, window, mask):
    """Block-sparse masks (asymmetric, ragged last blocks, combined with the
    causal band or a window): the autograd route with the Kronecker-expanded
    mask, and central differences of every entry."""
    q, k, v, dO = _small(n=1, T=Tq, d=3, seed=80 + Tq, Tk=Tk)
    s = 0.55
    kw = dict(window=window, block_mask=mask, block=block)
    g = oracle_mod.backward(q, k, v, dO, causal, s, **kw)
    t = _torch_reference(q, k, v, dO, causal, s, **kw)
    assert np.all(np.isfinite(t["LSE"]))  # the case has no empty row
    for key in ("O", "dQ", "dK", "dV"):
        assert rel_err(g[key], t[key]) <= 1e-12, key
    assert float(np.max(np.abs(g["LSE"] - t["LSE"]))) <= 1e-12

    def fd(which, idx, h=1e-6):
        args = {"q": q, "k": k, "v": v}
        plus = {kk: vv.copy() for kk, vv in args.items()}
        minus = {kk: vv.copy() for kk, vv in args.items()}
        plus[which][idx] += h
        minus[which][idx] -= h
        Lp = oracle_mod.loss(plus["q"], plus["k"], plus["v"], dO, causal, s, **kw)
        Lm = oracle_mod.loss(minus["q"], minus["k"], minus["v"], dO, causal, s, **kw)
        return (Lp - Lm) / (2 * h)

    for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        ref = max(np.max(np.abs(grad)), 1e-30)
        for idx in np.ndindex(*grad.shape):
            assert abs(fd(which, idx) - grad[idx]) <= 1e-7 * ref, (which, idx)


@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (False, (2, 3))])
def test_block_mask_of_ones_changes_nothing(oracle_mod, causal, window):
    q, k, v, dO = _small(n=2, T=11, d=4, seed=90)
    s = 0.5
    plain = oracle_mod.backward(q, k, v, dO, causal, s, window=window)
    ones = oracle_mod.backward(q, k, v, dO, causal, s, window=window,
                               block_mask=np.ones((3, 3)), block=4)
    for key in ("O", "LSE", "D", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(ones[key], plain[key])


@pytest.mark.parametrize("causal", [False, True])
def test_block_diagonal_mask_splits_into_independent_segments(oracle_mod, causal):
    """With only the diagonal blocks marked, each block of queries attends to
    its own block of keys alone: the result is that of separate problems."""
    T, b = 24, 8
    q, k, v, dO = _small(n=1, T=T, d=5, seed=91)
    s = 0.4
    g = oracle_mod.backward(q, k, v, dO, causal, s, block_mask=np.eye(3), block=b)
    for seg in range(3):
        sl = slice(seg * b, (seg + 1) * b)
        ref = oracle_mod.backward(q[:, sl], k[:, sl], v[:, sl], dO[:, sl], causal, s)
        for key in ("O", "LSE", "dQ", "dK", "dV"):
            np.testing.assert_allclose(g[key][:, sl], ref[key], rtol=1e-13, atol=1e-15)


def test_block_mask_rows_with_no_key(oracle_mod):
    """A query block with no marked key block: O = 0, LSE = -inf, dQ = D = 0,
    and dK / dV are those of the same problem without these queries."""
    Tq, Tk, b = 24, 20, 8
    mask = np.array([[1, 0, 1], [0, 1, 1], [0, 0, 0]])
    q, k, v, dO = _small(n=1, T=Tq, d=4, seed=92, Tk=Tk)
    s = 0.6
    g = oracle_mod.backward(q, k, v, dO, False, s, block_mask=mask, block=b)
    assert np.all(g["O"][0, 16:] == 0) and np.all(g["dQ"][0, 16:] == 0)
    assert np.all(g["LSE"][0, 16:] == -np.inf) and np.all(g["D"][0, 16:] == 0)
    assert np.all(np.isfinite(g["LSE"][0, :16]))
    cut = oracle_mod.backward(q[:, :16], k, v, dO[:, :16], False, s, block_mask=mask[:2],
                              block=b)
    for key in ("dK", "dV"):
        np.testing.assert_array_equal(g[key], cut[key])
    for key in ("O", "LSE", "dQ"):
        np.testing.assert_array_equal(g[key][:, :16], cut[key])
    # the forward alone agrees
    O, lse, D = oracle_mod.forward(q, k, v, False, s, dO=dO, block_mask=mask, block=b)
    np.testing.assert_array_equal(O, g["O"])
    np.testing.assert_array_equal(lse, g["LSE"])


def test_block_mask_masks_exactly_the_marked_pairs(oracle_mod):
    """P and dS vanish outside (marked blocks AND causal band); rows of P sum to
    one wherever a row sees a key."""
    T, b = 10, 3
    mask = np.array([[1, 0, 1, 1], [1, 1, 0, 0], [0, 1, 1, 0], [1, 0, 0, 1]])
    q, k, v, dO = _small(n=1, T=T, d=3, seed=93)
    r = oracle_mod.backward(q, k, v, dO, True, 0.7, mode="E", want_matrices=True,
                            block_mask=mask, block=b)
    for i in range(T):
        for j in range(T):
            inside = j <= i and mask[i // b, j // b] != 0
            assert (r["P"][0, i, j] > 0) == inside, (i, j)
            if not inside:
                assert r["dS"][0, i, j] == 0
    sums = r["P"][0].sum(-1)
    seen = np.array([any(j <= i and mask[i // b, j // b] for j in range(T)) for i in range(T)])
    np.testing.assert_allclose(sums[seen], 1.0, rtol=1e-14)
    assert np.all(sums[~seen] == 0)


def test_block_mask_key_rows_match_full(oracle_mod):
    q, k, v, dO = _small(n=1, T=12, d=4, seed=94, Tk=16)
    mask = np.array([[1, 0, 0, 1], [0, 0, 0, 0], [1, 1, 0, 1]])  # one empty query block
    kw = dict(block_mask=mask, block=4)
    g = oracle_mod.backward(q, k, v, dO, False, 0.4, **kw)
    _, lse, D = oracle_mod.forward(q, k, v, False, 0.4, dO=dO, **kw)
    dk, dv = oracle_mod.kv_rows(q[0], k[0], v[0], dO[0], np.asarray(lse)[0], np.asarray(D)[0],
                                np.arange(16), False, 0.4, **kw)
    np.testing.assert_allclose(dk, g["dK"][0], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dv, g["dV"][0], rtol=1e-12, atol=1e-15)
    assert np.all(dk[8:12] == 0) and np.all(dv[8:12] == 0)  # key block 2 is never marked


def test_block_mask_must_cover_the_problem(oracle_mod):
    q, k, v, dO = _small(n=1, T=9, d=3, seed=95)
    with pytest.raises(ValueError):
        oracle_mod.backward(q, k, v, dO, False, 0.5, block_mask=np.ones((2, 3)), block=4)
