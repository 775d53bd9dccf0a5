"""The pins catch plausible mistakes: each planted variant of the oracle
(compiled from the same C source with ORACLE_PLANT=n, on the CPU) must fail at
least one pin, while the oracle itself passes all of them."""
import math

import numpy as np
import pytest

from tests._common import rel_err
from tests.test_oracle_pins import _fd_grad, _small, _torch_reference


def _pins(oracle, lib):
    """name -> passed, for a compact battery of the pins in test_oracle_pins."""
    res = {}
    s = 0.45
    for causal in (False, True):
        q, k, v, dO = _small(n=1, T=6, d=3, seed=2)
        g = oracle.backward(q, k, v, dO, causal, s, lib=lib)
        ok = True
        for which, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
            for idx in np.ndindex(*grad.shape):
                fd = _fd_grad(oracle, q, k, v, dO, causal, s, which, idx, lib=lib)
                ok &= abs(fd - grad[idx]) <= 1e-7 * max(np.max(np.abs(grad)), 1e-30)
        res[f"fd_causal{int(causal)}"] = bool(ok)
        t = _torch_reference(q, k, v, dO, causal, s)
        res[f"autograd_causal{int(causal)}"] = all(
            rel_err(g[key], t[key]) <= 1e-10 for key in ("O", "dQ", "dK", "dV")
        ) and float(np.max(np.abs(g["LSE"] - t["LSE"]))) <= 1e-12
        r = oracle.backward(q, k, v, dO, causal, s, mode="E", want_matrices=True, lib=lib)
        res[f"rowsum_dS_causal{int(causal)}"] = bool(
            np.max(np.abs(r["dS"].sum(-1))) <= 1e-12 * np.linalg.norm(r["dS"]))
    # block-sparse mask (asymmetric) against the autograd route
    q, k, v, dO = _small(n=1, T=8, Tk=10, d=3, seed=5)
    bm = np.array([[1, 1, 0], [0, 1, 1], [1, 0, 1]])  # not symmetric
    g = oracle.backward(q, k, v, dO, False, s, block_mask=bm, block=4, lib=lib)
    t = _torch_reference(q, k, v, dO, False, s, block_mask=bm, block=4)
    res["autograd_block_mask"] = all(
        rel_err(g[key], t[key]) <= 1e-10 for key in ("O", "dQ", "dK", "dV"))
    # local window (Tq < Tk) against the autograd route
    q, k, v, dO = _small(n=1, T=6, Tk=9, d=3, seed=6)
    g = oracle.backward(q, k, v, dO, False, s, window=(2, 1), lib=lib)
    t = _torch_reference(q, k, v, dO, False, s, window=(2, 1))
    res["autograd_window"] = all(
        rel_err(g[key], t[key]) <= 1e-10 for key in ("O", "dQ", "dK", "dV"))
    # a query block that keeps no key block: LSE = -inf, O = 0
    q, k, v, dO = _small(n=1, T=8, d=3, seed=8)
    O, L, _ = oracle.forward(q, k, v, False, s, block_mask=[[1, 1], [0, 0]], block=4, lib=lib)
    res["empty_rows"] = bool(np.all(np.isneginf(L[0, 4:])) and np.all(O[0, 4:] == 0)
                             and np.all(np.isfinite(L[0, :4])))
    # last row: causal == non-causal
    q, k, v, dO = _small(n=1, T=6, d=3, seed=4)
    Oc, Lc, _ = oracle.forward(q, k, v, True, s, lib=lib)
    On, Ln, _ = oracle.forward(q, k, v, False, s, lib=lib)
    res["last_row"] = rel_err(Oc[:, -1], On[:, -1]) <= 1e-14
    # hand-derived two-token example
    l3 = math.log(3.0)
    q = np.array([[[0.0], [l3]]]); k = np.array([[[0.0], [1.0]]])
    v = np.array([[[0.0], [1.0]]]); dO = np.array([[[1.0], [1.0]]])
    r = oracle.backward(q, k, v, dO, False, 1.0, lib=lib)
    res["hand_example"] = bool(
        np.allclose(r["LSE"][0], [math.log(2), math.log(4)], rtol=1e-14)
        and np.allclose(r["dQ"][0, :, 0], [0.25, 3 / 16], rtol=1e-13)
        and np.allclose(r["dK"][0, :, 0], [-3 * l3 / 16, 3 * l3 / 16], rtol=1e-13)
        and np.allclose(r["dV"][0, :, 0], [0.75, 1.25], rtol=1e-14))
    return res


def test_oracle_passes_every_pin(oracle_mod):
    res = _pins(oracle_mod, None)
    assert all(res.values()), res


@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_planted_mistake_is_caught(oracle_mod, plant):
    lib = oracle_mod.planted(plant)
    res = _pins(oracle_mod, lib)
    failed = [k for k, ok in res.items() if not ok]
    assert failed, f"planted mistake {plant} passed every pin"
