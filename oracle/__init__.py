"""fp64 CPU oracle for attention forward/backward — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over
independent problems/rows).  This module compiles it with gcc, loads it with
ctypes and moves numpy fp64 arrays in and out.  A "problem" is one
(sequence, head) pair; arrays are ``[n_problems][T][d]`` float64, or, for
problems of unequal length, lists of ``[T][d]`` arrays.

Formulas followed (see the C file for the per-function citations):
"ops(8)：self-attention 的 CUDA 实现及优化 (下) - 深度分析", §2.1 and §2.2,
Appendix A.1-A.3.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, plant: int = 0) -> str:
    """Compile the oracle into ``oracle/_build/`` (gcc, -O2, OpenMP).

    ``plant`` > 0 builds a deliberately wrong variant for the mutation tests
    (see ORACLE_PLANT in attn_oracle.c); 0 is the oracle itself.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    path = _LIB_PATH if plant == 0 else os.path.join(_BUILD_DIR, f"liboracle_plant{plant}.so")
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           f"-DORACLE_PLANT={int(plant)}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _open(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_forward.argtypes = [I, P, P, P, P, I, I, I, I, I, P, I, I, I, D,
                                   P, P, P, P, P, P, P]
    lib.oracle_forward.restype = I
    lib.oracle_backward.argtypes = [I, I, P, P, P, P, I, I, I, I, I, P, I, I, I, D,
                                    P, P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_backward.restype = I
    lib.oracle_kv_rows.argtypes = [I, I, I, I, I, I, I, P, I, I, I, D, P, P, P, P, P, P,
                                   P, I, P, P]
    lib.oracle_kv_rows.restype = I
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
        return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class _Problems:
    """Concatenates per-problem [T][d] blocks and records their row offsets."""

    def __init__(self, q, k, v, dO=None):
        if isinstance(q, np.ndarray) and q.ndim == 3:
            q, k, v = list(q), list(k), list(v)
            dO = None if dO is None else list(dO)
        self.n = len(q)
        self.Tq = np.array([x.shape[0] for x in q], dtype=np.int32)
        self.Tk = np.array([x.shape[0] for x in k], dtype=np.int32)
        self.qrow0 = np.concatenate([[0], np.cumsum(self.Tq)[:-1]]).astype(np.int64)
        self.krow0 = np.concatenate([[0], np.cumsum(self.Tk)[:-1]]).astype(np.int64)
        self.dqk = q[0].shape[1]
        self.dv = v[0].shape[1]
        self.Q = _f64(np.concatenate(q, axis=0))
        self.K = _f64(np.concatenate(k, axis=0))
        self.V = _f64(np.concatenate(v, axis=0))
        self.dO = None if dO is None else _f64(np.concatenate(dO, axis=0))

    def split_q(self, a):
        return [a[o:o + t] for o, t in zip(self.qrow0, self.Tq)]

    def split_k(self, a):
        return [a[o:o + t] for o, t in zip(self.krow0, self.Tk)]


def _stack_if_uniform(parts):
    if len({p.shape for p in parts}) == 1:
        return np.stack(parts)
    return parts


def _window(window):
    """(left, right) bounds of a local window; -1 (or None) leaves a side open."""
    if window is None:
        return -1, -1
    wl, wr = window
    return (-1 if wl is None else int(wl)), (-1 if wr is None else int(wr))


def _blocks(block_mask, nprob, block):
    """uint8 [nprob][nqb][nkb] block masks (a 2-D mask is shared by every
    problem) and the ctypes arguments (pointer, nqb, nkb, block)."""
    if block_mask is None:
        return None, (None, 0, 0, 0)
    m = np.asarray(block_mask)
    if m.ndim == 2:
        m = np.broadcast_to(m, (nprob,) + m.shape)
    if m.ndim != 3 or m.shape[0] != nprob:
        raise ValueError("block_mask must be [nqb][nkb] or [nprob][nqb][nkb]")
    m = np.ascontiguousarray(m != 0, dtype=np.uint8)
    return m, (_ptr(m), int(m.shape[1]), int(m.shape[2]), int(block))


def forward(q, k, v, causal: bool, scale: float, dO=None, lib=None, window=None,
            block_mask=None, block: int = 128):
    """O, LSE (natural log) and, when dO is given, D_i = sum_j P_ij dP_ij.

    q: [nprob][Tq][dqk] (or list), k: [nprob][Tk][dqk], v: [nprob][Tk][dv].
    window: (left, right) local-attention bounds (see attn_oracle.c), or None.
    block_mask: optional [nqb][nkb] or [nprob][nqb][nkb] array; key j is
    visible to query i only where block_mask[i // block][j // block] != 0.
    Returns (O, LSE, D) with D None when dO is None.
    """
    lib = lib or _load()
    pr = _Problems(q, k, v, dO)
    nq = int(pr.Tq.sum())
    O = np.zeros((nq, pr.dv))
    LSE = np.zeros(nq)
    Dv = np.zeros(nq) if dO is not None else None
    wl, wr = _window(window)
    keep, bm = _blocks(block_mask, pr.n, block)
    rc = lib.oracle_forward(pr.n, _ptr(pr.qrow0), _ptr(pr.Tq), _ptr(pr.krow0),
                            _ptr(pr.Tk), pr.dqk, pr.dv, int(causal), wl, wr, *bm,
                            float(scale),
                            _ptr(pr.Q), _ptr(pr.K), _ptr(pr.V), _ptr(pr.dO),
                            _ptr(O), _ptr(LSE), _ptr(Dv))
    if rc != 0:
        raise ValueError(f"oracle_forward failed ({rc})")
    out_D = None if Dv is None else _stack_if_uniform(pr.split_q(Dv))
    return (_stack_if_uniform(pr.split_q(O)), _stack_if_uniform(pr.split_q(LSE)),
            out_D)


def backward(q, k, v, dO, causal: bool, scale: float, mode: str = "R",
             rows=None, want_matrices: bool = False, lib=None, window=None,
             block_mask=None, block: int = 128):
    """Full backward by the chain rule of §2.1.

    mode "R": dS_i = P_i * (dP_i - <P_i, dP_i>) (row Jacobian-vector product);
    mode "E": dS_i = J_i dP_i with the explicit softmax Jacobian (§2.2 loop).
    rows: optional list (one per problem) of query-row index arrays; then only
    those rows' outputs are produced and dK/dV hold only their contributions.
    window, block_mask, block: the visibility rule, as in forward().
    Returns a dict with dQ, dK, dV, O, LSE, D (and P, dS when
    want_matrices).  Arrays are stacked per problem when shapes agree.
    """
    lib = lib or _load()
    pr = _Problems(q, k, v, dO)
    nq, nk = int(pr.Tq.sum()), int(pr.Tk.sum())
    dQ = np.zeros((nq, pr.dqk))
    dK = np.zeros((nk, pr.dqk))
    dV = np.zeros((nk, pr.dv))
    O = np.zeros((nq, pr.dv))
    LSE = np.zeros(nq)
    Dv = np.zeros(nq)
    rows_arr = nrows = None
    if rows is not None:
        rows = [np.asarray(r, dtype=np.int32) for r in rows]
        nrows = np.array([len(r) for r in rows], dtype=np.int32)
        rows_arr = (np.concatenate(rows).astype(np.int32) if len(rows)
                    else np.zeros(0, np.int32))
    Pm = dSm = None
    if want_matrices:
        tot = int((pr.Tq.astype(np.int64) * pr.Tk).sum())
        Pm = np.zeros(tot)
        dSm = np.zeros(tot)
    wl, wr = _window(window)
    keep, bm = _blocks(block_mask, pr.n, block)
    rc = lib.oracle_backward(0 if mode == "R" else 1, pr.n, _ptr(pr.qrow0),
                             _ptr(pr.Tq), _ptr(pr.krow0), _ptr(pr.Tk), pr.dqk,
                             pr.dv, int(causal), wl, wr, *bm, float(scale), _ptr(pr.Q),
                             _ptr(pr.K), _ptr(pr.V), _ptr(pr.dO), _ptr(rows_arr),
                             _ptr(nrows), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(O),
                             _ptr(LSE), _ptr(Dv), _ptr(Pm), _ptr(dSm))
    if rc != 0:
        raise ValueError(f"oracle_backward failed ({rc})")
    out = {
        "dQ": _stack_if_uniform(pr.split_q(dQ)),
        "dK": _stack_if_uniform(pr.split_k(dK)),
        "dV": _stack_if_uniform(pr.split_k(dV)),
        "O": _stack_if_uniform(pr.split_q(O)),
        "LSE": _stack_if_uniform(pr.split_q(LSE)),
        "D": _stack_if_uniform(pr.split_q(Dv)),
    }
    if want_matrices:
        mats_P, mats_dS, off = [], [], 0
        for tq, tk in zip(pr.Tq, pr.Tk):
            n = int(tq) * int(tk)
            mats_P.append(Pm[off:off + n].reshape(tq, tk))
            mats_dS.append(dSm[off:off + n].reshape(tq, tk))
            off += n
        out["P"] = _stack_if_uniform(mats_P)
        out["dS"] = _stack_if_uniform(mats_dS)
    return out


def kv_rows(q, k, v, dO, lse, D, keys, causal: bool, scale: float, lib=None, window=None,
            block_mask=None, block: int = 128):
    """dK, dV at the listed key rows of ONE problem, given its LSE and D.

    q: [Tq][dqk], k: [Tk][dqk], v: [Tk][dv], dO: [Tq][dv], lse/D: [Tq].
    block_mask: optional [nqb][nkb] block mask of this problem.
    Returns (dK_rows [nkeys][dqk], dV_rows [nkeys][dv]).
    """
    lib = lib or _load()
    q, k, v, dO, lse, D = map(_f64, (q, k, v, dO, lse, D))
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    dk = np.zeros((len(keys), q.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    wl, wr = _window(window)
    keep, bm = _blocks(block_mask, 1, block)
    rc = lib.oracle_kv_rows(q.shape[0], k.shape[0], q.shape[1], v.shape[1],
                            int(causal), wl, wr, *bm, float(scale), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(dO), _ptr(lse), _ptr(D), _ptr(keys), len(keys),
                            _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_kv_rows failed ({rc})")
    return dk, dv


def loss(q, k, v, dO, causal: bool, scale: float, lib=None, window=None,
         block_mask=None, block: int = 128) -> float:
    """Scalar L = sum(O * dO) whose gradient the backward returns."""
    O, _, _ = forward(q, k, v, causal, scale, lib=lib, window=window,
                      block_mask=block_mask, block=block)
    if isinstance(O, list):
        return float(sum((o * d).sum() for o, d in zip(O, dO)))
    return float((O * np.asarray(dO)).sum())


def planted(n: int):
    """ctypes handle of a variant with planted mistake ``n`` (mutation tests)."""
    return _open(build(plant=n))
