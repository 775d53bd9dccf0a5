"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI
binding, run the oracle on the same bf16 inputs, compare with the stated
tolerances.  (Layout marshalling and comparisons only; no attention math.)"""
import numpy as np
import torch

import oracle
from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn
from tests._common import max_abs, rel_err, row_err

# Tolerances (bf16 inputs, fp32 accumulation): normwise relative error for
# O and for dQ/dK/dV, maximum absolute error for the natural-log LSE.
TOL_O = 5e-3
TOL_GRAD = 1e-2
TOL_LSE = 1e-4
# Per row of O, dQ, dK, dV (beside the normwise bounds): the error norm of a
# row may be at most 5 % of that row's norm (or of the rms row norm, for rows
# whose exact values are near zero), so a single wrong row or tile cannot hide
# in a whole-tensor norm.  A CPU model of the kernels' bf16 rounding points
# (P, dP - D, dS, O before D, the outputs) reproduces the GPU's errors and puts
# the worst row of 36 seeded problem sets at 2.8e-2 for dQ (short causal rows,
# whose dS entries cancel) and below 1e-2 for O, dK and dV.
TOL_ROW = 5e-2


def run_gpu(x, w, deterministic=None, with_lse=True, window=None):
    """Forward + backward of workload ``w`` on inputs ``x`` (CPU bf16 tensors)."""
    dev = torch.device("cuda:0")
    det = w.deterministic if deterministic is None else deterministic
    cu = x.get("cu_seqlens")
    cu_list = None if cu is None else [int(c) for c in cu]
    if w.layout == syn.LAYOUT_PACKED:
        qkv = x["qkv"].to(dev)
        q, k, v = qkv.select(-3, 0), qkv.select(-3, 1), qkv.select(-3, 2)
    else:
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    dO = x["dO"].to(dev)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu_list,
                             layout=w.layout, with_lse=True, window=window)
    dq, dk, dv = binding.backward(q, k, v, o, dO, lse, causal=w.causal, scale=w.scale,
                                  cu_seqlens=cu_list, layout=w.layout, deterministic=det,
                                  window=window)
    torch.cuda.synchronize()
    assert binding.attn_fwd_status() == 0
    out = {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}
    return {key: val.float().cpu() for key, val in out.items()}


def problems(t, w, cu=None):
    """Per-(sequence, head) float64 arrays of a (B,T,H,d) or (sum T,H,d) tensor."""
    t = t.float()
    if cu is None:
        x = t.permute(0, 2, 1, 3).contiguous()
        return list(x.reshape(-1, x.shape[2], x.shape[3]).double().numpy())
    out = []
    for s in range(len(cu) - 1):
        for h in range(t.shape[1]):
            out.append(t[cu[s]:cu[s + 1], h, :].double().numpy())
    return out


def lse_problems(lse, w, cu=None):
    if cu is None:
        return list(lse.double().numpy().reshape(-1, lse.shape[-1]))
    out = []
    for s in range(len(cu) - 1):
        for h in range(lse.shape[0]):
            out.append(lse[h, cu[s]:cu[s + 1]].double().numpy())
    return out


def inputs_as_problems(x, w):
    cu = None if "cu_seqlens" not in x else [int(c) for c in x["cu_seqlens"]]
    return [problems(x[n], w, cu) for n in ("q", "k", "v", "dO")], cu


def compare_full(x, w, g, pick=None, window=None, block_mask=None):
    """Full oracle on the problems in `pick` (all when None); returns error dict.

    block_mask: optional [n_problems][NQ][NK] array (problem order as in
    problems()), blocks of binding.BLOCK rows.  Rows the oracle gives LSE =
    -inf (no visible key) must be -inf on the GPU too; the LSE error is taken
    over the other rows."""
    (q, k, v, dO), cu = inputs_as_problems(x, w)
    idx = list(range(len(q))) if pick is None else list(pick)
    sel = lambda lst: [lst[i] for i in idx]
    bm = None if block_mask is None else np.asarray(block_mask)[idx]
    r = oracle.backward(sel(q), sel(k), sel(v), sel(dO), w.causal, w.scale, window=window,
                        block_mask=bm, block=binding.BLOCK)
    gp = {key: sel(problems(g[key], w, cu)) for key in ("O", "dQ", "dK", "dV")}
    gl = sel(lse_problems(g["LSE"], w, cu))
    cat = lambda a: np.concatenate([np.asarray(z).reshape(-1) for z in a])
    rows = lambda a: np.concatenate([np.asarray(z).reshape(-1, np.asarray(z).shape[-1])
                                     for z in a])
    as_list = lambda a: a if isinstance(a, list) else list(a)
    err = {key: rel_err(cat(gp[key]), cat(as_list(r[key]))) for key in ("O", "dQ", "dK", "dV")}
    for key in ("O", "dQ", "dK", "dV"):
        err[key + "_row"] = row_err(rows(gp[key]), rows(as_list(r[key])))
    ref_lse = cat(r["LSE"] if isinstance(r["LSE"], list) else list(r["LSE"]))
    got_lse = cat(gl)
    empty = np.isneginf(ref_lse)
    if not np.array_equal(np.isneginf(got_lse), empty):
        err["LSE"] = float("inf")
    else:
        err["LSE"] = max_abs(got_lse[~empty], ref_lse[~empty]) if (~empty).any() else 0.0
    return err


def sample_rows(T, n, seed):
    base = [0, 1, 63, 64, 127, 128, 129, T // 2, T - 129, T - 128, T - 2, T - 1]
    rng = np.random.default_rng(seed)
    extra = rng.choice(T, size=min(n, T), replace=False)
    rows = sorted({int(r) for r in base + list(extra) if 0 <= r < T})
    return np.array(rows, dtype=np.int32)


def compare_sampled(x, w, g, heads, n_rows=48, kv_heads=(), seed=0):
    """Oracle on sampled query rows (O, LSE, dQ) of `heads` and sampled key rows
    (dK, dV) of `kv_heads`, all computed one row / one key at a time."""
    (q, k, v, dO), cu = inputs_as_problems(x, w)
    gp = {key: problems(g[key], w, cu) for key in ("O", "dQ", "dK", "dV")}
    gl = lse_problems(g["LSE"], w, cu)
    acc = {key: ([], []) for key in ("O", "dQ", "dK", "dV", "LSE")}
    for p in heads:
        T = q[p].shape[0]
        rows = sample_rows(T, n_rows, seed + p)
        r = oracle.backward([q[p]], [k[p]], [v[p]], [dO[p]], w.causal, w.scale, rows=[rows])
        for key in ("O", "dQ"):
            acc[key][0].append(gp[key][p][rows])
            acc[key][1].append(np.asarray(r[key])[0][rows])
        acc["LSE"][0].append(gl[p][rows])
        acc["LSE"][1].append(np.asarray(r["LSE"])[0][rows])
    for p in kv_heads:
        T = k[p].shape[0]
        keys = sample_rows(T, n_rows, seed + 1000 + p)
        _, lse_all, D_all = oracle.forward([q[p]], [k[p]], [v[p]], w.causal, w.scale, dO=[dO[p]])
        dk, dv = oracle.kv_rows(q[p], k[p], v[p], dO[p], np.asarray(lse_all)[0],
                                np.asarray(D_all)[0], keys, w.causal, w.scale)
        acc["dK"][0].append(gp["dK"][p][keys]); acc["dK"][1].append(dk)
        acc["dV"][0].append(gp["dV"][p][keys]); acc["dV"][1].append(dv)
    err = {}
    for key, (a, b) in acc.items():
        if not a:
            continue
        if key != "LSE":
            err[key + "_row"] = row_err(np.concatenate([z.reshape(-1, z.shape[-1]) for z in a]),
                                        np.concatenate([z.reshape(-1, z.shape[-1]) for z in b]))
        a = np.concatenate([z.reshape(-1) for z in a])
        b = np.concatenate([z.reshape(-1) for z in b])
        err[key] = max_abs(a, b) if key == "LSE" else rel_err(a, b)
    return err


def compare_forward_sampled(x, w, o, heads, n_rows=48, seed=0):
    """O of the inference-mode forward (no LSE) at sampled query rows of
    `heads`, against the oracle's forward computed row by row."""
    (q, k, v, _), cu = inputs_as_problems(x, w)
    go = problems(o, w, cu)
    got, ref = [], []
    for p in heads:
        rows = sample_rows(q[p].shape[0], n_rows, seed + p)
        r = oracle.backward([q[p]], [k[p]], [v[p]], [np.zeros((q[p].shape[0], v[p].shape[1]))],
                            w.causal, w.scale, rows=[rows])
        got.append(go[p][rows])
        ref.append(np.asarray(r["O"])[0][rows])
    a, b = np.concatenate(got), np.concatenate(ref)
    return {"O": rel_err(a.reshape(-1), b.reshape(-1)), "O_row": row_err(a, b)}


def assert_within(err, where=""):
    limits = {"O": TOL_O, "dQ": TOL_GRAD, "dK": TOL_GRAD, "dV": TOL_GRAD, "LSE": TOL_LSE,
              "O_row": TOL_ROW, "dQ_row": TOL_ROW, "dK_row": TOL_ROW, "dV_row": TOL_ROW}
    bad = {k: v for k, v in err.items() if not (v <= limits[k])}
    assert not bad, f"{where}: {err}"
