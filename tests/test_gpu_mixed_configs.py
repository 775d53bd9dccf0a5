"""Seeded mixes of every option on the GPU against the oracle.

Each case draws (from a fixed seed) a head size, a batch form (fixed length
with Tq <= Tk or not, variable length with shared or separate offsets), causal
or not, a local window or none, a block mask or none, fast or deterministic
mode, and small ragged lengths; the CUDA path must meet the usual tolerances
and leave both status words clear.  The cases are listed by `mixed_cases()`
so that they can be read before they run."""
import numpy as np
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from tests import gpu_common as gc
from tests._common import max_abs, rel_err

BL = binding.BLOCK
DIMS = [(64, 64), (128, 128), (192, 128)]


def mixed_cases(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(n):
        d, dv = DIMS[c % 3]
        form = ["fixed", "varlen", "varlen_qk"][(c // 3) % 3]
        packed = c >= 12  # the last cases use the packed (.., 3, H, d) layout
        if packed:
            d = dv = (64, 128)[c % 2]
            form = ("fixed", "varlen")[(c // 2) % 2]
        causal = bool(rng.integers(2))
        window = None
        if rng.random() < 0.4:
            window = (int(rng.choice([-1, 0, 40, 150])), int(rng.choice([-1, 0, 25, 300])))
            if causal:
                window = (window[0], -1)
        banded = causal or (window is not None and (window[0] >= 0 or window[1] >= 0))
        H = int(rng.integers(1, 4))
        if form == "fixed":
            B = int(rng.integers(1, 3))
            Tk = int(rng.integers(1, 700))
            Tq = int(rng.integers(1, Tk + 1)) if banded else int(rng.integers(1, 700))
            if packed:
                Tq = Tk
            lq, lk = (Tq,) * B, (Tk,) * B
        else:
            B = int(rng.integers(1, 5))
            lk = tuple(int(x) for x in rng.integers(1, 520, B))
            if form == "varlen":
                lq = lk
            else:
                lq = tuple(int(rng.integers(0, k + 1)) if banded else int(rng.integers(0, 520))
                           for k in lk)
        density = [None, 0.35, 0.75][int(rng.integers(3))]
        det = bool(rng.integers(2))
        cases.append(dict(id=c, d=d, dv=dv, form=form, causal=causal, window=window, H=H,
                          lq=lq, lk=lk, density=density, det=det, packed=packed))
    return cases


def _split(t, cu):
    t = t.float()
    return [t[cu[s]:cu[s + 1], h, :].double().numpy()
            for s in range(len(cu) - 1) for h in range(t.shape[1])]


@pytest.mark.gpu
@pytest.mark.parametrize("case", mixed_cases(), ids=lambda c: f"case{c['id']}")
def test_mixed_case_against_oracle(case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import oracle
    from attention_backward_flashattention_gb300 import build
    build.build()
    oracle.build()
    d, dv, H, lq, lk = case["d"], case["dv"], case["H"], case["lq"], case["lk"]
    fixed = case["form"] == "fixed"
    g0 = torch.Generator().manual_seed(500 + case["id"])
    cq = [0] + [int(x) for x in np.cumsum(lq)]
    ck = [0] + [int(x) for x in np.cumsum(lk)]
    x = {"q": torch.randn(cq[-1], H, d, generator=g0).bfloat16(),
         "k": torch.randn(ck[-1], H, d, generator=g0).bfloat16(),
         "v": torch.randn(ck[-1], H, dv, generator=g0).bfloat16(),
         "dO": torch.randn(cq[-1], H, dv, generator=g0).bfloat16()}
    dev = "cuda:0"
    B = len(lq)
    if fixed:  # (B, T, H, d) views of the same rows
        t = {n: x[n].view(B, -1, H, x[n].shape[-1]).to(dev) for n in x}
        kw = {}
    else:
        t = {n: x[n].to(dev) for n in x}
        kw = dict(cu_seqlens=cq, cu_seqlens_k=ck if case["form"] == "varlen_qk" else None)
    if case["packed"]:  # q, k, v as slots of one (.., 3, H, d) buffer
        qkv = torch.stack([t["q"], t["k"], t["v"]], dim=-3).contiguous()
        t.update(q=qkv.select(-3, 0), k=qkv.select(-3, 1), v=qkv.select(-3, 2))
        kw["layout"] = binding.LAYOUT_PACKED_QKV
    mask = bm = None
    nq, nk = -(-max(max(lq), 1) // BL), -(-max(lk) // BL)
    if case["density"] is not None:
        mask = (np.random.default_rng(600 + case["id"]).random((1, H, nq, nk))
                < case["density"]).astype(np.uint8)
        bm = torch.from_numpy(mask).to(dev)
    scale = 1.0 / np.sqrt(d)
    o, lse = binding.forward(t["q"], t["k"], t["v"], causal=case["causal"], scale=scale,
                             window=case["window"], block_mask=bm, **kw)
    dq, dk, dvv = binding.backward(t["q"], t["k"], t["v"], o, t["dO"], lse,
                                   causal=case["causal"], scale=scale, window=case["window"],
                                   block_mask=bm, deterministic=case["det"], **kw)
    torch.cuda.synchronize()
    assert binding.attn_fwd_status() == 0
    flat = lambda a, rows: a.reshape(rows, H, a.shape[-1]).cpu()
    g = {"O": flat(o, cq[-1]), "dQ": flat(dq, cq[-1]), "dK": flat(dk, ck[-1]),
         "dV": flat(dvv, ck[-1])}
    lse = lse.cpu().double().numpy()
    got_lse = (np.concatenate([lse[b, h] for b in range(B) for h in range(H)]) if fixed else
               np.concatenate([lse[h, cq[s]:cq[s + 1]] for s in range(B) for h in range(H)]))
    qs, ks, vs, dOs = (_split(x[n], c) for n, c in (("q", cq), ("k", ck), ("v", ck), ("dO", cq)))
    pm = None if mask is None else np.broadcast_to(mask, (B, H, nq, nk)).reshape(B * H, nq, nk)
    r = oracle.backward(qs, ks, vs, dOs, case["causal"], scale, window=case["window"],
                        block_mask=pm, block=BL)
    cat = lambda a: np.concatenate([np.asarray(z).reshape(-1) for z in a])
    err = {key: rel_err(cat(_split(g[key], cu)), cat(r[key]))
           for key, cu in (("O", cq), ("dQ", cq), ("dK", ck), ("dV", ck))}
    ref = cat(r["LSE"])
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got_lse), empty), "rows without keys"
    err["LSE"] = max_abs(got_lse[~empty], ref[~empty]) if (~empty).any() else 0.0
    gc.assert_within(err, str(case))
