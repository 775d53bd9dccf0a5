"""Variable-length batches whose queries and keys have separate offsets
(cu_seqlens_q / cu_seqlens_k) on the GPU against the oracle.

Each sequence's queries are the last Lq of its Lk key positions (causal and
windows align bottom-right); the oracle takes each (sequence, head) as a
problem with its own Tq and Tk."""
import numpy as np
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from tests import gpu_common as gc
from tests._common import max_abs, rel_err

pytestmark = pytest.mark.gpu
BL = binding.BLOCK


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()
    import oracle
    oracle.build()


def _split(t, cu):
    """(sum L, H, d) tensor -> [L][d] float64 arrays in (sequence, head) order."""
    t = t.float()
    return [t[cu[s]:cu[s + 1], h, :].double().numpy()
            for s in range(len(cu) - 1) for h in range(t.shape[1])]


def _inputs(lq, lk, H, d, dv, seed):
    cq = [0] + list(np.cumsum(lq))
    ck = [0] + list(np.cumsum(lk))
    g0 = torch.Generator().manual_seed(seed)
    x = {"q": torch.randn(cq[-1], H, d, generator=g0).bfloat16(),
         "k": torch.randn(ck[-1], H, d, generator=g0).bfloat16(),
         "v": torch.randn(ck[-1], H, dv, generator=g0).bfloat16(),
         "dO": torch.randn(cq[-1], H, dv, generator=g0).bfloat16()}
    return x, [int(c) for c in cq], [int(c) for c in ck]


def _run(x, cq, ck, causal, scale, det, window=None, bm=None, share=False):
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    kw = dict(cu_seqlens=cq, cu_seqlens_k=None if share else ck, window=window, block_mask=bm)
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, **kw)
    dq, dk, dv = binding.backward(q, k, v, o, dO, lse, causal=causal, scale=scale,
                                  deterministic=det, **kw)
    torch.cuda.synchronize()
    assert binding.attn_fwd_status() == 0
    return {"O": o.cpu(), "LSE": lse.cpu(), "dQ": dq.cpu(), "dK": dk.cpu(), "dV": dv.cpu()}


CASES = [
    # query lengths, key lengths, H, d, dv, causal, window, block-mask density
    ((300, 1, 257, 142, 64), (500, 128, 257, 900, 64), 2, 128, 128, True, None, None),
    ((300, 1, 257, 142, 64), (500, 128, 257, 900, 64), 2, 128, 128, False, None, None),
    ((200, 0, 333, 17), (150, 100, 700, 17), 3, 64, 64, False, None, None),  # Lq > Lk; no queries
    ((129, 256, 300), (400, 256, 1000), 2, 128, 128, False, (90, 30), None),
    ((300, 142, 257), (700, 900, 257), 2, 192, 128, True, None, 0.6),
]


@pytest.mark.parametrize("lq,lk,H,d,dv,causal,window,density", CASES)
def test_varlen_separate_offsets_against_oracle(lq, lk, H, d, dv, causal, window, density):
    import oracle
    x, cq, ck = _inputs(lq, lk, H, d, dv, seed=400 + sum(lq))
    scale = 1.0 / np.sqrt(d)
    mask = bm = None
    if density is not None:
        nq, nk = -(-max(lq) // BL), -(-max(lk) // BL)
        mask = (np.random.default_rng(401).random((1, H, nq, nk)) < density).astype(np.uint8)
        bm = torch.from_numpy(mask).to("cuda:0")
    qs, ks, vs, dOs = (_split(x[n], c) for n, c in (("q", cq), ("k", ck), ("v", ck), ("dO", cq)))
    pm = None if mask is None else np.broadcast_to(mask, (len(lq), H) + mask.shape[2:]).reshape(
        (len(lq) * H,) + mask.shape[2:])
    r = oracle.backward(qs, ks, vs, dOs, causal, scale, window=window, block_mask=pm, block=BL)
    cat = lambda a: np.concatenate([np.asarray(z).reshape(-1) for z in a])
    for det in (False, True):
        g = _run(x, cq, ck, causal, scale, det, window, bm)
        err = {}
        for key, cu in (("O", cq), ("dQ", cq), ("dK", ck), ("dV", ck)):
            err[key] = rel_err(cat(_split(g[key], cu)), cat(r[key]))
        lse = g["LSE"].double().numpy()  # (H, sum Lq)
        got = cat([lse[h, cq[s]:cq[s + 1]] for s in range(len(lq)) for h in range(H)])
        ref = cat(r["LSE"])
        empty = np.isneginf(ref)
        assert np.array_equal(np.isneginf(got), empty), "rows without keys"
        err["LSE"] = max_abs(got[~empty], ref[~empty])
        gc.assert_within(err, f"lq={lq} lk={lk} causal={causal} window={window} det={det}")


def test_separate_offsets_equal_to_shared_are_the_same_call():
    """Key offsets equal to the query offsets (passed as a second array) give
    the bytes of the shared-offset call, deterministic mode."""
    lens = (300, 1, 257, 142)
    x, cq, _ = _inputs(lens, lens, 2, 128, 128, seed=402)
    a = _run(x, cq, list(cq), True, 1.0 / np.sqrt(128), True)
    b = _run(x, cq, cq, True, 1.0 / np.sqrt(128), True, share=True)
    for key in a:
        assert torch.equal(a[key], b[key]), key
