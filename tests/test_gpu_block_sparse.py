"""Block-sparse attention on the GPU against the oracle.

The block mask drops whole (query tile, key tile) pairs of 128 x 128; it
combines with the causal band, local windows, variable-length batches and the
deterministic dQ order.  Masks are seeded random with the given density, with
some query blocks and key blocks dropped entirely (rows that see no key: O = 0,
LSE = -inf, dQ = 0; keys no query sees: dK = dV = 0)."""
import numpy as np
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu
W = syn.Workload
BL = binding.BLOCK


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()
    import oracle
    oracle.build()


def random_mask(shape, density, seed, empty_row=None, empty_col=None):
    """uint8 mask of `shape` (..., NQ, NK) with about `density` kept pairs;
    optionally one query block (row) and one key block (column) dropped in
    every mask."""
    m = (np.random.default_rng(seed).random(shape) < density).astype(np.uint8)
    if empty_row is not None:
        m[..., empty_row, :] = 0
    if empty_col is not None:
        m[..., :, empty_col] = 0
    return m


def per_problem(mask4, B, H):
    """[Bm][Hm][NQ][NK] -> [B*H][NQ][NK] in (sequence, head) order."""
    full = np.broadcast_to(mask4, (B, H) + mask4.shape[2:])
    return full.reshape((B * H,) + mask4.shape[2:])


def _inputs(B, H, Tq, Tk, d, dv, seed):
    g0 = torch.Generator().manual_seed(seed)
    return {"q": torch.randn(B, Tq, H, d, generator=g0).bfloat16(),
            "k": torch.randn(B, Tk, H, d, generator=g0).bfloat16(),
            "v": torch.randn(B, Tk, H, dv, generator=g0).bfloat16(),
            "dO": torch.randn(B, Tq, H, dv, generator=g0).bfloat16()}


def _run(x, w, causal, window, mask4, det, ws=None):
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    bm = torch.from_numpy(np.ascontiguousarray(mask4)).to(dev)
    o, lse = binding.forward(q, k, v, causal=causal, scale=w.scale, window=window, block_mask=bm)
    assert binding.attn_fwd_status() == 0
    dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=causal, scale=w.scale,
                                   deterministic=det, window=window, block_mask=bm, workspace=ws)
    torch.cuda.synchronize()
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dvv}


CASES = [
    # B, H, Tq, Tk, d, dv, causal, window, (Bm, Hm), density
    (2, 3, 700, 700, 128, 128, False, None, (2, 3), 0.5),   # per (sequence, head) masks
    (1, 4, 1000, 1000, 64, 64, True, None, (1, 1), 0.6),    # one shared mask, causal band
    (1, 2, 300, 900, 128, 128, False, (200, 50), (1, 2), 0.7),  # window, Tq < Tk, per head
    (2, 2, 640, 640, 192, 128, True, None, (2, 1), 0.5),    # d192, per-sequence masks
    (1, 2, 1024, 1024, 128, 128, False, None, (1, 2), 0.15),  # sparse: few pairs per row
]


@pytest.mark.parametrize("B,H,Tq,Tk,d,dv,causal,window,mdims,density", CASES)
def test_block_sparse_against_oracle(B, H, Tq, Tk, d, dv, causal, window, mdims, density):
    x = _inputs(B, H, Tq, Tk, d, dv, seed=300 + Tq + d)
    w = W("blocksparse", B, H, Tq, d, dv, causal)
    nq, nk = -(-Tq // BL), -(-Tk // BL)
    mask4 = random_mask(mdims + (nq, nk), density, seed=Tq + H, empty_row=nq // 2,
                        empty_col=1)
    need = binding.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda:0")
    for det in (False, True):
        out = _run(x, w, causal, window, mask4, det, ws)
        assert binding.attn_bwd_status(ws) == 0
        g = {key: val.float().cpu() for key, val in out.items()}
        err = gc.compare_full(x, w, g, window=window, block_mask=per_problem(mask4, B, H))
        gc.assert_within(err, f"mask {mdims} density {density} det={det}")
        # the dropped query block: no key, O = 0, LSE = -inf, dQ = 0
        rows = slice((nq // 2) * BL, min(Tq, (nq // 2 + 1) * BL))
        assert torch.all(g["O"][:, rows] == 0) and torch.all(g["dQ"][:, rows] == 0)
        assert torch.all(torch.isneginf(g["LSE"][:, :, rows]))
        # the dropped key block: no query sees it, dK = dV = 0
        assert torch.all(g["dK"][:, BL:2 * BL] == 0) and torch.all(g["dV"][:, BL:2 * BL] == 0)


def test_block_sparse_varlen():
    lens = (300, 1, 257, 142)
    w = W("varlen_blocksparse", 4, 2, 300, 128, 128, True, varlen=lens)
    x = syn.make_inputs(w, seed=301)
    nb = -(-max(lens) // BL)
    mask4 = random_mask((1, 2, nb, nb), 0.7, seed=302)
    mask4[..., np.arange(nb), np.arange(nb)] = 1  # diagonal kept: every row sees a key
    dev = "cuda:0"
    cu = [0] + list(np.cumsum(lens))
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    bm = torch.from_numpy(mask4).to(dev)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu, block_mask=bm)
    dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                   cu_seqlens=cu, deterministic=True, block_mask=bm)
    torch.cuda.synchronize()
    assert binding.attn_fwd_status() == 0
    g = {"O": o.float().cpu(), "LSE": lse.cpu(), "dQ": dq.float().cpu(),
         "dK": dk.float().cpu(), "dV": dvv.float().cpu()}
    gc.assert_within(gc.compare_full(x, w, g, block_mask=per_problem(mask4, 4, 2)),
                     "varlen block-sparse")


def test_all_ones_mask_is_bitwise_the_dense_path():
    """Keeping every pair changes no arithmetic: deterministic results are
    byte-identical to the same call without a mask."""
    B, H, T, d = 1, 3, 777, 128
    x = _inputs(B, H, T, T, d, d, seed=303)
    w = W("ones", B, H, T, d, d, True)
    n = -(-T // BL)
    masked = _run(x, w, True, None, np.ones((1, 1, n, n), np.uint8), det=True)
    dev = "cuda:0"
    q, k, v, dO = (x[nm].to(dev) for nm in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                   deterministic=True)
    torch.cuda.synchronize()
    for key, ref in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dvv)):
        assert torch.equal(masked[key], ref), key


def test_deterministic_block_sparse_is_bitwise_repeatable():
    B, H, T, d = 1, 4, 2048, 128
    x = _inputs(B, H, T, T, d, d, seed=304)
    w = W("det", B, H, T, d, d, False)
    n = T // BL
    mask4 = random_mask((1, H, n, n), 0.4, seed=305)
    a = _run(x, w, False, None, mask4, det=True)
    b = _run(x, w, False, None, mask4, det=True)
    for key in ("dQ", "dK", "dV"):
        assert torch.equal(a[key], b[key]), key


def test_empty_mask_gives_zero_outputs():
    B, H, T, d = 1, 2, 300, 64
    x = _inputs(B, H, T, T, d, d, seed=306)
    w = W("empty", B, H, T, d, d, False)
    n = -(-T // BL)
    out = _run(x, w, False, None, np.zeros((1, 1, n, n), np.uint8), det=True)
    assert binding.attn_fwd_status() == 0
    assert torch.all(out["O"] == 0) and torch.all(torch.isneginf(out["LSE"]))
    for key in ("dQ", "dK", "dV"):
        assert torch.all(out[key] == 0), key


def test_block_mask_argument_checks():
    dev = "cuda:0"
    q = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, dtype=torch.float32, device=dev)
    bm = torch.ones(2, 2, dtype=torch.uint8, device=dev)
    for mb, mh in ((3, 1), (1, 3), (0, 1)):  # neither 1 nor B / H
        rc = binding.attn_fwd_ex(q, q, q, o, lse, 1, 2, 256, 256, 64, 64, 0, -1, -1, bm, mb, mh,
                                 0.125)
        assert rc == binding.ATTN_ERR_INVALID_ARG, (mb, mh)
