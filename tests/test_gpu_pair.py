"""The backward main kernel on CTA pairs (tcgen05 cta_group::2: two key tiles
per cluster of two CTAs, M = 256 pair MMAs, dQ contracted over both tiles
before its atomics) against the oracle, element by element on small shapes
(odd key-tile counts, ragged tails, variable lengths, fewer queries than keys,
a right-bounded band, packed QKV) and by sampled rows and keys on the 32K
workloads; against the one-CTA kernel (dK, dV bit-identical: their sums do not
depend on how dQ is reduced); deterministic mode bit-identical over 10 runs;
a device timeout reported with the context left usable."""
import hashlib

import numpy as np
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()
    import oracle
    oracle.build()


@pytest.fixture(autouse=True)
def _pair_kernel():
    binding.attn_debug_set_bwd_variant(binding.BWD_CTA_PAIR)
    yield
    binding.attn_debug_set_bwd_variant(binding.BWD_AUTO)


def W(name, B, H, T, causal, layout=0, varlen=(), det=False):
    return syn.Workload(name, B, H, T, 128, 128, causal, layout=layout, varlen=tuple(varlen),
                        deterministic=det)


SMALL = [
    W("pair_T256_causal", 1, 2, 256, True),
    W("pair_T200_noncausal", 2, 3, 200, False),
    W("pair_T384_causal", 1, 3, 384, True),      # three key tiles: the last pair has one
    W("pair_T129_causal", 2, 2, 129, True),      # ragged second tile
    W("pair_T1000_causal", 2, 2, 1000, True),
    W("pair_T640_noncausal", 1, 2, 640, False),  # five key tiles
    W("pair_packed", 1, 2, 300, True, layout=syn.LAYOUT_PACKED),
    W("pair_varlen", 5, 2, 300, True, varlen=(1, 100, 128, 129, 300)),
    W("pair_varlen_nc", 4, 3, 600, False, varlen=(600, 5, 257, 130)),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_pair_small_shapes_every_element(w):
    x = syn.make_inputs(w, seed=7)
    for det in (False, True):
        g = gc.run_gpu(x, w, deterministic=det)
        gc.assert_within(gc.compare_full(x, w, g), f"{w.name} det={det}")


def test_pair_dk_dv_equal_one_cta_kernel():
    w = W("pair_vs_one", 2, 4, 1000, True)
    x = syn.make_inputs(w, seed=8)
    g2 = gc.run_gpu(x, w, deterministic=True)
    binding.attn_debug_set_bwd_variant(binding.BWD_ONE_CTA)
    g1 = gc.run_gpu(x, w, deterministic=True)
    assert torch.equal(g1["dK"], g2["dK"]) and torch.equal(g1["dV"], g2["dV"])
    assert gc.rel_err(g2["dQ"].numpy(), g1["dQ"].numpy()) <= 2e-3


@pytest.mark.parametrize("B,H,Tq,Tk,causal,window", [
    (2, 2, 130, 300, True, None),          # causal, fewer queries than keys
    (1, 2, 200, 900, False, (-1, 10)),     # right-bounded band, keys no query sees
    (1, 2, 520, 520, False, (-1, 100)),
])
def test_pair_bands(B, H, Tq, Tk, causal, window):
    g0 = torch.Generator().manual_seed(90 + Tq)
    x = {"q": torch.randn(B, Tq, H, 128, generator=g0).bfloat16(),
         "k": torch.randn(B, Tk, H, 128, generator=g0).bfloat16(),
         "v": torch.randn(B, Tk, H, 128, generator=g0).bfloat16(),
         "dO": torch.randn(B, Tq, H, 128, generator=g0).bfloat16()}
    w = W("pair_band", B, H, Tq, causal)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=w.scale, window=window)
    need = binding.attn_bwd_workspace_size(B, H, Tq, Tk, 128, 128, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for det in (False, True):
        dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=causal, scale=w.scale,
                                       deterministic=det, window=window, workspace=ws)
        assert binding.attn_bwd_status(ws) == 0
        g = {"O": o.float().cpu(), "LSE": lse.cpu(), "dQ": dq.float().cpu(),
             "dK": dk.float().cpu(), "dV": dvv.float().cpu()}
        gc.assert_within(gc.compare_full(x, w, g, window=window), f"Tq={Tq} Tk={Tk} det={det}")


@pytest.mark.parametrize("w", [w for w in syn.SWEEP_D128 if w.T in (2048, 32768)],
                         ids=lambda w: w.name)
def test_pair_sweep_points(w):
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    if w.T <= 2048:
        pick = np.random.default_rng(5).choice(w.B * w.H, size=3, replace=False)
        gc.assert_within(gc.compare_full(x, w, g, pick=pick), w.name)
    else:
        err = gc.compare_sampled(x, w, g, heads=[0, 7, 15],
                                 kv_heads=[2, 5, 13] if w.causal else [5, 11])
        assert {"dK", "dV"} <= set(err)
        gc.assert_within(err, w.name)


def test_pair_varlen_deterministic_workload_bit_identical_10_runs():
    w = syn.VARLEN
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    lens = list(w.varlen)
    short = sorted(range(len(lens)), key=lambda s: lens[s])[:2]
    pick = [s * w.H + h for s in short for h in (0, w.H - 1)]
    gc.assert_within(gc.compare_full(x, w, g, pick=pick), "pair varlen short sequences")
    dev = "cuda:0"
    cu = [int(c) for c in x["cu_seqlens"]]
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu)
    digests = set()
    for _ in range(10):
        dq, dk, dv = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                      cu_seqlens=cu, deterministic=True)
        h = hashlib.sha256()
        for t in (dq, dk, dv):
            h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
        digests.add(h.hexdigest())
    assert len(digests) == 1


def test_pair_bounded_wait_reports_timeout_and_context_survives():
    w = W("pair_to", 1, 2, 512, True, det=True)
    x = syn.make_inputs(w)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    need = binding.attn_bwd_workspace_size(1, 2, 512, 512, 128, 128, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    binding.attn_debug_set_wait_bias(1000)
    try:
        rc = binding.attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, 1, 2, 512, 512, 128, 128, True,
                              w.scale, None, 0, True, ws, need)
        assert rc == binding.ATTN_OK
        assert binding.attn_bwd_status(ws) == binding.ATTN_ERR_TIMEOUT
    finally:
        binding.attn_debug_set_wait_bias(0)
    g = gc.run_gpu(x, w)
    gc.assert_within(gc.compare_full(x, w, g), "pair after timeout")
