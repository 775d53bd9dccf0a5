"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (in the test code): normwise relative error <= 1e-2 for dQ, dK,
dV and <= 5e-3 for O; max |LSE - LSE_ref| <= 1e-4.  Small cases compare every
element; the large workloads compare sampled rows and keys that the oracle
computes one at a time, in the same launch configuration the benchmark uses.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

from tests import gpu_common as gc


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()
    import oracle
    oracle.build()


def W(name, B, H, T, dqk, dv, causal, layout=0, varlen=(), det=False):
    return syn.Workload(name, B, H, T, dqk, dv, causal, layout=layout, varlen=tuple(varlen),
                        deterministic=det)


# ---------------------------------------------------------------------------
# every element, small shapes (several tiles, ragged tails, edge cases)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("w", syn.TINY, ids=lambda w: w.name)
def test_tiny_workload(w):
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    gc.assert_within(gc.compare_full(x, w, g), w.name)


SMALL = [
    W("d64_T200_causal", 2, 3, 200, 64, 64, True),
    W("d64_T200_noncausal", 2, 3, 200, 64, 64, False),
    W("d64_T1_causal", 1, 2, 1, 64, 64, True),
    W("d64_T1_noncausal", 3, 1, 1, 64, 64, False),
    W("d128_T129_causal", 1, 2, 129, 128, 128, True),
    W("d128_T300_noncausal", 2, 2, 300, 128, 128, False),
    W("d128_T384_causal", 1, 3, 384, 128, 128, True),
    W("d192_T257_causal", 1, 2, 257, 192, 128, True),
    W("d192_T200_noncausal", 2, 1, 200, 192, 128, False),
    W("d64_T200_packed", 2, 3, 200, 64, 64, True, layout=syn.LAYOUT_PACKED),
    W("d128_T130_packed_nc", 1, 2, 130, 128, 128, False, layout=syn.LAYOUT_PACKED),
    W("varlen_d128_causal", 5, 2, 300, 128, 128, True, varlen=(1, 100, 128, 129, 300)),
    W("varlen_d64_noncausal", 4, 3, 257, 64, 64, False, varlen=(257, 5, 130, 64)),
    W("varlen_d128_det", 5, 2, 300, 128, 128, True, varlen=(300, 1, 129, 128, 100), det=True),
    W("varlen_d192_causal", 3, 2, 260, 192, 128, True, varlen=(260, 17, 131)),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_shapes_every_element(w):
    x = syn.make_inputs(w, seed=3)
    for det in (False, True):
        g = gc.run_gpu(x, w, deterministic=det)
        gc.assert_within(gc.compare_full(x, w, g), f"{w.name} det={det}")


def test_noncausal_rectangular():
    """Tq != Tk (non-causal, fixed length)."""
    g0 = torch.Generator().manual_seed(5)
    B, H, Tq, Tk, d = 2, 2, 130, 300, 64
    x = {"q": torch.randn(B, Tq, H, d, generator=g0).bfloat16(),
         "k": torch.randn(B, Tk, H, d, generator=g0).bfloat16(),
         "v": torch.randn(B, Tk, H, d, generator=g0).bfloat16(),
         "dO": torch.randn(B, Tq, H, d, generator=g0).bfloat16()}
    w = W("rect", B, H, Tq, d, d, False)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=False, scale=w.scale)
    dq, dk, dv = binding.backward(q, k, v, o, dO, lse, causal=False, scale=w.scale)
    g = {"O": o.float().cpu(), "LSE": lse.cpu(), "dQ": dq.float().cpu(), "dK": dk.float().cpu(),
         "dV": dv.float().cpu()}
    gc.assert_within(gc.compare_full(x, w, g), "rect")


@pytest.mark.parametrize("B,H,Tq,Tk,d,dv", [
    (2, 3, 200, 456, 64, 64),      # offset 256: whole tiles
    (1, 2, 130, 300, 128, 128),    # offset 170: the diagonal band crosses tiles
    (2, 2, 1, 300, 128, 128),      # one query (a decoding step): sees every key
    (1, 2, 129, 131, 192, 128),    # offset 2, ragged on both sides
    (1, 1, 384, 1000, 64, 64),     # several q-tiles per kv-tile band
])
def test_causal_fewer_queries_than_keys(B, H, Tq, Tk, d, dv):
    """Causal with Tq < Tk: query i sees keys j <= i + Tk - Tq (bottom-right)."""
    g0 = torch.Generator().manual_seed(60 + Tq)
    x = {"q": torch.randn(B, Tq, H, d, generator=g0).bfloat16(),
         "k": torch.randn(B, Tk, H, d, generator=g0).bfloat16(),
         "v": torch.randn(B, Tk, H, dv, generator=g0).bfloat16(),
         "dO": torch.randn(B, Tq, H, dv, generator=g0).bfloat16()}
    w = W("rect_causal", B, H, Tq, d, dv, True)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    assert binding.attn_fwd_status() == 0
    need = binding.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for det in (False, True):
        dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                       deterministic=det, workspace=ws)
        assert binding.attn_bwd_status(ws) == 0
        g = {"O": o.float().cpu(), "LSE": lse.cpu(), "dQ": dq.float().cpu(),
             "dK": dk.float().cpu(), "dV": dvv.float().cpu()}
        gc.assert_within(gc.compare_full(x, w, g), f"Tq={Tq} Tk={Tk} det={det}")


@pytest.mark.parametrize("B,H,Tq,Tk,d,dv,causal,window", [
    (1, 2, 700, 700, 64, 64, True, (200, -1)),      # causal local window
    (1, 2, 700, 700, 128, 128, False, (100, 60)),   # two-sided band, edges inside tiles
    (2, 2, 300, 300, 128, 128, False, (0, 0)),      # each query sees its own key only
    (1, 2, 200, 900, 64, 64, False, (150, 10)),     # Tq < Tk: early keys seen by no query
    (1, 1, 384, 384, 192, 128, True, (128, -1)),    # band edge on a tile boundary, d192
    (1, 2, 520, 520, 128, 128, False, (-1, 100)),   # right bound only
])
def test_local_window(B, H, Tq, Tk, d, dv, causal, window):
    """Local (sliding-window) attention against the oracle, fast and deterministic."""
    g0 = torch.Generator().manual_seed(80 + Tq + (window[0] if window[0] > 0 else 0))
    x = {"q": torch.randn(B, Tq, H, d, generator=g0).bfloat16(),
         "k": torch.randn(B, Tk, H, d, generator=g0).bfloat16(),
         "v": torch.randn(B, Tk, H, dv, generator=g0).bfloat16(),
         "dO": torch.randn(B, Tq, H, dv, generator=g0).bfloat16()}
    w = W("window", B, H, Tq, d, dv, causal)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=causal, scale=w.scale, window=window)
    assert binding.attn_fwd_status() == 0
    need = binding.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for det in (False, True):
        dq, dk, dvv = binding.backward(q, k, v, o, dO, lse, causal=causal, scale=w.scale,
                                       deterministic=det, window=window, workspace=ws)
        assert binding.attn_bwd_status(ws) == 0
        g = {"O": o.float().cpu(), "LSE": lse.cpu(), "dQ": dq.float().cpu(),
             "dK": dk.float().cpu(), "dV": dvv.float().cpu()}
        gc.assert_within(gc.compare_full(x, w, g, window=window),
                         f"window={window} causal={causal} det={det}")


def test_local_window_varlen():
    w = W("varlen_window", 4, 2, 300, 128, 128, True, varlen=(300, 1, 257, 142))
    x = syn.make_inputs(w, seed=81)
    g = gc.run_gpu(x, w, window=(100, -1))
    gc.assert_within(gc.compare_full(x, w, g, window=(100, -1)), "varlen window")


# ---------------------------------------------------------------------------
# the five workload families at their full sizes
# ---------------------------------------------------------------------------
def test_gpt2_packed_every_element():
    w = syn.GPT2
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    gc.assert_within(gc.compare_full(x, w, g), w.name)


@pytest.mark.parametrize("w", [w for w in syn.SWEEP_D128 if w.T <= 8192], ids=lambda w: w.name)
def test_d128_sweep_every_element(w):
    """The d=128 sweep up to T=8K, causal and not: every element of a few
    seeded (b, h) heads (heads are independent problems, so a subset is
    exact)."""
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    n_pick = 4 if w.T <= 4096 else (3 if w.causal else 2)
    pick = np.random.default_rng(w.T).choice(w.B * w.H, size=n_pick, replace=False)
    gc.assert_within(gc.compare_full(x, w, g, pick=pick), w.name)


# (b, h) problems whose query rows (O, LSE, dQ) and key rows (dK, dV) are
# checked one by one at the long lengths; the 32K causal workload is the
# benchmark's, run in the benchmark's launch configuration.
LONG_HEADS = {
    "d128_T16K_causal": ([0, 9, 31], [4, 27]),
    "d128_T16K_noncausal": ([1, 14, 30], [6, 25]),
    "d128_T32K_causal": ([0, 7, 15], [2, 5, 13]),
    "d128_T32K_noncausal": ([0, 7, 15], [5, 11]),
}


@pytest.mark.parametrize("w", [w for w in syn.SWEEP_D128 if w.T >= 16384], ids=lambda w: w.name)
def test_d128_long(w):
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    heads, kv_heads = LONG_HEADS[w.name]
    err = gc.compare_sampled(x, w, g, heads=heads, kv_heads=kv_heads)
    assert {"dK", "dV", "dQ", "O", "LSE"} <= set(err)
    gc.assert_within(err, w.name)


@pytest.mark.parametrize("w", syn.D192, ids=lambda w: w.name)
def test_d192(w):
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    if w.T <= 2048:
        pick = np.random.default_rng(1).choice(w.B * w.H, size=3, replace=False)
        gc.assert_within(gc.compare_full(x, w, g, pick=pick), w.name)
    else:
        kv = [3] if w.T <= 8192 else [3, 12]
        err = gc.compare_sampled(x, w, g, heads=[1, 9], kv_heads=kv)
        assert {"dK", "dV"} <= set(err)
        gc.assert_within(err, w.name)


INFERENCE = (syn.TINY + [syn.GPT2] + [w for w in syn.SWEEP_D128 if w.T == 32768] + syn.D192)


@pytest.mark.parametrize("w", INFERENCE, ids=lambda w: w.name)
def test_inference_forward_against_oracle(w):
    """Inference mode (lse = NULL: no statistics written) against the oracle's
    O: every element on the tiny workload, sampled rows elsewhere; and equal,
    bit for bit, to the training forward's O."""
    x = syn.make_inputs(w)
    dev = "cuda:0"
    if w.layout == syn.LAYOUT_PACKED:
        qkv = x["qkv"].to(dev)
        q, k, v = qkv.select(-3, 0), qkv.select(-3, 1), qkv.select(-3, 2)
    else:
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o_inf, none = binding.forward(q, k, v, causal=w.causal, scale=w.scale, layout=w.layout,
                                  with_lse=False)
    o_train, _ = binding.forward(q, k, v, causal=w.causal, scale=w.scale, layout=w.layout)
    torch.cuda.synchronize()
    assert binding.attn_fwd_status() == 0
    assert none is None and torch.equal(o_inf, o_train)
    o = o_inf.float().cpu()
    if w.T <= 128:
        (qp, kp, vp, _), cu = gc.inputs_as_problems(x, w)
        O_ref, _, _ = oracle.forward(qp, kp, vp, w.causal, w.scale)
        got = np.stack(gc.problems(o, w, cu))
        err = {"O": gc.rel_err(got, O_ref), "O_row": gc.row_err(got, O_ref)}
    else:
        nprob = w.B * w.H
        heads = sorted({0, nprob // 2, nprob - 1})
        err = gc.compare_forward_sampled(x, w, o, heads)
    gc.assert_within(err, w.name)


def test_varlen_deterministic_workload():
    w = syn.VARLEN
    x = syn.make_inputs(w)
    g = gc.run_gpu(x, w)
    lens = list(w.varlen)
    H = w.H
    # every element of the shortest sequences' heads, sampled rows of the longest
    short = sorted(range(len(lens)), key=lambda s: lens[s])[:2]
    pick = [s * H + h for s in short for h in (0, H - 1)]
    gc.assert_within(gc.compare_full(x, w, g, pick=pick), "varlen short sequences")
    longest = max(range(len(lens)), key=lambda s: lens[s])
    err = gc.compare_sampled(x, w, g, heads=[longest * H + 3], kv_heads=[])
    gc.assert_within(err, "varlen longest sequence")


def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def test_deterministic_mode_bit_identical_10_runs():
    w = syn.VARLEN
    x = syn.make_inputs(w)
    dev = "cuda:0"
    cu = [int(c) for c in x["cu_seqlens"]]
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu)
    digests = set()
    ws = None
    for _ in range(10):
        dq, dk, dv = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                      cu_seqlens=cu, deterministic=True, workspace=ws)
        digests.add(_digest([dq, dk, dv]))
    assert len(digests) == 1


def test_deterministic_and_fast_agree():
    w = [w for w in syn.SWEEP_D128 if w.T == 4096 and w.causal][0]
    x = syn.make_inputs(w)
    a = gc.run_gpu(x, w, deterministic=False)
    b = gc.run_gpu(x, w, deterministic=True)
    for key in ("dQ", "dK", "dV"):
        assert gc.rel_err(a[key].numpy(), b[key].numpy()) <= 2e-3, key
    # dK and dV do not depend on the dQ reduction order
    assert torch.equal(a["dK"], b["dK"]) and torch.equal(a["dV"], b["dV"])


def test_bounded_wait_reports_timeout_and_context_survives():
    """Host-side fault injection: the ordered dQ wait targets a semaphore value
    that nothing will write; the kernel must give up, report ATTN_ERR_TIMEOUT
    and leave the context usable for the next call."""
    w = W("to", 1, 2, 512, 64, 64, True, det=True)
    x = syn.make_inputs(w)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    need = binding.attn_bwd_workspace_size(1, 2, 512, 512, 64, 64, False, True)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    binding.attn_debug_set_wait_bias(1000)
    try:
        rc = binding.attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, 1, 2, 512, 512, 64, 64, True,
                              w.scale, None, 0, True, ws, need)
        assert rc == binding.ATTN_OK
        assert binding.attn_bwd_status(ws) == binding.ATTN_ERR_TIMEOUT
    finally:
        binding.attn_debug_set_wait_bias(0)
    g = gc.run_gpu(x, w)
    gc.assert_within(gc.compare_full(x, w, g), "after timeout")
    dq2, dk2, dv2 = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                                     deterministic=True, workspace=ws)
    assert binding.attn_bwd_status(ws) == binding.ATTN_OK


@pytest.mark.parametrize("causal", [False, True])
def test_running_max_jumps_between_key_tiles(causal):
    """Keys of later tiles scaled up so that each row's maximum grows by far
    more than the forward's lazy-rescale bound (2^8) from one key tile to the
    next: the rows must be recomputed with the new maximum and O rescaled."""
    w = W("jump", 1, 2, 1024, 64, 64, causal)
    x = syn.make_inputs(w, seed=21)
    k = x["k"].float()
    for t in range(1, 8):  # key tile t scaled by 1.6^t (score spread grows tile by tile)
        k[:, t * 128:(t + 1) * 128] *= 1.6 ** t
    x["k"] = k.bfloat16()
    g = gc.run_gpu(x, w)
    gc.assert_within(gc.compare_full(x, w, g), f"jump causal={causal}")


@pytest.mark.parametrize("dqk,dv", [(128, 128), (192, 128)])
def test_gradient_buffers_only_16_byte_aligned(dqk, dv):
    """dK and dV rows are written with 32-byte stores when the buffers allow it
    and with 16-byte stores otherwise; both give the same bits (deterministic
    mode), and dQ is unaffected."""
    B, H, T = 1, 2, 300
    w = syn.Workload("align16", B=B, H=H, T=T, dqk=dqk, dv=dv, causal=True)
    x = syn.make_inputs(w, seed=21)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    ref = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale, deterministic=True)

    def shifted(t):  # same shape, data starting 16 bytes past a 256-byte boundary
        buf = torch.empty(t.numel() + 8, dtype=torch.bfloat16, device=dev)
        return buf[8:].view(t.shape)

    out = (shifted(q), shifted(k), shifted(v))
    assert all(t.data_ptr() % 32 == 16 for t in out)
    got = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale, deterministic=True,
                           out=out)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_forward_output_only_16_byte_aligned():
    """O rows are written with 32-byte stores when the buffer allows it and
    with 16-byte stores otherwise; both give the same bits."""
    B, H, T, d = 1, 2, 300, 128
    w = syn.Workload("align16_fwd", B=B, H=H, T=T, dqk=d, dv=d, causal=True)
    x = syn.make_inputs(w, seed=22)
    dev = "cuda:0"
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o_ref, lse_ref = binding.forward(q, k, v, causal=True, scale=w.scale)
    buf = torch.empty(o_ref.numel() + 8, dtype=torch.bfloat16, device=dev)
    o = buf[8:].view(o_ref.shape)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty_like(lse_ref)
    rc = binding.attn_fwd_ex(q, k, v, o, lse, B, H, T, T, d, d, True, -1, -1, None, 1, 1,
                             w.scale, None, None, binding.LAYOUT_BTHD, None)
    assert rc == binding.ATTN_OK
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
