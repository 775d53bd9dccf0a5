"""attn_step_host: host tensors in and out, copies overlapped with the kernels.

Deterministic mode must give exactly the bytes of attn_fwd + attn_bwd on the
whole device tensors (the heads are independent problems, and the dQ order is
fixed); fast mode is checked against the oracle with the usual tolerances."""
import pytest
import torch

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


def _pinned(x):
    return {n: (t.pin_memory() if n != "cu_seqlens" else t) for n, t in x.items()}


@pytest.mark.parametrize("B,H,T,d,dv,causal,G", [
    (2, 8, 1000, 128, 128, True, 3),     # ragged last group (3, 3, 2)
    (1, 5, 513, 64, 64, False, 2),
    (1, 4, 300, 192, 128, True, 0),      # library's choice of group size
])
def test_deterministic_matches_device_path_bytes(B, H, T, d, dv, causal, G):
    w = syn.Workload("hs", B, H, T, d, dv, causal)
    x = _pinned(syn.make_inputs(w, seed=11))
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o_ref, lse = binding.forward(q, k, v, causal=causal, scale=w.scale)
    ref = binding.backward(q, k, v, o_ref, dO, lse, causal=causal, scale=w.scale,
                           deterministic=True)
    dq, dk, dvt, o = binding.step_host(x["q"], x["k"], x["v"], x["dO"], causal=causal,
                                       scale=w.scale, deterministic=True, heads_per_group=G,
                                       with_o=True)
    for got, want, name in ((dq, ref[0], "dq"), (dk, ref[1], "dk"), (dvt, ref[2], "dv"),
                            (o, o_ref, "o")):
        assert torch.equal(got, want.cpu()), name


def test_fast_mode_against_oracle():
    w = syn.Workload("hs_fast", 2, 5, 300, 64, 64, True)
    x = _pinned(syn.make_inputs(w, seed=12))
    dev = torch.device("cuda:0")
    streams = (torch.cuda.current_stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev),
               torch.cuda.Stream(dev))
    need = binding.attn_step_host_scratch_size(w.B, w.H, w.T, w.dqk, w.dv, 2)
    scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dvt, o = binding.step_host(x["q"], x["k"], x["v"], x["dO"], causal=True,
                                       scale=w.scale, heads_per_group=2, with_o=True,
                                       scratch=scratch, streams=streams)
    streams[0].synchronize()
    assert binding.attn_step_host_status(scratch, w.B, w.H, w.T, w.dqk, w.dv, 2) == 0
    # LSE is not returned by the host step: compare the rest against the oracle
    g = {"O": o.float(), "dQ": dq.float(), "dK": dk.float(), "dV": dvt.float(),
         "LSE": torch.zeros(w.B, w.H, w.T)}
    err = gc.compare_full(x, w, g)
    err.pop("LSE")
    gc.assert_within(err, "step_host fast")
