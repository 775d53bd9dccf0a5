"""attn_bwd_noalloc — the backward for callers that cannot allocate device
memory (their framework owns it all, or cudaMalloc's device synchronisation is
not allowed where they run).  Its workspace is the library's own fixed 32 MiB
device array.  Checked through the C ABI against attn_bwd (caller workspace)
on two calls in a row, within the parity tolerance; this file is collected
last so that a run that stops at its first failure has run everything else."""
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn
from tests._common import rel_err

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_matches_attn_bwd_twice(deterministic):
    w = syn.Workload("noalloc", B=2, H=4, T=1000, dqk=128, dv=128, causal=True)
    x = syn.make_inputs(w, seed=11)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    B, H, T, d = w.B, w.H, w.T, w.dqk
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    ref = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                           deterministic=deterministic)
    for _ in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, 7), torch.empty_like(v)
        rc = binding.attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, T, T, d, d, True,
                                      w.scale, None, 0, deterministic)
        assert rc == binding.ATTN_OK, binding.attn_strerror(rc)
        torch.cuda.synchronize()
        for got, want in zip((dq, dk, dv), ref):
            assert rel_err(got.float().cpu().numpy(), want.float().cpu().numpy()) <= TOL_GRAD


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, T, d = 1, 16, 32768, 128  # needs ~272 MB of workspace
    assert binding.attn_bwd_workspace_size(B, H, T, T, d, d) > 32 << 20
    A = 0x10000
    rc = binding.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, H, T, T, d, d, True, 0.088)
    assert rc == binding.ATTN_ERR_SCRATCH_TOO_SMALL
    assert "32 MiB" in binding.attn_strerror(rc)
