"""attn_bwd_noalloc — the backward for callers that cannot allocate device
memory (their framework owns it all, or cudaMalloc's device synchronisation is
not allowed where they run).  Its workspace is the library's own fixed 32 MiB
device array.  Checked through the C ABI against attn_bwd (caller workspace)
on two calls in a row: within the parity tolerance in fast mode, bit for bit in
deterministic mode, with a call of another shape in between so that leftovers
of a differently laid-out call are exercised.  This file is collected last so
that a run that stops at its first failure has run everything else."""
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


def _problem(w, seed):
    x = syn.make_inputs(w, seed=seed)
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale)
    return q, k, v, dO, o, lse


def _noalloc(w, q, k, v, dO, o, lse, deterministic):
    dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, 7), torch.empty_like(v)
    rc = binding.attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, w.B, w.H, w.T, w.T, w.dqk,
                                  w.dv, w.causal, w.scale, None, 0, deterministic)
    assert rc == binding.ATTN_OK, binding.attn_strerror(rc)
    assert binding.attn_bwd_noalloc_status() == binding.ATTN_OK
    return dq, dk, dv


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_matches_attn_bwd_twice(deterministic):
    w = syn.Workload("noalloc", B=2, H=4, T=1000, dqk=128, dv=128, causal=True)
    other = syn.Workload("noalloc_other", B=1, H=6, T=700, dqk=64, dv=64, causal=False)
    q, k, v, dO, o, lse = _problem(w, 11)
    ref = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale,
                           deterministic=deterministic)
    qo, ko, vo, dOo, oo, lseo = _problem(other, 12)
    ref_o = binding.backward(qo, ko, vo, oo, dOo, lseo, causal=False, scale=other.scale,
                             deterministic=deterministic)
    for _ in range(2):
        got = _noalloc(w, q, k, v, dO, o, lse, deterministic)
        # a call of another shape leaves its own contents in the shared array
        got_o = _noalloc(other, qo, ko, vo, dOo, oo, lseo, deterministic)
        torch.cuda.synchronize()
        for g, want in ((got, ref), (got_o, ref_o)):
            for a, b in zip(g, want):
                if deterministic:
                    assert torch.equal(a, b)
                else:
                    assert rel_err(a.float().cpu().numpy(), b.float().cpu().numpy()) <= TOL_GRAD


def test_noalloc_reports_a_device_timeout():
    """Host-side fault injection, as for attn_bwd: the ordered dQ wait of a
    deterministic call targets a value nothing writes; the status call must
    report the timeout, and the next call must run clean."""
    w = syn.Workload("noalloc_to", B=1, H=2, T=512, dqk=64, dv=64, causal=True)
    q, k, v, dO, o, lse = _problem(w, 13)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    binding.attn_debug_set_wait_bias(1000)
    try:
        rc = binding.attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, w.B, w.H, w.T, w.T,
                                      w.dqk, w.dv, True, w.scale, None, 0, True)
        assert rc == binding.ATTN_OK
        assert binding.attn_bwd_noalloc_status() == binding.ATTN_ERR_TIMEOUT
    finally:
        binding.attn_debug_set_wait_bias(0)
    ref = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale, deterministic=True)
    got = _noalloc(w, q, k, v, dO, o, lse, True)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, T, d = 1, 16, 32768, 128  # needs ~272 MB of workspace
    assert binding.attn_bwd_workspace_size(B, H, T, T, d, d) > 32 << 20
    A = 0x10000
    rc = binding.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, H, T, T, d, d, True, 0.088)
    assert rc == binding.ATTN_ERR_SCRATCH_TOO_SMALL
    assert "32 MiB" in binding.attn_strerror(rc)
