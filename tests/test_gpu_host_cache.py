"""The host-side cache of tensor maps and variable-length schedule tables: a
call repeated with the same pointers, shapes and options re-encodes no tensor
map and rebuilds no table, and its results are unchanged."""
import pytest
import torch

from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from attention_backward_flashattention_gb300 import build
    build.build()


def test_repeated_calls_reuse_maps_and_tables():
    w = syn.Workload("cache_varlen", B=3, H=2, T=300, dqk=64, dv=64, causal=True,
                     varlen=(300, 77, 129))
    x = syn.make_inputs(w, seed=4)
    cu = [int(c) for c in x["cu_seqlens"]]
    dev = "cuda:0"
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu)
    ref = binding.backward(q, k, v, o, dO, lse, causal=True, scale=w.scale, cu_seqlens=cu,
                           deterministic=True)
    torch.cuda.synchronize()
    before = binding.attn_debug_cache_stats()
    o2, lse2 = binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu)
    got = binding.backward(q, k, v, o2, dO, lse2, causal=True, scale=w.scale, cu_seqlens=cu,
                           deterministic=True, out=[torch.empty_like(t) for t in (q, k, v)])
    torch.cuda.synchronize()
    after = binding.attn_debug_cache_stats()
    # the second forward + backward hit on q, k, v (forward) and q, k, v, dO
    # (backward) and on both tables; output pointers are not part of any map
    assert after["map_encodes"] == before["map_encodes"]
    assert after["map_hits"] - before["map_hits"] == 7
    assert after["table_builds"] == before["table_builds"]
    assert after["table_hits"] - before["table_hits"] == 2
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    # other offsets: a new table, maps still reused (same pointers and totals)
    cu3 = [0, 100, 377, 506]
    binding.forward(q, k, v, causal=True, scale=w.scale, cu_seqlens=cu3)
    torch.cuda.synchronize()
    last = binding.attn_debug_cache_stats()
    assert last["table_builds"] == after["table_builds"] + 1
    assert last["map_encodes"] == after["map_encodes"]
