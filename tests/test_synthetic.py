"""The seeded input recipe is reproducible and follows its stated rules."""
import math

import numpy as np
import torch

from attention_backward_flashattention_gb300 import synthetic as syn


def test_inputs_are_seeded_and_bf16():
    a = syn.make_inputs(syn.TINY[0])
    b = syn.make_inputs(syn.TINY[0])
    for n in ("q", "k", "v", "dO"):
        assert a[n].dtype == torch.bfloat16
        assert torch.equal(a[n], b[n])
    assert a["q"].shape == (1, 128, 2, 64)
    c = syn.make_inputs(syn.TINY[0], seed=1)
    assert not torch.equal(a["q"], c["q"])


def test_packed_layout_views():
    w = syn.Workload("p", 2, 3, 40, 16, 16, True, layout=syn.LAYOUT_PACKED, do_scale=0.1)
    x = syn.make_inputs(w)
    assert x["qkv"].shape == (2, 40, 3, 3, 16)
    assert torch.equal(x["k"], x["qkv"][:, :, 1])
    assert x["q"].data_ptr() == x["qkv"].data_ptr()
    # dO carries the 0.1 factor: its spread is about a tenth of Q's
    assert 0.05 < x["dO"].float().std().item() < 0.2


def test_varlen_lengths_rule():
    lens = syn.varlen_lengths()
    assert sum(lens) == 32768
    assert all(1 <= L <= 16384 for L in lens)
    assert all(L >= 512 for L in lens[:-1])
    assert lens == syn.varlen_lengths()           # seeded
    x = syn.make_inputs(syn.VARLEN)
    cu = x["cu_seqlens"].numpy()
    assert cu[0] == 0 and cu[-1] == 32768 and np.all(np.diff(cu) == np.array(lens))
    assert x["q"].shape == (32768, 16, 128)


def test_flop_formulas():
    w = syn.HEADLINE
    assert w.B == 1 and w.T == 32768 and w.H == 16 and w.causal
    assert math.isclose(w.bwd_flops(), 2 * 16 * 32768 ** 2 * (3 * 128 + 2 * 128) / 2)
    assert math.isclose(w.bwd_flops() / 1e12, 10.995116, rel_tol=1e-6)
