"""The C-ABI library builds, loads and exports every symbol include/attn.h
declares, and rejects bad arguments on the host before touching the GPU.
No compute calls here (no GPU needed)."""
import os
import re

import pytest

from attention_backward_flashattention_gb300 import binding
from attention_backward_flashattention_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 0x10000  # an aligned, never-dereferenced stand-in address


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return binding.load()


def _declared():
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(attn_\w+)\s*\(", src, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_strerror"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.EXPORTED) == set(names)


def test_strerror(lib):
    assert binding.attn_strerror(0) == "ok"
    assert binding.attn_strerror(binding.ATTN_ERR_TIMEOUT) == "device wait timed out"
    assert binding.attn_strerror(-99) == "unknown error"


def _fwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Tq=128, Tk=128, dqk=64, dv=64, causal=1,
                scale=0.125, cu_seqlens=None, layout=0, stream=0)
    args.update(kw)
    return binding.attn_fwd(**args)


def _bwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, dq=A, dk=A, dv_out=A, B=1, H=2, Tq=128,
                Tk=128, dqk=64, dv=64, causal=1, scale=0.125, cu_seqlens=None, layout=0,
                deterministic=0, workspace=A, workspace_bytes=1 << 30, stream=0)
    args.update(kw)
    return binding.attn_bwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(o=A + 8), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=A + 2), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tq=0, Tk=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(layout=7), binding.ATTN_ERR_INVALID_ARG),
    (dict(dqk=96, dv=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(dqk=128, dv=64), binding.ATTN_ERR_UNSUPPORTED),
    (dict(Tq=256, Tk=128), binding.ATTN_ERR_UNSUPPORTED),      # causal, Tq > Tk
    (dict(layout=1, dqk=192, dv=128), binding.ATTN_ERR_UNSUPPORTED),
    (dict(cu_seqlens=[0, 100, 90], B=2, Tq=90, Tk=90), binding.ATTN_ERR_INVALID_ARG),
    (dict(cu_seqlens=[0, 100, 200], B=2, Tq=300, Tk=300), binding.ATTN_ERR_INVALID_ARG),
    (dict(cu_seqlens=[1, 100, 200], B=2, Tq=200, Tk=200), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.125), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG),
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(lse=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(workspace=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(workspace=A + 16), binding.ATTN_ERR_INVALID_ARG),   # must be 256-byte aligned
    (dict(dq=A + 4), binding.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=1024), binding.ATTN_ERR_WORKSPACE_TOO_SMALL),
    (dict(dqk=192, dv=192), binding.ATTN_ERR_UNSUPPORTED),
    (dict(causal=1, Tk=64), binding.ATTN_ERR_UNSUPPORTED),
    (dict(scale=-1.0), binding.ATTN_ERR_INVALID_ARG),
])
def test_bwd_rejects(lib, kw, code):
    assert _bwd(**kw) == code


def test_varlen_too_many_sequences(lib):
    n = binding.MAX_VARLEN_SEQS + 1
    cu = list(range(n + 1))
    assert _fwd(cu_seqlens=cu, B=n, Tq=n, Tk=n) == binding.ATTN_ERR_UNSUPPORTED


def test_workspace_size_formula(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for (B, H, T, dqk, dv, varlen) in [(1, 16, 32768, 128, 128, 0), (8, 12, 1024, 64, 64, 0),
                                       (2, 3, 200, 192, 128, 0), (40, 16, 32768, 128, 128, 1)]:
        tiles = (-(-T // 128) + B) if varlen else B * -(-T // 128)
        # header, two semaphores per (q-tile, head) (one per tile half: the
        # CTA-pair kernel orders each half on its own), -LSE2 and -D rows, dQ
        expect = (256 + r256(tiles * H * 2 * 4) + 2 * r256(tiles * H * 128 * 4)
                  + r256(tiles * H * 128 * dqk * 4))
        assert binding.attn_bwd_workspace_size(B, H, T, T, dqk, dv, varlen, 0) == expect
    assert binding.attn_bwd_workspace_size(1, 1, 1, 1, 96, 96) == 0


def test_varlen_order_longest_first(lib):
    assert binding.attn_varlen_order([0, 5, 105, 106, 300]) == [3, 1, 0, 2]
    # ties keep index order
    assert binding.attn_varlen_order([0, 10, 20, 25, 35]) == [0, 1, 3, 2]
    with pytest.raises(binding.AttnError):
        binding.attn_varlen_order([0, 10, 5])


def _step(**kw):
    args = dict(q=A, k=A, v=A, dO=A, o=None, dq=A, dk=A, dv_out=A, B=1, H=4, T=256, dqk=64,
                dv=64, causal=1, scale=0.125, deterministic=0, heads_per_group=0, scratch=A,
                scratch_bytes=1 << 40, stream=0, stream2=0, h2d_stream=0, d2h_stream=0)
    args.update(kw)
    return binding.attn_step_host(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(dv_out=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(scratch=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(scratch=A + 16), binding.ATTN_ERR_INVALID_ARG),    # must be 256-byte aligned
    (dict(heads_per_group=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(T=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(dqk=96, dv=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(scratch_bytes=4096), binding.ATTN_ERR_WORKSPACE_TOO_SMALL),
])
def test_step_host_rejects(lib, kw, code):
    assert _step(**kw) == code


def test_step_host_scratch_formula(lib):
    """Two device sets of G heads (q, k, v, dO, o, lse, dq, dk, dv, backward
    workspace, each rounded to 256 bytes) plus a status word per head."""
    def r256(x):
        return (x + 255) // 256 * 256
    for (B, H, T, dqk, dv, G, det) in [(1, 16, 32768, 128, 128, 0, 0), (2, 12, 1000, 64, 64, 5, 1),
                                       (1, 3, 200, 192, 128, 1, 0), (1, 7, 64, 128, 128, 9, 0)]:
        g = min(G, H) if G else -(-H // 2)
        rows = B * T
        eq, ev = rows * g * dqk * 2, rows * g * dv * 2
        ws = binding.attn_bwd_workspace_size(B, g, T, T, dqk, dv, 0, det)
        one = 2 * r256(eq) + 2 * r256(ev) + r256(ev) + r256(rows * g * 4) + 2 * r256(eq) \
            + r256(ev) + r256(ws)
        assert binding.attn_step_host_scratch_size(B, H, T, dqk, dv, G, det) == \
            2 * one + r256(H * 4), (B, H, T, dqk, dv, G, det)
    assert binding.attn_step_host_scratch_size(1, 4, 128, 96, 96) == 0
    assert binding.attn_step_host_scratch_size(1, 4, 128, 64, 64, -1) == 0


def test_window_rejects(lib):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Tq=128, Tk=256, dqk=64, dv=64, causal=0,
                window_left=16, window_right=0, scale=0.125, cu_seqlens=None, layout=0, stream=0)
    bad = dict(args, window_left=-2)
    assert binding.attn_fwd_window(**bad) == binding.ATTN_ERR_INVALID_ARG
    bad = dict(args, window_right=-5)
    assert binding.attn_fwd_window(**bad) == binding.ATTN_ERR_INVALID_ARG
    more_q = dict(args, Tq=300)  # a window with more queries than keys
    assert binding.attn_fwd_window(**more_q) == binding.ATTN_ERR_UNSUPPORTED
    bargs = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, dq=A, dk=A, dv_out=A, B=1, H=2, Tq=300, Tk=256,
                 dqk=64, dv=64, causal=0, window_left=-1, window_right=4, scale=0.125,
                 cu_seqlens=None, layout=0, deterministic=0, workspace=A,
                 workspace_bytes=1 << 30, stream=0)
    assert binding.attn_bwd_window(**bargs) == binding.ATTN_ERR_UNSUPPORTED



def _ex_fwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=2, H=2, Tq=300, Tk=700, dqk=64, dv=64, causal=1,
                window_left=-1, window_right=-1, block_mask=None, mask_batches=1, mask_heads=1,
                scale=0.125, cu_seqlens_q=[0, 100, 300], cu_seqlens_k=[0, 200, 700], layout=0,
                stream=0)
    args.update(kw)
    return binding.attn_fwd_ex(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_seqlens_k=[0, 200, 699]), "INVALID_ARG"),        # does not end at Tk
    (dict(cu_seqlens_k=[1, 200, 700]), "INVALID_ARG"),        # does not start at 0
    (dict(cu_seqlens_k=[0, 300, 200]), "INVALID_ARG"),        # decreasing
    (dict(cu_seqlens_k=[0, 0, 700]), "INVALID_ARG"),          # queries without keys
    (dict(cu_seqlens_k=[0, 50, 700]), "UNSUPPORTED"),         # causal, Lq 100 > Lk 50
    (dict(causal=0, window_left=8, cu_seqlens_k=[0, 50, 700]), "UNSUPPORTED"),  # window too
    (dict(cu_seqlens_q=None), "INVALID_ARG"),                 # key offsets without query ones
    (dict(layout=1, Tq=700, cu_seqlens_q=[0, 200, 700],
          cu_seqlens_k=[0, 250, 700]), "UNSUPPORTED"),        # packed needs shared offsets
    (dict(block_mask=A, mask_batches=3), "INVALID_ARG"),      # neither 1 nor B
])
def test_ex_rejects(lib, kw, code):
    assert _ex_fwd(**kw) == getattr(binding, "ATTN_ERR_" + code)


def test_ex_backward_rejects_like_forward(lib):
    args = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, dq=A, dk=A, dv_out=A, B=2, H=2, Tq=300, Tk=700,
                dqk=64, dv=64, causal=1, window_left=-1, window_right=-1, block_mask=None,
                mask_batches=1, mask_heads=1, scale=0.125, cu_seqlens_q=[0, 100, 300],
                cu_seqlens_k=[0, 50, 700], layout=0, deterministic=0, workspace=A,
                workspace_bytes=1 << 30, stream=0)
    assert binding.attn_bwd_ex(**args) == binding.ATTN_ERR_UNSUPPORTED
    args["cu_seqlens_k"] = [0, 0, 700]
    assert binding.attn_bwd_ex(**args) == binding.ATTN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No fallback: with the library absent the binding raises at first use."""
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libattn_gb300.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(Exception, match="missing"):
        binding.load()
