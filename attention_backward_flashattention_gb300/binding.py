"""ctypes binding of the C ABI in ``include/attn.h`` (libattn_gb300.so).

The functions named like the C entry points (``attn_fwd``, ``attn_bwd``, ...)
only marshal arguments: tensors become device pointers, streams become
``cudaStream_t`` handles, and the integer status comes back unchanged.
``forward`` / ``backward`` are conveniences on top that allocate outputs and
the workspace with PyTorch (device memory only) and raise ``AttnError`` on a
non-zero status.  Every step of the computation runs in the library's CUDA
kernels: there is no CPU path, and a missing library raises at first use.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_WORKSPACE_TOO_SMALL = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5
ATTN_ERR_INTERNAL = -6
ATTN_ERR_SCRATCH_TOO_SMALL = -7
LAYOUT_BTHD = 0
LAYOUT_PACKED_QKV = 1
MAX_VARLEN_SEQS = 1024

EXPORTED = ("attn_fwd", "attn_bwd_workspace_size", "attn_bwd", "attn_bwd_status",
            "attn_fwd_status", "attn_strerror", "attn_varlen_order", "attn_debug_set_wait_bias",
            "attn_profile_main_kernel", "attn_profile_aux_kernels", "attn_bwd_noalloc",
            "attn_bwd_noalloc_status", "attn_step_host_scratch_size", "attn_step_host",
            "attn_step_host_status", "attn_fwd_window", "attn_bwd_window", "attn_fwd_ex",
            "attn_bwd_ex", "attn_debug_cache_stats", "attn_debug_set_bwd_variant")
BLOCK = 128  # rows per block of a block-sparse mask

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} ({code})")
        self.code = code


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m attention_backward_flashattention_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P, I, P]
        lib.attn_fwd.restype = I
        lib.attn_fwd_window.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, I, P]
        lib.attn_fwd_window.restype = I
        lib.attn_bwd_window.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F,
                                        P, I, I, P, SZ, P]
        lib.attn_bwd_window.restype = I
        lib.attn_fwd_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, I, I, F, P, P,
                                    I, P]
        lib.attn_fwd_ex.restype = I
        lib.attn_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, I, I,
                                    F, P, P, I, I, P, SZ, P]
        lib.attn_bwd_ex.restype = I
        lib.attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.attn_bwd_workspace_size.restype = SZ
        lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, I, I, P,
                                 SZ, P]
        lib.attn_bwd.restype = I
        lib.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, I,
                                         I, P]
        lib.attn_bwd_noalloc.restype = I
        lib.attn_bwd_noalloc_status.argtypes = [P]
        lib.attn_bwd_noalloc_status.restype = I
        lib.attn_bwd_status.argtypes = [P, P]
        lib.attn_bwd_status.restype = I
        lib.attn_fwd_status.argtypes = [P]
        lib.attn_fwd_status.restype = I
        lib.attn_strerror.argtypes = [I]
        lib.attn_strerror.restype = ctypes.c_char_p
        lib.attn_varlen_order.argtypes = [P, I, P]
        lib.attn_varlen_order.restype = I
        lib.attn_profile_main_kernel.argtypes = [P, P]
        lib.attn_profile_main_kernel.restype = I
        lib.attn_profile_aux_kernels.argtypes = [P, P, P, P]
        lib.attn_profile_aux_kernels.restype = I
        lib.attn_debug_set_bwd_variant.argtypes = [I]
        lib.attn_debug_set_bwd_variant.restype = I
        lib.attn_debug_cache_stats.argtypes = [P]
        lib.attn_debug_cache_stats.restype = I
        lib.attn_debug_set_wait_bias.argtypes = [I]
        lib.attn_debug_set_wait_bias.restype = I
        lib.attn_step_host_scratch_size.argtypes = [I, I, I, I, I, I, I]
        lib.attn_step_host_scratch_size.restype = SZ
        lib.attn_step_host.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, SZ,
                                       P, P, P, P]
        lib.attn_step_host.restype = I
        lib.attn_step_host_status.argtypes = [P, I, I, I, I, I, I, I, P]
        lib.attn_step_host_status.restype = I
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


class _HostInts:
    """Keeps a host int32 array alive for the duration of a call."""

    def __init__(self, values):
        if values is None:
            self.arr = None
        else:
            vals = [int(v) for v in (values.tolist() if hasattr(values, "tolist") else values)]
            self.arr = (ctypes.c_int * len(vals))(*vals)

    @property
    def ptr(self):
        return None if self.arr is None else ctypes.cast(self.arr, ctypes.c_void_p)


# ----------------------------------------------------------------------------
# C entry points (same names, argument marshalling only)
# ----------------------------------------------------------------------------
def attn_fwd(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, scale, cu_seqlens=None,
             layout=LAYOUT_BTHD, stream=None) -> int:
    cu = _HostInts(cu_seqlens)
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, dqk, dv,
                           int(causal), float(scale), cu.ptr, layout, _stream(stream))


def attn_fwd_window(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, window_left, window_right,
                    scale, cu_seqlens=None, layout=LAYOUT_BTHD, stream=None) -> int:
    cu = _HostInts(cu_seqlens)
    return load().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk,
                                  dqk, dv, int(causal), int(window_left), int(window_right),
                                  float(scale), cu.ptr, layout, _stream(stream))


def attn_bwd_window(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal,
                    window_left, window_right, scale, cu_seqlens=None, layout=LAYOUT_BTHD,
                    deterministic=False, workspace=None, workspace_bytes=0, stream=None) -> int:
    cu = _HostInts(cu_seqlens)
    return load().attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                  _ptr(dq), _ptr(dk), _ptr(dv_out), B, H, Tq, Tk, dqk, dv,
                                  int(causal), int(window_left), int(window_right),
                                  float(scale), cu.ptr, layout, int(deterministic),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_fwd_ex(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, window_left, window_right,
                block_mask, mask_batches, mask_heads, scale, cu_seqlens_q=None,
                cu_seqlens_k=None, layout=LAYOUT_BTHD, stream=None) -> int:
    cq, ck = _HostInts(cu_seqlens_q), _HostInts(cu_seqlens_k)
    return load().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, dqk,
                              dv, int(causal), int(window_left), int(window_right),
                              _ptr(block_mask), int(mask_batches), int(mask_heads), float(scale),
                              cq.ptr, ck.ptr, layout, _stream(stream))


def attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal, window_left,
                window_right, block_mask, mask_batches, mask_heads, scale, cu_seqlens_q=None,
                cu_seqlens_k=None, layout=LAYOUT_BTHD, deterministic=False, workspace=None,
                workspace_bytes=0, stream=None) -> int:
    cq, ck = _HostInts(cu_seqlens_q), _HostInts(cu_seqlens_k)
    return load().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv_out), B, H, Tq, Tk, dqk, dv, int(causal),
                              int(window_left), int(window_right), _ptr(block_mask),
                              int(mask_batches), int(mask_heads), float(scale), cq.ptr, ck.ptr,
                              layout, int(deterministic), _ptr(workspace), int(workspace_bytes),
                              _stream(stream))


def _mask_dims(block_mask):
    """(mask, mask_batches, mask_heads) of a [NQ][NK] or [Bm][Hm][NQ][NK] uint8
    device tensor (None: no block mask)."""
    if block_mask is None:
        return None, 1, 1
    if block_mask.dtype != torch.uint8 or not block_mask.is_contiguous():
        raise ValueError("block_mask must be a contiguous uint8 tensor")
    if block_mask.dim() == 2:
        return block_mask, 1, 1
    if block_mask.dim() != 4:
        raise ValueError("block_mask must be [NQ][NK] or [Bm][Hm][NQ][NK]")
    return block_mask, block_mask.shape[0], block_mask.shape[1]


def attn_bwd_workspace_size(B, H, Tq, Tk, dqk, dv, varlen=False, deterministic=False) -> int:
    return int(load().attn_bwd_workspace_size(B, H, Tq, Tk, dqk, dv, int(varlen),
                                              int(deterministic)))


def attn_bwd(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal, scale,
             cu_seqlens=None, layout=LAYOUT_BTHD, deterministic=False, workspace=None,
             workspace_bytes=0, stream=None) -> int:
    cu = _HostInts(cu_seqlens)
    return load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                           _ptr(dk), _ptr(dv_out), B, H, Tq, Tk, dqk, dv, int(causal),
                           float(scale), cu.ptr, layout, int(deterministic), _ptr(workspace),
                           int(workspace_bytes), _stream(stream))


def attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal, scale,
                     cu_seqlens=None, layout=LAYOUT_BTHD, deterministic=False,
                     stream=None) -> int:
    """attn_bwd without a caller workspace (the library's 32 MiB device array)."""
    cu = _HostInts(cu_seqlens)
    return load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv_out), B, H, Tq, Tk, dqk, dv,
                                   int(causal), float(scale), cu.ptr, layout, int(deterministic),
                                   _stream(stream))


def attn_bwd_noalloc_status(stream=None) -> int:
    return load().attn_bwd_noalloc_status(_stream(stream))


def attn_bwd_status(workspace, stream=None) -> int:
    return load().attn_bwd_status(_ptr(workspace), _stream(stream))


def attn_fwd_status(stream=None) -> int:
    return load().attn_fwd_status(_stream(stream))


def attn_strerror(code: int) -> str:
    return load().attn_strerror(int(code)).decode()


def strerror(code: int) -> str:
    try:
        return attn_strerror(code)
    except RuntimeError:
        return f"code {code}"


def attn_profile_main_kernel(event_start=None, event_stop=None) -> int:
    """Record torch.cuda.Event (or raw cudaEvent_t) pairs around the backward main kernel."""
    conv = lambda e: None if e is None else (e.cuda_event if hasattr(e, "cuda_event") else int(e))
    return load().attn_profile_main_kernel(conv(event_start), conv(event_stop))


def attn_profile_aux_kernels(pre_start=None, pre_stop=None, convert_start=None,
                             convert_stop=None) -> int:
    """Record event pairs around the backward's preprocess and dQ conversion kernels."""
    conv = lambda e: None if e is None else (e.cuda_event if hasattr(e, "cuda_event") else int(e))
    return load().attn_profile_aux_kernels(conv(pre_start), conv(pre_stop), conv(convert_start),
                                           conv(convert_stop))


BWD_AUTO, BWD_ONE_CTA, BWD_CTA_PAIR = 0, 1, 2


def attn_debug_set_bwd_variant(variant: int) -> int:
    """Backward main kernel where both apply: 0 library's choice, 1 one CTA, 2 CTA pairs."""
    return load().attn_debug_set_bwd_variant(int(variant))


def attn_debug_cache_stats() -> dict:
    """Host-side cache counters (tensor maps encoded / reused, tables built / reused)."""
    out = (ctypes.c_longlong * 4)()
    rc = load().attn_debug_cache_stats(ctypes.cast(out, ctypes.c_void_p))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_debug_cache_stats")
    return {"map_encodes": out[0], "map_hits": out[1], "table_builds": out[2],
            "table_hits": out[3]}


def attn_debug_set_wait_bias(bias: int) -> int:
    return load().attn_debug_set_wait_bias(int(bias))


def attn_step_host_scratch_size(B, H, T, dqk, dv, heads_per_group=0, deterministic=False) -> int:
    return int(load().attn_step_host_scratch_size(B, H, T, dqk, dv, int(heads_per_group),
                                                  int(deterministic)))


def attn_step_host(q, k, v, dO, o, dq, dk, dv_out, B, H, T, dqk, dv, causal, scale,
                   deterministic=False, heads_per_group=0, scratch=None, scratch_bytes=0,
                   stream=None, stream2=None, h2d_stream=None, d2h_stream=None) -> int:
    """Host tensors in and out (pinned CPU tensors); copies overlapped with the kernels."""
    opt = lambda s: None if s is None else _stream(s)
    return load().attn_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(o), _ptr(dq),
                                 _ptr(dk), _ptr(dv_out), B, H, T, dqk, dv, int(causal),
                                 float(scale), int(deterministic), int(heads_per_group),
                                 _ptr(scratch), int(scratch_bytes), _stream(stream),
                                 opt(stream2), opt(h2d_stream), opt(d2h_stream))


def attn_step_host_status(scratch, B, H, T, dqk, dv, heads_per_group=0, deterministic=False,
                          stream=None) -> int:
    return load().attn_step_host_status(_ptr(scratch), B, H, T, dqk, dv, int(heads_per_group),
                                        int(deterministic), _stream(stream))


def attn_varlen_order(cu_seqlens) -> list:
    cu = _HostInts(cu_seqlens)
    n = len(cu.arr) - 1
    out = (ctypes.c_int * max(n, 1))()
    rc = load().attn_varlen_order(cu.ptr, n, ctypes.cast(out, ctypes.c_void_p))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_varlen_order")
    return list(out)[:n]


# ----------------------------------------------------------------------------
# Conveniences: shapes from tensors, outputs allocated with torch
# ----------------------------------------------------------------------------
def _dims(q, k, v, cu_seqlens, layout):
    # the library sees only pointers: a tensor whose rank does not match the
    # layout would be read with the wrong sizes
    rank = (3 if cu_seqlens is not None else 4) + (1 if layout == LAYOUT_PACKED_QKV else 0)
    if layout == LAYOUT_PACKED_QKV:
        rank -= 1  # q, k, v are slot views: (..., H, d) of a (..., 3, H, d) buffer
    if any(t.dim() != rank for t in (q, k, v)):
        raise ValueError(f"q, k, v must have {rank} dimensions for this layout "
                         f"({'variable length' if cu_seqlens is not None else 'fixed length'})")
    if layout == LAYOUT_PACKED_QKV:
        # q, k, v are slot views of one (..., 3, H, d) buffer
        H, dqk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
    else:
        H, dqk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    if cu_seqlens is not None:
        B = len(cu_seqlens) - 1
        Tq, Tk = q.shape[0], k.shape[0]
    else:
        B, Tq, Tk = q.shape[0], q.shape[1], k.shape[1]
    return B, H, Tq, Tk, dqk, dv


def forward(q, k, v, causal=False, scale=None, cu_seqlens=None, layout=LAYOUT_BTHD,
            with_lse=True, stream=None, window=None, block_mask=None, cu_seqlens_k=None):
    """O (bf16, like q with v's head size) and LSE (fp32) or None.
    window: (left, right) local-attention bounds (-1: open side), or None.
    block_mask: device uint8 [NQ][NK] or [Bm][Hm][NQ][NK] (NQ, NK: blocks of
    BLOCK rows), non-zero = the block pair takes part, or None.
    cu_seqlens_k: key offsets of a variable-length batch when they differ
    from cu_seqlens (the query offsets), or None."""
    B, H, Tq, Tk, dqk, dv = _dims(q, k, v, cu_seqlens, layout)
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    o = torch.empty(q.shape[:-2] + (H, dv), dtype=torch.bfloat16, device=q.device)
    lse = None
    if with_lse:
        lse = torch.empty((H, Tq) if cu_seqlens is not None else (B, H, Tq),
                          dtype=torch.float32, device=q.device)
    wl, wr = (-1, -1) if window is None else window
    bm, mb, mh = _mask_dims(block_mask)
    rc = attn_fwd_ex(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, wl, wr, bm, mb, mh, scale,
                     cu_seqlens, cu_seqlens_k, layout, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return o, lse


def backward(q, k, v, o, dO, lse, causal=False, scale=None, cu_seqlens=None,
             layout=LAYOUT_BTHD, deterministic=False, workspace=None, stream=None, out=None,
             window=None, block_mask=None, cu_seqlens_k=None):
    """(dq, dk, dv) as bf16 tensors shaped like q, k, v (a packed buffer for layout 1).
    window, block_mask, cu_seqlens_k: as in forward()."""
    B, H, Tq, Tk, dqk, dv = _dims(q, k, v, cu_seqlens, layout)
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    if out is not None:
        dq, dk, dvt = out
    elif layout == LAYOUT_PACKED_QKV:
        g = torch.empty(q.shape[:-2] + (3, H, dqk), dtype=torch.bfloat16, device=q.device)
        dq, dk, dvt = g.select(-3, 0), g.select(-3, 1), g.select(-3, 2)
    else:
        dq = torch.empty_like(q)
        dk = torch.empty_like(k)
        dvt = torch.empty_like(v)
    need = attn_bwd_workspace_size(B, H, Tq, Tk, dqk, dv, cu_seqlens is not None, deterministic)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wl, wr = (-1, -1) if window is None else window
    bm, mb, mh = _mask_dims(block_mask)
    rc = attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dvt, B, H, Tq, Tk, dqk, dv, causal, wl, wr, bm,
                     mb, mh, scale, cu_seqlens, cu_seqlens_k, layout, deterministic, workspace,
                     workspace.numel() * workspace.element_size(), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dvt


def step_host(q, k, v, dO, causal=False, scale=None, deterministic=False, heads_per_group=0,
              with_o=False, out=None, scratch=None, streams=None, device=None):
    """Forward + backward of host (B,T,H,d) bf16 tensors through attn_step_host.

    Returns (dq, dk, dv, o) as host tensors (o is None unless with_o).  Pass
    pinned tensors for overlapped copies; `out` reuses (dq, dk, dv, o) host
    buffers, `scratch` a device uint8 buffer, `streams` a (compute, compute2,
    h2d, d2h) tuple (compute2 may be None).  The call is asynchronous: synchronise the compute stream before
    reading the outputs (this helper does so unless `streams` is given)."""
    B, T, H, dqk = q.shape
    dv = v.shape[-1]
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if out is None:
        mk = lambda t: torch.empty(t.shape, dtype=torch.bfloat16, pin_memory=True)
        out = (mk(q), mk(k), mk(v), mk(v) if with_o else None)
    need = attn_step_host_scratch_size(B, H, T, dqk, dv, heads_per_group, deterministic)
    if scratch is None or scratch.numel() * scratch.element_size() < need:
        scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    own = streams is None
    if own:
        streams = (torch.cuda.current_stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev),
                   torch.cuda.Stream(dev))
    cs, cs2, hs, ds = streams
    dq, dk, dvt, o = out
    rc = attn_step_host(q, k, v, dO, o, dq, dk, dvt, B, H, T, dqk, dv, causal, scale,
                        deterministic, heads_per_group, scratch,
                        scratch.numel() * scratch.element_size(), cs, cs2, hs, ds)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_step_host")
    if own:
        cs.synchronize()
    return dq, dk, dvt, o
