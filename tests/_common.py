"""Test helpers: layout marshalling and error metrics (no attention arithmetic)."""
import numpy as np
import torch


def to_problems(x: torch.Tensor) -> np.ndarray:
    """(B, T, H, d) tensor -> float64 [B*H][T][d] (one problem per (b, h))."""
    x = x.float().permute(0, 2, 1, 3).contiguous()
    return x.reshape(-1, x.shape[2], x.shape[3]).double().numpy()


def varlen_problems(x: torch.Tensor, cu) -> list:
    """(sum T, H, d) tensor + offsets -> list of [T_s][d] float64, (seq, head) order."""
    cu = [int(c) for c in cu]
    xf = x.float()
    out = []
    for s in range(len(cu) - 1):
        for h in range(x.shape[1]):
            out.append(xf[cu[s]:cu[s + 1], h, :].double().numpy())
    return out


def rel_err(x, ref) -> float:
    """Normwise relative error ||x - ref||_F / ||ref||_F."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def max_abs(x, ref) -> float:
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def row_err(x, ref) -> float:
    """Worst row of a [rows][d] comparison: max over rows of
    ||x_i - ref_i|| / max(||ref_i||, rms over rows of ||ref_i||).

    A wrong row or a wrong tile (a few rows among thousands) can hide under a
    normwise bound over the whole tensor; this bound sees it (such a row
    scores about 1).  The rms row norm is the floor of each row's scale, so
    rows whose exact value is (near) zero -- the first query of a causal
    problem has dQ = 0 -- are held to the tensor's typical magnitude rather
    than to their own.  The norm over a row, not its largest element, keeps
    the bf16 rounding of dS (whose row sums to zero, so short causal rows of
    dQ cancel) from dominating."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.size == 0:
        return 0.0
    x = x.reshape(-1, x.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(ref, axis=1)
    floor = float(np.sqrt(np.mean(rn * rn)))
    scale = np.maximum(rn, floor if floor > 0 else 1.0)
    return float(np.max(np.linalg.norm(x - ref, axis=1) / scale))
