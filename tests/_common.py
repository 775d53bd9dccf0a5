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
