"""Shared helpers of the parity tests: tolerance checks and device movement."""
import numpy as np
import torch

# Tolerances (relative Frobenius error over the whole tensor):
#   fp32 inputs: 1e-4 on o and on the final state;
#   bf16 inputs: 1e-2 on o, 5e-3 on the final state.
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 5e-3)}


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, np.float64)


def rel_fro(x, ref) -> float:
    x, ref = _np(x), _np(ref)
    den = np.linalg.norm(ref)
    if den == 0:
        return float(np.linalg.norm(x))
    return float(np.linalg.norm(x - ref) / den)


def worst_rel(x, ref, kind="tokens", cu_seqlens=None, n_seqs=1):
    """Largest relative Frobenius error over the (sequence, head) blocks.

    kind "tokens": [T, H, D] cut into documents by cu_seqlens (or n_seqs equal
    lengths); "state": [n, H, D, D] cut by (n, h); "decode": [N, W, H, D] cut by
    (b, h).  Blocks whose reference is zero are skipped.  Returns
    (worst error, (sequence, head))."""
    x, ref = _np(x), _np(ref)
    blocks = []
    if kind == "state":
        for n in range(ref.shape[0]):
            for h in range(ref.shape[1]):
                blocks.append(((n, h), x[n, h], ref[n, h]))
    elif kind == "decode":
        for n in range(ref.shape[0]):
            for h in range(ref.shape[2]):
                blocks.append(((n, h), x[n, :, h], ref[n, :, h]))
    else:
        T = ref.shape[0]
        if cu_seqlens is None:
            step = T // max(n_seqs, 1)
            cu = [i * step for i in range(n_seqs + 1)]
        else:
            cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        for n in range(len(cu) - 1):
            for h in range(ref.shape[1]):
                blocks.append(((n, h), x[cu[n]:cu[n + 1], h], ref[cu[n]:cu[n + 1], h]))
    worst, where = 0.0, None
    for key, a, b in blocks:
        den = np.linalg.norm(b)
        if den == 0:
            continue
        e = float(np.linalg.norm(a - b) / den)
        if where is None or e > worst:
            worst, where = e, key
    return worst, where


def err_report(x, ref, kind="tokens", cu_seqlens=None, n_seqs=1):
    """Whole-tensor relative error and a message that also names the worst
    (sequence, head) block, for assertions."""
    e = rel_fro(x, ref)
    w, where = worst_rel(x, ref, kind, cu_seqlens, n_seqs)
    return e, f"rel err {e:.3e}, worst (seq, head) {where}: {w:.3e}"


def to_dev(d: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "f32"
