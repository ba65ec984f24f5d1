"""Shared helpers of the parity tests: tolerance checks and device movement."""
import numpy as np
import torch

# Tolerances (relative Frobenius error over the whole tensor):
#   fp32 inputs: 1e-4 on o and on the final state;
#   bf16 inputs: 1e-2 on o, 5e-3 on the final state.
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 5e-3)}


def rel_fro(x, ref) -> float:
    x = x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    ref = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    if den == 0:
        return float(np.linalg.norm(x))
    return float(np.linalg.norm(x - ref) / den)


def to_dev(d: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "f32"
