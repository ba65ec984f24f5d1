"""Seeded synthetic inputs for the KDA forward workloads.

This module only draws random inputs; it holds none of the method's
arithmetic (no gate, no decay, no recurrence).  Both the CUDA path's tests /
benchmark and the oracle consume what it returns, so the two sides always see
bit-identical values.

Input recipe (all draws in fp32 from a seeded ``torch.Generator``, then cast):
  * q, k ~ N(0, 1), L2-normalised over d_k per (token, head) before the cast
    (the method takes normalised q, k; the kernels' L2-norm option, tested on
    unnormalised inputs of its own, can do it instead);
  * v ~ N(0, 1);
  * z (gate logits) ~ N(0, z_std) per channel, fp32;  A_h ~ N(0, A_std) per head
    (A_std = 0 gives A_h = 0);
  * beta = sigmoid(N(0, 1)), fp32 (the method takes beta after its sigmoid);
  * initial states ~ N(0, init_std) fp32, or none (zeros);
  * fused decode step: q, k, v ~ N(0, 1) before the short convolution (not
    normalised), beta logits ~ N(0, 1), output-gate logits ~ N(0, 1), convolution
    state ~ N(0, 1), convolution weights ~ U(-0.5, 0.5), output-norm weight
    1 + N(0, 0.1).
Standard deviations are the second argument of N(., .).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

D = 128  # d_k = d_v


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill", "segment", "decode"
    H: int
    T: int = 0           # total tokens (prefill / segment)
    dtype: str = "bf16"  # input dtype of q, k, v
    z_std: float = 1.0
    A_std: float = 0.0
    varlen: bool = False
    init_std: float = 0.0
    n_segments: int = 0
    N: int = 0           # decode batch
    W: int = 0           # decode window (1 + drafts)
    seed: int = 0


WORKLOADS = {
    # B=1, H=2, T=256, fp32, z~N(0,1), A=0, zero init, seed 0
    "tiny_fp32": Workload("tiny_fp32", "prefill", H=2, T=256, dtype="f32", seed=0),
    # B=1, H=16, T=8192, bf16, z~N(0,1.5), A~N(0,0.5), zero init
    "prefill_h16_t8k": Workload("prefill_h16_t8k", "prefill", H=16, T=8192, dtype="bf16",
                                z_std=1.5, A_std=0.5, seed=2),
    # 32768 packed tokens, H=32, doc lengths ~U[512, 8192], per-doc init ~N(0, 0.05)
    "varlen_32k_h32": Workload("varlen_32k_h32", "prefill", H=32, T=32768, dtype="bf16",
                               varlen=True, init_std=0.05, seed=3),
    # B=1, H=8, T=1,048,576, bf16, 148 segments
    "segscan_1m_h8": Workload("segscan_1m_h8", "segment", H=8, T=1 << 20, dtype="bf16",
                              n_segments=148, seed=4),
    # decode: N=256, H=96, window 1 + 4 drafts, fp32, state ~N(0, 0.05)
    "decode_mtp_b256_h96": Workload("decode_mtp_b256_h96", "decode", H=96, dtype="f32",
                                    init_std=0.05, N=256, W=5, seed=5),
}

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std=1.0, mean=0.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def draw_doc_lengths(total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Document lengths ~U{lo..hi} drawn until their sum reaches `total`; the
    last one is truncated so that the lengths add up to exactly `total`."""
    g = _gen(seed + 1000, "cpu")
    lens = []
    s = 0
    while s < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - s)
        lens.append(n)
        s += n
    return lens


def cu_from_lengths(lens) -> torch.Tensor:
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def prefill_inputs(T: int, H: int, dtype: str = "bf16", seed: int = 0, z_std: float = 1.0,
                   A_std: float = 0.0, cu_seqlens: Optional[torch.Tensor] = None,
                   init_std: float = 0.0, device="cpu", z_mean: float = 0.0,
                   beta_mean: float = 0.0, n_init: Optional[int] = None) -> dict:
    """q, k, v [T, H, D] (dtype), z [T, H, D] fp32, A [H] fp32, beta [T, H] fp32,
    cu_seqlens [n+1] int32 or None, init_state [n, H, D, D] fp32 or None."""
    g = _gen(seed, device)
    tdt = TORCH_DTYPE[dtype]
    q = _unit_rows(_randn((T, H, D), g, device)).to(tdt)
    k = _unit_rows(_randn((T, H, D), g, device)).to(tdt)
    v = _randn((T, H, D), g, device).to(tdt)
    z = _randn((T, H, D), g, device, std=z_std, mean=z_mean)
    A = _randn((H,), g, device, std=A_std) if A_std > 0 else torch.zeros(H, device=device)
    beta = torch.sigmoid(_randn((T, H), g, device, mean=beta_mean))
    n = (len(cu_seqlens) - 1) if cu_seqlens is not None else 1
    if n_init is not None:
        n = n_init
    init = _randn((n, H, D, D), g, device, std=init_std) if init_std > 0 else None
    return dict(q=q, k=k, v=v, z=z, A=A, beta=beta, cu_seqlens=cu_seqlens, init_state=init)


def workload_inputs(name: str, device="cpu", T: Optional[int] = None) -> dict:
    """Inputs of a named prefill / segment workload (T may be overridden to shrink it)."""
    w = WORKLOADS[name]
    T = T or w.T
    cu = None
    if w.varlen:
        cu = cu_from_lengths(draw_doc_lengths(T, 512, 8192, w.seed))
    return prefill_inputs(T, w.H, w.dtype, w.seed, w.z_std, w.A_std, cu, w.init_std, device)


def decode_state(N: int, H: int, seed: int, std: float = 0.05, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return _randn((N, H, D, D), g, device, std=std)


def decode_window(N: int, W: int, H: int, step: int, seed: int, dtype: str = "f32",
                  z_std: float = 1.0, A_std: float = 0.0, device="cpu", z_mean: float = 0.0) -> dict:
    """Projected inputs of one decode window [t0, d1 .. d_{W-1}]: q, k, v, z [N, W, H, D],
    beta [N, W, H], and num_accepted [N] ~ U{0 .. W-1} for this step."""
    g = _gen(seed * 7919 + 17 * step + 1, device)
    tdt = TORCH_DTYPE[dtype]
    q = _unit_rows(_randn((N, W, H, D), g, device)).to(tdt)
    k = _unit_rows(_randn((N, W, H, D), g, device)).to(tdt)
    v = _randn((N, W, H, D), g, device).to(tdt)
    z = _randn((N, W, H, D), g, device, std=z_std, mean=z_mean)
    beta = torch.sigmoid(_randn((N, W, H), g, device))
    nacc = torch.randint(0, W, (N,), generator=g, device=device, dtype=torch.int32)
    return dict(q=q, k=k, v=v, z=z, beta=beta, num_accepted=nacc)


def decode_A(H: int, seed: int, A_std: float = 0.0, device="cpu") -> torch.Tensor:
    if A_std <= 0:
        return torch.zeros(H, device=device)
    g = _gen(seed + 99, device)
    return _randn((H,), g, device, std=A_std)


def segment_bounds(n_chunks: int, n_segments: int) -> list[tuple[int, int]]:
    """Balanced chunk-aligned split of n_chunks into n_segments ranges, earlier
    segments one chunk longer when the division is not exact."""
    base, extra = divmod(n_chunks, n_segments)
    out = []
    c = 0
    for i in range(n_segments):
        n = base + (1 if i < extra else 0)
        out.append((c, c + n))
        c += n
    return out


def decode_fused_params(H: int, seed: int, device="cpu") -> dict:
    """Parameters of the fused decode step: short-convolution weights conv_w [3, H, D, 4]
    (q, k, v; tap 3 multiplies the current token) ~ U(-0.5, 0.5), the range of the usual
    fan-in initialisation of a width-4 depthwise convolution; output-norm weight
    o_norm_w [D] = 1 + N(0, 0.1)."""
    g = _gen(seed + 313, device)
    conv_w = torch.rand((3, H, D, 4), generator=g, device=device, dtype=torch.float32).sub_(0.5)
    o_norm_w = _randn((D,), g, device, std=0.1, mean=1.0)
    return dict(conv_w=conv_w, o_norm_w=o_norm_w)


def decode_conv_state(N: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """Short-convolution state [N, H, 3, 3, D] fp32 (q, k, v; the last three projected
    inputs, oldest first) ~ N(0, 1)."""
    g = _gen(seed + 717, device)
    return _randn((N, H, 3, 3, D), g, device)


def decode_fused_window(N: int, W: int, H: int, step: int, seed: int, dtype: str = "f32",
                        z_std: float = 1.0, device="cpu") -> dict:
    """Projected inputs of one window of the fused decode step, before the short
    convolution: q, k, v [N, W, H, D] ~ N(0, 1) (not normalised: the step normalises q
    and k after the convolution), z [N, W, H, D] ~ N(0, z_std), beta logits [N, W, H]
    ~ N(0, 1), output-gate logits o_gate [N, W, H, D] ~ N(0, 1) fp32, and
    num_accepted [N] ~ U{0 .. W-1}."""
    g = _gen(seed * 7919 + 17 * step + 5, device)
    tdt = TORCH_DTYPE[dtype]
    q = _randn((N, W, H, D), g, device).to(tdt)
    k = _randn((N, W, H, D), g, device).to(tdt)
    v = _randn((N, W, H, D), g, device).to(tdt)
    z = _randn((N, W, H, D), g, device, std=z_std)
    beta = _randn((N, W, H), g, device)
    o_gate = _randn((N, W, H, D), g, device)
    nacc = torch.randint(0, W, (N,), generator=g, device=device, dtype=torch.int32)
    return dict(q=q, k=k, v=v, z=z, beta=beta, o_gate=o_gate, num_accepted=nacc)
