"""Seeded synthetic inputs for the MoE routing + FP8 path.

This module only draws inputs.  It holds none of the path's arithmetic (no
top-k, no routing, no scaling or casting), so both the CUDA path and the CPU
oracle may take their inputs from it.

Five workloads, named by what they are:

``tiny``            T=64 tokens, E=16 experts, k=2, hidden 256; scores and x
                    ~N(0,1).
``decode_1k``       T=1024, E=256, k=8, hidden 4096; scores and x ~N(0,1).
``skewed_8k``       T=8192, E=256, k=8, hidden 7168; scores ~N(0,1) plus a per
                    expert bias 2*ln(p_r) with p_r the Zipf(s=1.1) probability
                    of rank r = e+1 over the 256 experts; x ~N(0,1) with 72
                    channels (round(1% of 7168), a seeded choice shared by all
                    tokens) multiplied by 50 in fp32 before the bf16 rounding.
``swiglu_64k``      65536 expert-sorted rows (T*k of ``skewed_8k``); each row
                    holds gate | up halves of 2048 bf16 each, ~N(0,1).  The op
                    is row-wise, so its values do not depend on the routing.
``prefill_64k``     T=65536, E=256, k=8, hidden 7168; scores ~N(0,1) plus a
                    per-expert bias ~U[-0.5, 0.5]; x ~N(0, 0.5^2).

Every tensor is drawn in fp32 from ``torch.Generator`` seeded with ``seed``
(0 by default) on the requested device, in the fixed order scores, bias, x,
outlier channels, then (on request) the SwiGLU input and the combine input y;
bf16 tensors are the round-to-nearest-even bf16 of those draws.  The combine
input y [T*k, H] stands in for the expert GEMM output, which the path does not
compute: bf16 ~N(0,1).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int = 0          # tokens
    E: int = 0          # experts
    k: int = 0          # experts per token
    H: int = 0          # hidden size (route/expand/combine)
    N: int = 0          # SwiGLU output width (input row = 2N)
    M: int = 0          # SwiGLU rows
    bias: str = "none"  # "none" | "zipf" | "uniform"
    x_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 50.0
    zipf_s: float = 1.1
    zipf_mult: float = 2.0

    @property
    def R(self) -> int:
        """Routed rows T*k."""
        return self.T * self.k

    @property
    def G(self) -> int:
        return self.H // 128


WORKLOADS = {
    "tiny": Workload("tiny", T=64, E=16, k=2, H=256),
    "decode_1k": Workload("decode_1k", T=1024, E=256, k=8, H=4096),
    "skewed_8k": Workload("skewed_8k", T=8192, E=256, k=8, H=7168, bias="zipf",
                          outlier_frac=0.01),
    "swiglu_64k": Workload("swiglu_64k", M=65536, N=2048),
    # the skewed workload with the Zipf bias multiplier 0.4 instead of 2: about
    # 10 % of the experts take half of the copies (a sensitivity variant)
    "skewed_8k_mild": Workload("skewed_8k_mild", T=8192, E=256, k=8, H=7168, bias="zipf",
                               zipf_mult=0.4, outlier_frac=0.01),
    "prefill_64k": Workload("prefill_64k", T=65536, E=256, k=8, H=7168, bias="uniform",
                            x_std=0.5),
}


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def zipf_log_bias(E: int, s: float = 1.1, mult: float = 2.0) -> torch.Tensor:
    """Per-expert bias mult * ln(p_r), p_r = r^-s / sum_{r'=1..E} r'^-s, with
    rank r = e + 1 (the identity ranking).  Computed in float64, returned fp32."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    p = r.pow(-s)
    p = p / p.sum()
    return (mult * torch.log(p)).to(torch.float32)


def make_scores(w: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router scores [T, E] fp32 (draw 1: N(0,1); draw 2: the bias, if any)."""
    g = _gen(seed, device)
    s = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32)
    if w.bias == "zipf":
        s += zipf_log_bias(w.E, w.zipf_s, w.zipf_mult).to(device)
    elif w.bias == "uniform":
        b = torch.rand(w.E, generator=g, device=device, dtype=torch.float32) - 0.5
        s += b
    return s


def make_inputs(w: Workload, seed: int = 0, device="cpu", with_y: bool = False,
                with_swiglu: bool = False, swiglu_rows: int | None = None,
                swiglu_n: int | None = None) -> dict:
    """Draw every input of one workload on ``device`` from one generator.

    Returns a dict with ``scores`` [T,E] f32 and ``x`` [T,H] bf16 (route
    workloads), ``swiglu_x`` [M, 2N] bf16 (SwiGLU workload, or with_swiglu),
    ``y`` [T*k, H] bf16 (with_y), and ``outlier_channels`` when used."""
    g = _gen(seed, device)
    out: dict = {}
    if w.T > 0:
        s = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32)
        if w.bias == "zipf":
            s += zipf_log_bias(w.E, w.zipf_s, w.zipf_mult).to(device)
        elif w.bias == "uniform":
            s += torch.rand(w.E, generator=g, device=device, dtype=torch.float32) - 0.5
        out["scores"] = s
        x = torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32)
        if w.x_std != 1.0:
            x *= w.x_std
        if w.outlier_frac > 0:
            n_out = int(round(w.outlier_frac * w.H))
            ch = torch.randperm(w.H, generator=g, device=device)[:n_out]
            x[:, ch] *= w.outlier_scale
            out["outlier_channels"] = ch
        out["x"] = x.to(torch.bfloat16)
        del x
    if w.M > 0 or with_swiglu:
        M = swiglu_rows if swiglu_rows is not None else (w.M if w.M > 0 else w.R)
        N = swiglu_n if swiglu_n is not None else (w.N if w.N > 0 else 2048)
        out["swiglu_x"] = _randn_bf16((M, 2 * N), g, device)
    if with_y:
        out["y"] = _randn_bf16((w.R, w.H), g, device)
    return out


def _randn_bf16(shape, g, device, chunk_rows: int = 8192) -> torch.Tensor:
    """N(0,1) bf16 drawn in row chunks (bounded fp32 temporaries)."""
    rows, cols = shape
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn(r1 - r0, cols, generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def random_small(T: int, E: int, k: int, H: int, seed: int, device="cpu",
                 ties: bool = False, zero_groups: bool = False) -> dict:
    """Small randomised cases for parity sweeps.

    ties: scores drawn from a few integer levels so many rows hold equal
    scores.  zero_groups: some 128-channel groups of x set to exactly zero and
    some to tiny values (below the 1e-4 scale floor)."""
    g = _gen(seed, device)
    if ties:
        s = torch.randint(-2, 3, (T, E), generator=g, device=device).to(torch.float32)
    else:
        s = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    if zero_groups and T > 0:
        G = H // 128
        sel = torch.rand(T, G, generator=g, device=device) < 0.25
        tiny = torch.rand(T, G, generator=g, device=device) < 0.25
        m = sel.repeat_interleave(128, dim=1)
        t = tiny.repeat_interleave(128, dim=1)
        x = torch.where(m, torch.zeros_like(x), x)
        x = torch.where(t & ~m, x * 1e-6, x)
    return {"scores": s, "x": x.to(torch.bfloat16)}


def random_permutation_pos(T: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    """A seeded bijection (t, j) -> row in [0, T*k), shaped [T, k] int32: a
    routing layout for testing expand and combine on their own."""
    g = _gen(seed, device)
    return torch.randperm(T * k, generator=g, device=device).to(torch.int32).view(T, k)


def skew_stats(counts) -> dict:
    """Summary of a per-expert count vector: how many experts take half the
    routed copies, how many are empty, min/max/mean."""
    c = torch.as_tensor(counts).to(torch.int64).flatten().sort(descending=True).values
    tot = int(c.sum())
    half = int((c.cumsum(0) < (tot + 1) // 2).sum()) + 1 if tot > 0 else 0
    return {
        "experts_taking_half": half,
        "empty_experts": int((c == 0).sum()),
        "max": int(c[0]) if c.numel() else 0,
        "min": int(c[-1]) if c.numel() else 0,
        "mean": tot / max(1, c.numel()),
    }


__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_scores", "zipf_log_bias",
           "random_small", "random_permutation_pos", "skew_stats"]

