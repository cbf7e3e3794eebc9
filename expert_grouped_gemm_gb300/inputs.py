"""Seeded synthetic inputs for the MoE expert block.

This module builds workloads only: shapes, random draws and the per-expert
retention quota that a caller hands to the layer. It holds none of the layer's
arithmetic (routing, expert MLP, combine, backward). Both the CUDA path and the
fp64 oracle take their inputs from here, so the two see identical bytes.

Recipe (one ``torch.Generator('cpu')`` per call, seeded; draws in this order):

* ``x[T,H]``        ~ N(0, x_std^2)   (unit-RMS hidden states by default)
* ``w_router[H,E]`` ~ N(0, w_std^2)
* ``w_gate[E,H,F]``, ``w_up[E,H,F]``  ~ N(0, w_std^2)
* ``w_down[E,F,H]`` ~ N(0, w_std^2)
* shared expert ``ws_gate[H,Fs]``, ``ws_up[H,Fs]``, ``ws_down[Fs,H]`` (only when Fs > 0)
* a permutation of the E experts that assigns popularity ranks
* ``dy[T,H]``       ~ N(0, 1)

Every draw is taken in fp32 and, for bf16 workloads, rounded to nearest-even
bf16 once. Expert popularity is skewed with a constant router bias
``b_e = -s * ln(rank_e)`` (rank 1 = most popular), which makes the softmax
probability of expert e proportional to ``rank_e^-s`` times its data-dependent
part: a Zipf(s) popularity that is not correlated with the expert index. The
``zero_experts`` lowest-ranked experts get a bias of -1e4 so that they never
win a top-k slot (the "some experts get no tokens" case).

The workload shapes follow the two model families the LRMoE paper evaluates
(Qwen3-30B-A3B: H=2048, F=768, E=128, top-8; GLM-4.5-106B-A12B: H=4096,
F=1408, E=128 routed + 1 shared, top-8), with token counts that are multiples
of the S=128 sequence length used in the keep_graph pull request's profile.
Trained weights and the NSMC text data are not available; these draws stand
in for them.
"""
from __future__ import annotations

import dataclasses
import fractions

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE-layer problem: shapes, dtype, popularity skew and backward mode."""

    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    F_shared: int = 0
    dtype: str = "bf16"            # "bf16" or "f32" (I/O and stored activations)
    zipf_s: float | None = None    # None: no router bias (uniform popularity)
    zero_experts: int = 0          # experts biased out of every top-k
    frozen: bool = False           # experts and router frozen: dX-only backward
    quota_factor: float | None = None  # retention quota = ceil(factor * mean load)
    x_std: float = 1.0
    w_std: float = 0.02

    @property
    def P(self) -> int:
        return self.T * self.k

    def quota_per_expert(self) -> int | None:
        """ceil(quota_factor * T*k/E), in integer arithmetic, or None (retain all)."""
        if self.quota_factor is None:
            return None
        f = fractions.Fraction(str(self.quota_factor))
        num = f.numerator * self.T * self.k
        den = f.denominator * self.E
        return -(-num // den)


def _wl(name, **kw) -> Workload:
    return Workload(name=name, **kw)


QWEN = dict(H=2048, F=768, E=128, k=8)
GLM = dict(H=4096, F=1408, E=128, k=8, F_shared=1408)

WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        _wl("tiny_f32", T=64, H=64, F=128, E=8, k=2, dtype="f32"),
        _wl("qwen3_t128_frozen", T=128, zipf_s=1.0, frozen=True, **QWEN),
        _wl("qwen3_t4096_full", T=4096, zipf_s=1.0, **QWEN),
        _wl("qwen3_t4096_retained_s0.5", T=4096, zipf_s=0.5, quota_factor=0.5, **QWEN),
        _wl("qwen3_t4096_retained_s1.0", T=4096, zipf_s=1.0, quota_factor=0.5, **QWEN),
        _wl("qwen3_t4096_retained_s1.5", T=4096, zipf_s=1.5, quota_factor=0.5, **QWEN),
        _wl("glm45_t8192_full", T=8192, zipf_s=1.2, zero_experts=4, **GLM),
        _wl("glm45_t8192_retained", T=8192, zipf_s=1.2, zero_experts=4, quota_factor=0.5, **GLM),
    ]
}


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit fields (used for small test shapes)."""
    return Workload(name=name, **kw)


def _draw(g: torch.Generator, shape, std: float) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_inputs(w: Workload, seed: int = 0) -> dict[str, torch.Tensor | None]:
    """Draw every input of the workload on the CPU, in the documented order.

    Returns CPU tensors in the workload's I/O dtype (bf16 or fp32); the router
    bias and the quota are fp32 / int32 whatever the I/O dtype.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    io = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out: dict[str, torch.Tensor | None] = {}
    out["x"] = _draw(g, (w.T, w.H), w.x_std).to(io)
    out["w_router"] = _draw(g, (w.H, w.E), w.w_std).to(io)
    out["w_gate"] = _draw(g, (w.E, w.H, w.F), w.w_std).to(io)
    out["w_up"] = _draw(g, (w.E, w.H, w.F), w.w_std).to(io)
    out["w_down"] = _draw(g, (w.E, w.F, w.H), w.w_std).to(io)
    if w.F_shared > 0:
        out["ws_gate"] = _draw(g, (w.H, w.F_shared), w.w_std).to(io)
        out["ws_up"] = _draw(g, (w.H, w.F_shared), w.w_std).to(io)
        out["ws_down"] = _draw(g, (w.F_shared, w.H), w.w_std).to(io)
    else:
        out["ws_gate"] = out["ws_up"] = out["ws_down"] = None
    perm = torch.randperm(w.E, generator=g)
    if w.zipf_s is not None:
        rank = (perm + 1).to(torch.float64)
        bias = -w.zipf_s * torch.log(rank)
        if w.zero_experts > 0:
            bias[rank > w.E - w.zero_experts] = -1.0e4
        out["router_bias"] = bias.to(torch.float32)
    else:
        out["router_bias"] = None
    out["dy"] = _draw(g, (w.T, w.H), 1.0).to(io)
    q = w.quota_per_expert()
    out["quota"] = None if q is None else torch.full((w.E,), q, dtype=torch.int32)
    return out


def describe(w: Workload) -> dict:
    """JSON-friendly description of a workload (for bench output)."""
    d = dataclasses.asdict(w)
    d["quota"] = w.quota_per_expert()
    return d


def bf16_bits_to_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


__all__ = ["Workload", "WORKLOADS", "custom", "make_inputs", "describe", "bf16_bits_to_f64"]
