"""The seeded input generator (the one module the oracle and the CUDA path share):
deterministic, in its stated draw order, with the stated distributions and quota."""
import math

import pytest
import torch

from expert_grouped_gemm_gb300.inputs import WORKLOADS, custom, make_inputs

SMALL = dict(T=48, H=64, F=32, E=8, k=2)


def test_same_seed_same_bits_other_seed_differs():
    w = custom("g", zipf_s=1.0, F_shared=16, quota_factor=0.5, **SMALL)
    a, b, c = make_inputs(w, 7), make_inputs(w, 7), make_inputs(w, 8)
    for n, t in a.items():
        if t is None:
            continue
        assert torch.equal(t, b[n]), n
    assert not torch.equal(a["x"], c["x"])


def test_draw_order_is_x_weights_shared_permutation_dy():
    """Adding a shared expert inserts its three draws after W_down and before the
    rank permutation and dY, and changes nothing drawn before them."""
    w0 = custom("g", zipf_s=1.0, **SMALL)
    w1 = custom("g", zipf_s=1.0, F_shared=16, **SMALL)
    a, b = make_inputs(w0, 3), make_inputs(w1, 3)
    for n in ("x", "w_router", "w_gate", "w_up", "w_down"):
        assert torch.equal(a[n], b[n]), n
    assert not torch.equal(a["dy"], b["dy"])
    # dY is drawn last: restating the documented order by hand gives the same tensor
    g = torch.Generator(device="cpu")
    g.manual_seed(3)
    for shape in ((48, 64), (64, 8), (8, 64, 32), (8, 64, 32), (8, 32, 64)):
        torch.randn(*shape, generator=g)
    torch.randperm(8, generator=g)
    assert torch.equal(a["dy"], torch.randn(48, 64, generator=g).to(torch.bfloat16))


def test_zipf_bias_and_zero_experts():
    w = custom("g", zipf_s=1.5, zero_experts=2, **SMALL)
    raw = make_inputs(w, 0)["router_bias"]
    assert raw.dtype == torch.float32
    b = raw.double()
    live = b[b > -1.0e3]
    assert (b <= -1.0e3).sum() == 2
    # the live biases are -s ln(rank) for ranks 1..E-2, each once
    ranks = sorted(round(math.exp(-v / 1.5)) for v in live.tolist())
    assert ranks == list(range(1, 7))


def test_quota_is_ceil_in_integer_arithmetic():
    for T, k, E, qf, want in ((4096, 8, 128, 0.5, 128), (300, 4, 16, 0.5, 38), (77, 3, 32, 0.5, 4), (10, 1, 3, 0.1, 1)):
        w = custom("q", T=T, H=64, F=32, E=E, k=k, quota_factor=qf)
        assert w.quota_per_expert() == want
        q = make_inputs(w, 0)["quota"]
        assert q.dtype == torch.int32 and torch.all(q == want)
    assert make_inputs(custom("q", **SMALL), 0)["quota"] is None


@pytest.mark.parametrize("name", ["tiny_f32", "qwen3_t128_frozen"])
def test_distributions_and_dtypes(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, 0)
    io = torch.float32 if w.dtype == "f32" else torch.bfloat16
    for n in ("x", "w_router", "w_gate", "w_up", "w_down", "dy"):
        assert inp[n].dtype == io, n
    assert abs(inp["x"].float().std().item() - w.x_std) < 0.05 * w.x_std
    assert abs(inp["w_gate"].float().std().item() - w.w_std) < 0.05 * w.w_std
    assert abs(inp["dy"].float().std().item() - 1.0) < 0.05
