"""GPU parity of the fused decode forward (moe_fwd_decode) against the fp64 oracle.

The issue #14 page (Evidence) measures inference with 1..8 routed experts per token;
at such token counts the layer is a weight stream, which the fused kernel reads once.
Comparison rules as in the other parity tests: the routing decisions must equal the
oracle's when it replays the kernel's own fp32 logits (bit-exact), and may differ from
the standalone fp64 oracle only at near ties; weights and Y are compared with the
oracle run on those decisions (relative Frobenius error).
"""
import numpy as np
import pytest
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import custom, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from oracle import moe_oracle as O
from tests.parity import TOL, near_tie_tokens, oracle_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


QWEN = dict(H=2048, F=768, E=128, zipf_s=1.0)


def run_decode(w, inp, layer=None):
    layer = layer or MoELayer(w, inp, record_routing=True)
    x = inp["x"].cuda()
    layer.forward_decode(x)
    status = _lib.moe_read_status(layer.ws)
    torch.cuda.synchronize()
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    return dict(status=status, Y=f(layer.y), idx=layer.topk_idx.cpu().numpy().astype(np.int64),
                w=layer.topk_w.cpu().numpy().astype(np.float64), logits=layer.logits.cpu().numpy()), layer


def check_decode(w, inp, g):
    assert g["status"] == 0, g["status"]
    i64 = oracle_inputs(inp)
    fwd = O.forward(i64, w.k, logits_override=g["logits"])
    assert np.array_equal(g["idx"], fwd["idx"]), "top-k differs from the oracle replaying the kernel's logits"
    l64 = fwd["logits"]
    idx64, _, _ = O.route_topk(l64, w.k)
    diff = np.any(np.sort(idx64, axis=1) != np.sort(g["idx"], axis=1), axis=1)
    tie = near_tie_tokens(l64, w.k)
    assert not np.any(diff & ~tie), f"{int(np.sum(diff & ~tie))} tokens route differently without a near tie"
    errs = {"logits": rel_fro(g["logits"], l64), "w": rel_fro(g["w"], fwd["w"]), "Y": rel_fro(g["Y"], fwd["Y"])}
    assert errs["logits"] <= TOL["f32"] and errs["w"] <= TOL["f32"], errs
    assert errs["Y"] <= TOL["bf16"], errs
    return errs


@pytest.mark.parametrize("T,k", [(1, 1), (1, 8), (4, 8), (8, 8), (16, 8), (16, 1)])
def test_decode_parity_qwen(T, k):
    w = custom(f"dec_t{T}_k{k}", T=T, k=k, **QWEN)
    inp = make_inputs(w, seed=7)
    g, layer = run_decode(w, inp)
    errs = check_decode(w, inp, g)
    # deterministic: a second call gives the same bits
    y1 = layer.y.clone()
    layer.forward_decode(inp["x"].cuda())
    torch.cuda.synchronize()
    assert torch.equal(layer.y, y1)
    print(w.name, errs)


def test_decode_parity_glm_shared_expert():
    w = custom("dec_glm_t4", T=4, H=4096, F=1408, E=128, k=8, F_shared=1408, zipf_s=1.2, zero_experts=4)
    inp = make_inputs(w, seed=3)
    g, _ = run_decode(w, inp)
    print(w.name, check_decode(w, inp, g))


def test_decode_parity_ragged_small():
    w = custom("dec_small", T=3, H=192, F=128, E=16, k=2, F_shared=64, zipf_s=1.5)
    inp = make_inputs(w, seed=11)
    g, _ = run_decode(w, inp)
    print(w.name, check_decode(w, inp, g))


def test_decode_matches_moe_fwd_and_keeps_no_backward_state():
    w = custom("dec_vs_fwd", T=8, k=8, **QWEN)
    inp = make_inputs(w, seed=5)
    layer = MoELayer(w, inp, record_routing=True)
    x = inp["x"].cuda()
    layer.forward(x)
    torch.cuda.synchronize()
    y_fwd, idx_fwd = layer.y.clone(), layer.topk_idx.clone()
    layer.forward_decode(x)
    torch.cuda.synchronize()
    same = (torch.sort(idx_fwd, dim=1).values == torch.sort(layer.topk_idx, dim=1).values).all(dim=1)
    keep = same.cpu().numpy()  # tokens whose expert sets agree (all of them unless a near tie)
    err = rel_fro(layer.y.float().cpu().numpy()[keep], y_fwd.float().cpu().numpy()[keep])
    assert err <= TOL["bf16"], err
    dy = inp["dy"].cuda()
    with pytest.raises(_lib.MoeError) as ei:
        layer.backward(dy, x, False)
    assert ei.value.code == _lib.MOE_ERR_STATE


def test_decode_rejects_unsupported_dims():
    w = custom("dec_big", T=17, H=128, F=128, E=16, k=2)
    inp = make_inputs(w, seed=1)
    layer = MoELayer(w, inp)
    with pytest.raises(_lib.MoeError) as ei:
        layer.forward_decode(inp["x"].cuda())
    assert ei.value.code == _lib.MOE_ERR_UNSUPPORTED


def test_decode_router_ties_go_to_the_lower_expert():
    """A zero router leaves logits = bias exactly; bias values repeat every 5 experts, so
    the top-8 is a tie among 26 experts at 0 and must take the lowest indices."""
    w = custom("dec_ties", T=4, k=8, **QWEN)
    inp = make_inputs(w, seed=9)
    inp["w_router"] = torch.zeros_like(inp["w_router"])
    inp["router_bias"] = -(torch.arange(w.E) % 5).to(torch.float32)
    g, _ = run_decode(w, inp)
    assert g["status"] == 0
    want = np.tile(np.arange(0, 40, 5), (w.T, 1))
    assert np.array_equal(g["idx"], want), g["idx"]
    assert np.all(g["w"] == np.float32(0.125))
    check_decode(w, inp, g)


@pytest.mark.parametrize("barrier", [1, 2, 3, 4])
def test_decode_wait_that_runs_out_reports_timeout(barrier):
    """A grid barrier that can never complete: the bounded wait runs out, the kernel reports
    MOE_ERR_TIMEOUT and returns, and the next call on the same workspace is correct."""
    w = custom("dec_stall", T=8, k=8, **QWEN)
    inp = make_inputs(w, seed=13)
    layer = MoELayer(w, inp, record_routing=True)
    p = layer.p
    x = inp["x"].cuda()
    _lib.moe_selftest_decode_wait(layer.dims, layer.ws, x, p["w_router"], p["router_bias"], p["w_gate"], p["w_up"],
                                  p["w_down"], p["ws_gate"], p["ws_up"], p["ws_down"], layer.y, barrier, 20000)
    assert _lib.moe_read_status(layer.ws) == _lib.MOE_ERR_TIMEOUT
    g, _ = run_decode(w, inp, layer)
    check_decode(w, inp, g)


def test_decode_selftest_rejects_bad_arguments():
    w = custom("dec_stall_args", T=2, k=2, **QWEN)
    inp = make_inputs(w, seed=1)
    layer = MoELayer(w, inp)
    p = layer.p
    for barrier, limit in ((0, 1000), (5, 1000), (1, 0), (1, 2000000)):
        with pytest.raises(_lib.MoeError) as ei:
            _lib.moe_selftest_decode_wait(layer.dims, layer.ws, inp["x"].cuda(), p["w_router"], p["router_bias"],
                                          p["w_gate"], p["w_up"], p["w_down"], p["ws_gate"], p["ws_up"],
                                          p["ws_down"], layer.y, barrier, limit)
        assert ei.value.code == _lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [
    dict(T=5, H=256, F=192, E=48, k=3),     # E not a multiple of 32: top-k lanes past E
    dict(T=16, H=512, F=256, E=64, k=16),   # T * k = 256 routed pairs, the most the kernel takes
    dict(T=2, H=1024, F=1024, E=256, k=8),  # E = 256; F in two column blocks of 512
    dict(T=3, H=320, F=1600, E=32, k=4, F_shared=832),  # F in three blocks, a shared expert in two
])
def test_decode_parity_edge_shapes(shape):
    w = custom("dec_edge_" + "_".join(f"{kk}{v}" for kk, v in shape.items()), zipf_s=0.8, **shape)
    inp = make_inputs(w, seed=17)
    g, _ = run_decode(w, inp)
    print(w.name, check_decode(w, inp, g))
