"""GPU tests of the bounded-wait machinery, the recompute mode and the device quota planner."""
import numpy as np
import pytest
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import WORKLOADS, custom, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from tests.parity import check_parity, planned_parity_case, run_gpu, run_oracle_replay

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


def test_bounded_wait_times_out_and_context_stays_usable():
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    st.fill_(123)
    _lib.moe_selftest_wait(True, 20000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.MOE_OK
    st.fill_(123)
    _lib.moe_selftest_wait(False, 20000, st)          # nothing arrives: the 20 ms wait runs out
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.MOE_ERR_TIMEOUT
    # the context is still healthy: a full layer step right after is parity-clean
    w = custom("after_timeout", T=64, H=128, F=128, E=16, k=2)
    g, _ = run_gpu(w, make_inputs(w, seed=1))
    assert g["status"] == 0


@pytest.mark.parametrize("quota", [False, True])
def test_recompute_mode_is_bitwise_equal(quota):
    w = custom("recompute", T=320, H=256, F=192, E=16, k=4, F_shared=128, zipf_s=1.0,
               quota_factor=0.5 if quota else None)
    inp = make_inputs(w, seed=7)
    ref, _ = run_gpu(w, inp)
    rec_layer = MoELayer(w, inp, record_routing=True, recompute=True)
    rec, _ = run_gpu(w, inp, layer=rec_layer)
    for n in ("Y", "dX", "dw_router", "dw_gate", "dw_up", "dw_down", "dws_gate", "dws_up", "dws_down"):
        assert np.array_equal(ref[n], rec[n]), n


# [PR44] Compatibility and limits: keep_graph=False (nothing kept between the forward and
# the backward) must give the same gradients; here the recompute mode is compared with the
# fp64 oracle itself, not only with the saved mode.
@pytest.mark.parametrize("name,kw", [
    ("medium_bf16_retained", dict(T=300, H=256, F=192, E=16, k=4, zipf_s=1.0, F_shared=128, quota_factor=0.5)),
    ("medium_bf16_full", dict(T=300, H=256, F=192, E=16, k=4, zipf_s=1.0, F_shared=128)),
    ("qwen3_t4096_retained_s1.0", None),
])
def test_recompute_mode_matches_oracle(name, kw):
    w = WORKLOADS[name] if kw is None else custom(name, **kw)
    inp = make_inputs(w, seed=0)
    layer = MoELayer(w, inp, record_routing=True, recompute=True)
    g, _ = run_gpu(w, inp, layer=layer)
    fwd, bwd = run_oracle_replay(w, inp, g)
    rep = check_parity(w, g, fwd, bwd, inp)
    print(name, "recompute", rep)


# [LRMoE] Abstract: the forward plans retention quotas under resource constraints. The
# device-planned quota, the selection it drives and the retained backward are compared
# with the oracle, which plans its own quota from the same routing.
@pytest.mark.parametrize("rho,budget", [((1, 2), None), ((1, 4), None), ((3, 2), None), ((1, 1), "mixed")])
def test_device_quota_planner_matches_oracle(rho, budget):
    w = custom("planner", T=500, H=128, F=128, E=32, k=4, zipf_s=1.2)
    bud = (np.arange(w.E) % 5 - 1) * 9 if budget == "mixed" else None   # includes negatives and zeros
    rep, g, _ = planned_parity_case(w, rho, bud, seed=8)
    print(rho, budget, rep)


def test_device_quota_planner_full_size():
    rep, g, _ = planned_parity_case(WORKLOADS["qwen3_t4096_full"], (1, 2), seed=0)
    assert rep["quota_sum"] == rep["R"]
    print(rep)


# moe_bwd forks its router-gradient and dX-reduce kernels onto a stream of its own and
# joins them back with events: a whole step captured in a CUDA graph and replayed must
# give the eager step's results bit for bit.
@pytest.mark.parametrize("quota", [False, True])
def test_step_captured_in_a_cuda_graph_is_bitwise_equal(quota):
    w = custom("graph_step", T=320, H=256, F=192, E=16, k=4, F_shared=128, zipf_s=1.0,
               quota_factor=0.5 if quota else None)
    inp = make_inputs(w, seed=3)
    ref, _ = run_gpu(w, inp)
    dev = torch.device("cuda")
    layer = MoELayer(w, inp, dev, record_routing=True)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    q = inp["quota"].to(dev) if quota else None
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.step(x, dy, q)  # first calls outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        layer.step(x, dy, q)
    layer.y.zero_()
    layer.dx.zero_()
    for t in layer.grads.values():
        t.zero_()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert _lib.moe_read_status(layer.ws) == _lib.MOE_OK
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    assert np.array_equal(f(layer.y), ref["Y"])
    assert np.array_equal(f(layer.dx), ref["dX"])
    for n, t in layer.grads.items():
        assert np.array_equal(f(t), ref[n]), n
