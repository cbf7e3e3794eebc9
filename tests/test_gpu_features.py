"""GPU tests of the bounded-wait machinery, the recompute mode and the device quota planner."""
import numpy as np
import pytest
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import custom, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from tests.parity import run_gpu

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


@pytest.mark.parametrize("rho", [(1, 2), (1, 4), (3, 2)])
def test_device_quota_planner(rho):
    w = custom("planner", T=500, H=128, F=128, E=32, k=4, zipf_s=1.2)
    inp = make_inputs(w, seed=8)
    layer = MoELayer(w, inp, record_routing=True)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    layer.forward(x)
    quota = torch.empty(w.E, dtype=torch.int32, device="cuda")
    _lib.moe_plan_quota(layer.dims, layer.ws, rho[0], rho[1], quota)
    count = np.diff(layer.offsets.cpu().numpy().astype(np.int64))
    cap = -(-rho[0] * w.T * w.k // (rho[1] * w.E))
    assert quota.cpu().numpy().tolist() == np.minimum(count, cap).tolist()
    budget = torch.tensor(np.arange(w.E) % 5 - 1, dtype=torch.int32, device="cuda")   # includes a negative
    _lib.moe_plan_quota(layer.dims, layer.ws, rho[0], rho[1], quota, budget=budget)
    expect = np.minimum(np.minimum(count, cap), np.maximum(budget.cpu().numpy(), 0))
    assert quota.cpu().numpy().tolist() == expect.tolist()
    layer.select(dy, quota)
    assert int(layer.ret_offsets[-1].item()) == int(expect.sum())
    layer.backward(dy, x, True)
    assert _lib.moe_read_status(layer.ws) == _lib.MOE_OK
