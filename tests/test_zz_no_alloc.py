"""moe_route_noalloc: the routing stage for callers that cannot allocate.

Some callers cannot call cudaMalloc or lend the library a workspace (a
runtime with a memory pool fixed up front, a plugin that must not touch its
host's allocator, a process held to a pre-sized memory budget). This entry
point gives them the routing that moe_fwd computes -- top-k experts and
weights, per-expert offsets, expert-contiguous rows -- using only a fixed
device array inside the library. The test calls it through the C ABI twice in
a row, with the output buffers overwritten before each call, and checks every
output against moe_fwd's on the same inputs: integers exactly, weights within
the fp32 tolerance of the other parity tests (they come out identical).

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import WORKLOADS, custom, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from tests.parity import TOL, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


CASES = [
    WORKLOADS["qwen3_t4096_full"],
    custom("ragged", T=77, H=192, F=320, E=32, k=3, zipf_s=1.5, zero_experts=3),
    WORKLOADS["tiny_f32"],
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_routing_matches_moe_fwd_twice(w):
    inp = make_inputs(w, seed=0)
    layer = MoELayer(w, inp, record_routing=True)
    x = inp["x"].cuda()
    layer.forward(x)
    torch.cuda.synchronize()
    ref = dict(idx=layer.topk_idx.clone(), w=layer.topk_w.clone(), off=layer.offsets.clone(),
               rop=layer.row_of_pair.clone())
    T, E, k = w.T, w.E, w.k
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rop = torch.empty(T * k, dtype=torch.int32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        for t in (idx, off, rop, status):
            t.fill_(-7)
        wt.fill_(float("nan"))
        _lib.moe_route_noalloc(layer.dims, x, layer.p["w_router"], layer.p["router_bias"], idx, wt, off, rop,
                               device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == _lib.MOE_OK, call
        assert torch.equal(idx, ref["idx"]), call
        assert torch.equal(off, ref["off"]), call
        assert torch.equal(rop, ref["rop"]), call
        err = rel_fro(wt.cpu().numpy(), ref["w"].cpu().numpy())
        assert err <= TOL["f32"], (call, err)
        assert np.isfinite(wt.cpu().numpy()).all()


def test_noalloc_rejects_dims_past_its_fixed_scratch():
    w = custom("big", T=65536, H=256, F=256, E=128, k=8)
    d = _lib.make_dims(w.T, w.H, w.F, w.E, w.k)
    dev = "cuda"
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device=dev)        # never read: rejected on the host
    wr = torch.zeros(256, 128, dtype=torch.bfloat16, device=dev)
    i32 = torch.zeros(8, dtype=torch.int32, device=dev)
    f32 = torch.zeros(8, dtype=torch.float32, device=dev)
    with pytest.raises(_lib.MoeError) as ei:
        _lib.moe_route_noalloc(d, x, wr, None, i32, f32, i32, i32)
    assert ei.value.code == _lib.MOE_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
