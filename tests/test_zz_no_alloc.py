"""moe_route_noalloc: the routing stage for callers that cannot allocate.

Some callers cannot call cudaMalloc or lend the library a workspace (a
runtime with a memory pool fixed up front, a plugin that must not touch its
host's allocator, a process held to a pre-sized memory budget). This entry
point gives them the routing that moe_fwd computes -- top-k experts and
weights, per-expert offsets, expert-contiguous rows -- using only a fixed
device array inside the library.

The tests call it through the C ABI, two calls in a row with the output
buffers overwritten before each call, and check every output
* against the fp64 oracle: each token's set of experts equal except at
  tokens whose k-th and (k+1)-th oracle logits are closer than the near-tie
  margin of the other parity tests, offsets and rows equal to the oracle's permutation of the
  returned indices, weights within the fp32 tolerance;
* against moe_fwd on the same inputs: integers exactly, weights within the
  same tolerance (both run the router GEMM with the same K split here, so
  they come out identical).
It also runs the largest documented size, a call that leaves the status word
in the scratch, and a small problem right after a large one (stale scratch
contents must never be read).

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import WORKLOADS, custom, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from oracle import moe_oracle as O
from tests.parity import TOL, near_tie_tokens, oracle_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


# routing depends on x, the router weights and bias only: the expert sizes of the
# largest case are kept small so that moe_fwd, which the test compares with, is cheap
CASES = [
    WORKLOADS["qwen3_t4096_full"],
    custom("glm_routing_t8192", T=8192, H=4096, F=64, E=128, k=8, zipf_s=1.2, zero_experts=4),
    custom("ragged", T=77, H=192, F=320, E=32, k=3, zipf_s=1.5, zero_experts=3),
    WORKLOADS["tiny_f32"],
]


def _moe_fwd_routing(w, inp):
    layer = MoELayer(w, inp, record_routing=True)
    x = inp["x"].cuda()
    layer.forward(x)
    torch.cuda.synchronize()
    return layer, x, dict(idx=layer.topk_idx.clone(), w=layer.topk_w.clone(), off=layer.offsets.clone(),
                          rop=layer.row_of_pair.clone())


def _noalloc(layer, x, w, status):
    T, E, k = w.T, w.E, w.k
    out = dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               off=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               rop=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    for n in ("idx", "off", "rop"):
        out[n].fill_(-7)
    out["w"].fill_(float("nan"))
    if status is not None:
        status.fill_(-7)
    _lib.moe_route_noalloc(layer.dims, x, layer.p["w_router"], layer.p["router_bias"], out["idx"], out["w"],
                           out["off"], out["rop"], device_status=status)
    torch.cuda.synchronize()
    return out


def _check_against_oracle(w, inp, got):
    i64 = oracle_inputs(inp)
    logits = O.router_logits(i64["x"], i64["w_router"], i64.get("router_bias"))
    idx_or, w_or, _ = O.route_topk(logits, w.k)
    idx = got["idx"].cpu().numpy().astype(np.int64)
    # sets per token (slot order of two selected experts may flip where their logits nearly tie)
    diff = np.any(np.sort(idx, axis=1) != np.sort(idx_or, axis=1), axis=1)
    tie = near_tie_tokens(logits, w.k)
    assert not np.any(diff & ~tie), f"{int(np.sum(diff & ~tie))} tokens route differently without a near tie"
    # offsets and rows are a function of the indices: the oracle's permutation of the returned ones
    _, off_or, rop_or, _ = O.permute(idx, w.E)
    assert np.array_equal(got["off"].cpu().numpy(), off_or)
    assert np.array_equal(got["rop"].cpu().numpy(), rop_or)
    # weights: softmax over all E logits renormalised over the returned experts, in fp64
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    psel = np.take_along_axis(p, idx, axis=1)
    err = rel_fro(got["w"].cpu().numpy(), psel / psel.sum(axis=1, keepdims=True))
    assert err <= TOL["f32"], err
    return int(np.sum(tie))


def _check_against_moe_fwd(got, ref):
    assert torch.equal(got["idx"], ref["idx"])
    assert torch.equal(got["off"], ref["off"])
    assert torch.equal(got["rop"], ref["rop"])
    err = rel_fro(got["w"].cpu().numpy(), ref["w"].cpu().numpy())
    assert err <= TOL["f32"], err
    assert np.isfinite(got["w"].cpu().numpy()).all()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_routing_matches_oracle_and_moe_fwd_twice(w):
    inp = make_inputs(w, seed=0)
    layer, x, ref = _moe_fwd_routing(w, inp)
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        got = _noalloc(layer, x, w, status)
        assert int(status.item()) == _lib.MOE_OK, call
        _check_against_moe_fwd(got, ref)
        ties = _check_against_oracle(w, inp, got)
        print(w.name, "call", call, "near-tie tokens", ties)


def test_noalloc_status_word_in_scratch_and_small_after_large():
    """A large problem, then a small one, then the large one again, none of them given a
    status word (the library keeps it in its scratch): each matches moe_fwd, so nothing
    the previous call left in the scratch is read."""
    big = WORKLOADS["qwen3_t4096_full"]
    small = custom("small_after_big", T=40, H=128, F=64, E=16, k=2, zipf_s=1.0)
    runs = []
    for w in (big, small):
        inp = make_inputs(w, seed=11)
        runs.append((w, inp, *_moe_fwd_routing(w, inp)))
    for w, inp, layer, x, ref in (runs[0], runs[1], runs[0]):
        got = _noalloc(layer, x, w, None)
        _check_against_moe_fwd(got, ref)
        _check_against_oracle(w, inp, got)


def test_noalloc_rejects_dims_past_its_fixed_scratch():
    w = custom("big", T=131072, H=256, F=256, E=128, k=8)
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
