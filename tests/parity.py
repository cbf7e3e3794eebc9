"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same seeded inputs, compare.

Comparison rules:
* integers (routing indices, expert offsets, row_of_pair, kept offsets and
  rows) are compared bit-exactly against the oracle replaying the GPU's own
  fp32 logits / fp32 scores (both sides take each discrete decision on the
  same fp32 numbers); against the standalone fp64 oracle they may differ only
  at tokens whose k-th / (k+1)-th logit gap is below NEAR_TIE;
* floating point outputs: relative Frobenius error ||gpu - oracle|| / ||oracle||
  against the oracle run on the GPU's discrete decisions, at most TOL[dtype];
  a tensor whose oracle value is exactly zero must be exactly zero on the GPU.
"""
from __future__ import annotations

import numpy as np
import torch

from expert_grouped_gemm_gb300 import _lib
from expert_grouped_gemm_gb300.inputs import Workload, bf16_bits_to_f64, make_inputs
from expert_grouped_gemm_gb300.layer import MoELayer
from oracle import moe_oracle as O

TOL = {"bf16": 2e-2, "f32": 1e-5}
NEAR_TIE = 1e-4


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    nd = np.linalg.norm(a - b)
    if nb == 0.0:
        return 0.0 if nd == 0.0 else float("inf")
    return float(nd / nb)


def run_gpu(w: Workload, inp: dict, use_quota: bool = True, layer: MoELayer | None = None):
    """One fwd (+ select) + bwd through the C ABI; returns CPU numpy results."""
    dev = torch.device("cuda")
    if layer is None:
        layer = MoELayer(w, inp, dev, record_routing=True)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    q = inp["quota"].to(dev) if (use_quota and inp["quota"] is not None) else None
    layer.forward(x)
    if q is not None:
        layer.select(dy, q)
    dx, grads = layer.backward(dy, x, q is not None)
    status = _lib.moe_read_status(layer.ws)
    torch.cuda.synchronize()
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    out = dict(status=status, Y=f(layer.y), dX=f(dx), idx=layer.topk_idx.cpu().numpy().astype(np.int64),
               w=layer.topk_w.cpu().numpy().astype(np.float64), offsets=layer.offsets.cpu().numpy().astype(np.int64),
               row_of_pair=layer.row_of_pair.cpu().numpy().astype(np.int64), logits=layer.logits.cpu().numpy(),
               used_quota=q is not None)
    if q is not None:
        out["ret_offsets"] = layer.ret_offsets.cpu().numpy().astype(np.int64)
        R = int(out["ret_offsets"][-1])
        out["ret_rows"] = layer.ret_rows[:R].cpu().numpy().astype(np.int64)
        out["scores"] = layer.scores.cpu().numpy()
    for n, t in grads.items():
        out[n] = f(t)
    return out, layer


def oracle_inputs(inp: dict) -> dict:
    return {k: (None if v is None else bf16_bits_to_f64(v)) for k, v in inp.items() if k not in ("quota",)}


def run_oracle_replay(w: Workload, inp: dict, g: dict):
    """Oracle fwd/bwd taking the GPU's discrete decisions (fp32 logits and scores)."""
    i64 = oracle_inputs(inp)
    fwd = O.forward(i64, w.k, logits_override=g["logits"])
    quota = None
    score_rows = None
    if g["used_quota"]:
        quota = inp["quota"].numpy().astype(np.int64)
        score_rows = np.empty(w.P, dtype=np.float32)
        score_rows[fwd["row_of_pair"]] = g["scores"]
    bwd = O.backward(i64, fwd, i64["dy"], quota=quota, frozen=w.frozen, score_override=score_rows)
    return fwd, bwd


def near_tie_tokens(logits64: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest oracle logits are closer than NEAR_TIE."""
    if k >= logits64.shape[1]:
        return np.zeros(logits64.shape[0], bool)
    s = -np.sort(-logits64, axis=1)
    return (s[:, k - 1] - s[:, k]) < NEAR_TIE


def check_parity(w: Workload, g: dict, fwd: dict, bwd: dict, inp: dict, report: dict | None = None):
    tol = TOL[w.dtype]
    rep = {} if report is None else report
    assert g["status"] == 0, f"device status {g['status']}"
    # ---- discrete: bit-exact against the replaying oracle
    assert np.array_equal(g["idx"], fwd["idx"]), "top-k indices differ from the oracle replay"
    assert np.array_equal(g["offsets"], fwd["offset"]), "expert offsets differ"
    assert np.array_equal(g["row_of_pair"], fwd["row_of_pair"]), "row_of_pair differs"
    if g["used_quota"]:
        assert np.array_equal(g["ret_offsets"], bwd["ret_offset"]), "retained offsets differ"
        assert np.array_equal(g["ret_rows"], bwd["ret_rows"]), "retained rows differ"
        rep["R"] = int(g["ret_offsets"][-1])
    # ---- discrete: against the standalone fp64 oracle, except near ties
    l64 = fwd["logits"]
    idx64, _, _ = O.route_topk(l64, w.k)
    diff = np.any(np.sort(idx64, axis=1) != np.sort(g["idx"], axis=1), axis=1)
    tie = near_tie_tokens(l64, w.k)
    assert not np.any(diff & ~tie), f"{int(np.sum(diff & ~tie))} tokens route differently without a near tie"
    rep["near_tie_tokens"] = int(np.sum(tie))
    rep["routing_diff_tokens"] = int(np.sum(diff))
    # ---- float
    errs = {"logits": rel_fro(g["logits"], l64), "w": rel_fro(g["w"], fwd["w"]), "Y": rel_fro(g["Y"], fwd["Y"]),
            "dX": rel_fro(g["dX"], bwd["dX"])}
    if g["used_quota"]:
        sc = np.empty(w.P)
        sc[:] = bwd["score"][fwd["row_of_pair"]]
        errs["scores"] = rel_fro(g["scores"], sc)
    if not w.frozen:
        for n in ("dw_router", "dw_gate", "dw_up", "dw_down", "dws_gate", "dws_up", "dws_down"):
            if n in bwd:
                errs[n] = rel_fro(g[n], bwd[n])
        # experts with no kept pair must get exact zeros
        ro = bwd["ret_offset"]
        for e in range(w.E):
            if ro[e + 1] == ro[e]:
                for n in ("dw_gate", "dw_up", "dw_down"):
                    assert np.all(g[n][e] == 0.0), f"{n}[{e}] not zero for an expert with no kept pair"
    rep["errors"] = errs
    bad = {k_: v for k_, v in errs.items() if not (v <= tol)}
    assert not bad, f"relative Frobenius errors above {tol}: {bad}"
    return rep


def parity_case(w: Workload, seed: int = 0, inp: dict | None = None):
    inp = make_inputs(w, seed) if inp is None else inp
    g, layer = run_gpu(w, inp)
    fwd, bwd = run_oracle_replay(w, inp, g)
    rep = check_parity(w, g, fwd, bwd, inp)
    return rep, g, layer, inp


def run_gpu_planned(w: Workload, inp: dict, rho: tuple[int, int], budget=None, layer: MoELayer | None = None):
    """fwd, device-planned quota (moe_plan_quota), select with it, bwd; CPU numpy results
    plus the planned quota."""
    dev = torch.device("cuda")
    if layer is None:
        layer = MoELayer(w, inp, dev, record_routing=True)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    layer.forward(x)
    quota = torch.empty(w.E, dtype=torch.int32, device=dev)
    bud = None if budget is None else torch.as_tensor(budget, dtype=torch.int32).to(dev)
    _lib.moe_plan_quota(layer.dims, layer.ws, rho[0], rho[1], quota, budget=bud)
    layer.select(dy, quota)
    dx, grads = layer.backward(dy, x, True)
    status = _lib.moe_read_status(layer.ws)
    torch.cuda.synchronize()
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    out = dict(status=status, Y=f(layer.y), dX=f(dx), idx=layer.topk_idx.cpu().numpy().astype(np.int64),
               w=layer.topk_w.cpu().numpy().astype(np.float64), offsets=layer.offsets.cpu().numpy().astype(np.int64),
               row_of_pair=layer.row_of_pair.cpu().numpy().astype(np.int64), logits=layer.logits.cpu().numpy(),
               used_quota=True, quota=quota.cpu().numpy().astype(np.int64))
    out["ret_offsets"] = layer.ret_offsets.cpu().numpy().astype(np.int64)
    out["ret_rows"] = layer.ret_rows[:int(out["ret_offsets"][-1])].cpu().numpy().astype(np.int64)
    out["scores"] = layer.scores.cpu().numpy()
    for n, t in grads.items():
        out[n] = f(t)
    return out, layer


def planned_parity_case(w: Workload, rho: tuple[int, int], budget=None, seed: int = 0):
    """Parity of the device quota planner and the retained backward it drives: the
    oracle plans its own quota (oracle.plan_quota) from the replayed routing's counts,
    the planned quotas must be equal, then the select + backward are compared as in
    every other parity case."""
    inp = make_inputs(w, seed)
    g, layer = run_gpu_planned(w, inp, rho, budget)
    i64 = oracle_inputs(inp)
    fwd = O.forward(i64, w.k, logits_override=g["logits"])
    q_or = O.plan_quota(fwd["count"], rho[0], rho[1], None if budget is None else np.asarray(budget))
    assert np.array_equal(g["quota"], q_or), "planned quotas differ from the oracle's"
    score_rows = np.empty(w.P, dtype=np.float32)
    score_rows[fwd["row_of_pair"]] = g["scores"]
    bwd = O.backward(i64, fwd, i64["dy"], quota=q_or, frozen=w.frozen, score_override=score_rows)
    rep = check_parity(w, g, fwd, bwd, inp)
    rep["quota_sum"] = int(q_or.sum())
    return rep, g, layer
