"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks the oracle against one of: hand-derived fixtures
(tests/golden), closed forms, brute force on tiny inputs, central finite
differences of L = <dY, Y>, an independent torch-autograd formulation, or an
invariant the mathematics fixes. A plausible slip anywhere in the oracle (a
dropped term, a wrong sign or index, a transposed operand, a wrong tie rule)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(rng, T, H, F, E, k, Fs=0, bias=True, x_std=1.0, w_std=0.3):
    inp = dict(
        x=rng.normal(0, x_std, (T, H)),
        w_router=rng.normal(0, w_std, (H, E)),
        router_bias=rng.normal(0, 0.5, E) if bias else None,
        w_gate=rng.normal(0, w_std, (E, H, F)),
        w_up=rng.normal(0, w_std, (E, H, F)),
        w_down=rng.normal(0, w_std, (E, F, H)),
        ws_gate=None, ws_up=None, ws_down=None,
    )
    if Fs:
        inp["ws_gate"] = rng.normal(0, w_std, (H, Fs))
        inp["ws_up"] = rng.normal(0, w_std, (H, Fs))
        inp["ws_down"] = rng.normal(0, w_std, (Fs, H))
    return inp


# ---------------------------------------------------------------- routing

def test_routing_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "routing_ties.json")))
    for c in g["cases"]:
        l = np.array([c["log2_logits"]], dtype=np.float64) * math.log(2.0)
        idx, w, _ = O.route_topk(l, c["k"])
        assert idx[0].tolist() == c["idx"], c
        np.testing.assert_allclose(w[0], c["w"], rtol=1e-15, atol=0)


def test_topk_brute_force_subsets():
    rng = np.random.default_rng(1)
    for E in range(1, 7):
        for k in range(1, E + 1):
            # integer logits force many ties; float logits none
            for l in (rng.integers(-2, 3, (12, E)).astype(np.float64), rng.normal(size=(12, E))):
                idx, _, _ = O.route_topk(l, k)
                for t in range(l.shape[0]):
                    best = max(itertools.combinations(range(E), k),
                               key=lambda S: (sum(l[t, list(S)]), tuple(-e for e in S)))
                    assert sorted(idx[t].tolist()) == list(best)
                    # slot order: logit descending, lower index first on ties
                    for j in range(k - 1):
                        a, b = idx[t, j], idx[t, j + 1]
                        assert l[t, a] > l[t, b] or (l[t, a] == l[t, b] and a < b)
                    assert len(set(idx[t].tolist())) == k


def test_weights_are_softmax_of_selected_logits():
    rng = np.random.default_rng(2)
    l = rng.normal(0, 3, (40, 9))
    for k in (1, 3, 9):
        idx, w, p = O.route_topk(l, k)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        sel = np.take_along_axis(l, idx, axis=1)
        direct = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)   # shift invariance
        np.testing.assert_allclose(w, direct, rtol=1e-13)
        if k == l.shape[1]:          # renormalisation over all experts is the identity
            np.testing.assert_allclose(np.take_along_axis(p, idx, axis=1), w, rtol=1e-14)
        if k == 1:
            assert np.all(w == 1.0)


# ---------------------------------------------------------------- permute

def test_permute_golden():
    g = json.load(open(os.path.join(GOLDEN, "permute_small.json")))
    count, offset, rop, por = O.permute(np.array(g["idx"]), g["E"])
    assert count.tolist() == g["count"]
    assert offset.tolist() == g["offset"]
    assert rop.tolist() == g["row_of_pair"]
    assert por.tolist() == g["pair_of_row"]


@pytest.mark.parametrize("case", ["random", "one_expert", "zero_load", "E1"])
def test_permute_invariants(case):
    rng = np.random.default_rng(3)
    T, k, E = 37, 3, 7
    if case == "E1":
        E, k = 1, 1
        idx = np.zeros((T, 1), np.int64)
    elif case == "one_expert":
        idx = np.stack([np.array([4, 0, 6])] * T)      # every token picks the same experts
    elif case == "zero_load":
        idx = np.stack([rng.choice([1, 3, 5], k, replace=False) for _ in range(T)])
    else:
        idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    count, offset, rop, por = O.permute(idx, E)
    assert count.sum() == T * k
    assert np.all(np.diff(offset) >= 0) and offset[0] == 0 and offset[-1] == T * k
    assert np.array_equal(por[rop], np.arange(T * k))
    assert np.array_equal(rop[por], np.arange(T * k))
    for e in range(E):
        rows = np.arange(offset[e], offset[e + 1])
        assert np.all(idx.reshape(-1)[por[rows]] == e)            # expert-contiguous
        assert np.all(np.diff(por[rows] // k) > 0)                 # token order inside expert
    x = rng.normal(size=(T, 5))
    xperm = x[por // k]                                            # gather
    back = np.zeros((T, 5))
    for p in range(T * k):                                         # scatter-add
        back[p // k] += xperm[rop[p]]
    np.testing.assert_allclose(back, k * x, rtol=1e-15)


# ---------------------------------------------------------------- forward

def test_scalar_swiglu_closed_form():
    """T=H=F=E=k=1: every quantity is a closed form in e^-1."""
    inp = dict(x=np.array([[2.0]]), w_router=np.array([[0.7]]), router_bias=None,
               w_gate=np.array([[[0.5]]]), w_up=np.array([[[3.0]]]), w_down=np.array([[[-1.0]]]),
               ws_gate=None, ws_up=None, ws_down=None)
    f = O.forward(inp, 1)
    s1 = 1.0 / (1.0 + math.exp(-1.0))        # sigmoid(a) with a = 2*0.5 = 1
    h = 1.0 * s1 * 6.0                        # silu(1) * b, b = 2*3 = 6
    assert f["a"][0, 0] == 1.0 and f["b"][0, 0] == 6.0
    assert math.isclose(f["Y"][0, 0], -h, rel_tol=1e-15)
    dy = np.array([[1.0]])
    b = O.backward(inp, f, dy)
    dh = -1.0
    da = dh * 6.0 * s1 * (1.0 + 1.0 * (1.0 - s1))
    db = dh * s1
    assert math.isclose(b["dX"][0, 0], 0.5 * da + 3.0 * db, rel_tol=1e-14)
    assert math.isclose(b["dw_gate"][0, 0, 0], 2.0 * da, rel_tol=1e-14)
    assert math.isclose(b["dw_up"][0, 0, 0], 2.0 * db, rel_tol=1e-14)
    assert math.isclose(b["dw_down"][0, 0, 0], h, rel_tol=1e-14)
    assert b["dw_router"][0, 0] == 0.0


def _torch_dense_swiglu(x, wg, wu, wd):
    """Textbook SwiGLU MLP via torch.nn.functional (Linear uses y = x A^T)."""
    a = torch.nn.functional.linear(x, wg.t())
    b = torch.nn.functional.linear(x, wu.t())
    return torch.nn.functional.linear(torch.nn.functional.silu(a) * b, wd.t())


def test_single_expert_is_dense_swiglu_with_autograd():
    rng = np.random.default_rng(4)
    T, H, F = 9, 6, 10
    inp = _rand_layer(rng, T, H, F, 1, 1, bias=False)
    dy = rng.normal(size=(T, H))
    f = O.forward(inp, 1)
    b = O.backward(inp, f, dy)
    tx = torch.tensor(inp["x"], requires_grad=True)
    tg = torch.tensor(inp["w_gate"][0], requires_grad=True)
    tu = torch.tensor(inp["w_up"][0], requires_grad=True)
    td = torch.tensor(inp["w_down"][0], requires_grad=True)
    Y = _torch_dense_swiglu(tx, tg, tu, td)
    np.testing.assert_allclose(f["Y"], Y.detach().numpy(), rtol=1e-13, atol=1e-15)
    (Y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(b["dX"], tx.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["dw_gate"][0], tg.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["dw_up"][0], tu.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["dw_down"][0], td.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.all(b["dw_router"] == 0.0) and np.all(b["dX_router"] == 0.0)


def test_dense_softmax_moe_when_k_equals_E():
    """k = E: every expert is used with weight softmax(l); Y = sum_e p_e MLP_e(x)."""
    rng = np.random.default_rng(5)
    T, H, F, E = 7, 5, 6, 4
    inp = _rand_layer(rng, T, H, F, E, E)
    f = O.forward(inp, E)
    tx = torch.tensor(inp["x"])
    logits = tx @ torch.tensor(inp["w_router"]) + torch.tensor(inp["router_bias"])
    p = torch.softmax(logits, dim=1)
    ref = sum(p[:, e:e + 1] * _torch_dense_swiglu(tx, torch.tensor(inp["w_gate"][e]),
                                                  torch.tensor(inp["w_up"][e]), torch.tensor(inp["w_down"][e]))
              for e in range(E))
    np.testing.assert_allclose(f["Y"], ref.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- backward

def _loss(inp, k, dy, fixed_idx=None):
    f = O.forward(inp, k)
    if fixed_idx is not None:
        assert np.array_equal(f["idx"], fixed_idx), "top-k set moved under the finite-difference step"
    return float((f["Y"] * dy).sum())


@pytest.mark.parametrize("Fs", [0, 5])
def test_finite_differences_all_parameters(Fs):
    rng = np.random.default_rng(6 + Fs)
    T, H, F, E, k = 4, 8, 16, 4, 2
    inp = _rand_layer(rng, T, H, F, E, k, Fs=Fs)
    dy = rng.normal(size=(T, H))
    f = O.forward(inp, k)
    b = O.backward(inp, f, dy)
    names = {"x": "dX", "w_router": "dw_router", "w_gate": "dw_gate", "w_up": "dw_up", "w_down": "dw_down"}
    if Fs:
        names.update(ws_gate="dws_gate", ws_up="dws_up", ws_down="dws_down")
    step = 1e-6
    for pname, gname in names.items():
        base = inp[pname]
        num = np.zeros_like(base)
        for i in np.ndindex(base.shape):
            old = base[i]
            base[i] = old + step
            lp = _loss(inp, k, dy, f["idx"])
            base[i] = old - step
            lm = _loss(inp, k, dy, f["idx"])
            base[i] = old
            num[i] = (lp - lm) / (2 * step)
        an = b[gname]
        err = np.linalg.norm(an - num) / np.linalg.norm(num)
        assert err <= 1e-6, (pname, err)


def test_torch_autograd_restatement_tiny_config():
    """Independent forward in torch with an explicit loop over (token, slot) pairs."""
    from expert_grouped_gemm_gb300.inputs import WORKLOADS, make_inputs, bf16_bits_to_f64
    w = WORKLOADS["tiny_f32"]
    raw = make_inputs(w, seed=0)
    inp = {k_: (None if v is None else bf16_bits_to_f64(v)) for k_, v in raw.items()}
    f = O.forward(inp, w.k)
    b = O.backward(inp, f, inp["dy"])
    T = w.T
    tx = torch.tensor(inp["x"], requires_grad=True)
    tr = torch.tensor(inp["w_router"], requires_grad=True)
    tg = torch.tensor(inp["w_gate"], requires_grad=True)
    tu = torch.tensor(inp["w_up"], requires_grad=True)
    td = torch.tensor(inp["w_down"], requires_grad=True)
    logits = tx @ tr
    idx = torch.tensor(f["idx"])
    rows = []
    for t in range(T):
        sel = logits[t, idx[t]]
        wt = torch.softmax(sel, dim=0)
        acc = torch.zeros(w.H, dtype=torch.float64)
        for j in range(w.k):
            e = int(idx[t, j])
            acc = acc + wt[j] * _torch_dense_swiglu(tx[t:t + 1], tg[e], tu[e], td[e])[0]
        rows.append(acc)
    Y = torch.stack(rows)
    np.testing.assert_allclose(f["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-15)
    (Y * torch.tensor(inp["dy"])).sum().backward()
    for mine, theirs in [(b["dX"], tx.grad), (b["dw_router"], tr.grad), (b["dw_gate"], tg.grad),
                         (b["dw_up"], tu.grad), (b["dw_down"], td.grad)]:
        np.testing.assert_allclose(mine, theirs.numpy(), rtol=1e-10, atol=1e-14)


def test_router_gradient_invariants():
    rng = np.random.default_rng(8)
    T, H, F, E, k = 11, 6, 8, 5, 3
    inp = _rand_layer(rng, T, H, F, E, k)
    dy = rng.normal(size=(T, H))
    f = O.forward(inp, k)
    b = O.backward(inp, f, dy)
    dl = b["dl"]
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-15)          # sum_e dl[t,e] = 0
    np.testing.assert_allclose(b["dw_router"].sum(axis=1), 0.0, atol=1e-14)
    mask = np.zeros((T, E), bool)
    for j in range(k):
        mask[np.arange(T), f["idx"][:, j]] = True
    assert np.all(dl[~mask] == 0.0)


def test_k1_router_gradient_is_exactly_zero():
    rng = np.random.default_rng(9)
    inp = _rand_layer(rng, 13, 6, 8, 5, 1)
    f = O.forward(inp, 1)
    b = O.backward(inp, f, rng.normal(size=(13, 6)))
    assert np.all(b["dw_router"] == 0.0) and np.all(b["dX_router"] == 0.0)


# ---------------------------------------------------------------- retention

def test_selection_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "retention_ties.json")))
    for c in g["cases"]:
        ro, rr = O.select_retained(np.array(g["score"]), np.array(g["offset"]),
                                   np.array(g["pair_of_row"]), g["k"], c["quota"])
        assert ro.tolist() == c["ret_offset"] and rr.tolist() == c["ret_rows"], c


def test_selection_dominance_and_sizes():
    rng = np.random.default_rng(10)
    T, k, E = 60, 2, 5
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    count, offset, rop, por = O.permute(idx, E)
    score = rng.integers(0, 4, T * k).astype(np.float64)     # many ties
    quota = rng.integers(0, 30, E)
    ro, rr = O.select_retained(score, offset, por, k, quota)
    for e in range(E):
        kept = set(rr[ro[e]:ro[e + 1]].tolist())
        assert len(kept) == min(quota[e], count[e])
        assert list(rr[ro[e]:ro[e + 1]]) == sorted(kept)
        rows = range(offset[e], offset[e + 1])
        for r in kept:
            for r2 in set(rows) - kept:          # every kept row outranks every dropped row
                assert (score[r] > score[r2]) or (score[r] == score[r2] and por[r] // k < por[r2] // k)


def _retained_problem(seed, quota_val, Fs=0):
    rng = np.random.default_rng(seed)
    T, H, F, E, k = 24, 6, 8, 4, 2
    inp = _rand_layer(rng, T, H, F, E, k, Fs=Fs)
    dy = rng.normal(size=(T, H))
    f = O.forward(inp, k)
    quota = None if quota_val is None else np.full(E, quota_val)
    return inp, dy, f, quota


def test_all_retained_equals_full_bitwise():
    inp, dy, f, _ = _retained_problem(11, None, Fs=3)
    full = O.backward(inp, f, dy)
    big = O.backward(inp, f, dy, quota=np.full(4, 10**6))
    exact = O.backward(inp, f, dy, quota=f["count"])
    for key in full:
        if isinstance(full[key], np.ndarray):
            assert np.array_equal(full[key], big[key]), key
            assert np.array_equal(full[key], exact[key]), key


def test_quota_zero_leaves_router_and_shared_only():
    inp, dy, f, _ = _retained_problem(12, None, Fs=3)
    b0 = O.backward(inp, f, dy, quota=np.zeros(4, np.int64))
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert np.all(b0[key] == 0.0)
    full = O.backward(inp, f, dy)
    # router and shared parts do not depend on retention
    np.testing.assert_array_equal(b0["dw_router"], full["dw_router"])
    np.testing.assert_array_equal(b0["dws_gate"], full["dws_gate"])
    x = inp["x"]
    sa, sb, _, _ = f["shared"]
    s = O.sigmoid(sa)
    dhs = dy @ inp["ws_down"].T
    dxs = (dhs * sb * s * (1 + sa * (1 - s))) @ inp["ws_gate"].T + (dhs * sa * s) @ inp["ws_up"].T
    np.testing.assert_allclose(b0["dX"], b0["dX_router"] + dxs, rtol=1e-12, atol=1e-14)
    assert x.shape == b0["dX"].shape


def test_retained_backward_is_sum_of_single_pair_problems():
    """dW and expert dX under a quota equal the sum over retained pairs of the
    full backward of a one-token, one-expert layer fed dY' = w_r * dY_t."""
    inp, dy, f, quota = _retained_problem(13, 3)
    k, E = 2, 4
    b = O.backward(inp, f, dy, quota=quota)
    H, F = inp["x"].shape[1], inp["w_gate"].shape[2]
    acc = {n: np.zeros_like(b[n]) for n in ("dw_gate", "dw_up", "dw_down")}
    dx_exp = np.zeros_like(b["dX"])
    wflat = f["w"].reshape(-1)
    for e in range(E):
        for r in b["ret_rows"][b["ret_offset"][e]:b["ret_offset"][e + 1]]:
            p = f["pair_of_row"][r]
            t = p // k
            one = dict(x=inp["x"][t:t + 1], w_router=np.zeros((H, 1)), router_bias=None,
                       w_gate=inp["w_gate"][e:e + 1], w_up=inp["w_up"][e:e + 1], w_down=inp["w_down"][e:e + 1],
                       ws_gate=None, ws_up=None, ws_down=None)
            fo = O.forward(one, 1)
            bo = O.backward(one, fo, wflat[p] * dy[t:t + 1])
            acc["dw_gate"][e] += bo["dw_gate"][0]
            acc["dw_up"][e] += bo["dw_up"][0]
            acc["dw_down"][e] += bo["dw_down"][0]
            dx_exp[t] += bo["dX"][0]
    for n in acc:
        np.testing.assert_allclose(b[n], acc[n], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["dX"] - b["dX_router"], dx_exp, rtol=1e-11, atol=1e-13)
    assert len(b["ret_rows"]) == sum(min(3, c) for c in f["count"])


def test_linearity_in_dy_keeps_retained_set():
    inp, dy, f, quota = _retained_problem(14, 2, Fs=2)
    b1 = O.backward(inp, f, dy, quota=quota)
    b2 = O.backward(inp, f, 2.5 * dy, quota=quota)
    assert np.array_equal(b1["ret_rows"], b2["ret_rows"])
    for key in ("dX", "dw_gate", "dw_up", "dw_down", "dw_router", "dws_gate", "dws_up", "dws_down"):
        np.testing.assert_allclose(b2[key], 2.5 * b1[key], rtol=1e-12, atol=1e-14)


def test_replay_mode_reproduces_own_decisions():
    inp, dy, f, quota = _retained_problem(15, 2)
    f2 = O.forward(inp, 2, logits_override=f["logits"].astype(np.float32))
    # fp32-rounded logits keep the same decisions on this seed
    assert np.array_equal(f2["idx"], f["idx"])
    b1 = O.backward(inp, f, dy, quota=quota)
    b2 = O.backward(inp, f2, dy, quota=quota, score_override=b1["score"].astype(np.float32))
    assert np.array_equal(b1["ret_rows"], b2["ret_rows"])


def test_pair_scores_closed_form():
    """Hand values: ||(3,4)|| = 5, ||(0,2)|| = 2, ||(1,0)|| = 1, ||(6,8)|| = 10."""
    dy = np.array([[3.0, 4.0], [0.0, 2.0]])
    x = np.array([[1.0, 0.0], [6.0, 8.0]])
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    row_of_pair = np.array([2, 0, 3, 1])          # pairs (t,j) -> rows
    y_pair = np.array([[1.0, 1.0], [2.0, -1.0], [0.5, 0.0], [0.0, 3.0]])
    g, score = O.pair_scores(dy, x, w, y_pair, row_of_pair)
    # row 2 <- (t0,j0): g = <(3,4),(0.5,0)> = 1.5; score = .75*5*1
    # row 0 <- (t0,j1): g = 7;                      score = .25*5*1
    # row 3 <- (t1,j0): g = <(0,2),(0,3)> = 6;      score = .5*2*10
    # row 1 <- (t1,j1): g = -2;                     score = .5*2*10
    assert g.tolist() == [7.0, -2.0, 1.5, 6.0]
    assert score.tolist() == [1.25, 10.0, 3.75, 10.0]


# ---------------------------------------------------------------- quota planner

def test_plan_quota_golden():
    g = json.load(open(os.path.join(GOLDEN, "plan_quota.json")))
    for c in g["cases"]:
        q = O.plan_quota(np.array(c["count"]), c["rho"][0], c["rho"][1],
                         None if c["budget"] is None else np.array(c["budget"]))
        assert q.tolist() == c["quota"], c


def test_plan_quota_cap_is_the_least_integer_above_the_scaled_mean():
    """Brute force: the cap is the smallest integer c with c * E * den >= num * pairs
    (found by counting up, not by a ceiling formula); every quota is the minimum of
    the load, that cap and the clamped budget."""
    rng = np.random.default_rng(21)
    for _ in range(200):
        E = int(rng.integers(1, 12))
        count = rng.integers(0, 60, E)
        num, den = int(rng.integers(0, 9)), int(rng.integers(1, 9))
        budget = rng.integers(-3, 40, E) if rng.random() < 0.5 else None
        q = O.plan_quota(count, num, den, budget)
        pairs = int(count.sum())
        c = 0
        while c * E * den < num * pairs:
            c += 1
        for e in range(E):
            want = min(int(count[e]), c)
            if budget is not None:
                want = min(want, max(int(budget[e]), 0))
            assert q[e] == want
        assert np.all(q >= 0) and np.all(q <= count)


def test_plan_quota_large_rho_keeps_every_pair():
    count = np.array([5, 0, 17, 3])
    q = O.plan_quota(count, 1 << 20, 1)
    assert q.tolist() == count.tolist()


# ---------------------------------------------------------------- shared expert

def test_torch_autograd_restatement_with_shared_expert():
    """The shared expert computed independently with torch.nn.functional and added
    after the routed sum: a gate/up swap, a missing silu or a wrong transpose in the
    oracle's shared path (forward or backward) fails here."""
    from expert_grouped_gemm_gb300.inputs import custom, make_inputs, bf16_bits_to_f64
    w = custom("tiny_shared_f32", T=24, H=16, F=24, E=6, k=2, F_shared=20, dtype="f32", zipf_s=0.7)
    raw = make_inputs(w, seed=3)
    inp = {k_: (None if v is None else bf16_bits_to_f64(v)) for k_, v in raw.items()}
    f = O.forward(inp, w.k)
    b = O.backward(inp, f, inp["dy"])
    tx = torch.tensor(inp["x"], requires_grad=True)
    tr = torch.tensor(inp["w_router"], requires_grad=True)
    tg = torch.tensor(inp["w_gate"], requires_grad=True)
    tu = torch.tensor(inp["w_up"], requires_grad=True)
    td = torch.tensor(inp["w_down"], requires_grad=True)
    sg = torch.tensor(inp["ws_gate"], requires_grad=True)
    su = torch.tensor(inp["ws_up"], requires_grad=True)
    sd = torch.tensor(inp["ws_down"], requires_grad=True)
    logits = tx @ tr + torch.tensor(inp["router_bias"])
    idx = torch.tensor(f["idx"])
    rows = []
    for t in range(w.T):
        wt = torch.softmax(logits[t, idx[t]], dim=0)
        acc = torch.zeros(w.H, dtype=torch.float64)
        for j in range(w.k):
            e = int(idx[t, j])
            acc = acc + wt[j] * _torch_dense_swiglu(tx[t:t + 1], tg[e], tu[e], td[e])[0]
        rows.append(acc)
    Y = torch.stack(rows) + _torch_dense_swiglu(tx, sg, su, sd)
    np.testing.assert_allclose(f["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-15)
    (Y * torch.tensor(inp["dy"])).sum().backward()
    for mine, theirs in [(b["dX"], tx.grad), (b["dw_router"], tr.grad), (b["dw_gate"], tg.grad),
                         (b["dw_up"], tu.grad), (b["dw_down"], td.grad), (b["dws_gate"], sg.grad),
                         (b["dws_up"], su.grad), (b["dws_down"], sd.grad)]:
        np.testing.assert_allclose(mine, theirs.numpy(), rtol=1e-10, atol=1e-14)
