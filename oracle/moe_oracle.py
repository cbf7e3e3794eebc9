"""fp64 CPU oracle of the MoE expert block, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg do. It
shares no code with the CUDA library.

It is the plain definition of what the layer computes, written out step by
step in float64 from the exact values of the (bf16 or fp32) inputs, with no
blocking, fusion or reordering beyond the definition. numpy's matmul is used
as a library step for the dense products.

Sources (three web pages on one subject):

* [I14]  issue "[MoE] Hot experts on RNGD during training (host dispatch,
         device expert graphs) #14", section Proposal: routing and token
         dispatch, rows gathered per expert, expert forward graphs, backward
         "dx; and dW for full FT", results scattered back; section Scope:
         experts frozen (LoRA) first, then full fine-tuning.
* [PR44] pull request "PR #44" (HostMLP(keep_graph=True)), section Changes:
         the forward keeps what the backward needs and the backward reuses it.
* [LRMoE] "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training
         on Memory-Constrained Nodes" (arXiv 2610.37720), Abstract: forward
         keeps every routed computation; backward scores each token-expert
         pair by its estimated contribution to the expert update, keeps pairs
         within per-expert quotas and physically compacts them into smaller
         variable-size grouped GEMMs.

Readings where the pages are silent (each is listed again in the design notes):

* Router: logits l = x W_r + b with an optional constant per-expert bias b
  (no gradient); p = softmax over all E logits; the k experts with the
  largest logit are selected, ties to the lower expert index, slot j in that
  order; weights w = p_sel / sum(p_sel) ("softmax then renormalise").
* Permute: rows grouped by expert, expert-contiguous, token order inside an
  expert (stable).
* Expert MLP: SwiGLU, h = silu(x W_gate[e]) * (x W_up[e]), y = h W_down[e].
* Combine: Y_t = sum_j w[t,j] y_{row(t,j)} in slot order, then the shared
  expert's output (if any) is added.
* Retention score (the pages do not define the metric): the proxy
  score = w * ||dY_t||_2 * ||x_t||_2 of each pair.
* Retention: per expert keep the first min(quota_e, count_e) rows ordered by
  (score descending, token ascending); kept rows listed in ascending row order.
  Retention removes dropped pairs from the expert backward only (dW_expert and
  the expert part of dX). The router backward always uses every pair, and the
  shared expert is never subject to retention.
* Frozen: no dW_expert, dW_router, shared dW; dX is still complete.
* dW is overwritten (experts with no retained row get exact zeros).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "router_logits",
    "route_topk",
    "permute",
    "expert_forward",
    "combine",
    "shared_forward",
    "forward",
    "pair_scores",
    "plan_quota",
    "select_retained",
    "backward",
    "sigmoid",
    "silu",
]


# --------------------------------------------------------------------------
# elementary functions
# --------------------------------------------------------------------------

def sigmoid(z):
    """Logistic function 1 / (1 + e^-z), evaluated without overflow."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(z):
    """silu(z) = z * sigmoid(z), the gate nonlinearity of a SwiGLU expert."""
    return np.asarray(z, dtype=np.float64) * sigmoid(z)


# --------------------------------------------------------------------------
# forward: route, dispatch, expert MLP, combine   ([I14] Proposal)
# --------------------------------------------------------------------------

def router_logits(x, w_router, router_bias=None):
    """Router logits l[t,e] = sum_h x[t,h] W_r[h,e] + b[e]  ([I14] Proposal: routing)."""
    l = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64)
    if router_bias is not None:
        l = l + np.asarray(router_bias, np.float64)[None, :]
    return l


def route_topk(logits, k):
    """Top-k routing with softmax-then-renormalise weights.

    Selection: for each token, experts sorted by (logit descending, expert
    index ascending); the first k are kept, in that order (slot j).
    Weights: p = softmax over all E logits (max-subtracted), then
    w[t,j] = p[t, idx[t,j]] / sum_j' p[t, idx[t,j']].
    Comparisons are exact in whatever precision ``logits`` carries, so the
    same function replays the GPU's decisions when fed its fp32 logits.
    Returns (idx[T,k] int64, w[T,k] float64, p[T,E] float64).
    """
    l = np.asarray(logits)
    T, E = l.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-l[t, e], e))
        idx[t] = order[:k]
    l64 = l.astype(np.float64)
    m = l64.max(axis=1, keepdims=True)
    ex = np.exp(l64 - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    psel = np.take_along_axis(p, idx, axis=1)
    w = psel / psel.sum(axis=1, keepdims=True)
    return idx, w, p


def permute(idx, E):
    """Expert-contiguous, token-stable placement of the T*k token-expert pairs.

    count[e] = number of pairs routed to e; offset = exclusive prefix sum;
    visiting tokens in ascending order and slots j in ascending order, pair
    (t, j) with expert e gets row offset[e] + (running count of e so far).
    ([I14] Proposal: rows gathered per expert; results scattered back.)
    Returns count[E], offset[E+1], row_of_pair[T*k], pair_of_row[T*k].
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    count = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            count[idx[t, j]] += 1
    offset = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offset[e + 1] = offset[e] + count[e]
    cursor = np.zeros(E, dtype=np.int64)
    row_of_pair = np.empty(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            row_of_pair[t * k + j] = offset[e] + cursor[e]
            cursor[e] += 1
    pair_of_row = np.empty(T * k, dtype=np.int64)
    pair_of_row[row_of_pair] = np.arange(T * k)
    return count, offset, row_of_pair, pair_of_row


def expert_forward(x, w_gate, w_up, w_down, offset, pair_of_row, k):
    """SwiGLU expert MLP on every permuted row ([I14] Proposal: expert forward graphs).

    For row r of expert e (token t = pair // k):
    a = x_t W_gate[e], b = x_t W_up[e], h = silu(a) * b, y_r = h W_down[e].
    Returns a, b, h [P,F] and y [P,H] in permuted-row order.
    """
    x = np.asarray(x, np.float64)
    E = len(offset) - 1
    P = len(pair_of_row)
    F = w_gate.shape[2]
    H = x.shape[1]
    a = np.zeros((P, F))
    b = np.zeros((P, F))
    h = np.zeros((P, F))
    y = np.zeros((P, H))
    for e in range(E):
        r0, r1 = offset[e], offset[e + 1]
        if r1 == r0:
            continue
        tok = pair_of_row[r0:r1] // k
        xe = x[tok]
        ae = xe @ np.asarray(w_gate[e], np.float64)
        be = xe @ np.asarray(w_up[e], np.float64)
        he = silu(ae) * be
        a[r0:r1], b[r0:r1], h[r0:r1] = ae, be, he
        y[r0:r1] = he @ np.asarray(w_down[e], np.float64)
    return a, b, h, y


def shared_forward(x, ws_gate, ws_up, ws_down):
    """Always-on shared SwiGLU expert on every token (weight 1)."""
    x = np.asarray(x, np.float64)
    a = x @ np.asarray(ws_gate, np.float64)
    b = x @ np.asarray(ws_up, np.float64)
    h = silu(a) * b
    return a, b, h, h @ np.asarray(ws_down, np.float64)


def combine(w, y_pair, row_of_pair, shared_y=None):
    """Weighted combine back to tokens ([I14] Proposal: results scattered back).

    Y_t = sum_{j=0}^{k-1} w[t,j] * y_{row(t,j)}, slots in ascending order,
    then + shared-expert output.
    """
    T, k = w.shape
    Y = np.zeros((T, y_pair.shape[1]))
    for j in range(k):
        Y += w[:, j:j + 1] * y_pair[row_of_pair.reshape(T, k)[:, j]]
    if shared_y is not None:
        Y = Y + shared_y
    return Y


def forward(inp, k, logits_override=None):
    """Whole forward; returns a dict holding every intermediate.

    ``inp`` maps names to float64 arrays (x, w_router, router_bias or None,
    w_gate, w_up, w_down, ws_gate/ws_up/ws_down or None).
    ``logits_override`` replays the discrete routing on given logits (e.g. a
    GPU's fp32 logits) instead of the oracle's own; the float arithmetic after
    routing is unchanged.
    """
    x = inp["x"]
    E = inp["w_router"].shape[1]
    logits = router_logits(x, inp["w_router"], inp.get("router_bias"))
    route_on = logits if logits_override is None else logits_override
    idx, _, _ = route_topk(route_on, k)
    # weights always from the oracle's own fp64 logits (softmax then renormalise)
    l64 = logits
    m = l64.max(axis=1, keepdims=True)
    p = np.exp(l64 - m)
    p = p / p.sum(axis=1, keepdims=True)
    psel = np.take_along_axis(p, idx, axis=1)
    w = psel / psel.sum(axis=1, keepdims=True)
    count, offset, row_of_pair, pair_of_row = permute(idx, E)
    a, b, h, y = expert_forward(x, inp["w_gate"], inp["w_up"], inp["w_down"], offset, pair_of_row, k)
    shared = None
    if inp.get("ws_gate") is not None:
        shared = shared_forward(x, inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    Y = combine(w, y, row_of_pair, None if shared is None else shared[3])
    return dict(logits=logits, idx=idx, w=w, p=p, count=count, offset=offset,
                row_of_pair=row_of_pair, pair_of_row=pair_of_row,
                a=a, b=b, h=h, y_pair=y, shared=shared, Y=Y, k=k, E=E)


# --------------------------------------------------------------------------
# backward: pair scores, retention, expert and router gradients
# --------------------------------------------------------------------------

def pair_scores(dy, x, w, y_pair, row_of_pair):
    """Per pair (in permuted-row order): router-gradient dot and retention score.

    g_r = <dY_t, y_r>  (gradient of L=<dY,Y> w.r.t. the routing weight w_r);
    score_r = w_r * ||dY_t||_2 * ||x_t||_2  ([LRMoE] Abstract: a per-pair
    estimate of the contribution to the expert update; the proxy reading).
    Returns g[P], score[P] indexed by row.
    """
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    T, k = w.shape
    P = T * k
    g = np.zeros(P)
    score = np.zeros(P)
    dyn = np.sqrt((dy * dy).sum(axis=1))
    xn = np.sqrt((x * x).sum(axis=1))
    for t in range(T):
        for j in range(k):
            r = row_of_pair[t * k + j]
            g[r] = float(dy[t] @ y_pair[r])
            score[r] = w[t, j] * dyn[t] * xn[t]
    return g, score


def plan_quota(count, rho_num, rho_den, budget=None):
    """Per-expert retention quotas planned from the forward's routing.

    ([LRMoE] Abstract: the forward plans retention quotas under resource
    constraints.) The pages give no formula; the reading used is a fraction
    rho = rho_num / rho_den of the mean load, rounded up, capped at the
    expert's own load and, when a per-expert budget is given, at that budget
    (a negative budget counts as zero):

        mean = (sum_e count_e) / E
        quota_e = min(count_e, ceil(rho * mean) [, max(budget_e, 0)])

    Computed in exact rational arithmetic (Python integers), so the rounding
    of the ceiling is the mathematical one.
    """
    from fractions import Fraction

    count = [int(c) for c in count]
    E = len(count)
    pairs = sum(count)
    cap = Fraction(int(rho_num), int(rho_den)) * Fraction(pairs, E)
    cap_int = -((-cap.numerator) // cap.denominator)          # ceil of a non-negative rational
    out = []
    for e in range(E):
        q = min(count[e], cap_int)
        if budget is not None:
            q = min(q, max(int(budget[e]), 0))
        out.append(q)
    return np.asarray(out, dtype=np.int64)


def select_retained(score, offset, pair_of_row, k, quota=None):
    """Per-expert quota selection ([LRMoE] Abstract: select pairs within quotas).

    For expert e with count_e rows, q_e = min(quota[e], count_e) (count_e when
    no quota). Its rows are ranked by (score descending, token ascending) and
    the first q_e are kept; kept rows are listed in ascending row order.
    Comparisons are exact in the precision ``score`` carries, so the same
    function replays a GPU's decisions on its fp32 scores.
    Returns ret_offset[E+1], ret_rows[R] (row indices into permuted order).
    """
    score = np.asarray(score)
    E = len(offset) - 1
    ret_offset = np.zeros(E + 1, dtype=np.int64)
    kept = []
    for e in range(E):
        r0, r1 = int(offset[e]), int(offset[e + 1])
        cnt = r1 - r0
        q = cnt if quota is None else max(0, min(int(quota[e]), cnt))
        rows = list(range(r0, r1))
        rows.sort(key=lambda r: (-score[r], pair_of_row[r] // k))
        sel = sorted(rows[:q])
        kept.extend(sel)
        ret_offset[e + 1] = ret_offset[e] + q
    return ret_offset, np.asarray(kept, dtype=np.int64)


def _swiglu_backward(dh, a, b):
    """d/da and d/db of h = silu(a)*b given dh: da = dh*b*s*(1+a(1-s)), db = dh*silu(a)."""
    s = sigmoid(a)
    da = dh * b * s * (1.0 + a * (1.0 - s))
    db = dh * (a * s)
    return da, db


def backward(inp, fwd, dy, quota=None, frozen=False, score_override=None):
    """Backward of L = <dY, Y> restricted to retained pairs for the expert part.

    ([I14] Proposal/Scope: dx, and dW for full fine-tuning; [LRMoE] Abstract:
    scored pairs selected within per-expert quotas, compacted, variable-size
    grouped GEMMs; [PR44] Changes: the forward's saved state feeds the backward.)

    For every retained row r of expert e, token t, slot weight w_r:
      dy_r = w_r dY_t; dh = dy_r W_down[e]^T; (da, db) = SwiGLU'(dh; a, b);
      dx_r = da W_gate[e]^T + db W_up[e]^T;
      dW_down[e] += h_r^T dy_r; dW_gate[e] += x_t^T da; dW_up[e] += x_t^T db.
    Router, over all pairs: dl[t, idx_j] = w_j (g_j - sum_i w_i g_i), 0 elsewhere;
      dX_t += dl_t W_r^T; dW_r = x^T dl. No gradient to the router bias.
    Shared expert: full backward with dY (never subject to retention).
    ``score_override`` replays retention on given (e.g. GPU fp32) scores.
    """
    x = np.asarray(inp["x"], np.float64)
    dy = np.asarray(dy, np.float64)
    w_r = np.asarray(inp["w_router"], np.float64)
    w_gate, w_up, w_down = inp["w_gate"], inp["w_up"], inp["w_down"]
    k, E = fwd["k"], fwd["E"]
    T, H = x.shape
    F = w_gate.shape[2]
    w, idx = fwd["w"], fwd["idx"]
    row_of_pair, pair_of_row, offset = fwd["row_of_pair"], fwd["pair_of_row"], fwd["offset"]
    a, b, h, y_pair = fwd["a"], fwd["b"], fwd["h"], fwd["y_pair"]

    g, score = pair_scores(dy, x, w, y_pair, row_of_pair)
    sel_score = score if score_override is None else score_override
    ret_offset, ret_rows = select_retained(sel_score, offset, pair_of_row, k, quota)

    dX = np.zeros((T, H))
    grads = {}
    if not frozen:
        grads["dw_gate"] = np.zeros((E, H, F))
        grads["dw_up"] = np.zeros((E, H, F))
        grads["dw_down"] = np.zeros((E, F, H))
    w_flat = w.reshape(-1)
    for e in range(E):
        rows = ret_rows[ret_offset[e]:ret_offset[e + 1]]
        if len(rows) == 0:
            continue
        pairs = pair_of_row[rows]
        tok = pairs // k
        dye = w_flat[pairs][:, None] * dy[tok]
        dh = dye @ np.asarray(w_down[e], np.float64).T
        da, db = _swiglu_backward(dh, a[rows], b[rows])
        dxe = da @ np.asarray(w_gate[e], np.float64).T + db @ np.asarray(w_up[e], np.float64).T
        # tokens are distinct inside one expert, so this scatter never collides
        dX[tok] += dxe
        if not frozen:
            xe = x[tok]
            grads["dw_gate"][e] = xe.T @ da
            grads["dw_up"][e] = xe.T @ db
            grads["dw_down"][e] = h[rows].T @ dye

    # router backward over all pairs
    gp = np.empty((T, k))
    for t in range(T):
        for j in range(k):
            gp[t, j] = g[row_of_pair[t * k + j]]
    mean_g = (w * gp).sum(axis=1, keepdims=True)
    dl_sel = w * (gp - mean_g)
    dl = np.zeros((T, E))
    for j in range(k):
        dl[np.arange(T), idx[:, j]] = dl_sel[:, j]
    dX_router = dl @ w_r.T
    dX = dX + dX_router
    if not frozen:
        grads["dw_router"] = x.T @ dl

    if fwd["shared"] is not None:
        sa, sb, sh, _ = fwd["shared"]
        dhs = dy @ np.asarray(inp["ws_down"], np.float64).T
        das, dbs = _swiglu_backward(dhs, sa, sb)
        dX = dX + das @ np.asarray(inp["ws_gate"], np.float64).T + dbs @ np.asarray(inp["ws_up"], np.float64).T
        if not frozen:
            grads["dws_gate"] = x.T @ das
            grads["dws_up"] = x.T @ dbs
            grads["dws_down"] = sh.T @ dy

    return dict(dX=dX, g=g, score=score, ret_offset=ret_offset, ret_rows=ret_rows,
                dl=dl, dX_router=dX_router, **grads)
