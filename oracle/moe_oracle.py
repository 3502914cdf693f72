"""Plain, slow, fp64 oracle of one Mixture-of-Experts layer forward.

TEST INFRASTRUCTURE.  This module is the checker that the CUDA path is
compared against.  It is imported only by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.  It
shares no code with the CUDA kernels or their binding and never calls them.

Source of the method: "Scalable Pretraining of Large MoE LMs on Aurora Super
Computer", §3.1 FastSparseMoE, Algorithm 1 (FastSparseMoEBlock):
  stage 1  router logits -> Softmax -> TopK           (weights, indices [S,K])
  stage 2  per-expert token counts and prefix sums    (group boundaries)
  stage 3  index generation: input_indices (row -> token) and
           output_indices ((token, slot) -> row)
  stage 4  mlp_in = input[input_indices]; gate/up grouped GEMMs; Silu(gate)*up;
           down grouped GEMM
  stage 5  output reduction: out[t] = sum over the token's slots of
           weights[t][slot] * mlp_out[row of (t, slot)]
Renormalisation of the k selected gates is not in Algorithm 1; it is the
workload's stated routing ("softmax top-k renormalised") and is a flag here.

Each function is the plain definition of its step, written out with numpy
primitives (sort, cumsum, matmul) and no blocking or fusion.  All floating
point is fp64; inputs that are bf16 or fp32 on the GPU are passed in as
float arrays holding exactly those values.

Readings of points the pages leave open (each is pinned by a test):
  * experts are ranked by the fp32 router logit (softmax is monotone, so the
    set and order equal those of ranking by probability), ties broken by the
    smaller expert index; -0.0 equals +0.0;
  * slot j of a token holds its (j+1)-th best expert;
  * within an expert's group, rows are in ascending token order (the order
    Algorithm 1's thread-block layout of partial counts produces);
  * the expert MLP and the reduction are exact fp64 on the bf16 inputs, with
    no intermediate rounding.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- stage 1
def softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Row softmax in fp64: p[t,e] = exp(l[t,e] - m_t) / sum_e' exp(l[t,e'] - m_t).

    Algorithm 1, stage 1 (probs = Softmax(logits)).
    """
    l = np.asarray(logits, dtype=np.float64)
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    return z / z.sum(axis=1, keepdims=True)


def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k routing of each token.

    Algorithm 1, stage 1 (weights, indices = TopK(probs)).  Returns
    ``idx`` int32 [T,k] and ``w`` float64 [T,k].

    The k experts with the largest logits are chosen under the total order
    (logit descending, expert index ascending); slot j holds the (j+1)-th.
    ``w[t,j]`` is the softmax probability of that expert, divided by the sum
    of the k selected probabilities when ``renormalize``.
    """
    l32 = np.asarray(logits, dtype=np.float32)
    T, E = l32.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    # a stable sort of the negated values orders by value descending with
    # ties kept in ascending expert order; -0.0 and +0.0 compare equal
    order = np.argsort(-l32, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    probs = softmax_rows(l32)
    w = np.take_along_axis(probs, idx.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, w


def route_topk_grouped(logits: np.ndarray, k: int, n_groups: int, renormalize: bool = True):
    """Group-limited top-k routing.

    "Training a 1T-Params MoE on EU public infrastructure", Group-limited
    expert routing: the experts are split into n_groups equal groups
    (consecutive expert indices) and the router selects the same number of
    experts, k / n_groups, from every group.  Inside a group the choice is
    the ordinary top-(k/n_groups) under (logit descending, expert index
    ascending).  The k selected experts fill the slots in that same order
    across groups, and the gates are their softmax probabilities over all
    E experts (divided by the sum over the k selected when
    ``renormalize``), as in ``route_topk``.
    """
    l32 = np.asarray(logits, dtype=np.float32)
    T, E = l32.shape
    if n_groups < 1 or E % n_groups or k % n_groups:
        raise ValueError("n_groups must divide E and k")
    size, per = E // n_groups, k // n_groups
    if per > size:
        raise ValueError("k / n_groups exceeds the group size")
    chosen = []
    for g in range(n_groups):
        block = l32[:, g * size:(g + 1) * size]
        order = np.argsort(-block, axis=1, kind="stable")[:, :per]
        chosen.append(order + g * size)
    cand = np.concatenate(chosen, axis=1)                       # [T, k], group order
    vals = np.take_along_axis(l32, cand, axis=1)
    # slot order over the selection: value descending, then expert ascending
    slot = np.lexsort((cand, -vals), axis=1)
    idx = np.take_along_axis(cand, slot, axis=1).astype(np.int32)
    probs = softmax_rows(l32)
    w = np.take_along_axis(probs, idx.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, w


def router_topk(x, w_router, k: int, renormalize: bool = True):
    """Router linear layer, then Softmax and TopK, all in fp64.

    Algorithm 1, stage 1: logits = Router(input) with Router a linear layer
    (logits[t, e] = sum_i x[t, i] * w_router[i, e]), probs = Softmax(logits),
    weights, indices = TopK(probs).  The logits are exact fp64 products of
    the bf16 inputs and are ranked in fp64 (logit descending, expert index
    ascending).  Returns (idx int32 [T,k], w float64 [T,k], logits float64
    [T,E]).
    """
    logits = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    order = np.argsort(-logits, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    probs = softmax_rows(logits)
    w = np.take_along_axis(probs, idx.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, w, logits


# ---------------------------------------------------------- stages 2 and 3
def dispatch(idx: np.ndarray, E: int):
    """Counts, group boundaries and the two index maps.

    Algorithm 1, stages 2-3, written as the stable counting sort they
    compute.  With pairs p = t*k + j taken in increasing p:
      counts[e]    number of pairs routed to e (token counts)
      offsets      exclusive prefix sum of counts, length E+1 (cum_token_counts)
      dest_row[p]  offsets[e] + number of earlier pairs q < p with idx[q] == e
                   (output_indices)
      src_token[r] token of the pair placed at row r (input_indices)
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    pair_of_row = np.argsort(flat, kind="stable")     # rows grouped by expert, pair order kept
    dest_row = np.empty(T * k, dtype=np.int64)
    dest_row[pair_of_row] = np.arange(T * k, dtype=np.int64)
    src_token = pair_of_row // k
    return counts, offsets, src_token, dest_row


# ---------------------------------------------------------------- stage 4
def permute(x: np.ndarray, src_token: np.ndarray) -> np.ndarray:
    """mlp_in = input[input_indices] (Algorithm 1, stage 4): a row gather."""
    return np.asarray(x)[np.asarray(src_token, dtype=np.int64)]


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def expert_mlp(x_perm, offsets, w_gate, w_up, w_down, experts=None):
    """Grouped SwiGLU expert MLP on expert-contiguous rows.

    Algorithm 1, stage 4: for expert e and its rows [offsets[e], offsets[e+1]):
      gate = X_e @ Wg[e]       Wg[e] is [d, f]
      up   = X_e @ Wu[e]
      h    = Silu(gate) * up
      y    = h @ Wd[e]         Wd[e] is [f, d]
    Returns (h [P,f], y [P,d]) in fp64.  ``experts`` limits the work to a
    subset (rows of other experts stay zero).
    """
    x_perm = np.asarray(x_perm, dtype=np.float64)
    P = x_perm.shape[0]
    E = len(offsets) - 1
    f = w_gate.shape[2]
    d = w_down.shape[2]
    h = np.zeros((P, f), dtype=np.float64)
    y = np.zeros((P, d), dtype=np.float64)
    for e in (range(E) if experts is None else experts):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        X = x_perm[a:b]
        gate = X @ np.asarray(w_gate[e], dtype=np.float64)
        up = X @ np.asarray(w_up[e], dtype=np.float64)
        he = silu(gate) * up
        h[a:b] = he
        y[a:b] = he @ np.asarray(w_down[e], dtype=np.float64)
    return h, y


def silu_grad(z: np.ndarray) -> np.ndarray:
    """d/dz SiLU(z) = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    z = np.asarray(z, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def expert_gate_up(x_perm, offsets, w_gate, w_up):
    """The gate and up pre-activations of every row (Algorithm 1, stage 4:
    gate_out = X_e @ Wg[e], up_out = X_e @ Wu[e]), [P, f] each, fp64."""
    x_perm = np.asarray(x_perm, dtype=np.float64)
    f = w_gate.shape[2]
    gate = np.zeros((x_perm.shape[0], f))
    up = np.zeros((x_perm.shape[0], f))
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a < b:
            gate[a:b] = x_perm[a:b] @ np.asarray(w_gate[e], dtype=np.float64)
            up[a:b] = x_perm[a:b] @ np.asarray(w_up[e], dtype=np.float64)
    return gate, up


def expert_mlp_backward(x_perm, offsets, w_gate, w_up, w_down, dy, return_preact_grads=False):
    """Backward of the grouped SwiGLU expert MLP (Algorithm 1, stage 4,
    differentiated), expert by expert on its rows [offsets[e], offsets[e+1]):
      dH  = dY @ Wd[e]^T
      dG  = dH * up * Silu'(gate)        dU = dH * Silu(gate)
      dX  = dG @ Wg[e]^T + dU @ Wu[e]^T
      dWd[e] = h^T @ dY     dWg[e] = X^T @ dG     dWu[e] = X^T @ dU
    ``dy`` is the gradient of the expert outputs (rows of mlp_out).  Returns
    (dx_perm [P,d], dw_gate [E,d,f], dw_up [E,d,f], dw_down [E,f,d]) in fp64;
    experts without rows get zero weight gradients.  With
    ``return_preact_grads`` the tuple ends with dgate, dup [P,f].
    """
    x_perm = np.asarray(x_perm, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    E = len(offsets) - 1
    d, f = w_gate.shape[1], w_gate.shape[2]
    dx = np.zeros_like(x_perm)
    dwg = np.zeros((E, d, f))
    dwu = np.zeros((E, d, f))
    dwd = np.zeros((E, f, d))
    dgate = np.zeros((x_perm.shape[0], f))
    dup = np.zeros((x_perm.shape[0], f))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        X, dY = x_perm[a:b], dy[a:b]
        Wg = np.asarray(w_gate[e], dtype=np.float64)
        Wu = np.asarray(w_up[e], dtype=np.float64)
        Wd = np.asarray(w_down[e], dtype=np.float64)
        gate, up = X @ Wg, X @ Wu
        h = silu(gate) * up
        dH = dY @ Wd.T
        dG = dH * up * silu_grad(gate)
        dU = dH * silu(gate)
        dx[a:b] = dG @ Wg.T + dU @ Wu.T
        dwd[e] = h.T @ dY
        dwg[e] = X.T @ dG
        dwu[e] = X.T @ dU
        dgate[a:b] = dG
        dup[a:b] = dU
    if return_preact_grads:
        return dx, dwg, dwu, dwd, dgate, dup
    return dx, dwg, dwu, dwd


# ---------------------------------------------------------------- stage 5
def combine(y, dest_row, w):
    """Output reduction (Algorithm 1, stage 5, forward):
    out[t] = sum_j w[t,j] * y[dest_row[t*k + j]], slots in order j = 0..k-1.
    """
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    rows = np.asarray(dest_row, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[rows[:, j]]
    return out


# ------------------------------------------------------------- backward
def combine_backward(dout, mlp_out, dest_row, w):
    """Output reduction, backward (Algorithm 1, stage 5, backward function):
    for every routed pair p = (t, j) with row r = dest_row[p],
      mlp_out_grad[r] = w[t, j] * output_grad[t]
      weights_grad[t, j] = <mlp_out[r], output_grad[t]>
    ``mlp_out`` is the expert output before the gate.  Returns
    (mlp_out_grad [P, d], weights_grad [T, k]) in fp64.
    """
    dout = np.asarray(dout, dtype=np.float64)
    y = np.asarray(mlp_out, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    rows = np.asarray(dest_row, dtype=np.int64).reshape(T, k)
    dy = np.zeros_like(y)
    dw = np.zeros((T, k))
    for j in range(k):
        dy[rows[:, j]] = w[:, j:j + 1] * dout
        dw[:, j] = np.einsum("td,td->t", y[rows[:, j]], dout)
    return dy, dw


def route_backward(logits, idx, dw, renormalize=True):
    """Gradient of the router logits from the gradient of the gates.

    With the selection fixed, w_j = exp(l_{e_j}) / Z where Z sums exp(l)
    over all E experts, or over the k selected when renormalised, so
    dl_e = [e selected as slot j] w_j dw_j - q_e * sum_j w_j dw_j, with
    q_e = exp(l_e) / Z on the normalisation set and 0 elsewhere.
    Returns d_logits [T, E] in fp64.
    """
    l = np.asarray(logits, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    dw = np.asarray(dw, dtype=np.float64)
    T, E = l.shape
    out = np.zeros((T, E))
    for t in range(T):
        sel = idx[t]
        if renormalize:
            z = np.exp(l[t, sel] - l[t, sel].max())
            wt = z / z.sum()
            q = np.zeros(E)
            q[sel] = wt
        else:
            q = np.exp(l[t] - l[t].max())
            q = q / q.sum()
            wt = q[sel]
        s = np.dot(wt, dw[t])
        out[t] = -q * s
        out[t, sel] += wt * dw[t]
    return out


# ------------------------------------------------------------ whole layer
def moe_forward(x, logits, w_gate, w_up, w_down, k, renormalize=True):
    """Every stage of the layer forward, in order, with all intermediates."""
    E = w_gate.shape[0]
    idx, w = route_topk(logits, k, renormalize)
    counts, offsets, src_token, dest_row = dispatch(idx, E)
    x_perm = permute(x, src_token)
    h, y = expert_mlp(x_perm, offsets, w_gate, w_up, w_down)
    out = combine(y, dest_row, w)
    row_w = np.empty(len(dest_row), dtype=np.float64)
    row_w[dest_row] = w.reshape(-1)
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, src_token=src_token,
                dest_row=dest_row, row_w=row_w, x_perm=x_perm, h=h, y=y, out=out)


def moe_forward_tokens(x_rows, logits_rows, w_gate, w_up, w_down, k, renormalize=True, routing=None):
    """Layer output for a few tokens only.

    Routing, the expert MLP and the reduction of one token depend on that
    token's own row of x and logits alone, so the layer restricted to a
    token subset is the layer applied to those rows.  ``routing`` = (idx, w)
    replaces the routing of ``logits_rows`` when given.  Returns idx, w,
    per-slot h [n,k,f] and y [n,k,d] (unscaled) and out [n,d].
    """
    x_rows = np.asarray(x_rows, dtype=np.float64)
    if routing is None:
        idx, w = route_topk(logits_rows, k, renormalize)
    else:
        idx, w = (np.asarray(a) for a in routing)
    n = x_rows.shape[0]
    f = w_gate.shape[2]
    d = w_down.shape[2]
    h = np.zeros((n, k, f))
    y = np.zeros((n, k, d))
    for e in np.unique(idx):
        sel = np.nonzero(idx == e)          # (token, slot) pairs routed to e
        X = x_rows[sel[0]]
        gate = X @ np.asarray(w_gate[e], dtype=np.float64)
        up = X @ np.asarray(w_up[e], dtype=np.float64)
        he = silu(gate) * up
        h[sel] = he
        y[sel] = he @ np.asarray(w_down[e], dtype=np.float64)
    out = np.einsum("nk,nkd->nd", w, y)
    return dict(idx=idx, w=w, h=h, y=y, out=out)


def moe_backward(x, logits, w_gate, w_up, w_down, dout, k, renormalize=True):
    """Gradients of one layer's output (moe_forward) with respect to its
    inputs, for an output gradient ``dout`` [T,d], the top-k selection held
    fixed.  Runs the forward of Algorithm 1, then its stages backwards:
    output reduction backward (stage 5), the expert MLP backward (stage 4),
    the un-permute of the row gradients to their tokens (the transpose of
    mlp_in = input[input_indices]: every row adds into its token), and the
    gate gradient taken back to the router logits (stage 1).
    Returns a dict with dx [T,d], d_logits [T,E], dw_gate, dw_up [E,d,f],
    dw_down [E,f,d] (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    E = np.asarray(logits).shape[1]
    idx, w = route_topk(logits, k, renormalize)
    counts, offsets, src, dst = dispatch(idx, E)
    xp = permute(x, src)
    _, y = expert_mlp(xp, offsets, w_gate, w_up, w_down)
    dy, dw = combine_backward(dout, y, dst, w)
    dxp, dwg, dwu, dwd = expert_mlp_backward(xp, offsets, w_gate, w_up, w_down, dy)
    dx = np.zeros_like(x)
    np.add.at(dx, src, dxp)
    d_logits = route_backward(np.asarray(logits, dtype=np.float64), idx, dw, renormalize)
    return {"dx": dx, "d_logits": d_logits, "dw_gate": dwg, "dw_up": dwu, "dw_down": dwd}
