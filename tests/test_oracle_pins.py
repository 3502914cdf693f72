"""Pins of the fp64 oracle to facts other than its own code.

Each test checks an oracle step against something the pages or mathematics
fix: hand-worked examples (tests/golden), brute force on tiny inputs, a
restatement of Algorithm 1's thread-block procedure, library routines for
special cases (scipy softmax, torch's SiLU and matmul), closed forms of the
forced-uniform workload and invariants of a permutation.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads
from tests.alg1_emulation import index_generation


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_values(a):
    """Round an fp32/fp64 array to bf16 and return it as fp32 (exact values)."""
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _random_logits(rng, T, E, ties=False):
    l = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        # coarse values force many exact ties; sprinkle signed zeros
        l = np.round(l * 2.0) / 2.0
        l[rng.random((T, E)) < 0.1] = -0.0
        l[rng.random((T, E)) < 0.1] = 0.0
    return l


# ------------------------------------------------------------------ routing
def _brute_topk(row, k):
    """Pick k times the best remaining expert: larger value, then smaller index."""
    left = list(range(len(row)))
    chosen = []
    for _ in range(k):
        best = left[0]
        for e in left[1:]:
            if row[e] > row[best] or (row[e] == row[best] and e < best):
                best = e
        chosen.append(best)
        left.remove(best)
    return chosen


@pytest.mark.parametrize("T,E,k,ties", [(40, 8, 2, False), (40, 8, 8, True), (30, 16, 5, True),
                                        (25, 64, 8, False), (10, 1, 1, False)])
def test_route_indices_match_brute_force(T, E, k, ties):
    l = _random_logits(_rng(T * E + k), T, E, ties)
    idx, _ = oracle.route_topk(l, k)
    for t in range(T):
        assert list(idx[t]) == _brute_topk([float(v) for v in l[t]], k)


@pytest.mark.parametrize("renorm", [True, False])
def test_route_weights_closed_form(renorm):
    T, E, k = 50, 12, 4
    l = _random_logits(_rng(7), T, E)
    idx, w = oracle.route_topk(l, k, renorm)
    for t in range(T):
        sel = l[t, idx[t]].astype(np.float64)
        if renorm:
            # renormalised gates are the softmax over the selected logits alone
            ref = scipy.special.softmax(sel)
        else:
            ref = scipy.special.softmax(l[t].astype(np.float64))[idx[t]]
        np.testing.assert_allclose(w[t], ref, rtol=1e-14, atol=1e-16)
    if renorm:
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_route_golden(golden):
    g = golden("route_example.json")
    for case in g["cases"]:
        l = np.array([case["logits"]], dtype=np.float32)
        idx, w = oracle.route_topk(l, case["k"], case["renormalize"])
        assert list(idx[0]) == case["idx"]
        np.testing.assert_allclose(w[0], case["w"], rtol=1e-15, atol=0)


def test_softmax_rows_properties():
    l = _random_logits(_rng(3), 20, 9)
    p = oracle.softmax_rows(l)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-15)
    np.testing.assert_allclose(p, scipy.special.softmax(l.astype(np.float64), axis=1), rtol=1e-14)
    # shift invariance
    np.testing.assert_allclose(oracle.softmax_rows(l.astype(np.float64) + 100.0), p, rtol=1e-12)


# ----------------------------------------------------------- counts / index
def test_index_golden_matches_hand_example(golden):
    g = golden("alg1_index_example.json")
    idx = np.array(g["indices"])
    counts, offsets, src, dst = oracle.dispatch(idx, g["N"])
    assert list(counts) == g["no_ep"]["token_counts"]
    assert list(offsets) == g["no_ep"]["cum_token_counts"]
    assert list(src) == g["no_ep"]["input_indices"]
    assert list(dst) == g["no_ep"]["output_indices"]


def test_alg1_emulation_matches_hand_example(golden):
    """The restated thread-block procedure reproduces the hand-worked example
    with and without expert parallelism (small token blocks make several
    threads matter)."""
    g = golden("alg1_index_example.json")
    for tbs in (1, 2, 8):
        ctc, _, _, inp, outp, _ = index_generation(g["indices"], g["N"], tbs=tbs)
        assert ctc == g["no_ep"]["cum_token_counts"]
        assert inp == g["no_ep"]["input_indices"]
        assert outp == g["no_ep"]["output_indices"]
        for r in (0, 1):
            want = g["ep2"][f"rank{r}"]
            ctc, ec, _, inp, outp, sel = index_generation(g["indices"], g["N"], ep=2, rank=r, tbs=tbs)
            assert ctc == want["cum_token_counts"]
            assert ec == want["expert_counts"]
            assert inp == want["input_indices"]
            assert outp == want["output_indices"]
            assert sel == want["selected_expert_indices"]


@pytest.mark.parametrize("T,E,k,tbs", [(37, 8, 2, 8), (64, 16, 4, 8), (100, 5, 5, 3), (9, 32, 7, 8),
                                       (1, 4, 1, 8), (50, 1, 1, 8)])
def test_dispatch_matches_alg1_thread_blocks(T, E, k, tbs):
    l = _random_logits(_rng(T + 31 * E + k), T, E, ties=True)
    idx, _ = oracle.route_topk(l, k)
    counts, offsets, src, dst = oracle.dispatch(idx, E)
    ctc, ec, cec, inp, outp, sel = index_generation(idx.tolist(), E, tbs=tbs)
    assert list(offsets) == ctc
    assert list(src) == inp
    assert list(dst) == outp
    assert ec == [k] * T and cec == [t * k for t in range(T + 1)]
    assert sel == [j for _ in range(T) for j in range(k)]


@pytest.mark.parametrize("ep", [2, 4])
def test_dispatch_matches_alg1_expert_parallel_ranks(ep):
    """Each EP rank's local indices are the oracle's rows of that rank's
    expert range, renumbered from the range's first row."""
    T, E, k = 45, 16, 4
    idx, _ = oracle.route_topk(_random_logits(_rng(ep), T, E), k)
    counts, offsets, src, dst = oracle.dispatch(idx, E)
    nr = E // ep
    for r in range(ep):
        lo, hi = r * nr, r * nr + nr
        ctc, ec, cec, inp, outp, sel = index_generation(idx.tolist(), E, ep=ep, rank=r)
        base = offsets[lo]
        assert [c + base for c in ctc] == list(offsets[lo:hi + 1])
        assert inp == list(src[offsets[lo]:offsets[hi]])
        local_pairs = [t * k + j for t in range(T) for j in range(k) if lo <= idx[t, j] < hi]
        assert outp == [int(dst[p] - base) for p in local_pairs]
        assert sel == [p % k for p in local_pairs]


def test_dispatch_invariants():
    T, E, k = 300, 24, 6
    idx, _ = oracle.route_topk(_random_logits(_rng(11), T, E, ties=True), k)
    counts, offsets, src, dst = oracle.dispatch(idx, E)
    P = T * k
    assert counts.sum() == P and offsets[0] == 0 and offsets[-1] == P
    assert np.all(np.diff(offsets) == counts)
    assert sorted(dst.tolist()) == list(range(P))                 # bijection
    assert np.array_equal(src[dst], np.arange(P) // k)            # row -> token inverse
    for e in range(E):                                             # ascending tokens in a group
        grp = src[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(grp) > 0)
        assert np.all(idx.reshape(-1)[np.argsort(dst)][offsets[e]:offsets[e + 1]] == e)


def test_dispatch_empty_experts_and_single_expert():
    idx = np.array([[2], [2], [0], [2]])
    counts, offsets, src, dst = oracle.dispatch(idx, 5)
    assert list(counts) == [1, 0, 3, 0, 0]
    assert list(offsets) == [0, 1, 1, 4, 4, 4]
    assert list(src) == [2, 0, 1, 3] and list(dst) == [1, 2, 0, 3]
    counts, offsets, src, dst = oracle.dispatch(np.zeros((0, 3), dtype=np.int32), 4)
    assert list(offsets) == [0, 0, 0, 0, 0] and len(src) == 0


def test_forced_uniform_closed_form():
    """Forced-uniform routing: pair p goes to expert p mod E, so expert e gets
    P//E pairs plus one when e < P mod E (T=65,536, k=8, E=384)."""
    cfg = workloads.get("long")
    l = workloads.generate_logits(cfg).numpy()
    idx, _ = oracle.route_topk(l, cfg.k)
    assert np.array_equal(np.sort(idx, axis=1), np.sort(workloads.fur_assignment(cfg.T, cfg.E, cfg.k).numpy(), axis=1))
    counts, offsets, _, _ = oracle.dispatch(idx, cfg.E)
    P = cfg.T * cfg.k
    want = np.array([P // cfg.E + (1 if e < P % cfg.E else 0) for e in range(cfg.E)])
    assert np.array_equal(counts, want)
    assert set(counts.tolist()) == {1365, 1366}


# ------------------------------------------------------------- expert MLP
def test_swiglu_scalar_golden(golden):
    g = golden("swiglu_scalar.json")
    wg = np.array([[[g["wg"]]]]); wu = np.array([[[g["wu"]]]]); wd = np.array([[[g["wd"]]]])
    for c in g["cases"]:
        h, y = oracle.expert_mlp(np.array([[c["x"]]]), [0, 1], wg, wu, wd)
        np.testing.assert_allclose(oracle.silu(np.array([c["g"]])), [c["silu_g"]], rtol=1e-15)
        np.testing.assert_allclose(h[0, 0], c["h"], rtol=1e-15)
        np.testing.assert_allclose(y[0, 0], c["y"], rtol=1e-15)


def test_single_expert_layer_is_dense_swiglu_mlp():
    """E=1, k=1 with renormalised gates (w = 1): the layer is a dense SwiGLU
    MLP, computed here with torch's float64 SiLU and matmul."""
    rng = _rng(5)
    T, d, f = 33, 24, 40
    x = _bf16_values(rng.standard_normal((T, d)))
    wg = _bf16_values(rng.standard_normal((1, d, f)) / math.sqrt(d))
    wu = _bf16_values(rng.standard_normal((1, d, f)) / math.sqrt(d))
    wd = _bf16_values(rng.standard_normal((1, f, d)) / math.sqrt(f))
    logits = rng.standard_normal((T, 1)).astype(np.float32)
    res = oracle.moe_forward(x, logits, wg, wu, wd, k=1)
    X = torch.from_numpy(x).double()
    ref = (torch.nn.functional.silu(X @ torch.from_numpy(wg[0]).double()) *
           (X @ torch.from_numpy(wu[0]).double())) @ torch.from_numpy(wd[0]).double()
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["w"], 1.0)


def _brute_force_layer(x, logits, wg, wu, wd, k, renorm):
    """Every token through every expert, then a routing mask: no grouping,
    no permutation, no index maps."""
    T, E = logits.shape
    out = np.zeros((T, wd.shape[2]))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        chosen = _brute_topk(row, k)
        m = max(row)
        z = [math.exp(v - m) for v in row]
        denom = sum(z[e] for e in chosen) if renorm else sum(z)
        xt = x[t].astype(np.float64)
        for e in range(E):
            if e not in chosen:
                continue
            g = xt @ wg[e].astype(np.float64)
            u = xt @ wu[e].astype(np.float64)
            h = np.array([gi / (1.0 + math.exp(-gi)) for gi in g]) * u
            out[t] += (z[e] / denom) * (h @ wd[e].astype(np.float64))
    return out


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("T,d,E,k,f", [(21, 16, 6, 2, 24), (12, 8, 4, 4, 8), (17, 24, 5, 1, 16)])
def test_layer_matches_per_token_brute_force(T, d, E, k, f, renorm):
    rng = _rng(T * d + E * k + f)
    x = _bf16_values(rng.standard_normal((T, d)))
    wg = _bf16_values(rng.standard_normal((E, d, f)) / math.sqrt(d))
    wu = _bf16_values(rng.standard_normal((E, d, f)) / math.sqrt(d))
    wd = _bf16_values(rng.standard_normal((E, f, d)) / math.sqrt(f))
    logits = _random_logits(rng, T, E)
    res = oracle.moe_forward(x, logits, wg, wu, wd, k, renorm)
    ref = _brute_force_layer(x, logits, wg, wu, wd, k, renorm)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-13)


def test_token_subset_matches_full_layer():
    rng = _rng(9)
    T, d, E, k, f = 40, 16, 6, 3, 8
    x = _bf16_values(rng.standard_normal((T, d)))
    wg = _bf16_values(rng.standard_normal((E, d, f)))
    wu = _bf16_values(rng.standard_normal((E, d, f)))
    wd = _bf16_values(rng.standard_normal((E, f, d)))
    logits = _random_logits(rng, T, E)
    full = oracle.moe_forward(x, logits, wg, wu, wd, k)
    toks = np.array([0, 5, 17, 39])
    sub = oracle.moe_forward_tokens(x[toks], logits[toks], wg, wu, wd, k)
    np.testing.assert_allclose(sub["out"], full["out"][toks], rtol=1e-13, atol=1e-14)
    rows = full["dest_row"].reshape(T, k)[toks]
    np.testing.assert_allclose(sub["y"], full["y"][rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sub["h"], full["h"][rows], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- combine
def test_combine_of_identity_experts_returns_input():
    """With identity experts (y = mlp_in) and renormalised gates the output
    reduction returns each token's input: sum_j w_j x_t = x_t."""
    rng = _rng(13)
    T, d, E, k = 64, 12, 10, 3
    x = rng.standard_normal((T, d))
    idx, w = oracle.route_topk(_random_logits(rng, T, E), k)
    _, _, src, dst = oracle.dispatch(idx, E)
    out = oracle.combine(oracle.permute(x, src), dst, w)
    np.testing.assert_allclose(out, x, rtol=1e-14, atol=1e-14)


def test_combine_k1_is_gate_times_row():
    rng = _rng(17)
    T, d, E = 20, 8, 5
    y = rng.standard_normal((T, d))
    idx, w = oracle.route_topk(_random_logits(rng, T, E), 1, renormalize=False)
    _, _, src, dst = oracle.dispatch(idx, E)
    out = oracle.combine(y, dst, w)
    assert np.array_equal(out, w[:, :1] * y[dst])


def test_permute_is_row_gather():
    x = np.arange(12.0).reshape(4, 3)
    assert np.array_equal(oracle.permute(x, [3, 0, 0, 2]), x[[3, 0, 0, 2]])


# ------------------------------------------------------- grouped routing
def _brute_grouped(row, k, G):
    E = len(row)
    size, per = E // G, k // G
    picked = []
    for g in range(G):
        sub = list(range(g * size, (g + 1) * size))
        picked += [sub[i] for i in _brute_topk([row[e] for e in sub], per)]
    # slots: value descending, then index ascending
    return sorted(picked, key=lambda e: (-row[e], e))


@pytest.mark.parametrize("T,E,k,G,ties", [(30, 8, 4, 2, False), (30, 16, 8, 4, True), (20, 12, 6, 3, True),
                                          (10, 64, 8, 8, False), (15, 8, 8, 2, False)])
def test_grouped_route_matches_brute_force(T, E, k, G, ties):
    l = _random_logits(_rng(T + E + k + G), T, E, ties)
    idx, w = oracle.route_topk_grouped(l, k, G)
    for t in range(T):
        assert list(idx[t]) == _brute_grouped([float(v) for v in l[t]], k, G)
        np.testing.assert_allclose(w[t], scipy.special.softmax(l[t, idx[t]].astype(np.float64)), rtol=1e-14)


def test_grouped_route_with_one_group_is_plain_topk():
    l = _random_logits(_rng(21), 40, 16, ties=True)
    for renorm in (True, False):
        gi, gw = oracle.route_topk_grouped(l, 4, 1, renorm)
        ri, rw = oracle.route_topk(l, 4, renorm)
        assert np.array_equal(gi, ri)
        np.testing.assert_allclose(gw, rw, rtol=1e-15)


def test_grouped_route_balances_the_groups():
    """Every group receives the same number of (token, expert) pairs,
    T*k/G: the property the page uses to give every GPU the same load."""
    T, E, k, G = 500, 384, 8, 4
    l = _random_logits(_rng(5), T, E)
    l[:, :96] += 2.0  # a router that prefers group 0 still gives it only T*k/G
    idx, _ = oracle.route_topk_grouped(l, k, G)
    counts, _, _, _ = oracle.dispatch(idx, E)
    assert list(counts.reshape(G, -1).sum(axis=1)) == [T * k // G] * G
    plain, _ = oracle.route_topk(l, k)
    pc, _, _, _ = oracle.dispatch(plain, E)
    assert pc.reshape(G, -1).sum(axis=1)[0] > T * k // G  # the unconstrained router is unbalanced


def test_grouped_route_golden(golden):
    g = golden("route_example.json")
    for case in g["grouped_cases"]:
        idx, w = oracle.route_topk_grouped(np.array([case["logits"]], dtype=np.float32), case["k"], case["n_groups"],
                                           case["renormalize"])
        assert list(idx[0]) == case["idx"]
        np.testing.assert_allclose(w[0], case["w"], rtol=1e-15)


# -------------------------------------------------------- router + top-k
def test_router_logits_match_per_token_dot_products():
    """Brute force: each logit is the plain dot product of the token row and
    the expert's router column."""
    rng = _rng(31)
    T, d, E = 7, 12, 5
    x = _bf16_values(rng.standard_normal((T, d)))
    wr = _bf16_values(rng.standard_normal((d, E)))
    _, _, logits = oracle.router_topk(x, wr, 2)
    for t in range(T):
        for e in range(E):
            assert logits[t, e] == pytest.approx(sum(float(x[t, i]) * float(wr[i, e]) for i in range(d)), rel=1e-13)


def test_router_with_one_hot_tokens_selects_router_rows():
    """x = e_i makes the logits the i-th row of the router matrix (closed form)."""
    rng = _rng(33)
    d, E, k = 6, 9, 3
    wr = rng.standard_normal((d, E))
    idx, w, logits = oracle.router_topk(np.eye(d), wr, k)
    assert np.array_equal(logits, wr)
    for i in range(d):
        assert list(idx[i]) == _brute_topk(list(wr[i]), k)
        np.testing.assert_allclose(w[i], scipy.special.softmax(wr[i, idx[i]]), rtol=1e-14)


def test_router_topk_equals_routing_of_its_logits():
    rng = _rng(35)
    x = _bf16_values(rng.standard_normal((50, 32)))
    wr = _bf16_values(rng.standard_normal((32, 16)) / np.sqrt(32))
    for renorm in (True, False):
        idx, w, logits = oracle.router_topk(x, wr, 4, renorm)
        # logits here are exactly representable in fp32 for the ranking check
        order = np.argsort(-logits, axis=1, kind="stable")[:, :4]
        assert np.array_equal(idx, order)
        ref = scipy.special.softmax(logits, axis=1)
        ref = np.take_along_axis(ref, order, axis=1)
        if renorm:
            ref = ref / ref.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(w, ref, rtol=1e-13)


# --------------------------------------------------------------- backward
def _finite_diff(fn, x, eps=1e-6):
    """Central differences of a scalar function of an fp64 array."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp = x.copy(); xp[i] += eps
        xm = x.copy(); xm[i] -= eps
        g[i] = (fn(xp) - fn(xm)) / (2 * eps)
    return g


def test_combine_backward_matches_finite_differences():
    """The output reduction is linear in the expert outputs and the gates;
    its backward must equal the numerical derivative of
    L = <G, combine(y, dest_row, w)> for a fixed output gradient G."""
    rng = _rng(41)
    T, d, E, k = 6, 5, 4, 2
    idx, w = oracle.route_topk(_random_logits(rng, T, E), k)
    _, _, _, dst = oracle.dispatch(idx, E)
    y = rng.standard_normal((T * k, d))
    G = rng.standard_normal((T, d))
    dy, dw = oracle.combine_backward(G, y, dst, w)
    np.testing.assert_allclose(dy, _finite_diff(lambda yy: np.sum(G * oracle.combine(yy, dst, w)), y), atol=1e-8)
    np.testing.assert_allclose(dw, _finite_diff(lambda ww: np.sum(G * oracle.combine(y, dst, ww)), w), atol=1e-8)


@pytest.mark.parametrize("renorm", [True, False])
def test_route_backward_matches_finite_differences(renorm):
    """With the selection held fixed, the gate gradient w.r.t. the logits is
    the derivative of the oracle's own gates."""
    rng = _rng(43)
    T, E, k = 5, 7, 3
    l = rng.standard_normal((T, E))
    idx, _ = oracle.route_topk(l.astype(np.float32), k, renorm)
    dw = rng.standard_normal((T, k))

    def gates(ll):
        if renorm:
            z = np.exp(np.take_along_axis(ll, idx.astype(np.int64), axis=1))
            return z / z.sum(axis=1, keepdims=True)
        p = oracle.softmax_rows(ll)
        return np.take_along_axis(p, idx.astype(np.int64), axis=1)
    ref = _finite_diff(lambda ll: np.sum(dw * gates(ll)), l)
    np.testing.assert_allclose(oracle.route_backward(l, idx, dw, renorm), ref, atol=1e-8)


def test_combine_backward_golden_scalar():
    """One token, two slots, d = 1, worked by hand: rows 0 and 1, gates
    0.25 and 0.75, expert outputs 2 and -4, output gradient 3:
    mlp_out_grad = (0.75, 2.25) and weights_grad = (6, -12)."""
    dy, dw = oracle.combine_backward(np.array([[3.0]]), np.array([[2.0], [-4.0]]), np.array([0, 1]),
                                     np.array([[0.25, 0.75]]))
    assert dy.ravel().tolist() == [0.75, 2.25] and dw.ravel().tolist() == [6.0, -12.0]


# ------------------------------------------------------- layer backward
def test_silu_grad_matches_finite_differences_and_limits():
    z = np.linspace(-12.0, 12.0, 97)
    fd = (oracle.silu(z + 1e-6) - oracle.silu(z - 1e-6)) / 2e-6
    np.testing.assert_allclose(oracle.silu_grad(z), fd, atol=1e-8)
    assert oracle.silu_grad(np.array([0.0]))[0] == 0.5          # sigmoid(0) * (1 + 0)
    assert abs(oracle.silu_grad(np.array([-60.0]))[0]) < 1e-20  # flat far left
    assert abs(oracle.silu_grad(np.array([60.0]))[0] - 1.0) < 1e-20  # identity far right


def _small_layer(seed, T, d, E, k, f):
    rng = _rng(seed)
    x = _bf16_values(rng.standard_normal((T, d)))
    wg = _bf16_values(rng.standard_normal((E, d, f)) / math.sqrt(d))
    wu = _bf16_values(rng.standard_normal((E, d, f)) / math.sqrt(d))
    wd = _bf16_values(rng.standard_normal((E, f, d)) / math.sqrt(f))
    logits = _random_logits(rng, T, E).astype(np.float64)
    dout = rng.standard_normal((T, d))
    return x.astype(np.float64), logits, wg.astype(np.float64), wu.astype(np.float64), wd.astype(np.float64), dout


@pytest.mark.parametrize("renorm", [True, False])
def test_layer_backward_matches_finite_differences(renorm):
    """Every gradient of the layer against central differences of the
    per-token brute-force forward (every token through its experts, no
    grouping or index maps), L = <dout, out>.  E = 4 with k = 2 leaves one
    expert with few rows; the selection does not move under the 1e-6 steps."""
    T, d, E, k, f = 7, 4, 4, 2, 3
    x, l, wg, wu, wd, dout = _small_layer(61, T, d, E, k, f)
    g = oracle.moe_backward(x, l.astype(np.float32), wg, wu, wd, dout, k, renorm)

    def loss(xx=x, ll=l, gg=wg, uu=wu, dd=wd):
        return float(np.sum(dout * _brute_force_layer(xx, ll, gg, uu, dd, k, renorm)))
    np.testing.assert_allclose(g["dx"], _finite_diff(lambda v: loss(xx=v), x), atol=1e-7)
    np.testing.assert_allclose(g["d_logits"], _finite_diff(lambda v: loss(ll=v), l), atol=1e-7)
    np.testing.assert_allclose(g["dw_gate"], _finite_diff(lambda v: loss(gg=v), wg), atol=1e-7)
    np.testing.assert_allclose(g["dw_up"], _finite_diff(lambda v: loss(uu=v), wu), atol=1e-7)
    np.testing.assert_allclose(g["dw_down"], _finite_diff(lambda v: loss(dd=v), wd), atol=1e-7)


def test_layer_backward_scalar_closed_form():
    """d = f = 1, one token, one expert: out = wd * SiLU(wg x) * (wu x), so
    d out/dx = wd (SiLU'(wg x) wg wu x + SiLU(wg x) wu) and
    d out/d wd = SiLU(wg x) wu x, written with math.exp at x=1, wg=1, wu=2,
    wd=3."""
    s = 1.0 / (1.0 + math.exp(-1.0))
    silu1, dsilu1 = s, s * (1.0 + (1.0 - s))
    g = oracle.moe_backward(np.array([[1.0]]), np.array([[0.3]], dtype=np.float32), np.array([[[1.0]]]),
                            np.array([[[2.0]]]), np.array([[[3.0]]]), np.array([[1.0]]), 1, True)
    assert g["dx"][0, 0] == pytest.approx(3.0 * (dsilu1 * 2.0 + silu1 * 2.0), rel=1e-14)
    assert g["dw_down"][0, 0, 0] == pytest.approx(silu1 * 2.0, rel=1e-14)
    assert g["dw_gate"][0, 0, 0] == pytest.approx(3.0 * 2.0 * dsilu1, rel=1e-14)
    assert g["dw_up"][0, 0, 0] == pytest.approx(3.0 * silu1, rel=1e-14)
    assert g["d_logits"][0, 0] == 0.0     # one expert, renormalised: the gate is constant 1


def test_expert_without_rows_gets_zero_weight_gradient():
    T, d, E, k, f = 5, 4, 6, 1, 3
    x, l, wg, wu, wd, dout = _small_layer(67, T, d, E, k, f)
    l[:, 5] = -30.0                       # expert 5 is never chosen
    g = oracle.moe_backward(x, l.astype(np.float32), wg, wu, wd, dout, k)
    assert not g["dw_gate"][5].any() and not g["dw_up"][5].any() and not g["dw_down"][5].any()


def test_gate_up_preactivations_give_the_mlp_hidden_state():
    """h of the expert MLP is Silu(gate) * up of the pre-activations, and the
    pre-activation gradients put together give the same dx_perm."""
    T, d, E, k, f = 9, 6, 3, 2, 5
    x, l, wg, wu, wd, _ = _small_layer(71, T, d, E, k, f)
    idx, _ = oracle.route_topk(l.astype(np.float32), k)
    _, offsets, src, _ = oracle.dispatch(idx, E)
    xp = oracle.permute(x, src)
    gate, up = oracle.expert_gate_up(xp, offsets, wg, wu)
    h, _ = oracle.expert_mlp(xp, offsets, wg, wu, wd)
    np.testing.assert_allclose(oracle.silu(gate) * up, h, rtol=1e-13, atol=1e-14)
    dy = _rng(72).standard_normal((T * k, d))
    dx, _, _, _, dG, dU = oracle.expert_mlp_backward(xp, offsets, wg, wu, wd, dy, return_preact_grads=True)
    ref = np.zeros_like(dx)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        ref[a:b] = dG[a:b] @ wg[e].T + dU[a:b] @ wu[e].T
    np.testing.assert_allclose(dx, ref, rtol=1e-12, atol=1e-13)
