"""Planted mistakes in the oracle must be caught by its pins.

Each test swaps one oracle step for a plausibly wrong variant (on the CPU,
through monkeypatch) and checks that a pin of tests/test_oracle_pins.py
then fails.  This shows the pins are sensitive to a dropped term, a wrong
order or sign, and a transposed operand.
"""
import numpy as np
import pytest

import oracle
import oracle.moe_oracle as om
from tests import test_oracle_pins as pins
from tests.conftest import load_golden


def _fails(fn, *args, **kw):
    with pytest.raises((AssertionError, ValueError)):
        fn(*args, **kw)


def test_silu_without_input_factor_is_caught(monkeypatch):
    monkeypatch.setattr(om, "silu", lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64))))
    _fails(pins.test_swiglu_scalar_golden, load_golden)
    _fails(pins.test_layer_matches_per_token_brute_force, 21, 16, 6, 2, 24, True)


def test_silu_wrong_sign_is_caught(monkeypatch):
    monkeypatch.setattr(om, "silu", lambda z: np.asarray(z) / (1.0 + np.exp(np.asarray(z, dtype=np.float64))))
    _fails(pins.test_swiglu_scalar_golden, load_golden)


def test_dropped_up_projection_is_caught(monkeypatch):
    real = om.expert_mlp

    def no_up(x_perm, offsets, w_gate, w_up, w_down, experts=None):
        return real(x_perm, offsets, w_gate, np.ones_like(w_up) / w_up.shape[1], w_down, experts)
    monkeypatch.setattr(om, "expert_mlp", no_up)
    _fails(pins.test_single_expert_layer_is_dense_swiglu_mlp)


def test_transposed_down_projection_is_caught(monkeypatch):
    real = om.expert_mlp

    def transposed(x_perm, offsets, w_gate, w_up, w_down, experts=None):
        wd = np.ascontiguousarray(np.transpose(w_down, (0, 2, 1)))
        if wd.shape[1] != w_gate.shape[2]:
            raise ValueError("shape mismatch")
        return real(x_perm, offsets, w_gate, w_up, wd, experts)
    monkeypatch.setattr(om, "expert_mlp", transposed)
    _fails(pins.test_layer_matches_per_token_brute_force, 12, 8, 4, 4, 8, True)


def test_reversed_tie_break_is_caught(monkeypatch):
    def bad_route(logits, k, renormalize=True):
        l32 = np.asarray(logits, dtype=np.float32)
        E = l32.shape[1]
        order = (E - 1 - np.argsort(-l32[:, ::-1], axis=1, kind="stable"))  # ties -> larger index
        idx = order[:, :k].astype(np.int32)
        w = np.take_along_axis(om.softmax_rows(l32), idx.astype(np.int64), axis=1)
        return idx, (w / w.sum(axis=1, keepdims=True) if renormalize else w)
    monkeypatch.setattr(om, "route_topk", bad_route)
    import oracle
    monkeypatch.setattr(oracle, "route_topk", bad_route)
    _fails(pins.test_route_indices_match_brute_force, 40, 8, 8, True)
    _fails(pins.test_route_golden, load_golden)


def test_missing_renormalisation_is_caught(monkeypatch):
    real = om.route_topk
    import oracle
    monkeypatch.setattr(oracle, "route_topk", lambda l, k, renormalize=True: real(l, k, False))
    _fails(pins.test_route_weights_closed_form, True)


def test_unstable_group_order_is_caught(monkeypatch):
    import oracle
    real = om.dispatch

    def bad_dispatch(idx, E):
        counts, offsets, src, dst = real(idx, E)
        # reverse the rows inside every expert group
        new_dst = dst.copy()
        for e in range(E):
            a, b = offsets[e], offsets[e + 1]
            sel = (dst >= a) & (dst < b)
            new_dst[sel] = a + b - 1 - dst[sel]
        new_src = np.empty_like(src)
        new_src[new_dst] = np.arange(len(new_dst)) // idx.shape[1]
        return counts, offsets, new_src, new_dst
    monkeypatch.setattr(oracle, "dispatch", bad_dispatch)
    _fails(pins.test_dispatch_matches_alg1_thread_blocks, 64, 16, 4, 8)
    _fails(pins.test_index_golden_matches_hand_example, load_golden)


def test_combine_without_gates_is_caught(monkeypatch):
    import oracle
    real = om.combine
    monkeypatch.setattr(oracle, "combine", lambda y, dest_row, w: real(y, dest_row, np.ones_like(w)))
    _fails(pins.test_combine_of_identity_experts_returns_input)


def test_grouped_route_ignoring_groups_is_caught(monkeypatch):
    import oracle
    real = om.route_topk
    monkeypatch.setattr(oracle, "route_topk_grouped", lambda l, k, G, renormalize=True: real(l, k, renormalize))
    _fails(pins.test_grouped_route_balances_the_groups)
    _fails(pins.test_grouped_route_golden, load_golden)


def test_router_with_transposed_weights_is_caught(monkeypatch):
    import oracle
    real = om.router_topk
    monkeypatch.setattr(oracle, "router_topk", lambda x, w, k, renormalize=True: real(x, np.asarray(w)[::-1], k,
                                                                                       renormalize))
    _fails(pins.test_router_logits_match_per_token_dot_products)
    _fails(pins.test_router_with_one_hot_tokens_selects_router_rows)


def test_fp8_round_half_up_is_caught(monkeypatch):
    from oracle import fp8_oracle as f8
    from tests import test_fp8_oracle as fp8_pins
    real = f8.e4m3_round

    def half_up(x):
        x = np.asarray(x, dtype=np.float32).astype(np.float64)
        a = np.abs(x)
        _, e2 = np.frexp(a)
        q = np.exp2(np.maximum(e2 - 1, -6) - 3.0)
        r = np.minimum(np.floor(a / q + 0.5) * q, 448.0)
        return np.where(np.signbit(x), -r, r).astype(np.float32)
    monkeypatch.setattr(f8, "e4m3_round", half_up)
    _fails(fp8_pins.test_rounding_matches_torch_including_every_tie)
    monkeypatch.setattr(f8, "e4m3_round", real)


def test_fp8_wrong_scale_range_is_caught(monkeypatch):
    from oracle import fp8_oracle as f8
    from tests import test_fp8_oracle as fp8_pins
    monkeypatch.setattr(f8, "E4M3_MAX", 240.0)
    _fails(fp8_pins.test_blockwise_scale_puts_the_block_maximum_at_448)


def test_combine_backward_without_gate_is_caught(monkeypatch):
    real = om.combine_backward

    def no_gate(dout, mlp_out, dest_row, w):
        dy, dw = real(dout, mlp_out, dest_row, np.ones_like(np.asarray(w, dtype=np.float64)))
        return dy, dw
    monkeypatch.setattr(oracle, "combine_backward", no_gate)
    _fails(pins.test_combine_backward_matches_finite_differences)
    _fails(pins.test_combine_backward_golden_scalar)


def test_route_backward_wrong_sign_is_caught(monkeypatch):
    real = om.route_backward

    def flipped(logits, idx, dw, renormalize=True):
        g = real(logits, idx, dw, renormalize)
        base = real(logits, idx, np.zeros_like(np.asarray(dw, dtype=np.float64)), renormalize)
        return 2 * base - g          # negates the whole gradient
    monkeypatch.setattr(oracle, "route_backward", flipped)
    _fails(pins.test_route_backward_matches_finite_differences, True)
    _fails(pins.test_route_backward_matches_finite_differences, False)


def test_route_backward_softmax_over_wrong_set_is_caught(monkeypatch):
    real = om.route_backward

    def other_set(logits, idx, dw, renormalize=True):
        return real(logits, idx, dw, not renormalize)
    monkeypatch.setattr(oracle, "route_backward", other_set)
    _fails(pins.test_route_backward_matches_finite_differences, True)
    _fails(pins.test_route_backward_matches_finite_differences, False)


def test_silu_grad_without_product_term_is_caught(monkeypatch):
    sigmoid_only = lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))  # noqa: E731
    monkeypatch.setattr(om, "silu_grad", sigmoid_only)
    monkeypatch.setattr(oracle, "silu_grad", sigmoid_only)
    _fails(pins.test_layer_backward_matches_finite_differences, True)
    _fails(pins.test_silu_grad_matches_finite_differences_and_limits)


def test_unpermute_overwriting_instead_of_adding_is_caught(monkeypatch):
    real = om.expert_mlp_backward

    def dropped(x_perm, offsets, w_gate, w_up, w_down, dy):
        dx, dwg, dwu, dwd = real(x_perm, offsets, w_gate, w_up, w_down, dy)
        return dx * 0.5, dwg, dwu, dwd     # as if one of two slots were lost
    monkeypatch.setattr(om, "expert_mlp_backward", dropped)
    _fails(pins.test_layer_backward_matches_finite_differences, False)


def test_up_gradient_with_wrong_factor_is_caught(monkeypatch):
    real = om.expert_mlp_backward

    def wrong(x_perm, offsets, w_gate, w_up, w_down, dy):
        # dU = dH * up instead of dH * Silu(gate): swap the roles of gate and up
        return real(x_perm, offsets, w_up, w_gate, w_down, dy)
    monkeypatch.setattr(om, "expert_mlp_backward", wrong)
    _fails(pins.test_layer_backward_scalar_closed_form)
