"""Plant a plausible mistake in the CPU oracle (never in the CUDA path) and check
that at least one pin of ``test_oracle_pins`` catches it."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_oracle
from tests.test_oracle_pins import PINS
from tests.test_oracle_sigmoid_pins import SIGMOID_PINS

_route = moe_oracle.route
_dispatch = moe_oracle.dispatch
_combine = moe_oracle.combine
_rows = moe_oracle._swiglu_rows
_grouped = moe_oracle.route_sigmoid_grouped


def _route_ignoring_renormalize(logits, top_k, renormalize, out_dtype=None):
    return _route(logits, top_k, False, out_dtype)


def _route_ties_to_higher_id(logits, top_k, renormalize, out_dtype=None):
    rt = _route(torch.flip(logits, dims=[1]), top_k, renormalize, out_dtype)
    E = logits.shape[1]
    rt.indices = (E - 1 - rt.indices.astype(np.int64)).astype(np.uint32)
    return rt


def _route_ascending_slots(logits, top_k, renormalize, out_dtype=None):
    rt = _route(logits, top_k, renormalize, out_dtype)
    rt.indices = rt.indices[:, ::-1].copy()
    rt.weights32 = rt.weights32[:, ::-1].copy()
    rt.weights = rt.weights[:, ::-1].copy()
    rt.weights64 = rt.weights64[:, ::-1].copy()
    return rt


def _route_uniform_fallback(logits, top_k, renormalize, out_dtype=None):
    rt = _route(logits, top_k, renormalize, out_dtype)
    E = logits.shape[1]
    for arr in (rt.weights32, rt.weights, rt.weights64):
        arr[rt.bad] = 1.0 / (top_k if renormalize else E)
    return rt


def _dispatch_descending(indices, E):
    d = _dispatch(indices, E)
    for e in range(E):
        lo, hi = int(d.offsets[e]), int(d.offsets[e + 1])
        d.row_src[lo:hi] = d.row_src[lo:hi][::-1].copy()
    d.inv[d.row_src] = np.arange(len(d.row_src), dtype=np.uint32)
    return d


def _dispatch_inclusive_offsets(indices, E):
    d = _dispatch(indices, E)
    d.offsets = np.concatenate([d.offsets[1:], d.offsets[-1:]])
    return d


def _combine_unweighted(y, inv, weights, T, top_k):
    return _combine(y, inv, np.where(np.isnan(weights), np.nan, 1.0), T, top_k)


def _combine_with_row_src(y, inv, weights, T, top_k):
    order = np.argsort(np.asarray(inv, dtype=np.int64))
    return _combine(y, order.astype(np.uint32), weights, T, top_k)


def _rows_swap_gate_up(x, gate, up, down):
    return _rows(x, up, gate, down)


def _rows_drop_up(x, gate, up, down):
    g = x @ gate.T
    return moe_oracle.silu(g) @ down.T


def _silu_wrong_sign(g):
    return g / (1.0 + np.exp(g))


def _forward_expert0_down(x, logits, gate, up, down, top_k, renormalize):
    down0 = down[0:1].expand_as(down) if isinstance(down, torch.Tensor) else np.broadcast_to(down[0:1], down.shape)
    return moe_oracle.__dict__["_forward_orig"](x, logits, gate, up, down0, top_k, renormalize)


def _grouped_with(**changes):
    def fn(logits, bias, o, out_dtype=None):
        return _grouped(logits, bias, dataclasses.replace(o, **changes), out_dtype)
    return fn


def _grouped_no_group_limit(logits, bias, o, out_dtype=None):
    return _grouped(logits, bias, dataclasses.replace(o, groups=1, selected_groups=1, group_top_two=False),
                    out_dtype)


def _grouped_bias_ignored(logits, bias, o, out_dtype=None):
    return _grouped(logits, None, o, out_dtype)


def _grouped_bias_in_weights(logits, bias, o, out_dtype=None):
    rt = _grouped(logits, bias, o, out_dtype)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32)[rt.indices.astype(np.int64)]
        rt.weights32 = (rt.weights32 + b).astype(np.float32)
        rt.weights64 = rt.weights64 + b
    return rt


def _grouped_sigmoid_wrong_sign(logits, bias, o, out_dtype=None):
    return _grouped(-logits, bias, o, out_dtype)


MUTATIONS = {
    "no_renormalize": ("route", _route_ignoring_renormalize),
    "ties_to_higher_id": ("route", _route_ties_to_higher_id),
    "ascending_slot_order": ("route", _route_ascending_slots),
    "uniform_fallback_on_nonfinite": ("route", _route_uniform_fallback),
    "dispatch_descending_within_expert": ("dispatch", _dispatch_descending),
    "dispatch_inclusive_offsets": ("dispatch", _dispatch_inclusive_offsets),
    "combine_ignores_weights": ("combine", _combine_unweighted),
    "combine_indexes_with_row_src": ("combine", _combine_with_row_src),
    "swap_gate_and_up": ("_swiglu_rows", _rows_swap_gate_up),
    "drop_up_projection": ("_swiglu_rows", _rows_drop_up),
    "silu_wrong_sign": ("silu", _silu_wrong_sign),
    "every_expert_uses_down_of_expert_0": ("forward", _forward_expert0_down),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setitem(moe_oracle.__dict__, "_forward_orig", moe_oracle.forward)
    monkeypatch.setattr(moe_oracle, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin(moe_oracle)
        except Exception as exc:  # an assertion or a shape error both count
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin catches the planted mistake {name!r}"


SIGMOID_MUTATIONS = {
    "grouped_ignores_renormalize": _grouped_with(renormalize=False),
    "grouped_ignores_scale": _grouped_with(scale=1.0),
    "grouped_max_instead_of_top_two": _grouped_with(group_top_two=False),
    "grouped_no_group_limit": _grouped_no_group_limit,
    "grouped_bias_ignored": _grouped_bias_ignored,
    "grouped_bias_in_weights": _grouped_bias_in_weights,
    "grouped_sigmoid_wrong_sign": _grouped_sigmoid_wrong_sign,
}


@pytest.mark.parametrize("name", sorted(SIGMOID_MUTATIONS))
def test_planted_routing_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(moe_oracle, "route_sigmoid_grouped", SIGMOID_MUTATIONS[name])
    caught = []
    for pin in SIGMOID_PINS:
        try:
            pin(moe_oracle)
        except Exception as exc:
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin catches the planted mistake {name!r}"


# ---------------------------------------------------------------- training oracle
from oracle import training as _training  # noqa: E402
from tests.test_oracle_training_pins import TRAINING_PINS  # noqa: E402

_jac = _training.router_jacobian
_cb = _training.combine_backward
_eb = _training.experts_backward
_db = _training.dispatch_backward


def _jac_without_softmax_cross_term(l64_row, idx_row, o):
    if o.scoring != "softmax":
        return _jac(l64_row, idx_row, o)
    ex = np.exp(l64_row - l64_row.max())
    P = ex / ex.sum()
    J = np.zeros((idx_row.size, l64_row.size))
    J[np.arange(idx_row.size), idx_row] = P[idx_row]        # drops -P_i P_m
    if o.renormalize:
        v = P[idx_row]
        Z = v.sum()
        J = (J * Z - np.outer(v, J.sum(axis=0))) / (Z * Z)
    return J * float(o.scale)


def _jac_ignoring_scale(l64_row, idx_row, o):
    return _jac(l64_row, idx_row, dataclasses.replace(o, scale=1.0))


def _jac_renorm_sign_flipped(l64_row, idx_row, o):
    if not o.renormalize:
        return _jac(l64_row, idx_row, o)
    J0 = _jac(l64_row, idx_row, dataclasses.replace(o, renormalize=False, scale=1.0))
    ex = np.exp(l64_row - l64_row.max())
    P = ex / ex.sum() if o.scoring == "softmax" else 1 / (1 + np.exp(-l64_row))
    v = P[idx_row]
    Z = v.sum()
    return (J0 * Z + np.outer(v, J0.sum(axis=0))) / (Z * Z) * float(o.scale)


def _combine_backward_unweighted(y, inv, weights, grad_out, T, top_k):
    return _cb(y, inv, np.ones_like(np.asarray(weights, dtype=np.float64)), grad_out, T, top_k)


def _experts_backward_silu_for_derivative(x, gate, up, down, offsets, dexpert):
    saved = _training._silu_grad
    _training._silu_grad = _training._silu
    try:
        return _eb(x, gate, up, down, offsets, dexpert)
    finally:
        _training._silu_grad = saved


def _experts_backward_swapped_gate_up(x, gate, up, down, offsets, dexpert):
    g = _eb(x, up, gate, down, offsets, dexpert)
    return _training.ExpertGrads(g.dx_dispatched, g.dup, g.dgate, g.ddown)


_tfc = _training.training_forward_cache


def _training_cache_gate_up_swapped(x, gate, up, offsets):
    return _tfc(x, up, gate, offsets)


def _training_cache_h_from_up(x, gate, up, offsets):
    g, u, _ = _tfc(x, gate, up, offsets)
    return g, u, _training._silu(u) * g


def _dispatch_backward_mean(dinput, inv, T, top_k):
    return _db(dinput, inv, T, top_k) / top_k


TRAINING_MUTATIONS = {
    "softmax_jacobian_without_cross_term": ("router_jacobian", _jac_without_softmax_cross_term),
    "router_backward_ignores_scale": ("router_jacobian", _jac_ignoring_scale),
    "renormalize_quotient_rule_sign": ("router_jacobian", _jac_renorm_sign_flipped),
    "combine_backward_drops_weight": ("combine_backward", _combine_backward_unweighted),
    "silu_used_for_its_derivative": ("experts_backward", _experts_backward_silu_for_derivative),
    "gate_and_up_gradients_swapped": ("experts_backward", _experts_backward_swapped_gate_up),
    "dispatch_backward_averages_slots": ("dispatch_backward", _dispatch_backward_mean),
    "training_cache_gate_up_swapped": ("training_forward_cache", _training_cache_gate_up_swapped),
    "training_cache_silu_of_up": ("training_forward_cache", _training_cache_h_from_up),
}


@pytest.mark.parametrize("name", sorted(TRAINING_MUTATIONS))
def test_planted_training_mistake_is_caught(name, monkeypatch):
    import oracle as pkg

    attr, fn = TRAINING_MUTATIONS[name]
    monkeypatch.setattr(_training, attr, fn)
    if hasattr(pkg, attr):
        monkeypatch.setattr(pkg, attr, fn)
    caught = []
    for pin in TRAINING_PINS:
        try:
            pin(pkg)
        except Exception as exc:
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin catches the planted mistake {name!r}"
