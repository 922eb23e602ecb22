"""Pins for the oracle's grouped, bias-corrected sigmoid routing (ruDNN user
guide, section 10): closed forms, hand-worked group choices, brute force,
and the DeepSeek-style restatement in "PyTorch general ops" (group max,
top groups, mask, top-k). Each pin is a function of the oracle module so the
planted-mistake tests can reuse it."""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle

Opt = moe_oracle.GroupRoutingOptions


def _logit(p):
    return math.log(p / (1.0 - p))


def pin_sigmoid_closed_form(m):
    """logits ln(p / (1 - p)) give sigmoid scores p: the weights are p * scale,
    or p / sum(p) * scale when renormalized (FP32 within 1e-6)."""
    p = np.array([0.9, 0.2, 0.75, 0.6, 0.35, 0.5])
    l = torch.tensor([[_logit(v) for v in p]], dtype=torch.float32)
    for renorm, scale in [(False, 1.0), (False, 2.5), (True, 1.0), (True, 0.5)]:
        rt = m.route_sigmoid_grouped(l, None, Opt(3, 1, 1, False, renorm, scale))
        assert rt.indices[0].tolist() == [0, 2, 3]
        want = p[[0, 2, 3]]
        want = want / want.sum() * scale if renorm else want * scale
        np.testing.assert_allclose(rt.weights32[0], want, rtol=1e-6)
        np.testing.assert_allclose(rt.weights64[0], want, rtol=2e-7)


def pin_bias_steers_selection_only(m):
    """scores [0.9, 0.8, 0.7, 0.6] with bias [0, 0, 0.5, 0]: corrected
    [0.9, 0.8, 1.2, 0.6] picks experts [2, 0], but the weights are the
    uncorrected scores [0.7, 0.9]."""
    l = torch.tensor([[_logit(v) for v in (0.9, 0.8, 0.7, 0.6)]], dtype=torch.float32)
    b = torch.tensor([0.0, 0.0, 0.5, 0.0])
    rt = m.route_sigmoid_grouped(l, b, Opt(2, 1, 1, False, False, 1.0))
    assert rt.indices[0].tolist() == [2, 0]
    np.testing.assert_allclose(rt.weights32[0], [0.7, 0.9], rtol=1e-6)
    rt = m.route_sigmoid_grouped(l, None, Opt(2, 1, 1, False, False, 1.0))
    assert rt.indices[0].tolist() == [0, 1]


def pin_group_max_versus_top_two(m):
    """Four groups of two. Scores g0 [0.9, 0.1], g1 [0.6, 0.6], g2 [0.5, 0.5],
    g3 [0.2, 0.3]: one group by max picks g0 (0.9 > 0.6); by the top-two sum
    it picks g1 (1.2 > 1.0); top-2 experts then come from that group only."""
    s = [0.9, 0.1, 0.6, 0.6, 0.5, 0.5, 0.2, 0.3]
    l = torch.tensor([[_logit(v) for v in s]], dtype=torch.float32)
    rt = m.route_sigmoid_grouped(l, None, Opt(2, 4, 1, False, False, 1.0))
    assert rt.indices[0].tolist() == [0, 1]
    rt = m.route_sigmoid_grouped(l, None, Opt(2, 4, 1, True, False, 1.0))
    assert rt.indices[0].tolist() == [2, 3]                  # equal scores: lower id first
    rt = m.route_sigmoid_grouped(l, None, Opt(3, 4, 2, True, False, 1.0))
    assert rt.indices[0].tolist() == [0, 2, 3]                # groups g1 and g0


def pin_one_group_equals_plain_topk(m):
    """groups = 1, no bias: sigmoid is increasing, so the selection equals the
    softmax routing's top-k of the logits (an independent statement of the
    same order, ties to the lower id)."""
    rng = np.random.default_rng(23)
    l = torch.from_numpy((np.round(rng.standard_normal((300, 40)) * 4) / 4).astype(np.float32))
    for k in (1, 5, 16):
        a = m.route_sigmoid_grouped(l, None, Opt(k, 1, 1, False, True, 1.0))
        b = m.route(l, k, True)
        assert np.array_equal(a.indices, b.indices)


def pin_renormalized_sum_is_scale(m):
    rng = np.random.default_rng(29)
    l = torch.from_numpy(rng.standard_normal((200, 64)).astype(np.float32))
    for scale in (1.0, 2.5):
        rt = m.route_sigmoid_grouped(l, None, Opt(6, 8, 3, True, True, scale))
        np.testing.assert_allclose(rt.weights32.astype(np.float64).sum(1), scale, rtol=2e-6)


def _brute(c, o):
    """Exhaustive: the best selected_groups-subset of groups (ordered by group
    score desc, id asc), then the best ordered k-tuple of experts inside."""
    E = len(c)
    G = E // o.groups
    gs = []
    for g in range(o.groups):
        vals = sorted(c[g * G:(g + 1) * G], reverse=True)
        gs.append(np.float32(np.float32(vals[0]) + np.float32(vals[1])) if o.group_top_two else vals[0])
    best_g, best_key = None, None
    for tup in itertools.permutations(range(o.groups), o.selected_groups):
        key = tuple(v for g in tup for v in (gs[g], -g))
        if best_key is None or key > best_key:
            best_g, best_key = tup, key
    allowed = [i for i in range(E) if i // G in best_g]
    best_e, best_key = None, None
    for tup in itertools.permutations(allowed, o.top_k):
        key = tuple(v for i in tup for v in (c[i], -i))
        if best_key is None or key > best_key:
            best_e, best_key = tup, key
    return list(best_e)


def pin_brute_force_grouped_selection(m):
    """Tiny rows full of ties (quantised scores, a quantised bias) against an
    exhaustive search over group subsets and expert tuples."""
    rng = np.random.default_rng(31)
    for E, groups in [(4, 2), (6, 3), (6, 2), (8, 4), (6, 1)]:
        G = E // groups
        for sel in range(1, groups + 1):
            for top_two in ([False, True] if G >= 2 else [False]):
                for k in range(1, min(sel * G, 4) + 1):
                    o = Opt(k, groups, sel, top_two, False, 1.0)
                    p = rng.choice([0.25, 0.5, 0.75], size=(6, E))
                    l = torch.tensor(np.log(p / (1 - p)), dtype=torch.float32)
                    b = torch.tensor(rng.choice([0.0, 0.25, 0.0, 0.25, -np.inf], size=E), dtype=torch.float32)
                    rt = m.route_sigmoid_grouped(l, b, o)
                    s = (np.float32(1) / (np.float32(1) + np.exp(-l.numpy().astype(np.float64)).astype(np.float32))
                         ).astype(np.float32)
                    c = (s + b.numpy()).astype(np.float32)
                    for t in range(6):
                        assert rt.indices[t].tolist() == _brute(c[t].tolist(), o), (E, groups, sel, top_two, k)


def pin_deepseek_style_restatement(m):
    """The grouped top-k of "PyTorch general ops": group max (view + max),
    top groups (topk), group mask expanded to experts, masked_fill(0), topk,
    then the FP32-summed renormalize, restated in f64 with torch ops on
    tie-free scores (no bias, max variant)."""
    rng = np.random.default_rng(37)
    T, E, groups, sel, k = 64, 32, 8, 3, 4
    l = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32))
    rt = m.route_sigmoid_grouped(l, None, Opt(k, groups, sel, False, True, 1.0))
    scores = torch.sigmoid(l.double())
    group_scores = scores.view(T, groups, -1).max(dim=-1).values
    group_idx = torch.topk(group_scores, k=sel, dim=-1).indices
    group_mask = torch.zeros_like(group_scores).scatter_(1, group_idx, 1)
    score_mask = group_mask.unsqueeze(-1).expand(T, groups, E // groups).reshape(T, -1)
    tmp = scores.masked_fill(~score_mask.bool(), 0.0)
    w, ids = torch.topk(tmp, k=k, dim=-1)
    w = w / w.sum(dim=-1, keepdim=True)
    assert np.array_equal(rt.indices.astype(np.int64), ids.numpy())
    np.testing.assert_allclose(rt.weights32, w.numpy(), rtol=2e-6)


def pin_minus_inf_bias_stays_in_its_group(m):
    """An expert of a selected group whose bias is -inf still ranks ahead of
    every expert outside the selected groups: scores [0.5, 0.5 | 0.9, s3]
    with bias [0, 0, 0, -inf], one group of two by max, top-2 -> [2, 3]."""
    l = torch.tensor([[0.0, 0.0, _logit(0.9), 0.3]])
    b = torch.tensor([0.0, 0.0, 0.0, -np.inf], dtype=torch.float32)
    rt = m.route_sigmoid_grouped(l, b, Opt(2, 2, 1, False, False, 1.0))
    assert rt.indices[0].tolist() == [2, 3]
    assert np.isfinite(rt.weights32[0]).all()


def pin_sigmoid_nan_rows(m):
    """Reading: a NaN logit makes the row's weights NaN (indices 0..k-1);
    +inf and -inf logits are finite scores 1 and 0."""
    l = torch.tensor([[0.5, float("nan"), 0.0, 1.0], [float("inf"), float("-inf"), 0.0, 1.0]])
    rt = m.route_sigmoid_grouped(l, None, Opt(2, 2, 2, False, False, 1.0))
    assert np.isnan(rt.weights32[0]).all() and rt.indices[0].tolist() == [0, 1]
    assert rt.indices[1].tolist() == [0, 3] and rt.weights32[1, 0] == 1.0


def pin_option_ranges(m):
    bad = [Opt(0, 1, 1, False, True, 1.0), Opt(65, 1, 1, False, True, 1.0), Opt(2, 3, 1, False, True, 1.0),
           Opt(2, 2, 3, False, True, 1.0), Opt(5, 4, 1, False, True, 1.0), Opt(1, 8, 1, True, True, 1.0),
           Opt(2, 2, 1, False, True, 0.0), Opt(2, 2, 1, False, True, float("inf")), Opt(2, 129, 1, False, True, 1.0)]
    for o in bad:
        with pytest.raises(ValueError):
            m.check_group_options(8, o)
    m.check_group_options(8, Opt(4, 2, 1, True, True, 1.0))


def pin_grouped_forward_per_token(m):
    """The grouped-routing forward equals, token by token, the sum over its
    slots of weight * down(SiLU(gate x) * (up x)) written out with explicit
    loops (f64), and the sampled-token form agrees with the whole batch."""
    rng = np.random.default_rng(41)
    T, H, I, E = 9, 6, 5, 8
    x = torch.from_numpy(rng.standard_normal((T, H)))
    gate = torch.from_numpy(rng.standard_normal((E, I, H)) * 0.5)
    up = torch.from_numpy(rng.standard_normal((E, I, H)) * 0.5)
    down = torch.from_numpy(rng.standard_normal((E, H, I)) * 0.5)
    l = torch.from_numpy(rng.standard_normal((T, E)))
    b = torch.from_numpy(rng.standard_normal(E).astype(np.float32) * 0.1)
    o = Opt(3, 4, 2, True, True, 1.5)
    rt = m.route_sigmoid_grouped(l, b, o, out_dtype=torch.float64)
    fr = m.forward_with_routing(x, gate, up, down, rt)
    X, G, U, D = (a.numpy() for a in (x, gate, up, down))
    for t in range(T):
        want = np.zeros(H)
        for j in range(3):
            e = int(rt.indices[t, j])
            h = [0.0] * I
            for i in range(I):
                g = sum(G[e, i, c] * X[t, c] for c in range(H))
                u = sum(U[e, i, c] * X[t, c] for c in range(H))
                h[i] = g / (1.0 + math.exp(-g)) * u
            for c in range(H):
                want[c] += rt.weights[t, j] * sum(D[e, c, i] * h[i] for i in range(I))
        np.testing.assert_allclose(fr.out[t], want, rtol=1e-12, atol=1e-12)
    toks = np.array([7, 2, 5])
    part = m.forward_tokens_routed(x, gate, up, down, m.route_sigmoid_grouped(l[toks], b, o, torch.float64), toks)
    np.testing.assert_allclose(part, fr.out[toks], rtol=1e-12, atol=1e-12)


SIGMOID_PINS = [
    pin_sigmoid_closed_form,
    pin_bias_steers_selection_only,
    pin_group_max_versus_top_two,
    pin_one_group_equals_plain_topk,
    pin_renormalized_sum_is_scale,
    pin_brute_force_grouped_selection,
    pin_deepseek_style_restatement,
    pin_minus_inf_bias_stays_in_its_group,
    pin_sigmoid_nan_rows,
    pin_option_ranges,
    pin_grouped_forward_per_token,
]


@pytest.mark.parametrize("pin", SIGMOID_PINS, ids=[p.__name__ for p in SIGMOID_PINS])
def test_sigmoid_oracle_pin(pin):
    pin(moe_oracle)
