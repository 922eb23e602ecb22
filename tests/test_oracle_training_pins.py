"""Pins for the training oracle (ruDNN user guide, section 12): closed forms,
finite differences of the oracle's own forward definitions, invariants of
the softmax and sigmoid Jacobians, brute force on the maps, and one f64
torch-autograd restatement of the whole chain. Each pin is a function of the
oracle package so the planted-mistake tests can reuse it."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle

Opt = oracle.RouterWeightOptions
VARIANTS = [Opt("softmax", False, 1.0), Opt("softmax", True, 1.0), Opt("sigmoid", False, 1.5),
            Opt("sigmoid", True, 2.5)]


def _logit(p):
    return math.log(p / (1.0 - p))


def _quarter_logits(rng, T, E):
    """Logits on a 1/256 grid within [-4, 4]: exact in FP32, and exact after
    the +-2^-10 steps the finite differences take."""
    return np.round(rng.uniform(-4, 4, size=(T, E)) * 256) / 256


def pin_router_softmax_matches_forward_routing(m):
    """Softmax weights of the selection the forward routing made equal the
    forward routing's FP32 weights exactly (the same FP32 operations)."""
    rng = np.random.default_rng(3)
    l = torch.from_numpy(rng.standard_normal((64, 12)).astype(np.float32))
    for renorm in (False, True):
        rt = moe_oracle.route(l, 4, renorm)
        w32, _ = m.selected_router_weights(l, rt.indices, Opt("softmax", renorm, 1.0))
        assert np.array_equal(w32, rt.weights32)


def pin_router_sigmoid_closed_form(m):
    p = np.array([0.9, 0.2, 0.75, 0.6])
    l = torch.tensor([[_logit(v) for v in p]], dtype=torch.float32)
    idx = np.array([[2, 0, 3]])
    w32, _ = m.selected_router_weights(l, idx, Opt("sigmoid", False, 2.0))
    np.testing.assert_allclose(w32[0], 2.0 * p[[2, 0, 3]], rtol=1e-6)
    w32, _ = m.selected_router_weights(l, idx, Opt("sigmoid", True, 1.0))
    np.testing.assert_allclose(w32[0], p[[2, 0, 3]] / p[[2, 0, 3]].sum(), rtol=1e-6)


def pin_router_duplicate_indices_gather(m):
    """A repeated index is gathered twice: equal weights, and renormalize
    counts it twice (one expert selected twice renormalizes to 1/2, 1/2)."""
    l = torch.tensor([[0.3, -1.0, 2.0]])
    for sc in ("softmax", "sigmoid"):
        w32, _ = m.selected_router_weights(l, np.array([[2, 2]]), Opt(sc, True, 1.0))
        assert w32[0].tolist() == [0.5, 0.5]
        w32, _ = m.selected_router_weights(l, np.array([[2, 0, 2]]), Opt(sc, False, 1.0))
        assert w32[0, 0] == w32[0, 2]


def pin_router_invalid_index_nan_row(m):
    l = torch.tensor([[0.3, -1.0, 2.0], [1.0, 2.0, 3.0]])
    idx = np.array([[0, 3], [1, 2]])
    g = torch.ones(2, 2)
    for o in VARIANTS:
        w32, _ = m.selected_router_weights(l, idx, o)
        assert np.isnan(w32[0]).all() and np.isfinite(w32[1]).all()
        d64, _ = m.selected_router_backward(l, idx, g, o)
        assert np.isnan(d64[0]).all() and np.isfinite(d64[1]).all()


def pin_router_backward_finite_differences(m):
    """Central differences of the oracle's f64 weights (step 2^-10) against
    J^T g, all four scoring/renormalize variants, with repeated indices."""
    rng = np.random.default_rng(5)
    T, E, k = 3, 5, 3
    l = _quarter_logits(rng, T, E)
    idx = np.array([[0, 3, 3], [4, 1, 2], [2, 2, 0]])
    g = rng.standard_normal((T, k)).astype(np.float32)
    h = 2.0 ** -10
    for o in VARIANTS:
        d64, _ = m.selected_router_backward(torch.from_numpy(l.astype(np.float32)), idx, torch.from_numpy(g), o)
        fd = np.zeros((T, E))
        for t in range(T):
            for e in range(E):
                lp, lm = l.copy(), l.copy()
                lp[t, e] += h
                lm[t, e] -= h
                _, wp = m.selected_router_weights(torch.from_numpy(lp.astype(np.float32)), idx, o)
                _, wm = m.selected_router_weights(torch.from_numpy(lm.astype(np.float32)), idx, o)
                fd[t, e] = float(((wp[t] - wm[t]) / (2 * h)) @ g[t].astype(np.float64))
        np.testing.assert_allclose(d64, fd, rtol=1e-5, atol=1e-7)


def pin_router_backward_invariants(m):
    """Softmax weights do not change when every logit of a row shifts by the
    same amount, so each dlogits row sums to 0; sigmoid weights depend only on
    the selected logits, so dlogits is 0 elsewhere; the gradient is linear in
    scale."""
    rng = np.random.default_rng(7)
    l = torch.from_numpy(rng.standard_normal((20, 9)).astype(np.float32))
    idx = np.stack([rng.choice(9, size=4, replace=False) for _ in range(20)])
    g = torch.from_numpy(rng.standard_normal((20, 4)).astype(np.float32))
    for renorm in (False, True):
        d64, _ = m.selected_router_backward(l, idx, g, Opt("softmax", renorm, 1.0))
        np.testing.assert_allclose(d64.sum(axis=1), 0.0, atol=1e-12)
        d64, _ = m.selected_router_backward(l, idx, g, Opt("sigmoid", renorm, 1.0))
        mask = np.zeros((20, 9), dtype=bool)
        np.put_along_axis(mask, idx, True, axis=1)
        assert np.all(d64[~mask] == 0.0) and np.any(d64[mask] != 0.0)
        a, _ = m.selected_router_backward(l, idx, g, Opt("sigmoid", renorm, 1.0))
        b, _ = m.selected_router_backward(l, idx, g, Opt("sigmoid", renorm, 2.5))
        np.testing.assert_allclose(b, 2.5 * a, rtol=1e-14)


def pin_combine_backward_finite_differences(m):
    """d<G, out>/dy and d<G, out>/dw by central differences of the forward
    combine (moe_oracle.combine), which is linear in both."""
    rng = np.random.default_rng(11)
    T, k, H = 4, 2, 3
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1]])
    dp = moe_oracle.dispatch(idx, 3)
    n = T * k
    y = rng.standard_normal((n, H))
    w = rng.standard_normal((T, k))
    G = rng.standard_normal((T, H))
    dexp, dw = m.combine_backward(torch.from_numpy(y), dp.inv, w, torch.from_numpy(G), T, k)
    h = 1e-3
    for r in range(n):
        for c in range(H):
            yp, ym = y.copy(), y.copy()
            yp[r, c] += h
            ym[r, c] -= h
            fd = (np.sum(G * moe_oracle.combine(yp, dp.inv, w, T, k)) -
                  np.sum(G * moe_oracle.combine(ym, dp.inv, w, T, k))) / (2 * h)
            assert abs(fd - dexp[r, c]) < 1e-9
    for t in range(T):
        for j in range(k):
            wp, wm = w.copy(), w.copy()
            wp[t, j] += h
            wm[t, j] -= h
            fd = (np.sum(G * moe_oracle.combine(y, dp.inv, wp, T, k)) -
                  np.sum(G * moe_oracle.combine(y, dp.inv, wm, T, k))) / (2 * h)
            assert abs(fd - dw[t, j]) < 1e-9


def _tiny_experts(rng, E=3, H=4, I=5):
    gate = rng.standard_normal((E, I, H)) * 0.7
    up = rng.standard_normal((E, I, H)) * 0.7
    down = rng.standard_normal((E, H, I)) * 0.7
    return gate, up, down


def pin_experts_backward_finite_differences(m):
    """d<dY, y>/dtheta by central differences of the forward experts
    (moe_oracle.experts_forward_dispatched) for every entry of x, gate, up
    and down, with one expert empty."""
    rng = np.random.default_rng(13)
    gate, up, down = _tiny_experts(rng)
    idx = np.array([[0, 2], [2, 0], [0, 2]])          # expert 1 gets no rows
    T, k = idx.shape
    dp = moe_oracle.dispatch(idx, 3)
    x = rng.standard_normal((T, 4))
    xd = x[dp.row_src.astype(np.int64) // k]
    dY = rng.standard_normal((T * k, 4))
    gr = m.experts_backward(torch.from_numpy(xd), torch.from_numpy(gate), torch.from_numpy(up),
                            torch.from_numpy(down), dp.offsets, dY)

    def loss(g_, u_, d_):
        y = moe_oracle.experts_forward_dispatched(
            torch.from_numpy(x), torch.from_numpy(g_), torch.from_numpy(u_), torch.from_numpy(d_), dp, k)
        return float(np.sum(dY * y))

    # x enters the forward through the dispatched rows: perturb x[t] moves
    # every row of token t, so compare against the sum of the row gradients.
    h = 1e-5
    for name, arr, ref in (("gate", gate, gr.dgate), ("up", up, gr.dup), ("down", down, gr.ddown)):
        for pos in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[pos] += h
            am[pos] -= h
            args_p = {"gate": gate, "up": up, "down": down}
            args_m = dict(args_p)
            args_p[name], args_m[name] = ap, am
            fd = (loss(args_p["gate"], args_p["up"], args_p["down"]) -
                  loss(args_m["gate"], args_m["up"], args_m["down"])) / (2 * h)
            assert abs(fd - ref[pos]) < 1e-6 * max(1.0, abs(fd)), (name, pos, fd, ref[pos])
    assert np.all(gr.dgate[1] == 0) and np.all(gr.ddown[1] == 0)
    dx_tok = np.zeros_like(x)
    np.add.at(dx_tok, dp.row_src.astype(np.int64) // k, gr.dx_dispatched)
    for pos in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[pos] += h
        xm[pos] -= h
        yp = moe_oracle.experts_forward_dispatched(torch.from_numpy(xp), torch.from_numpy(gate), torch.from_numpy(up),
                                                   torch.from_numpy(down), dp, k)
        ym = moe_oracle.experts_forward_dispatched(torch.from_numpy(xm), torch.from_numpy(gate), torch.from_numpy(up),
                                                   torch.from_numpy(down), dp, k)
        fd = float(np.sum(dY * (yp - ym))) / (2 * h)
        assert abs(fd - dx_tok[pos]) < 1e-6 * max(1.0, abs(fd))


def pin_training_forward_cache_hand_worked(m):
    """A hand-worked cache, H = 2, I = 3, two experts (the second with gate
    and up exchanged, an empty expert between them): x = (1, 2) gives
    g = (1, 2, 3), u = (2, 1, 0) on expert 0, so h = (2 SiLU(1), SiLU(2), 0)
    with SiLU(a) = a / (1 + e^-a); expert 2 sees the same x with the roles
    swapped: g = (2, 1, 0), u = (1, 2, 3), h = (SiLU(2), 2 SiLU(1), 0)."""
    A = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    B = np.array([[0.0, 1.0], [1.0, 0.0], [2.0, -1.0]])
    gate = np.stack([A, np.zeros((3, 2)), B])
    up = np.stack([B, np.zeros((3, 2)), A])
    x = np.array([[1.0, 2.0], [1.0, 2.0]])
    g, u, h = m.training_forward_cache(torch.from_numpy(x), torch.from_numpy(gate), torch.from_numpy(up),
                                       np.array([0, 1, 1, 2]))
    s1, s2 = 1.0 / (1.0 + np.exp(-1.0)), 2.0 / (1.0 + np.exp(-2.0))
    np.testing.assert_array_equal(g, [[1, 2, 3], [2, 1, 0]])
    np.testing.assert_array_equal(u, [[2, 1, 0], [1, 2, 3]])
    np.testing.assert_allclose(h, [[2 * s1, s2, 0.0], [s2, 2 * s1, 0.0]], rtol=1e-15, atol=0)


def pin_dispatch_backward_brute_force(m):
    rng = np.random.default_rng(17)
    idx = np.array([[0, 2], [1, 0], [2, 2], [5, 1]])   # token 3 holds an invalid index
    T, k = idx.shape
    dp = moe_oracle.dispatch(idx, 3)
    d = rng.standard_normal((T * k, 3))
    dx = m.dispatch_backward(d, dp.inv, T, k)
    for t in range(3):
        want = sum(d[dp.inv[t * k + j]] for j in range(k))
        np.testing.assert_allclose(dx[t], want, rtol=0, atol=1e-15)
    assert np.isnan(dx[3]).all()


def pin_whole_backward_against_autograd(m):
    """The composed oracle backward (combine -> experts -> dispatch, plus the
    router gradient of dweights) equals torch autograd (f64) of the forward
    out[t] = sum_j w_j(l) * MLP_{e_j}(x_t) with the selection held fixed, for
    both scorings."""
    rng = np.random.default_rng(19)
    T, E, H, I, k = 5, 4, 3, 4, 2
    gate, up, down = _tiny_experts(rng, E, H, I)
    x = rng.standard_normal((T, H))
    l = _quarter_logits(rng, T, E)
    idx = np.array([[0, 1], [3, 0], [2, 2], [1, 3], [0, 2]])
    G = rng.standard_normal((T, H))
    for o in (Opt("softmax", True, 1.0), Opt("softmax", False, 2.0), Opt("sigmoid", True, 1.5)):
        lt = torch.from_numpy(l).requires_grad_(True)
        xt = torch.from_numpy(x).requires_grad_(True)
        gt, ut, dt = (torch.from_numpy(a).requires_grad_(True) for a in (gate, up, down))
        it = torch.from_numpy(idx)
        if o.scoring == "softmax":
            v = torch.gather(torch.softmax(lt, dim=1), 1, it)
        else:
            v = torch.sigmoid(torch.gather(lt, 1, it))
        if o.renormalize:
            v = v / v.sum(dim=1, keepdim=True)
        w = v * o.scale
        out = torch.zeros(T, H, dtype=torch.float64)
        for t in range(T):
            for j in range(k):
                e = int(idx[t, j])
                hh = torch.nn.functional.silu(gt[e] @ xt[t]) * (ut[e] @ xt[t])
                out[t] = out[t] + w[t, j] * (dt[e] @ hh)
        (out * torch.from_numpy(G)).sum().backward()

        dp = moe_oracle.dispatch(idx, E)
        xd = x[dp.row_src.astype(np.int64) // k]
        _, w64 = m.selected_router_weights(torch.from_numpy(l.astype(np.float32)), idx, o)
        yd = moe_oracle.experts_forward_dispatched(torch.from_numpy(x), torch.from_numpy(gate),
                                                   torch.from_numpy(up), torch.from_numpy(down), dp, k)
        dexp, dw = m.combine_backward(torch.from_numpy(yd), dp.inv, w64, torch.from_numpy(G), T, k)
        gr = m.experts_backward(torch.from_numpy(xd), torch.from_numpy(gate), torch.from_numpy(up),
                                torch.from_numpy(down), dp.offsets, dexp)
        dx = m.dispatch_backward(gr.dx_dispatched, dp.inv, T, k)
        dl, _ = m.selected_router_backward(torch.from_numpy(l.astype(np.float32)), idx,
                                           torch.from_numpy(dw.astype(np.float32)), o)
        np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gr.dgate, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gr.dup, ut.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gr.ddown, dt.grad.numpy(), rtol=1e-10, atol=1e-12)
        # dweights passes through FP32 on its way to the router (its dtype on the pages)
        np.testing.assert_allclose(dl, lt.grad.numpy(), rtol=1e-6, atol=1e-7)


def pin_router_option_ranges(m):
    for E, k, o in [(4, 0, Opt("softmax", True, 1.0)), (4, 5, Opt("softmax", True, 1.0)),
                    (100, 65, Opt("sigmoid", True, 1.0)), (4, 2, Opt("tanh", True, 1.0)),
                    (4, 2, Opt("softmax", True, 0.0)), (4, 2, Opt("softmax", True, float("nan")))]:
        with pytest.raises(ValueError):
            m.check_router_options(E, k, o)
    m.check_router_options(100, 64, Opt("sigmoid", False, 3.0))


TRAINING_PINS = [
    pin_router_softmax_matches_forward_routing,
    pin_router_sigmoid_closed_form,
    pin_router_duplicate_indices_gather,
    pin_router_invalid_index_nan_row,
    pin_router_backward_finite_differences,
    pin_router_backward_invariants,
    pin_combine_backward_finite_differences,
    pin_experts_backward_finite_differences,
    pin_training_forward_cache_hand_worked,
    pin_dispatch_backward_brute_force,
    pin_whole_backward_against_autograd,
    pin_router_option_ranges,
]


@pytest.mark.parametrize("pin", TRAINING_PINS, ids=[p.__name__ for p in TRAINING_PINS])
def test_training_oracle_pin(pin):
    pin(oracle)
