"""Pins that tie the CPU oracle to facts fixed by the pages and by mathematics,
not to itself: hand-worked cases, closed forms, invariants, brute force and an
independent restatement (the einsum form). Each pin is a plain function of the
oracle module so that ``test_oracle_mutations`` can plant a mistake in the
oracle and check that some pin catches it."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s):
    a, b = s.split("/")
    return int(a) / int(b)


def _parse_logits(s):
    vals = []
    for tok in s.split(","):
        tok = tok.strip()
        vals.append(math.log(float(tok[2:])) if tok.startswith("ln") else float(tok))
    return vals


# --- routing -------------------------------------------------------------------------------

def pin_hand_worked_routing(m):
    """tests/golden/routing_hand_worked.json: E=3 logits [0, ln2, ln3] and an
    all-equal row, worked by hand from the routing contract."""
    with open(os.path.join(GOLDEN, "routing_hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        l = torch.tensor([_parse_logits(c["logits"])], dtype=torch.float32)
        rt = m.route(l, c["top_k"], c["renormalize"])
        assert rt.indices[0].tolist() == c["indices"], c
        want = np.array([_frac(w) for w in c["weights"]])
        np.testing.assert_allclose(rt.weights32[0], want, rtol=1e-6, atol=0)
        np.testing.assert_allclose(rt.weights64[0], want, rtol=2e-7, atol=0)  # logits are FP32-rounded


def pin_exact_tie_lower_id(m):
    """Two equal maxima at ids a < b: indices [a, b]; renormalized FP32 weights
    are exactly 0.5 (p + p is exact and p / 2p = 0.5)."""
    rng = np.random.default_rng(7)
    for a, b, E in [(1, 6, 8), (0, 3, 4), (2, 5, 16), (10, 11, 64)]:
        row = rng.standard_normal(E).astype(np.float32)
        row[a] = row[b] = row.max() + 1.0
        rt = m.route(torch.from_numpy(row[None]), 2, True)
        assert rt.indices[0].tolist() == [a, b]
        assert rt.weights32[0].tolist() == [0.5, 0.5]
    # the contract row of the F32 workload
    inp = workloads.generate(workloads.CONFIGS[0], weights=False)
    rt = m.route(inp["logits"], 2, True)
    assert rt.indices[0].tolist() == [1, 6]
    assert rt.weights32[0].tolist() == [0.5, 0.5]


def pin_nonfinite_rows(m):
    """Rows with a NaN, a +inf, or only -inf keep NaN weights (no uniform
    fallback); their indices are 0..k-1. A single -inf in a finite row is a
    probability of 0."""
    E, k = 6, 3
    l = np.zeros((5, E), dtype=np.float32)
    l[0] = [0.5, 1, 2, 3, 0, -1]
    l[1] = [0.5, np.nan, 2, 3, 0, -1]
    l[2] = [0.5, 1, 2, np.inf, 0, -1]
    l[3] = -np.inf
    l[4] = [0.5, -np.inf, 2, 3, 0, -1]
    for renorm in (True, False):
        rt = m.route(torch.from_numpy(l), k, renorm)
        assert not np.isnan(rt.weights32[0]).any()
        for r in (1, 2, 3):
            assert np.isnan(rt.weights32[r]).all() and np.isnan(rt.weights[r]).all()
            assert rt.indices[r].tolist() == [0, 1, 2]
        assert rt.bad.tolist() == [False, True, True, True, False]
        assert rt.indices[4].tolist() == [3, 2, 0]
    rt = m.route(torch.from_numpy(l[4:5]), E, False)
    assert rt.indices[0].tolist() == [3, 2, 0, 4, 5, 1]
    assert rt.weights32[0, -1] == 0.0 and rt.weights32[0, :-1].min() > 0


def pin_renormalized_sum(m):
    """With renormalize the selected weights sum to 1 (FP32 within 1e-6)."""
    rng = np.random.default_rng(11)
    for E, k in [(8, 2), (64, 6), (128, 8)]:
        l = torch.from_numpy(rng.standard_normal((200, E)).astype(np.float32))
        rt = m.route(l, k, True)
        np.testing.assert_allclose(rt.weights32.astype(np.float64).sum(1), 1.0, atol=1e-6)
        np.testing.assert_allclose(rt.weights64.sum(1), 1.0, atol=1e-12)
        rt = m.route(l, k, False)
        assert (rt.weights64.sum(1) < 1.0).all()


def pin_topk_equals_E_is_full_softmax(m):
    """top_k = E with renormalize: the weights are the whole softmax in
    descending order. logits ln(q) give softmax q / sum(q) in closed form."""
    rng = np.random.default_rng(3)
    for E in (3, 8, 40):
        q = rng.permutation(np.arange(1, E + 1)).astype(np.float64)
        l = torch.tensor(np.log(q)[None], dtype=torch.float32)
        want_idx = np.argsort(-q, kind="stable")
        want = np.sort(q)[::-1] / q.sum()
        for renorm in (True, False):
            rt = m.route(l, E, renorm)
            assert rt.indices[0].tolist() == want_idx.tolist()
            np.testing.assert_allclose(rt.weights32[0], want, rtol=2e-6)


def pin_overflow_safe_softmax(m):
    """The max shift keeps exp from overflowing: logits [200, 200+ln2, 200+ln3]
    still give p = [1/6, 1/3, 1/2] (up to the FP32 rounding of the shifted logits)."""
    l = torch.tensor([[200.0, 200.0 + math.log(2), 200.0 + math.log(3)]], dtype=torch.float32)
    rt = m.route(l, 3, False)
    assert rt.indices[0].tolist() == [2, 1, 0]
    np.testing.assert_allclose(rt.weights32[0], [1 / 2, 1 / 3, 1 / 6], rtol=1e-4)


def _brute_force_topk(row, k):
    """Among all ordered k-tuples of distinct ids, the lexicographically greatest
    under the key (logit descending, id ascending)."""
    best, best_key = None, None
    for tup in itertools.permutations(range(len(row)), k):
        key = tuple(v for i in tup for v in (row[i], -i))
        if best_key is None or key > best_key:
            best, best_key = tup, key
    return list(best)


def pin_brute_force_selection(m):
    """Exhaustive search on tiny rows full of ties and -inf entries."""
    rng = np.random.default_rng(5)
    levels = np.array([-np.inf, -1.0, -0.5, 0.0, 0.5, 1.0], dtype=np.float32)
    for E in range(1, 7):
        rows = levels[rng.integers(1, len(levels), size=(12, E))]
        rows[rng.random((12, E)) < 0.15] = -np.inf
        rows[0, :] = levels[1 + rng.integers(0, 5)]        # an all-equal row
        if E > 1:
            rows[1, :] = -np.inf
            rows[1, E // 2] = 0.0                            # one finite entry
        for k in range(1, E + 1):
            rt = m.route(torch.from_numpy(rows), k, True)
            for t in range(rows.shape[0]):
                if rt.bad[t]:
                    continue
                assert rt.indices[t].tolist() == _brute_force_topk(rows[t].tolist(), k), (rows[t], k)


def pin_fp32_within_rounding_bound(m):
    """FP32 routing weights stay within the first-order rounding bound of the
    same softmax evaluated in f64: (E + k + 8) units of 2^-24, relative."""
    rng = np.random.default_rng(13)
    for E, k, renorm in [(8, 2, True), (128, 8, True), (64, 6, False), (1024, 16, False)]:
        l = torch.from_numpy((rng.standard_normal((300, E)) * 3).astype(np.float32))
        rt = m.route(l, k, renorm)
        bound = (E + k + 8) * 2.0 ** -24
        rel = np.abs(rt.weights32 - rt.weights64) / rt.weights64
        assert rel.max() <= bound, (E, k, rel.max(), bound)


def pin_contract_rows_of_f32_workload(m):
    """The four special rows of the F32 routing-contract workload."""
    inp = workloads.generate(workloads.CONFIGS[0], weights=False)
    rt = m.route(inp["logits"], 2, True)
    assert rt.indices[0].tolist() == [1, 6]
    for r in (1, 2, 3):
        assert rt.bad[r] and np.isnan(rt.weights[r]).all() and rt.indices[r].tolist() == [0, 1]
    assert not rt.bad[4:].any() and not np.isnan(rt.weights[4:]).any()


# --- dispatch ------------------------------------------------------------------------------

def pin_dispatch_invariants(m):
    """No dropping (sum of counts = T*k), offsets are the exclusive prefix,
    inv and row_src are inverse permutations, every row sits in its expert's
    range, and rows of one expert ascend in t*k + j (a stable sort by expert)."""
    rng = np.random.default_rng(17)
    for T, k, E in [(200, 3, 9), (1, 1, 1), (57, 5, 64), (300, 2, 4)]:
        p = rng.random(E) ** 3
        p[rng.random(E) < 0.3] = 0
        p = p + (p.sum() == 0)
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) if np.count_nonzero(p) >= k
                        else rng.permutation(E)[:k] for _ in range(T)]).astype(np.uint32)
        d = m.dispatch(idx, E)
        flat = idx.reshape(-1).astype(np.int64)
        assert int(d.counts.sum()) == T * k
        assert d.offsets[0] == 0 and (np.diff(d.offsets.astype(np.int64)) == d.counts).all()
        assert (d.inv[d.row_src] == np.arange(T * k)).all()
        assert (d.row_src[d.inv] == np.arange(T * k)).all()
        for e in range(E):
            rows = d.row_src[d.offsets[e]:d.offsets[e + 1]].astype(np.int64)
            assert (flat[rows] == e).all() and (np.diff(rows) > 0).all()
        assert (d.row_src == np.argsort(flat, kind="stable")).all()


# --- experts and combine -------------------------------------------------------------------

def _identity_experts(E, n, scale=None):
    eye = torch.eye(n, dtype=torch.float64)
    gate = eye.repeat(E, 1, 1)
    down = eye.repeat(E, 1, 1)
    if scale is not None:
        down = down * torch.tensor(scale, dtype=torch.float64)[:, None, None]
    return gate, gate.clone(), down


def pin_identity_experts_closed_form(m):
    """gate = up = down = I: h = SiLU(x) * x and out[t] = (sum_j w_j c_e) * SiLU(x) * x.
    With x = ln(a), SiLU(x) = ln(a) * a / (1 + a) in closed form; logits ln(q)
    give the routing weights q / sum(q) in closed form."""
    E, n, T, k = 4, 5, 3, 2
    a = np.array([[0.5, 1.0, 2.0, 3.0, 9.0], [1 / 3, 4.0, 1.5, 1.0, 0.25], [7.0, 2.0, 0.125, 5.0, 1.0]])
    x = torch.tensor(np.log(a))
    siluxx = np.log(a) ** 2 * a / (1 + a)
    q = np.array([[1.0, 2.0, 3.0, 4.0], [4.0, 1.0, 1.0, 2.0], [1.0, 5.0, 2.0, 2.0]])
    logits = torch.tensor(np.log(q), dtype=torch.float32)
    c = [1.0, -2.0, 0.5, 3.0]
    for renorm in (True, False):
        for scale in (None, c):
            gate, up, down = _identity_experts(E, n, scale)
            res = m.forward(x, logits, gate, up, down, k, renorm)
            cs = np.ones(E) if scale is None else np.array(scale)
            want = np.zeros((T, n))
            for t in range(T):
                order = np.argsort(-q[t], kind="stable")[:k]
                w = q[t, order] / (q[t, order].sum() if renorm else q[t].sum())
                want[t] = (w * cs[order]).sum() * siluxx[t]
            np.testing.assert_allclose(res.out, want, rtol=1e-6, atol=1e-12)
    gate, up, _ = _identity_experts(E, n)
    res = m.forward(x, logits, gate, up, torch.zeros(E, n, n, dtype=torch.float64), k, True)
    assert (res.out == 0).all()


def pin_hand_worked_swiglu(m):
    """A non-square case worked by hand (H=2, I=3, E=2). gate rows pick
    x0, x1, x0+x1; up rows pick x1, x0, 0; down = [[1,0,0],[0,1,1]]; expert 1
    is expert 0 with down doubled. x = [ln3, 2]:
      g = [ln3, 2, ln3+2], u = [2, ln3, 0],
      h = [2 SiLU(ln3), ln3 SiLU(2), 0] = [1.5 ln3, 2 sigma(2) ln3, 0],
      y0 = [1.5 ln3, 2 sigma(2) ln3], y1 = 2 y0.
    logits [0, ln3], k = 2, renormalize: w = [3/4, 1/4] on experts [1, 0], so
    out = (3/4 * 2 + 1/4) y0 = 1.75 y0; without renormalize the same (the two
    experts hold all the probability)."""
    g0 = [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]
    u0 = [[0.0, 1.0], [1.0, 0.0], [0.0, 0.0]]
    d0 = [[1.0, 0.0, 0.0], [0.0, 1.0, 1.0]]
    gate = torch.tensor([g0, g0], dtype=torch.float64)
    up = torch.tensor([u0, u0], dtype=torch.float64)
    down = torch.tensor([d0, [[2 * v for v in r] for r in d0]], dtype=torch.float64)
    x = torch.tensor([[math.log(3), 2.0]], dtype=torch.float64)
    logits = torch.tensor([[0.0, math.log(3)]], dtype=torch.float32)
    sig2 = 1 / (1 + math.exp(-2))
    y0 = np.array([1.5 * math.log(3), 2 * sig2 * math.log(3)])
    for renorm in (True, False):
        res = m.forward(x, logits, gate, up, down, 2, renorm)
        assert res.route.indices[0].tolist() == [1, 0]
        np.testing.assert_allclose(res.out[0], 1.75 * y0, rtol=1e-6)
        np.testing.assert_allclose(res.y_dispatched[res.dispatch.inv[1]], y0, rtol=1e-12)
        np.testing.assert_allclose(res.y_dispatched[res.dispatch.inv[0]], 2 * y0, rtol=1e-12)
    res = m.forward(x, logits, gate, up, down, 1, False)
    np.testing.assert_allclose(res.out[0], 0.75 * 2 * y0, rtol=1e-6)


def pin_einsum_cross_statement(m):
    """The expert-major oracle equals the token-major einsum statement of the
    same computation ("PyTorch general ops", section "two ways to write a
    contraction"): gather each token's expert weights, contract the hidden
    dim, apply SiLU(gate) * up, contract the intermediate dim, then the
    routing-weighted sum over the selected experts."""
    rng = np.random.default_rng(19)
    T, E, k, H, I = 9, 5, 3, 6, 7
    x = torch.tensor(rng.standard_normal((T, H)))
    logits = torch.tensor(rng.standard_normal((T, E)), dtype=torch.float32)
    gate = torch.tensor(rng.standard_normal((E, I, H)))
    up = torch.tensor(rng.standard_normal((E, I, H)))
    down = torch.tensor(rng.standard_normal((E, H, I)))
    for renorm in (True, False):
        res = m.forward(x, logits, gate, up, down, k, renorm)
        ids = res.route.indices.astype(np.int64)
        w1 = gate.numpy()[ids]              # [t, a, o, i]
        w3 = up.numpy()[ids]
        w2 = down.numpy()[ids]              # [t, a, i, o]
        xx = x.numpy()
        x1 = np.einsum("ti,taoi->tao", xx, w1)
        x3 = np.einsum("ti,taoi->tao", xx, w3)
        act = x1 / (1 + np.exp(-x1))
        eo = np.einsum("tao,taio->tai", act * x3, w2)
        want = np.einsum("tai,ta->ti", eo, res.route.weights)
        np.testing.assert_allclose(res.out, want, rtol=1e-10, atol=1e-12)


def pin_forward_tokens_consistent(m):
    """Sampled-token evaluation equals the full forward on those tokens
    (including the NaN rows of the contract workload)."""
    cfg = workloads.CONFIGS[0]
    inp = workloads.generate(cfg)
    full = m.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k, True)
    toks = np.array([0, 1, 2, 3, 17, 63])
    part = m.forward_tokens(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"],
                            cfg.top_k, True, toks)
    np.testing.assert_allclose(part, full.out[toks], rtol=1e-12, atol=1e-14)
    assert np.isnan(full.out[1:4]).all() and not np.isnan(full.out[4:]).any()


PINS = [
    pin_hand_worked_routing,
    pin_exact_tie_lower_id,
    pin_nonfinite_rows,
    pin_renormalized_sum,
    pin_topk_equals_E_is_full_softmax,
    pin_overflow_safe_softmax,
    pin_brute_force_selection,
    pin_fp32_within_rounding_bound,
    pin_contract_rows_of_f32_workload,
    pin_dispatch_invariants,
    pin_identity_experts_closed_form,
    pin_hand_worked_swiglu,
    pin_einsum_cross_statement,
    pin_forward_tokens_consistent,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(moe_oracle)
