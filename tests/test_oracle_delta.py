"""Pins for the gated delta-rule oracle (oracle/delta.py).

Each check rests on something other than the function it checks:
- associative memory: with alpha = beta = 1 and orthonormal keys the state
  returns every written value exactly, and a rewrite replaces only its slot;
- a write with beta = 1 and a unit key leaves S_t k_t = v_t for any decay and
  any prior state (the rule's projection property);
- beta = 0 reduces the rule to pure decay, o = (prod alpha) S_0 q;
- a scalar case (P = N = 1) worked by hand;
- the replay formula and the fold, two different computations, against the
  step-by-step definition;
- the pointer bookkeeping against the outer-product oracle's, bit for bit;
- the pseudo-value w of a step against the step itself: S_t - alpha S = w k^T;
- a two-step example worked by hand (tests/golden/hand_delta_two_step.txt), one
  step with a key coupled to the earlier one.
"""
import os

import numpy as np

import oracle
from oracle import delta


def _one(x):
    """[.] -> [B=1, H=1 or G=1, .]"""
    return np.asarray(x, np.float64)[None, None]


def test_associative_memory_with_orthonormal_keys():
    rng = np.random.default_rng(0)
    N, P = 8, 5
    Q, _ = np.linalg.qr(rng.standard_normal((N, N)))
    keys, vals = Q[:, :4].T, rng.standard_normal((4, P))
    S = np.zeros((1, 1, P, N))
    one = np.ones((1, 1))
    for kk, vv in zip(keys, vals):
        S, _ = delta.delta_step(S, one, one, _one(vv), _one(kk), _one(kk))
    for kk, vv in zip(keys, vals):
        assert np.allclose(S[0, 0] @ kk, vv, atol=1e-12)
    v_new = rng.standard_normal(P)
    S, o = delta.delta_step(S, one, one, _one(v_new), _one(keys[1]), _one(keys[2]))
    assert np.allclose(S[0, 0] @ keys[1], v_new, atol=1e-12)
    assert np.allclose(S[0, 0] @ keys[0], vals[0], atol=1e-12)
    assert np.allclose(o[0, 0], vals[2], atol=1e-12)


def test_full_strength_write_is_exact_for_any_decay():
    rng = np.random.default_rng(1)
    S = rng.standard_normal((2, 3, 4, 6))
    k = rng.standard_normal((2, 3, 6))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((2, 3, 4))
    alpha = rng.uniform(0.1, 1.0, (2, 3))
    S1, _ = delta.delta_step(S, alpha, np.ones((2, 3)), v, k, k)
    assert np.allclose(np.einsum("bhpn,bhn->bhp", S1, k), v, atol=1e-12)


def test_zero_write_strength_is_pure_decay():
    rng = np.random.default_rng(2)
    S0 = rng.standard_normal((2, 4, 3, 8))
    S, gam = S0.copy(), np.ones((2, 4))
    for _ in range(5):
        a = rng.uniform(0.5, 1.0, (2, 4))
        k, q = rng.standard_normal((2, 2, 8)), rng.standard_normal((2, 2, 8))
        S, o = delta.delta_step(S, a, np.zeros((2, 4)), rng.standard_normal((2, 4, 3)), k, q)
        gam *= a
    g = oracle.head_groups(4, 2)
    assert np.allclose(S, gam[:, :, None, None] * S0)
    assert np.allclose(o, gam[:, :, None] * np.einsum("bhpn,bhn->bhp", S0, q[:, g]))


def test_scalar_case_by_hand():
    # s1 = 0.9 * 0.5 * (1 - 0.5 * 1) + 0.5 * 2 * 1 = 1.225,  o1 = s1 * 1
    # s2 = 0.8 * 1.225 * (1 - 0.25 * 1) + 0.25 * (-1) * (-1) = 0.985,  o2 = 0.985 * 0.5
    S = np.full((1, 1, 1, 1), 0.5)
    S, o1 = delta.delta_step(S, np.full((1, 1), 0.9), np.full((1, 1), 0.5), _one([2.0]), _one([1.0]), _one([1.0]))
    assert np.isclose(S.item(), 1.225) and np.isclose(o1.item(), 1.225)
    S, o2 = delta.delta_step(S, np.full((1, 1), 0.8), np.full((1, 1), 0.25), _one([-1.0]), _one([-1.0]), _one([0.5]))
    assert np.isclose(S.item(), 0.985) and np.isclose(o2.item(), 0.4925)


def test_replay_formula_and_fold_match_the_definition():
    rng = np.random.default_rng(3)
    H, G, P, N = 4, 2, 6, 8
    S0 = rng.standard_normal((H, P, N))
    for h in (1, 2, 7, 12):
        a = rng.uniform(0.3, 1.0, (h, H))
        b = rng.uniform(0.0, 1.0, (h, H))
        v = rng.standard_normal((h, H, P))
        k = rng.standard_normal((h, G, N))
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q = rng.standard_normal((G, N))
        S = S0[None].copy()
        for j in range(h):
            S, o_def = delta.delta_step(S, a[j][None], b[j][None], v[j][None], k[j][None], q[None])
        o_rep = delta.delta_replay_output(S0, a, b, v, k, q)
        assert np.allclose(o_rep, o_def[0], rtol=1e-12, atol=1e-12), f"h={h}"
        assert np.allclose(delta.delta_fold(S0, a, b, v, k), S[0], rtol=1e-12, atol=1e-12)


def test_pointers_follow_the_outer_product_oracle():
    rng = np.random.default_rng(4)
    B, H, G, P, N, L = 3, 2, 1, 4, 4, 4
    S0 = rng.standard_normal((B, H, P, N))
    d = delta.DeltaReplayOracle(S0, L=L, R=L, G=G)
    r = oracle.ReplayOracle(S0, L=L, R=L, G=G)
    for t in range(11):
        a = rng.uniform(0.5, 1.0, (B, H))
        v, k, q = rng.standard_normal((B, H, P)), rng.standard_normal((B, G, N)), rng.standard_normal((B, G, N))
        _, f1 = d.decode(a, rng.uniform(0, 1, (B, H)), v, k, q)
        _, f2 = r.decode(a, v, k, q)
        assert np.array_equal(f1, f2) and np.array_equal(d.start, r.start) and np.array_equal(d.count, r.count)
    assert np.array_equal(d.flush(1), r.flush(1))
    assert np.array_equal(d.start, r.start) and np.array_equal(d.count, r.count)


def test_pseudo_value_is_the_steps_write_term():
    rng = np.random.default_rng(5)
    B, H, G, P, N = 2, 4, 2, 5, 7
    S = rng.standard_normal((B, H, P, N))
    a, b = rng.uniform(0.2, 1.0, (B, H)), rng.uniform(0.0, 1.0, (B, H))
    v, k, q = rng.standard_normal((B, H, P)), rng.standard_normal((B, G, N)), rng.standard_normal((B, G, N))
    S1, _ = delta.delta_step(S, a, b, v, k, q)
    w = delta.delta_pseudo_value(S, a, b, v, k)
    g = oracle.head_groups(H, G)
    assert np.allclose(S1 - a[:, :, None, None] * S, w[..., None] * k[:, g, None, :], atol=1e-12)


def _golden_delta():
    """name -> fields of tests/golden/hand_delta_two_step.txt."""
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_delta_two_step.txt")
    rows = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            name, *rest = line.split()
            rows[name] = rest
    return rows


def _step_inputs(fields):
    """'alpha a beta b v v0 v1 k k0 k1 q q0 q1' -> the [1,1,...] arrays delta_step takes."""
    d, i = {}, 0
    while i < len(fields):
        n = 2 if fields[i] in ("v", "k", "q") else 1
        d[fields[i]] = np.array([float(x) for x in fields[i + 1: i + 1 + n]])
        i += 1 + n
    return (d["alpha"].reshape(1, 1), d["beta"].reshape(1, 1), d["v"][None, None], d["k"][None, None],
            d["q"][None, None])


def test_hand_computed_two_step_example():
    """tests/golden/hand_delta_two_step.txt: steps, pseudo-values, replay output and fold."""
    g = _golden_delta()
    num = lambda xs: np.array([float(x) for x in xs])  # noqa: E731
    S0 = num(g["S0"]).reshape(1, 1, 2, 2)
    steps = [_step_inputs(g["step1"]), _step_inputs(g["step2"])]
    S = S0
    for n, (a, b, v, k, q) in enumerate(steps, 1):
        w = delta.delta_pseudo_value(S, a, b, v, k)
        assert np.allclose(w[0, 0], num(g[f"w{n}"]), atol=1e-12)
        S, o = delta.delta_step(S, a, b, v, k, q)
        assert np.allclose(S[0, 0].ravel(), num(g[f"S{n}"]), atol=1e-12)
        assert np.allclose(o[0, 0], num(g[f"o{n}"]), atol=1e-12)
    al, be = np.stack([x[0][0] for x in steps]), np.stack([x[1][0] for x in steps])
    vs, ks = np.stack([x[2][0] for x in steps]), np.stack([x[3][0] for x in steps])
    q2 = steps[1][4][0]
    assert np.allclose(delta.delta_replay_output(S0[0], al, be, vs, ks, q2)[0], num(g["o2"]), atol=1e-12)
    assert np.allclose(delta.delta_fold(S0[0], al, be, vs, ks)[0].ravel(), num(g["S2"]), atol=1e-12)
