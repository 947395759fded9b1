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
  step with a key coupled to the earlier one;
- speculative verify and commit: the hand example as two drafts, the projection
  and associative-memory properties within a verify, each draft's output
  against the replay formula, commit of an accepted prefix against the fold
  (with junk in the rejected drafts), and the pointers against the
  outer-product oracle's verify and commit.

Planted mistakes (an undecayed or sign-flipped erase, no erase, a write
without beta, an erase along the query, the old state's output, swapped k and
q, interleaved groups, and wrong orders in the replay and the fold) are each
caught by at least one of these pins.
"""
import os

import numpy as np
import pytest

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


# Speculative verify and commit on a gated delta-rule layer.


def _drafts(rng, B, T, H, G, P, N):
    return (rng.uniform(0.5, 1.0, (B, T, H)), rng.uniform(0.0, 1.0, (B, T, H)), rng.standard_normal((B, T, H, P)),
            rng.standard_normal((B, T, G, N)), rng.standard_normal((B, T, G, N)))


def test_verify_and_commit_of_the_hand_example():
    """The two golden steps as two drafts: outputs o1, o2; commit(1) leaves S1, commit(2) S2."""
    g = _golden_delta()
    num = lambda xs: np.array([float(x) for x in xs])  # noqa: E731
    S0 = num(g["S0"]).reshape(1, 1, 2, 2)
    steps = [_step_inputs(g["step1"]), _step_inputs(g["step2"])]
    drafts = [np.stack([s[i] for s in steps], axis=1) for i in range(5)]  # [1, T=2, ...]
    for a, S_name in ((1, "S1"), (2, "S2")):
        d = delta.DeltaReplayOracle(S0, L=4, R=4, G=1)
        O = d.verify(*drafts)
        assert np.allclose(O[0, 0, 0], num(g["o1"]), atol=1e-12)
        assert np.allclose(O[0, 1, 0], num(g["o2"]), atol=1e-12)
        assert np.array_equal(d.S, S0) and d.count[0] == 0
        d.commit([a])
        assert np.allclose(d.S[0, 0].ravel(), num(g[S_name]), atol=1e-12) and d.count[0] == a


def test_verify_keeps_the_projection_and_memory_properties():
    """beta = 1 and unit keys: draft t's output at q = k_t is v_t for any state and decay;
    with alpha = 1 and orthonormal keys a later draft's query k_i reads back v_i."""
    rng = np.random.default_rng(6)
    B, T, H, G, P, N = 2, 4, 3, 1, 5, 8
    d = delta.DeltaReplayOracle(rng.standard_normal((B, H, P, N)), L=8, R=8, G=G)
    d.decode(rng.uniform(0.5, 1, (B, H)), rng.uniform(0, 1, (B, H)), rng.standard_normal((B, H, P)),
             rng.standard_normal((B, G, N)), rng.standard_normal((B, G, N)))
    alpha, _, v, _, _ = _drafts(rng, B, T, H, G, P, N)
    k = rng.standard_normal((B, T, G, N))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    O = d.verify(alpha, np.ones((B, T, H)), v, k, k.copy())
    assert np.allclose(O, v, atol=1e-12)
    Q = np.stack([np.linalg.qr(rng.standard_normal((N, N)))[0][:, :T].T for _ in range(B)])  # [B, T, N]
    kq = Q[:, :, None, :]
    q = kq.copy()
    q[:, 3] = kq[:, 0]  # the last draft reads back the first draft's value
    O = d.verify(np.ones((B, T, H)), np.ones((B, T, H)), v, kq, q)
    assert np.allclose(O[:, 3], v[:, 0], atol=1e-12)
    assert np.allclose(O[:, :3], v[:, :3], atol=1e-12)


def test_verify_matches_the_replay_formula():
    """Draft t's output equals the backward query carry over the committed records and drafts 1..t."""
    rng = np.random.default_rng(7)
    B, T, H, G, P, N, L = 3, 3, 4, 2, 5, 6, 8
    S0 = rng.standard_normal((B, H, P, N))
    d = delta.DeltaReplayOracle(S0, L=L, R=L, G=G)
    recs = []
    for _ in range(2):
        a, b, v, k, q = (x[:, 0] for x in _drafts(rng, B, 1, H, G, P, N))
        d.decode(a, b, v, k, q)
        recs.append((a, b, v, k))
    dr = _drafts(rng, B, T, H, G, P, N)
    O = d.verify(*dr)
    for t in range(T):
        rows = recs + [tuple(x[:, j] for x in dr[:4]) for j in range(t + 1)]
        for bb in range(B):
            al, be, vs, ks = (np.stack([r[i][bb] for r in rows]) for i in range(4))
            o = delta.delta_replay_output(S0[bb], al, be, vs, ks, dr[4][bb, t])
            assert np.allclose(O[bb, t], o, rtol=1e-11, atol=1e-11), (bb, t)


def test_commit_applies_only_the_accepted_prefix():
    """The rejected drafts' inputs do not reach the state; the state equals the fold of the accepted records."""
    rng = np.random.default_rng(8)
    B, T, H, G, P, N, L = 5, 4, 2, 1, 4, 6, 8
    S0 = rng.standard_normal((B, H, P, N))
    dr = _drafts(rng, B, T, H, G, P, N)
    acc = np.array([0, 1, 2, 3, 4])
    junk = [x.copy() for x in dr]
    for bb, a in enumerate(acc):
        for x in junk:
            x[bb, a:] = rng.standard_normal(x[bb, a:].shape)
    d1, d2 = (delta.DeltaReplayOracle(S0, L=L, R=L, G=G) for _ in range(2))
    d1.verify(*dr)
    d2.verify(*junk)
    d1.commit(acc)
    d2.commit(acc)
    assert np.array_equal(d1.S, d2.S) and np.array_equal(d1.count, acc)
    for bb, a in enumerate(acc):
        al, be, vs, ks = (x[bb, :a] for x in dr[:4])
        want = delta.delta_fold(S0[bb], al, be, vs, ks) if a else S0[bb]
        assert np.allclose(d1.S[bb], want, rtol=1e-12, atol=1e-12), bb
    assert np.array_equal(d1.S[0], S0[0])  # commit of 0 drafts leaves the state bit for bit


def test_verify_commit_pointers_follow_the_outer_product_oracle():
    rng = np.random.default_rng(9)
    B, T, H, G, P, N, L = 4, 3, 2, 1, 3, 4, 6
    S0 = rng.standard_normal((B, H, P, N))
    d = delta.DeltaReplayOracle(S0, L=L, R=L + T, G=G)
    r = oracle.ReplayOracle(S0, L=L, R=L + T, G=G)
    for rnd in range(12):
        a, b, v, k, q = _drafts(rng, B, T, H, G, P, N)
        d.verify(a, b, v, k, q)
        r.verify(a, v, k, q)
        acc = rng.integers(0, T + 1, B)
        d.commit(acc)
        r.commit(acc)
        assert np.array_equal(d.flush(L), r.flush(L))
        assert np.array_equal(d.start, r.start) and np.array_equal(d.count, r.count), rnd


def test_verify_and_commit_refusals():
    rng = np.random.default_rng(10)
    B, T, H, G, P, N = 2, 3, 2, 1, 3, 4
    d = delta.DeltaReplayOracle(rng.standard_normal((B, H, P, N)), L=4, R=4, G=G)
    dr = _drafts(rng, B, T, H, G, P, N)
    with pytest.raises(oracle.CapacityError):
        d.commit([0, 0])  # no verify yet
    d.decode(*(x[:, 0] for x in dr))
    d.decode(*(x[:, 1] for x in dr))
    with pytest.raises(oracle.CapacityError):
        d.verify(*dr)  # 2 + 3 records > R = 4
    d.verify(*(x[:, :2] for x in dr))
    with pytest.raises(oracle.CapacityError):
        d.commit([3, 0])  # more than drafted
    with pytest.raises(oracle.CapacityError):
        d.commit([-1, 0])
    d.commit([2, 1])
    with pytest.raises(oracle.CapacityError):
        d.commit([0, 0])  # a verify is committed once
    d.flush(1)
    d.verify(*(x[:, :2] for x in dr))
    d.decode(*(x[:, 0] for x in dr))
    with pytest.raises(oracle.CapacityError):
        d.commit([1, 1])  # a decode step discards the pending drafts


# Planted mistakes: each plausible slip in the step, the replay formula or the
# fold, substituted into the oracle module, must fail at least one pin above.

_STEP = delta.delta_step
_REPLAY = delta.delta_replay_output
_FOLD = delta.delta_fold


def _parts(S, k, q):
    g = oracle.head_groups(S.shape[1], k.shape[1])
    kh, qh = k[:, g, :], q[:, g, :]
    return kh, qh, np.einsum("bhpn,bhn->bhp", S, kh)


def _finish(S_new, qh):
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, qh)


def _m_erase_not_decayed(S, a, b, v, k, q):  # alpha S - beta (S k) k^T + beta v k^T
    kh, qh, Sk = _parts(S, k, q)
    a4, b4 = a[:, :, None, None], b[:, :, None, None]
    return _finish(a4 * S - b4 * Sk[..., None] * kh[:, :, None, :] + b4 * v[..., None] * kh[:, :, None, :], qh)


def _m_no_erase(S, a, b, v, k, q):  # the outer-product rule with a write strength
    kh, qh, _ = _parts(S, k, q)
    return _finish(a[:, :, None, None] * S + b[:, :, None, None] * v[..., None] * kh[:, :, None, :], qh)


def _m_erase_sign(S, a, b, v, k, q):
    kh, qh, Sk = _parts(S, k, q)
    a4, b4 = a[:, :, None, None], b[:, :, None, None]
    return _finish(a4 * (S + b4 * Sk[..., None] * kh[:, :, None, :]) + b4 * v[..., None] * kh[:, :, None, :], qh)


def _m_write_without_beta(S, a, b, v, k, q):
    kh, qh, Sk = _parts(S, k, q)
    a4, b4 = a[:, :, None, None], b[:, :, None, None]
    return _finish(a4 * (S - b4 * Sk[..., None] * kh[:, :, None, :]) + v[..., None] * kh[:, :, None, :], qh)


def _m_erase_along_query(S, a, b, v, k, q):  # (S q) k^T in place of (S k) k^T
    kh, qh, _ = _parts(S, k, q)
    Sq = np.einsum("bhpn,bhn->bhp", S, qh)
    a4, b4 = a[:, :, None, None], b[:, :, None, None]
    return _finish(a4 * (S - b4 * Sq[..., None] * kh[:, :, None, :]) + b4 * v[..., None] * kh[:, :, None, :], qh)


def _m_old_state_output(S, a, b, v, k, q):
    S_new, _ = _STEP(S, a, b, v, k, q)
    _, qh, _ = _parts(S, k, q)
    return S_new, np.einsum("bhpn,bhn->bhp", S, qh)


def _m_swap_kq(S, a, b, v, k, q):
    return _STEP(S, a, b, v, q, k)


def _m_interleaved_groups(S, a, b, v, k, q):
    H, G = S.shape[1], k.shape[1]
    g = np.arange(H) % G
    kh, qh = k[:, g, :], q[:, g, :]
    Sk = np.einsum("bhpn,bhn->bhp", S, kh)
    a4, b4 = a[:, :, None, None], b[:, :, None, None]
    return _finish(a4 * (S - b4 * Sk[..., None] * kh[:, :, None, :]) + b4 * v[..., None] * kh[:, :, None, :], qh)


def _m_replay_forward_order(S_ckpt, alphas, betas, vs, ks, q):  # the query carried through the records forwards
    return _REPLAY(S_ckpt, alphas[::-1], betas[::-1], vs[::-1], ks[::-1], q)


def _m_replay_decay_before_erase(S_ckpt, alphas, betas, vs, ks, q):  # u <- alpha u - c k
    H = S_ckpt.shape[0]
    g = oracle.head_groups(H, q.shape[0])
    o = np.empty((H, S_ckpt.shape[1]))
    for head in range(H):
        u, val = np.array(q[g[head]], np.float64), np.zeros(S_ckpt.shape[1])
        for j in range(len(alphas) - 1, -1, -1):
            kj = ks[j, g[head]]
            c = betas[j, head] * float(kj @ u)
            val += c * vs[j, head]
            u = alphas[j, head] * u - c * kj
        o[head] = S_ckpt[head] @ u + val
    return o


def _m_fold_reversed(S_ckpt, alphas, betas, vs, ks):
    return _FOLD(S_ckpt, alphas[::-1], betas[::-1], vs[::-1], ks[::-1])


STEP_MUTANTS = [_m_erase_not_decayed, _m_no_erase, _m_erase_sign, _m_write_without_beta, _m_erase_along_query,
                _m_old_state_output, _m_swap_kq, _m_interleaved_groups]
FORM_MUTANTS = [("delta_replay_output", _m_replay_forward_order), ("delta_replay_output", _m_replay_decay_before_erase),
                ("delta_fold", _m_fold_reversed)]
PINS = [test_associative_memory_with_orthonormal_keys, test_full_strength_write_is_exact_for_any_decay,
        test_zero_write_strength_is_pure_decay, test_scalar_case_by_hand, test_replay_formula_and_fold_match_the_definition,
        test_pseudo_value_is_the_steps_write_term, test_hand_computed_two_step_example,
        test_verify_and_commit_of_the_hand_example, test_verify_keeps_the_projection_and_memory_properties,
        test_verify_matches_the_replay_formula, test_commit_applies_only_the_accepted_prefix]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(delta, name, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
            caught.append(False)
        except (AssertionError, ValueError, IndexError):
            caught.append(True)  # a failed pin, or a shape error, catches the mistake
    return caught


@pytest.mark.parametrize("mutant", STEP_MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_planted_mistakes_in_the_step(monkeypatch, mutant):
    assert any(_caught(monkeypatch, "delta_step", mutant)), f"no pin catches {mutant.__name__}"


@pytest.mark.parametrize("name,mutant", FORM_MUTANTS, ids=lambda x: getattr(x, "__name__", x))
def test_pins_catch_planted_mistakes_in_replay_and_fold(monkeypatch, name, mutant):
    assert any(_caught(monkeypatch, name, mutant)), f"no pin catches {mutant.__name__}"


def test_the_unmutated_oracle_passes_every_pin(monkeypatch):
    assert not any(_caught(monkeypatch, "delta_step", _STEP))


def test_pseudo_value_verify_form_matches_the_oracle():
    """The verify form a kernel evaluates from the checkpoint, the buffered pseudo-values
    and the drafts (checkpoint dots with each draft key and query, then a chain over the
    drafts) gives the oracle's verify outputs, and its w are the ones decode would write."""
    rng = np.random.default_rng(11)
    B, T, H, G, P, N, L = 2, 4, 4, 2, 5, 6, 8
    S0 = rng.standard_normal((B, H, P, N))
    d = delta.DeltaReplayOracle(S0, L=L, R=L + T, G=G)
    g = oracle.head_groups(H, G)
    recs = []  # committed (alpha, w, k) per step, w from the state before the step
    for _ in range(3):
        a, b, v, k, q = (x[:, 0] for x in _drafts(rng, B, 1, H, G, P, N))
        recs.append((a, delta.delta_pseudo_value(d.S, a, b, v, k), k))
        d.decode(a, b, v, k, q)
    al, be, v, k, q = _drafts(rng, B, T, H, G, P, N)
    O = d.verify(al, be, v, k, q)
    alphas = [r[0] for r in recs] + [al[:, t] for t in range(T)]  # [B,H] per record m = 1..c+T
    keys = [r[2] for r in recs] + [k[:, t] for t in range(T)]     # [B,G,N]
    ws = [r[1] for r in recs]                                      # grows by one per draft
    c = len(recs)

    def decay(i, m):  # product of alphas of records i+1..m (1-based; empty = 1)
        out = np.ones((B, H))
        for j in range(i + 1, m + 1):
            out = out * alphas[j - 1]
        return out

    def dot(x, y):  # group dots x_g . y_g, spread to the group's heads: [B,H]
        return np.einsum("bgn,bgn->bg", x, y)[:, g]

    for t in range(T):
        m = c + t + 1
        y = decay(0, m - 1)[..., None] * np.einsum("bhpn,bhn->bhp", S0, k[:, t][:, g])
        for i in range(1, m):
            y = y + (decay(i, m - 1) * dot(keys[i - 1], k[:, t]))[..., None] * ws[i - 1]
        ws.append(be[:, t][..., None] * (v[:, t] - al[:, t][..., None] * y))
        o = decay(0, m)[..., None] * np.einsum("bhpn,bhn->bhp", S0, q[:, t][:, g])
        for i in range(1, m + 1):
            o = o + (decay(i, m) * dot(keys[i - 1], q[:, t]))[..., None] * ws[i - 1]
        assert np.allclose(o, O[:, t], rtol=1e-11, atol=1e-11), t
    d.commit(np.array([2, 4]))
    for bb, a in enumerate((2, 4)):
        S_fold = S0[bb].copy()
        for i in range(c + a):
            S_fold = alphas[i][bb][:, None, None] * S_fold + ws[i][bb][..., None] * keys[i][bb][g][:, None, :]
        assert np.allclose(d.S[bb], S_fold, rtol=1e-11, atol=1e-11), bb
