"""Pins for the float64 oracle. These checks depend on no GPU.

Each pin ties the oracle to something other than itself: a hand-computed golden
case, the unrolled closed form, brute force with exact small-integer
arithmetic, degenerate special cases, and invariants the pages state. The
mutation test at the end plants plausible mistakes in copies of the oracle's
step, on the CPU, and checks that at least one pin catches each of them.
"""
import numpy as np
import pytest

import oracle
from oracle import conventional_step, head_groups, replay_output, unrolled_state, verify_outputs
from tests.golden_io import read_keyed

RNG = np.random.default_rng(1234)


def _rand_problem(B=2, H=4, P=5, N=3, G=2, rng=RNG):
    S = rng.normal(size=(B, H, P, N))
    return S


def _rand_step(B, H, P, N, G, rng=RNG, lo=0.2, hi=1.0):
    a = rng.uniform(lo, hi, size=(B, H))
    v = rng.normal(size=(B, H, P))
    k = rng.normal(size=(B, G, N))
    q = rng.normal(size=(B, G, N))
    return a, v, k, q


# ----------------------------------------------------------------------------- pins
def pin_golden(step) -> bool:
    """Hand-computed two-step example (tests/golden/hand_two_step.txt)."""
    g = read_keyed("hand_two_step.txt")
    S = g["S0"].reshape(1, 1, 2, 2)
    a = g["alpha"]
    S1, o1 = step(S, np.array([[a[0]]]), g["v1"].reshape(1, 1, 2), g["k1"].reshape(1, 1, 2), g["q1"].reshape(1, 1, 2))
    S2, o2 = step(S1, np.array([[a[1]]]), g["v2"].reshape(1, 1, 2), g["k2"].reshape(1, 1, 2), g["q2"].reshape(1, 1, 2))
    return (np.array_equal(S1.ravel(), g["S1"]) and np.array_equal(o1.ravel(), g["o1"])
            and np.array_equal(S2.ravel(), g["S2"]) and np.array_equal(o2.ravel(), g["o2"]))


def pin_closed_form(step, h=9) -> bool:
    """Recurrence == unrolled window sum, rel <= 1e-12 (unrolled equation, window of h records)."""
    B, H, P, N, G = 2, 4, 5, 3, 2
    rng = np.random.default_rng(7)
    S0 = rng.normal(size=(B, H, P, N))
    S = S0.copy()
    recs = []
    for _ in range(h):
        a, v, k, q = _rand_step(B, H, P, N, G, rng)
        S, _ = step(S, a, v, k, q)
        recs.append((a, v, k))
    ok = True
    for b in range(B):
        al = np.stack([r[0][b] for r in recs])
        vs = np.stack([r[1][b] for r in recs])
        ks = np.stack([r[2][b] for r in recs])
        ref = unrolled_state(S0[b], al, vs, ks)
        ok &= bool(np.max(np.abs(S[b] - ref)) <= 1e-12 * np.max(np.abs(ref)))
    return ok


def pin_bruteforce(step) -> bool:
    """alpha = 1 and orthonormal keys k_j = e_j: column j of S grows by exactly v_j.

    With small-integer v and S0 every operation is exact, so S_h = S0 + sum_j v_j e_j^T
    and o for q = e_i equals S0[:, i] + v_i (for i <= h).
    """
    B, H, P, N, G = 1, 2, 3, 4, 1
    rng = np.random.default_rng(3)
    S0 = rng.integers(-5, 6, size=(B, H, P, N)).astype(np.float64)
    S = S0.copy()
    expect = S0.copy()
    ok = True
    for j in range(N):
        v = rng.integers(-4, 5, size=(B, H, P)).astype(np.float64)
        k = np.zeros((B, G, N))
        k[0, 0, j] = 1.0
        q = np.zeros((B, G, N))
        q[0, 0, j] = 1.0
        S, o = step(S, np.ones((B, H)), v, k, q)
        expect[:, :, :, j] += v
        ok &= bool(np.array_equal(S, expect))
        ok &= bool(np.array_equal(o, S0[:, :, :, j] + v))
    return ok


def pin_zero_state(step) -> bool:
    """From a zero state one record gives o = (v k^T) q = v (k^T q) (output-only form, §05)."""
    B, H, P, N, G = 2, 2, 4, 3, 1
    rng = np.random.default_rng(5)
    a, v, k, q = _rand_step(B, H, P, N, G, rng)
    S, o = step(np.zeros((B, H, P, N)), a, v, k, q)
    kq = (k * q).sum(-1)  # [B,G]
    return bool(np.allclose(o, v * kq[:, :, None], rtol=1e-14, atol=0)) and bool(
        np.allclose(S, v[..., None] * k[:, :, None, :], rtol=1e-14, atol=0))


def pin_alpha_zero(step) -> bool:
    """alpha = 0 forgets everything: the state collapses to the last record."""
    B, H, P, N, G = 1, 2, 3, 3, 1
    rng = np.random.default_rng(9)
    S = rng.normal(size=(B, H, P, N))
    _, v, k, q = _rand_step(B, H, P, N, G, rng)
    S1, o = step(S, np.zeros((B, H)), v, k, q)
    return bool(np.array_equal(S1, v[..., None] * k[:, :, None, :]))


def pin_groups(step) -> bool:
    """Contiguous head groups: with H=4, G=2 heads 0,1 read group 0 and heads 2,3 read group 1."""
    B, H, P, N, G = 1, 4, 2, 3, 2
    S = np.zeros((B, H, P, N))
    v = np.ones((B, H, P))
    k = np.zeros((B, G, N))
    k[0, 0] = [1, 0, 0]
    k[0, 1] = [0, 0, 1]
    q = k.copy()
    S1, o = step(S, np.ones((B, H)), v, k, q)
    return (bool(np.all(S1[0, 0, :, 0] == 1) and np.all(S1[0, 1, :, 0] == 1))
            and bool(np.all(S1[0, 2, :, 2] == 1) and np.all(S1[0, 3, :, 2] == 1))
            and bool(np.all(o == 1)))


ALL_PINS = [pin_golden, pin_closed_form, pin_bruteforce, pin_zero_state, pin_alpha_zero, pin_groups]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_conventional_step_pins(pin):
    assert pin(conventional_step)


def test_head_groups_contiguous():
    assert list(head_groups(8, 2)) == [0, 0, 0, 0, 1, 1, 1, 1]
    with pytest.raises(ValueError):
        head_groups(6, 4)


def test_golden_output_only_form():
    """The output-only form reproduces o2 of the hand example from S0 and both records."""
    g = read_keyed("hand_two_step.txt")
    o2 = replay_output(g["S0"].reshape(1, 2, 2), g["alpha"].reshape(2, 1),
                       np.stack([g["v1"], g["v2"]]).reshape(2, 1, 2),
                       np.stack([g["k1"], g["k2"]]).reshape(2, 1, 2), g["q2"].reshape(1, 2))
    assert np.array_equal(o2.ravel(), g["o2"])


# ----------------------------------------------------------------- replay invariants
def _decode_run(L, R, steps, B=3, H=4, P=5, N=6, G=2, seed=0):
    rng = np.random.default_rng(seed)
    S0 = rng.normal(size=(B, H, P, N))
    orc = oracle.ReplayOracle(S0, L=L, R=R, G=G)
    return rng, orc


@pytest.mark.parametrize("L", [1, 2, 4, 5])
def test_replay_formula_equals_conventional_every_step(L):
    """Output-only replay from checkpoint + buffer equals the recurrence at every step,
    flush steps included (§03: outputs agree up to floating point)."""
    rng, orc = _decode_run(L, L, 0)
    B, H, P, N, G = orc.B, orc.H, orc.P, orc.N, orc.G
    for t in range(3 * L + 2):
        a, v, k, q = _rand_step(B, H, P, N, G, rng)
        ckpt_before = orc.ckpt.copy()
        recs_before = [list(r) for r in orc.records]
        o, flushed = orc.decode(a, v, k, q)
        assert np.array_equal(flushed, np.full(B, (t + 1) % L == 0))
        for b in range(B):
            recs = recs_before[b] + [(a[b], v[b], k[b])]
            al, vs, ks = (np.stack(x) for x in zip(*recs))
            o_rep = replay_output(ckpt_before[b], al, vs, ks, q[b])
            assert np.max(np.abs(o_rep - o[b])) <= 1e-12 * max(1.0, np.max(np.abs(o[b])))
            if flushed[b]:  # the new checkpoint is the unrolled state of all records
                S_unr = unrolled_state(ckpt_before[b], al, vs, ks)
                assert np.max(np.abs(S_unr - orc.ckpt[b])) <= 1e-12 * np.max(np.abs(S_unr))


def test_verify_formula_equals_scratch_recurrence():
    """O = S_ckpt Q D + V (W ⊙ K^T Q) equals running the drafts on a scratch state."""
    rng = np.random.default_rng(11)
    B, H, P, N, G, L, T = 2, 4, 3, 5, 2, 6, 3
    S0 = rng.normal(size=(B, H, P, N))
    orc = oracle.ReplayOracle(S0, L=L, R=L + T - 1, G=G)
    for _ in range(4):  # four committed records, no flush
        orc.decode(*_rand_step(B, H, P, N, G, rng))
    al = rng.uniform(0.2, 1, size=(B, T, H))
    v = rng.normal(size=(B, T, H, P))
    k = rng.normal(size=(B, T, G, N))
    q = rng.normal(size=(B, T, G, N))
    O = orc.verify(al, v, k, q)
    for b in range(B):
        recs = orc.records[b] + [(al[b, t], v[b, t], k[b, t]) for t in range(T)]
        a_, v_, k_ = (np.stack(x) for x in zip(*recs))
        O_f = verify_outputs(orc.ckpt[b], a_, v_, k_, q[b], int(orc.count[b]))
        assert np.max(np.abs(O_f - O[b])) <= 1e-12 * np.max(np.abs(O[b]))


def test_rollback_ignores_rejected_drafts():
    """After commit(a), later outputs do not depend on the rejected drafts (§05):
    replace them with garbage and every later output is bit-identical."""
    B, H, P, N, G, L, T = 3, 2, 4, 4, 1, 4, 3
    outs = []
    for garbage in (False, True):
        rng = np.random.default_rng(21)
        orc = oracle.ReplayOracle(rng.normal(size=(B, H, P, N)), L=L, R=L + T - 1, G=G)
        res = []
        for rnd in range(6):
            al = rng.uniform(0.2, 1, size=(B, T, H))
            v = rng.normal(size=(B, T, H, P))
            k = rng.normal(size=(B, T, G, N))
            q = rng.normal(size=(B, T, G, N))
            a = rng.integers(0, T + 1, size=B)
            if garbage:
                for b in range(B):
                    al[b, a[b]:] = 0.5
                    v[b, a[b]:] = 1e6
                    k[b, a[b]:] = -3e5
            O = orc.verify(al, v, k, q)
            orc.commit(a)
            orc.flush(L)
            # outputs of accepted drafts, which must be identical
            res.append([O[b, :a[b]].copy() for b in range(B)])
            o, _ = orc.decode(*_rand_step(B, H, P, N, G, rng))
            res.append(o.copy())
        outs.append((res, orc.S.copy(), orc.start.copy(), orc.count.copy()))
    (r0, S0, st0, c0), (r1, S1, st1, c1) = outs
    assert np.array_equal(S0, S1) and np.array_equal(st0, st1) and np.array_equal(c0, c1)
    for x, y in zip(r0, r1):
        if isinstance(x, list):
            for xb, yb in zip(x, y):
                assert np.array_equal(xb, yb)
        else:
            assert np.array_equal(x, y)


def test_pointer_bookkeeping_against_record_list():
    """Brute-force ring model: keep the live records as a list of absolute positions.

    The ring holds the records since the last flush, at slots (start + i) mod R.
    This model tracks absolute append positions and must agree with the oracle's
    (start, count) and flush events for random decode / verify / commit / flush sequences.
    """
    rng = np.random.default_rng(31)
    B, H, P, N, G, L, T = 4, 1, 2, 2, 1, 4, 3
    R = L + T - 1
    orc = oracle.ReplayOracle(rng.normal(size=(B, H, P, N)), L=L, R=R, G=G)
    folded = np.zeros(B, np.int64)  # absolute index of the first live record
    live = np.zeros(B, np.int64)  # number of live committed records
    for it in range(200):
        kind = rng.integers(0, 2)
        if kind == 0 and np.all(live + 1 <= R):
            _, flushed = orc.decode(*_rand_step(B, H, P, N, G, rng))
            live += 1
            exp_flush = live >= L
            assert np.array_equal(flushed, exp_flush)
            folded[exp_flush] += live[exp_flush]
            live[exp_flush] = 0
        elif np.all(live + T <= R):
            al = rng.uniform(0.2, 1, size=(B, T, H))
            orc.verify(al, rng.normal(size=(B, T, H, P)), rng.normal(size=(B, T, G, N)),
                       rng.normal(size=(B, T, G, N)))
            a = rng.integers(0, T + 1, size=B)
            orc.commit(a)
            live += a
            m = orc.flush(L)
            assert np.array_equal(m, live >= L)
            folded[live >= L] += live[live >= L]
            live[live >= L] = 0
        assert np.array_equal(orc.count, live)
        assert np.array_equal(orc.start, folded % R)


def test_capacity_and_commit_errors():
    B, H, P, N, G, L, T = 1, 1, 2, 2, 1, 4, 3
    orc = oracle.ReplayOracle(np.zeros((B, H, P, N)), L=L, R=L + T - 1, G=G)
    z = np.zeros
    with pytest.raises(oracle.CapacityError):
        orc.commit(np.array([0]))
    orc.verify(np.ones((B, T, H)), z((B, T, H, P)), z((B, T, G, N)), z((B, T, G, N)))
    with pytest.raises(oracle.CapacityError):
        orc.commit(np.array([T + 1]))
    orc.commit(np.array([T]))
    with pytest.raises(oracle.CapacityError):  # count 3 + T 3 = 6 = R is fine, 7 is not
        orc.verify(np.ones((B, T + 1, H)), z((B, T + 1, H, P)), z((B, T + 1, G, N)), z((B, T + 1, G, N)))
    with pytest.raises(ValueError):
        orc.flush(0)


def test_commit_equals_decode_of_accepted_prefix():
    """Committing a drafts leaves the same state as decoding those a records one by one
    (no flush in between), which is what 'oracle replaying only accepted tokens' means."""
    rng = np.random.default_rng(41)
    B, H, P, N, G, L, T = 2, 2, 3, 4, 1, 8, 4
    S0 = rng.normal(size=(B, H, P, N))
    A = oracle.ReplayOracle(S0, L=L, R=L + T - 1, G=G)
    al = rng.uniform(0.2, 1, size=(B, T, H))
    v = rng.normal(size=(B, T, H, P))
    k = rng.normal(size=(B, T, G, N))
    q = rng.normal(size=(B, T, G, N))
    A.verify(al, v, k, q)
    A.commit(np.array([T, T]))
    S = S0.copy()
    for t in range(T):
        S, _ = conventional_step(S, al[:, t], v[:, t], k[:, t], q[:, t])
    assert np.array_equal(A.S, S)


# ------------------------------------------------------------------- mutation test
def _m_decay_after(S, a, v, k, q):
    g = head_groups(S.shape[1], k.shape[1])
    Sn = a[:, :, None, None] * (S + v[..., None] * k[:, g][:, :, None, :])
    return Sn, (Sn * q[:, g][:, :, None, :]).sum(-1)


def _m_old_state_output(S, a, v, k, q):
    Sn, _ = conventional_step(S, a, v, k, q)
    g = head_groups(S.shape[1], k.shape[1])
    return Sn, (S * q[:, g][:, :, None, :]).sum(-1)


def _m_swap_kq(S, a, v, k, q):
    return conventional_step(S, a, v, q, k)


def _m_interleaved_groups(S, a, v, k, q):
    H, G = S.shape[1], k.shape[1]
    g = np.arange(H) % G
    Sn = a[:, :, None, None] * S + v[..., None] * k[:, g][:, :, None, :]
    return Sn, (Sn * q[:, g][:, :, None, :]).sum(-1)


def _m_no_decay(S, a, v, k, q):
    return conventional_step(S, np.ones_like(a), v, k, q)


def _m_minus(S, a, v, k, q):
    return conventional_step(S, a, -v, k, q)


def _m_transposed(S, a, v, k, q):
    g = head_groups(S.shape[1], k.shape[1])
    outer = k[:, g][:, :, :, None] * v[:, :, None, :]  # k v^T: only conforms when P == N
    Sn = a[:, :, None, None] * S + outer
    return Sn, (Sn * q[:, g][:, :, None, :]).sum(-1)


def _m_decay_squared(S, a, v, k, q):
    return conventional_step(S, a * a, v, k, q)


MUTANTS = [_m_decay_after, _m_old_state_output, _m_swap_kq, _m_interleaved_groups,
           _m_no_decay, _m_minus, _m_transposed, _m_decay_squared]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_planted_mistakes(mutant):
    caught = []
    for pin in ALL_PINS:
        try:
            caught.append(not pin(mutant))
        except (ValueError, IndexError):
            caught.append(True)  # a shape error is a caught mistake too
    assert any(caught), f"no pin catches {mutant.__name__}"


def _replay_wrong_w(S_ckpt, alphas, vs, ks, q):
    """Planted index mistake: w_j = gamma_{j:h} instead of gamma_{j+1:h}."""
    H = S_ckpt.shape[0]
    g = head_groups(H, q.shape[0])
    h = len(alphas)
    o = np.empty((H, S_ckpt.shape[1]))
    for head in range(H):
        a = alphas[:, head]
        o[head] = np.prod(a) * (S_ckpt[head] @ q[g[head]])
        for j in range(1, h + 1):
            o[head] += np.prod(a[j - 1:]) * float(ks[j - 1, g[head]] @ q[g[head]]) * vs[j - 1, head]
    return o


def test_invariant_catches_planted_replay_index_mistake():
    rng = np.random.default_rng(2)
    H, P, N = 2, 3, 4
    S = rng.normal(size=(H, P, N))
    al = rng.uniform(0.2, 0.9, size=(3, H))
    vs = rng.normal(size=(3, H, P))
    ks = rng.normal(size=(3, 1, N))
    q = rng.normal(size=(1, N))
    good = replay_output(S, al, vs, ks, q)
    bad = _replay_wrong_w(S, al, vs, ks, q)
    St = S.copy()[None]
    for j in range(3):
        St, o = conventional_step(St, al[j][None], vs[j][None], ks[j][None], q[None])
    assert np.allclose(good, o[0], rtol=1e-12)
    assert not np.allclose(bad, o[0], rtol=1e-6)
