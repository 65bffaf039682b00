"""Pins of the oracle's random-number, sampling and verification code.

Each test checks the oracle against something other than itself: published
known-answer vectors, exact integer arithmetic, closed forms from the
speculative-sampling rule ("DFlash vs DFlash 2" blog, section "The problem:
one expensive token at a time"), or chi-square tests of the lossless claim.
"""

import os

import numpy as np
import pytest
from scipy import stats

from oracle import fixedpoint, philox, sampling, verify

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ Philox

def test_philox_known_answer_vectors():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([int(t, 16) for t in line.replace("->", " ").split()])
    assert len(rows) == 3
    for r in rows:
        out = philox.philox4x32_10(r[0:4], r[4:6])
        assert [int(x) for x in out] == r[6:10]


def test_philox_uniformity_chi_square():
    n = 200_000
    u24 = philox.uniform24(12345, 7, np.arange(n, dtype=np.uint64), philox.PURPOSE_ACCEPT)
    counts = np.bincount((u24 >> np.uint64(18)).astype(np.int64), minlength=64)
    chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < stats.chi2.ppf(1 - 1e-4, 63)
    u64 = philox.uniform64(99, 3, np.arange(n, dtype=np.uint64), philox.PURPOSE_RESIDUAL)
    counts = np.bincount((u64 >> np.uint64(58)).astype(np.int64), minlength=64)
    chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < stats.chi2.ppf(1 - 1e-4, 63)


def test_philox_streams_differ_by_purpose_and_position():
    a = philox.block(5, 0, 0, 0)
    b = philox.block(5, 0, 0, 1)
    c = philox.block(5, 0, 1, 0)
    d = philox.block(6, 0, 0, 0)
    e = philox.block(5, 1 << 32, 0, 0)     # high word of the step
    outs = {tuple(int(x) for x in v) for v in (a, b, c, d, e)}
    assert len(outs) == 5


# -------------------------------------------------------------- fixed point

def test_mulhi64_matches_python_integers():
    rng = np.random.default_rng(0)
    a = rng.integers(0, 2 ** 63, 1000, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    b = rng.integers(0, 2 ** 63, 1000, dtype=np.uint64)
    edge = np.array([0, 1, 2 ** 32 - 1, 2 ** 32, 2 ** 64 - 1], dtype=np.uint64)
    a = np.concatenate([a, edge, edge])
    b = np.concatenate([b, edge, edge[::-1]])
    got = fixedpoint.mulhi64(a, b)
    want = [(int(x) * int(y)) >> 64 for x, y in zip(a, b)]
    assert [int(g) for g in got] == want


def test_fixed_point_draw_matches_scalar_integer_draw():
    rng = np.random.default_rng(1)
    for _ in range(200):
        V = int(rng.integers(1, 12))
        w = rng.random(V).astype(np.float32)
        w[rng.random(V) < 0.3] = 0.0
        if w.sum() == 0:
            w[0] = 0.5
        w = (w / w.sum()).astype(np.float32)
        u = rng.integers(0, 2 ** 64 - 1, dtype=np.uint64, endpoint=True)
        got = fixedpoint.sample_rows(fixedpoint.to_fixed(w)[None], np.array([u]))[0]
        assert got == fixedpoint.sample_row_exact(w, u)


def test_fixed_point_draw_boundaries_are_exact():
    """The set of u64 that selects v is exactly [ceil(C_{v-1} 2^64 / Z),
    ceil(C_v 2^64 / Z)), so P(v) differs from R_v / Z by less than 2^-64."""
    w = np.array([0.1, 0.0, 0.25, 0.4, 0.25], dtype=np.float32)
    R = [int(x) for x in fixedpoint.to_fixed(w)]
    Z = sum(R)
    cdf = np.cumsum(R).tolist()
    for v in range(len(R)):
        if R[v] == 0:
            continue
        lo = -((-(cdf[v] - R[v]) << 64) // Z)      # ceil
        hi = -((-(cdf[v]) << 64) // Z)
        assert abs((hi - lo) / 2 ** 64 - R[v] / Z) < 2 ** -63
        for u in (lo, hi - 1):
            assert fixedpoint.sample_rows(np.array([R], dtype=np.uint64),
                                          np.array([u], dtype=np.uint64))[0] == v
        if lo > 0:
            assert fixedpoint.sample_rows(np.array([R], dtype=np.uint64),
                                          np.array([lo - 1], dtype=np.uint64))[0] < v


def test_to_fixed_is_exact_floor():
    vals = np.array([0.0, 2.0 ** -45, 2.0 ** -46, 0.5, 1.0, 0.3], dtype=np.float32)
    got = fixedpoint.to_fixed(vals)
    from fractions import Fraction
    want = [int(Fraction(float(v)) * 2 ** 45) for v in vals]   # int() floors positives
    assert [int(g) for g in got] == want


# ------------------------------------------------------------------ top-p

def test_top_p_matches_subset_brute_force():
    """The nucleus is the subset of minimal size reaching mass top_p and,
    among those, the one of maximal mass (unique for distinct values)."""
    import itertools
    rng = np.random.default_rng(2)
    for _ in range(40):
        V = 7
        p = rng.dirichlet(np.ones(V) * 0.7)
        top_p = float(rng.uniform(0.3, 0.99))
        best = None
        for m in range(1, V + 1):
            cands = [s for s in itertools.combinations(range(V), m) if p[list(s)].sum() >= top_p]
            if cands:
                best = max(cands, key=lambda s: p[list(s)].sum())
                break
        keep = sampling.top_p_keep(p[None], top_p)[0]
        assert set(np.flatnonzero(keep)) == set(best)


def test_probs_temperature_softmax_matches_scipy():
    from scipy.special import softmax as sp_softmax
    rng = np.random.default_rng(3)
    z = rng.normal(0, 2, (5, 50))
    np.testing.assert_allclose(sampling.probs(z, 0.7, 1.0), sp_softmax(z / 0.7, axis=-1), rtol=1e-12)
    p = sampling.probs(z, 0.7, 0.9)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-12)
    assert (p > 0).sum() < p.size


def test_top_p_ties_go_to_lower_id():
    p = np.array([[0.3, 0.2, 0.2, 0.2, 0.1]])
    keep = sampling.top_p_keep(p, 0.65)
    assert keep.tolist() == [[True, True, True, False, False]]


# ------------------------------------------------------------ greedy verify

def test_greedy_accepts_longest_matching_prefix():
    rng = np.random.default_rng(4)
    B, gamma, V = 9, 6, 40
    t = rng.normal(size=(B, gamma, V)).astype(np.float32)
    a = t.argmax(-1)
    y = np.empty((B, gamma - 1), dtype=np.int64)
    for b in range(B):
        k = min(b, gamma - 1)                 # request b matches exactly k drafts
        y[b] = a[b, :gamma - 1]
        if k < gamma - 1:
            y[b, k] = (a[b, k] + 1) % V
            y[b, k + 1:] = rng.integers(0, V, gamma - 2 - k)
    n, tok = verify.greedy(t, y)
    for b in range(B):
        k = min(b, gamma - 1)
        assert n[b] == k
        assert tok[b, :k].tolist() == a[b, :k].tolist()
        assert tok[b, k] == a[b, k]             # correction, or the bonus when k = gamma-1
        assert (tok[b, k + 1:] == -1).all()


def test_greedy_ties_go_to_lowest_id():
    t = np.zeros((1, 3, 8), dtype=np.float32)
    t[0, :, 3] = 1.0
    t[0, :, 5] = 1.0
    n, tok = verify.greedy(t, np.array([[3, 5]]))
    assert n[0] == 1 and tok[0].tolist() == [3, 3, -1]


# ----------------------------------------------------------- sampled verify

def _dists(rng, gamma, V, conc=1.0):
    p = rng.dirichlet(np.ones(V) * conc, size=(1, gamma)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * conc, size=(1, gamma - 1)).astype(np.float32)
    return p, q


def _trials(p, q, T, seed=77):
    """T independent cycles: steps 0..T-1 of one request with the same p, q."""
    B = T
    P = np.broadcast_to(p, (B,) + p.shape[1:])
    Q = np.broadcast_to(q, (B,) + q.shape[1:])
    # every trial is a distinct Philox stream: vary the seed per trial
    seeds = (np.arange(B, dtype=np.uint64) * np.uint64(2654435761) + np.uint64(seed))
    y = sampling.draft_draw(Q, seeds, 11)
    n, tok = verify.sampled(P, Q, y, seeds, 11)
    return n, tok


def _chi2_ok(samples, probs):
    V = len(probs)
    counts = np.bincount(samples, minlength=V)
    exp = probs * len(samples)
    m = exp > 0
    assert counts[~m].sum() == 0
    chi2 = ((counts[m] - exp[m]) ** 2 / exp[m]).sum()
    return chi2 < stats.chi2.ppf(1 - 1e-3, m.sum() - 1)


def test_committed_tokens_are_distributed_as_target_chi_square():
    rng = np.random.default_rng(5)
    gamma, V, T = 4, 16, 1_000_000
    p, q = _dists(rng, gamma, V)
    n, tok = _trials(p, q, T)
    P = p[0].astype(np.float64)
    assert _chi2_ok(tok[:, 0], P[0] / P[0].sum())
    for k in range(1, gamma):
        reached = n >= k
        assert _chi2_ok(tok[reached, k], P[k] / P[k].sum())
    bonus = n == gamma - 1
    assert bonus.sum() > 1000
    assert _chi2_ok(tok[bonus, gamma - 1], P[gamma - 1] / P[gamma - 1].sum())


def test_acceptance_rate_and_expected_tau_closed_forms():
    rng = np.random.default_rng(6)
    gamma, V, T = 5, 16, 400_000
    p, q = _dists(rng, gamma, V, conc=2.0)
    n, _ = _trials(p, q, T, seed=3)
    beta = [verify.acceptance_probability(p[0, i], q[0, i]) for i in range(gamma - 1)]
    rate0 = (n >= 1).mean()
    assert abs(rate0 - beta[0]) < 5 * np.sqrt(beta[0] * (1 - beta[0]) / T)
    tau = n + 1
    assert abs(tau.mean() - verify.expected_tau(beta)) < 5 * tau.std() / np.sqrt(T)


def test_p_equal_q_always_accepts_and_draws_bonus_from_p():
    rng = np.random.default_rng(7)
    gamma, V, T = 4, 16, 200_000
    p, _ = _dists(rng, gamma, V)
    q = p[:, :gamma - 1].copy()
    n, tok = _trials(p, q, T, seed=9)
    assert (n == gamma - 1).all()
    P = p[0, gamma - 1].astype(np.float64)
    assert _chi2_ok(tok[:, gamma - 1], P / P.sum())


def test_one_hot_q_on_impossible_token_always_rejects_to_p():
    rng = np.random.default_rng(8)
    gamma, V, T = 3, 16, 200_000
    p, _ = _dists(rng, gamma, V)
    p[0, 0, 4] = 0.0
    p[0, 0] /= p[0, 0].sum()
    q = np.zeros((1, gamma - 1, V), dtype=np.float32)
    q[0, :, 4] = 1.0
    n, tok = _trials(p, q, T, seed=10)
    assert (n == 0).all()
    P = p[0, 0].astype(np.float64)
    assert _chi2_ok(tok[:, 0], P / P.sum())


def test_accept_test_is_exact_at_the_boundary():
    """u*q < p decides exactly: construct p(y) = u*q(y) for the drawn u."""
    seed, step = np.array([42], dtype=np.uint64), 5
    u24 = int(philox.uniform24(seed, step, 0, philox.PURPOSE_ACCEPT)[0])
    qy = np.float32(0.5)
    py_equal = np.float32(u24 * 2.0 ** -24 * 0.5)         # exactly u*q
    assert float(py_equal) == u24 * 2.0 ** -24 * 0.5
    V = 4
    for py, want_accept in ((py_equal, False), (np.nextafter(py_equal, np.float32(1)), True)):
        p = np.full((1, 2, V), 0.0, dtype=np.float32)
        p[0, 0, 1] = py
        p[0, 0, 2] = 1 - py
        p[0, 1, :] = 0.25
        q = np.zeros((1, 1, V), dtype=np.float32)
        q[0, 0, 1] = qy
        q[0, 0, 3] = 0.5
        n, _ = verify.sampled(p, q, np.array([[1]]), seed, step)
        assert (n[0] == 1) == want_accept


def test_draft_draw_follows_q():
    rng = np.random.default_rng(12)
    V, T = 16, 300_000
    q = rng.dirichlet(np.ones(V), size=(1, 1)).astype(np.float32)
    Q = np.broadcast_to(q, (T, 1, V))
    seeds = np.arange(T, dtype=np.uint64) + np.uint64(1000)
    y = sampling.draft_draw(Q, seeds, 0)[:, 0]
    Qd = q[0, 0].astype(np.float64)
    assert _chi2_ok(y, Qd / Qd.sum())


@pytest.mark.parametrize("gamma", [2, 8])
def test_sampled_token_layout(gamma):
    rng = np.random.default_rng(13)
    B, V = 64, 32
    p = rng.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, gamma - 1)).astype(np.float32)
    seeds = np.arange(B, dtype=np.uint64)
    y = sampling.draft_draw(q, seeds, 1)
    n, tok = verify.sampled(p, q, y, seeds, 1)
    for b in range(B):
        assert (tok[b, :n[b]] == y[b, :n[b]]).all()
        assert 0 <= tok[b, n[b]] < V
        assert (tok[b, n[b] + 1:] == -1).all()
