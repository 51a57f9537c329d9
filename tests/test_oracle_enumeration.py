"""Exact-enumeration and decision-margin pins of the oracle (CPU).

Exact enumeration ("Speculative Decoding: How Draft-Model Parallelism Cuts LLM
Inference Latency", sections "The proof of exactness" and "Acceptance rate
equals 1 minus total variation distance"): on tiny vocabularies the oracle is
run on EVERY draft-token tuple (weighted by its draft probability prod_i
q_i(x_i), i.e. the tokens a draft model draws) and on every point of a
stratified midpoint grid of the accept uniforms r_i ((j + 1/2) / N per
position).  The fraction of grid points on which the oracle's own accept /
stop decisions produce an outcome is then that outcome's probability up to
the grid error, and is compared with what the page fixes:

  * P(x_1 accepted and x_1 = x) = min(p_1(x), q_1(x))   (the accepted part of
    the exactness proof: the remainder p - min(p, q) = (p - q)+ is what the
    residual draw supplies);
  * P(x_1..x_j all accepted, x_i = t_i) = prod_i min(p_i(t_i), q_i(t_i));
  * P(k = j) = alpha_1 ... alpha_j (1 - alpha_{j+1}), P(k = gamma) =
    alpha_1 ... alpha_gamma, alpha_i = sum_x min(p_i, q_i) = 1 - TVD(p_i, q_i)
    (Theorem 3.5 and the first-rejection stop);
  * the emitted prefix is the accepted draft tokens.

A single threshold a = min(1, p/q) is hit by floor(a N + 1/2) of the N
midpoints, so each factor is within 1/(2N) of a and a product of m factors
within m/(2N): that is the bound on arbitrary (p, q).  The designed cases put
every ratio p(x)/q(x) on a multiple of 1/16 (the logits are log-probabilities
rounded to float32, off by ~1e-7), where a 16-point grid is exact up to that
rounding, so they are checked to 1e-6 at gamma up to 3.

The residual draw's trials are enumerated the same way: with the race forced
to draw a given x (its uniform set to 1, i.e. an arrival at time zero) and the
trial's acceptance uniform v on a midpoint grid, the fraction of accepted
trials is max(0, 1 - q(x)/p(x)) within 1/(2N); the race draws x with
probability p(x) (pinned by the chi-square tests of test_oracle_pins), so a
trial emits x with probability (p - q)+(x).

Decision margins (the near-tie accounting of the GPU-vs-oracle rule): cases
whose margins are known by construction -- r set to p/q (1 -+ 1e-7); a race
whose two earliest arrivals are in the ratio 1 + 1e-7; a trial whose
acceptance uniform puts 1 - v at q/p (1 + 1e-7) -- must report exactly that
margin, and only decisions on the path that produced the output count.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GRID_DESIGNED = 16


# ------------------------------------------------------------------ helpers
def _designed_pair(rng, V):
    """(p, q) with every ratio p(x)/q(x) < 1 a multiple of 1/16 and at least
    one id with p >= q (it takes the rest of p's mass)."""
    q = rng.integers(1, 9, size=V).astype(float)
    q /= q.sum()
    m = rng.integers(1, GRID_DESIGNED + 1, size=V)
    m[rng.integers(V)] = GRID_DESIGNED
    p = np.where(m < GRID_DESIGNED, m / GRID_DESIGNED * q, q)
    extra = 1.0 - p.sum()
    top = m == GRID_DESIGNED
    p[top] += extra / top.sum()
    return p, q


def _logits(prob):
    return np.log(prob).astype(np.float32)


def _probs(z):
    """p = softmax of the float32 logits in float64 (library routine)."""
    return softmax(np.asarray(z, np.float64))


def _enumerate(zt, zd, N):
    """Run the oracle on every draft tuple and every point of the r grid.
    zt [gamma+1, V], zd [gamma, V] float32.  Returns (tuples [n_t, gamma],
    weights [n_t], per tuple: accept counts [n_t, N^gamma] and out tokens)."""
    g, V = zd.shape
    q = [_probs(zd[i]) for i in range(g)]
    tuples = np.array(list(itertools.product(range(V), repeat=g)), np.int32)
    weights = np.array([np.prod([q[i][t[i]] for i in range(g)]) for t in tuples])
    mids = ((np.arange(N) + 0.5) / N).astype(np.float32)
    grid = np.array(list(itertools.product(mids, repeat=g)), np.float32)  # [N^g, g]
    n_t, n_r = len(tuples), len(grid)
    B = n_t * n_r
    tgt = np.broadcast_to(zt, (B, g + 1, V))
    drf = np.broadcast_to(zd, (B, g, V))
    toks = np.repeat(tuples, n_r, axis=0)
    r = np.tile(grid, (n_t, 1))
    keys = np.arange(B, dtype=np.uint64)
    out = oracle.verify_chain(tgt, drf, toks, r, keys, 1.0)
    assert (out["status"] == 0).all()
    k = out["accept_count"].reshape(n_t, n_r)
    toks_out = out["out_tokens"].reshape(n_t, n_r, g + 1)
    return tuples, weights, k, toks_out, grid


def _check_enumeration(zt, zd, N, tol_fn):
    g, V = zd.shape
    p = [_probs(zt[i]) for i in range(g + 1)]
    q = [_probs(zd[i]) for i in range(g)]
    mins = [np.minimum(p[i], q[i]) for i in range(g)]
    alpha = [m.sum() for m in mins]
    tuples, weights, k, toks_out, _ = _enumerate(zt, zd, N)

    # the emitted prefix is the accepted draft tokens, then one id, then -1
    for ti, t in enumerate(tuples):
        for j in range(g + 1):
            sel = k[ti] == j
            if not sel.any():
                continue
            assert (toks_out[ti][sel][:, :j] == t[:j]).all()
            last = toks_out[ti][sel][:, j]
            assert ((last >= 0) & (last < V)).all()
            assert (toks_out[ti][sel][:, j + 1:] == -1).all()

    # P(k = j): first-rejection stop with per-position acceptance alpha_i
    for j in range(g + 1):
        got = float((weights[:, None] * (k == j)).sum(axis=1).sum() / k.shape[1])
        want = np.prod(alpha[:j]) * (1.0 - alpha[j] if j < g else 1.0)
        assert abs(got - want) <= tol_fn(j + 1 if j < g else g), (j, got, want)

    # P(x_1 accepted, x_1 = x) = min(p_1(x), q_1(x))
    for x in range(V):
        sel = tuples[:, 0] == x
        got = float((weights[sel, None] * (k[sel] >= 1)).sum() / k.shape[1])
        assert abs(got - mins[0][x]) <= tol_fn(1), (x, got, mins[0][x])

    # P(x_1..x_j accepted with these tokens) = prod_i min(p_i, q_i)(t_i)
    for j in range(1, g + 1):
        for pre in itertools.product(range(V), repeat=j):
            sel = (tuples[:, :j] == pre).all(axis=1)
            got = float((weights[sel, None] * (k[sel] >= j)).sum() / k.shape[1])
            want = np.prod([mins[i][pre[i]] for i in range(j)])
            assert abs(got - want) <= tol_fn(j), (pre, got, want)


# --------------------------------------------------------- exact enumeration
@pytest.mark.parametrize("gamma,V,seed", [(1, 4, 0), (1, 8, 1), (2, 3, 2), (2, 5, 3), (3, 3, 4), (3, 4, 5)])
def test_enumeration_designed_thresholds(gamma, V, seed):
    """Every ratio p/q on the 16-point grid: the enumeration is exact up to
    the float32 rounding of the logits."""
    rng = np.random.default_rng(seed)
    zt = np.zeros((gamma + 1, V), np.float32)
    zd = np.zeros((gamma, V), np.float32)
    for i in range(gamma):
        p, q = _designed_pair(rng, V)
        zt[i], zd[i] = _logits(p), _logits(q)
    zt[gamma] = rng.normal(0, 1, V).astype(np.float32)
    _check_enumeration(zt, zd, GRID_DESIGNED, lambda m: 1e-6)


@pytest.mark.parametrize("gamma,V,N,seed", [(1, 3, 4096, 10), (1, 5, 4096, 11), (1, 8, 4096, 12),
                                            (2, 4, 256, 13), (3, 3, 32, 14)])
def test_enumeration_arbitrary_pairs(gamma, V, N, seed):
    """Arbitrary (p, q): each enumerated probability within the grid bound
    m / (2N) of its closed form (m = accept / reject factors involved)."""
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, (gamma + 1, V)).astype(np.float32)
    zd = (zt[:gamma] + rng.normal(0, 1.0, (gamma, V))).astype(np.float32)
    _check_enumeration(zt, zd, N, lambda m: m / (2.0 * N) + 1e-12)


def test_enumeration_identical_models_accept_everything():
    """q = p: every grid point of every tuple accepts every draft token."""
    zt = np.array([[0.3, -1.0, 2.0], [1.0, 0.0, -0.5], [0.0, 0.0, 0.0]], np.float32)
    zd = zt[:2].copy()
    tuples, weights, k, _, _ = _enumerate(zt, zd, 8)
    assert (k == 2).all()


def test_enumeration_zero_target_probability_always_rejects():
    """p(x) = 0 (a -inf target logit): a draft token x is rejected at every
    grid point, including r at the top of its range."""
    zt = np.array([[-np.inf, 0.0, 1.0], [0.0, 0.0, 0.0]], np.float32)
    zd = np.array([[2.0, 0.0, 1.0]], np.float32)
    tuples, weights, k, toks_out, _ = _enumerate(zt, zd, 64)
    assert (k[tuples[:, 0] == 0] == 0).all()
    assert (toks_out[tuples[:, 0] == 0][:, :, 0] != 0).all()  # the rejected id is never emitted


# ------------------------------------------------- residual trials, enumerated
TOKEN, ACCEPT = oracle.STREAM_TOKEN, oracle.STREAM_ACCEPT


def _forced_trial_hook(x_first, x_later, N):
    """Trial 0's race draws x_first (uniform 1: arrival at time zero) and its
    acceptance uniform is grid point `key`; later trials draw x_later with
    v = 2^-24 (accepted whenever p(x_later) > q(x_later))."""
    def fn(key, stream, trial, pos, n):
        if stream == TOKEN:
            want = x_first if trial == 0 else x_later
            return 1.0 if n == want else 0.5
        if stream == ACCEPT:
            return (key + 0.5) / N if trial == 0 else 2.0 ** -24
        return 0.5
    return fn


@pytest.mark.parametrize("V,seed", [(3, 20), (5, 21), (8, 22)])
def test_trial_acceptance_enumerated(V, seed):
    """A residual trial that drew x accepts with probability
    max(0, 1 - q(x)/p(x)) (grid of N acceptance uniforms), so it emits x with
    probability p(x) max(0, 1 - q/p) = (p - q)+(x), whose sum is Z."""
    N = 1024
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.0, (2, V)).astype(np.float32)
    zd = (zt[:1] + rng.normal(0, 1.0, (1, V))).astype(np.float32)
    p, q = _probs(zt[0]), _probs(zd[0])
    x_rej = int(np.argmax(q / p))         # the draft token: q > p, rejected at r = 1
    x_later = int(np.argmax(p / q))       # p > q: later trials accept it
    assert q[x_rej] > p[x_rej] and p[x_later] > 1.001 * q[x_later]
    emitted = np.zeros(V)
    for x in range(V):
        B = N
        tgt = np.broadcast_to(zt, (B, 2, V))
        drf = np.broadcast_to(zd, (B, 1, V))
        toks = np.full((B, 1), x_rej, np.int32)
        r = np.ones((B, 1), np.float32)
        keys = np.arange(B, dtype=np.uint64)
        with oracle.uniform_override(_forced_trial_hook(x, x_later, N)):
            out = oracle.verify_chain(tgt, drf, toks, r, keys, 1.0, threads=1)
        assert (out["accept_count"] == 0).all()
        first = out["trials"] == 1
        assert (out["out_tokens"][first, 0] == x).all()
        assert (out["out_tokens"][~first, 0] == x_later).all()
        frac = first.mean()
        want = max(0.0, 1.0 - q[x] / p[x])
        assert abs(frac - want) <= 1.0 / (2 * N) + 1e-12, (x, frac, want)
        emitted[x] = p[x] * frac
    resid = np.maximum(p - q, 0.0)
    np.testing.assert_allclose(emitted, resid, atol=1.0 / (2 * N))
    assert abs(emitted.sum() - 0.5 * np.abs(p - q).sum()) <= V / (2 * N)


# ------------------------------------------------------------- decision margins
def _run_one(zt, zd, toks, r, hook, want_Z=False):
    g = zd.shape[0]
    with oracle.uniform_override(hook):
        return oracle.verify_chain(zt[None], zd[None], np.asarray(toks, np.int32)[None],
                                   np.asarray(r, np.float32)[None], np.array([7], np.uint64), 1.0,
                                   want_Z=want_Z, threads=1)


def _table_hook(table, default=0.5):
    """Uniform (stream, n) -> value for every trial and position."""
    def fn(key, stream, trial, pos, n):
        return table.get((stream, n), default)
    return fn


def test_accept_margin_is_the_ratio_gap():
    """|r - p/q| with r = p/q (1 - 1e-7) (accepted) and (1 + 1e-7) (rejected,
    then a trial with a wide margin and the race forced)."""
    zt = np.array([[0.0, 0.8, -0.4], [0.1, 0.2, 0.3]], np.float32)
    zd = np.array([[0.5, 0.1, -0.2]], np.float32)
    p, q = _probs(zt[0]), _probs(zd[0])
    x = 0
    ratio = p[x] / q[x]
    assert ratio < 1
    for sgn in (-1, +1):
        r = np.float32(ratio * (1 + sgn * 1e-7))
        want = abs(float(r) - ratio)
        assert 5e-9 < want < 2e-7
        # accepted: bonus race forced onto id 0 (margin +inf); rejected: the
        # trial draws id 1 (p > q there) with v putting 1 - v far from q/p.
        x_res = int(np.argmax(p / q))
        v = 0.5 * (1 - q[x_res] / p[x_res])
        hook = _table_hook({(TOKEN, 0 if sgn < 0 else x_res): 1.0, (ACCEPT, 0): v})
        out = _run_one(zt, zd, [x], [r], hook)
        assert out["accept_count"][0] == (1 if sgn < 0 else 0)
        assert abs(out["margin"][0] - want) <= 1e-12, (out["margin"][0], want)


def test_race_margin_is_the_log_gap_of_the_two_earliest_arrivals():
    """Bonus race over three ids with arrivals E_x / p(x): the two earliest in
    the ratio 1 + d give the margin ln(1 + d); the earlier one wins."""
    zt = np.array([[0.2, 0.2, 0.2], [0.0, 1.0, -1.0]], np.float32)
    zd = zt[:1].copy()                     # q = p: accepted for any r (margin |r - 1|)
    pb = _probs(zt[1])
    for d, first in ((1e-7, 0), (1e-7, 1), (0.25, 2)):
        second = (first + 1) % 3
        E_first = 0.7
        E_second = (1 + d) * E_first * pb[second] / pb[first]  # A_second / A_first = 1 + d
        third = 3 - first - second
        table = {(TOKEN, first): np.exp(-E_first), (TOKEN, second): np.exp(-E_second),
                 (TOKEN, third): np.exp(-50.0)}
        out = _run_one(zt, zd, [1], [0.5], _table_hook(table))
        assert out["accept_count"][0] == 1
        assert out["out_tokens"][0, 1] == first
        assert abs(out["margin"][0] - np.log1p(d)) <= 1e-9 * max(1.0, np.log1p(d)), (out["margin"][0], d)


def test_trial_margin_is_the_gap_of_one_minus_v_to_q_over_p():
    """A residual trial that drew x and accepts with 1 - v = q/p (1 + 1e-7):
    margin |(1 - v) - q/p| = 1e-7 q/p."""
    zt = np.array([[0.0, 1.0, -0.5], [0.0, 0.0, 0.0]], np.float32)
    zd = np.array([[1.2, 0.7, -0.6]], np.float32)
    p, q = _probs(zt[0]), _probs(zd[0])
    x_draft = 0
    assert q[x_draft] > 2 * p[x_draft]     # r = 1 rejects with margin 1 - p/q > 0.5
    x = 1
    ratio = q[x] / p[x]
    assert ratio < 1
    for d in (1e-7, -1e-7):
        v = 1.0 - ratio * (1 + d)
        want = abs((1.0 - v) - ratio)
        hook = _table_hook({(TOKEN, x): 1.0, (ACCEPT, 0): v}, default=0.5)
        out = _run_one(zt, zd, [x_draft], [1.0], hook)
        assert out["accept_count"][0] == 0
        if d > 0:
            assert out["trials"][0] == 1 and out["out_tokens"][0, 0] == x
            assert abs(out["margin"][0] - want) <= 1e-12, (out["margin"][0], want)
        else:
            # every trial draws x with the same v and is rejected; the direct
            # residual race then decides (its margins count too)
            assert out["trials"][0] == oracle.MAX_TRIALS + 1
            assert out["margin"][0] <= want + 1e-12


def test_margin_counts_only_the_decisions_on_the_output_path():
    """A rejection at position 0 ends the chain: a near-tie r at position 1 and
    near-tie arrivals of races that are never run do not enter the margin."""
    zt = np.array([[0.0, 1.0, -0.5], [0.3, 0.1, 0.0], [0.0, 0.0, 0.0]], np.float32)
    zd = np.array([[1.2, 0.7, -0.6], [0.3, 0.2, 0.0]], np.float32)
    p0, q0 = _probs(zt[0]), _probs(zd[0])
    p1, q1 = _probs(zt[1]), _probs(zd[1])
    tie1 = np.float32(p1[0] / q1[0] * (1 + 1e-7))   # a near-tie at position 1
    x = 1
    v = 0.5 * (1 - q0[x] / p0[x])
    hook = _table_hook({(TOKEN, x): 1.0, (ACCEPT, 0): v})
    out = _run_one(zt, zd, [0, 0], [1.0, tie1], hook)
    assert out["accept_count"][0] == 0
    want = min(abs(1.0 - p0[0] / q0[0]), abs((1 - v) - q0[x] / p0[x]))
    assert abs(out["margin"][0] - want) <= 1e-12, (out["margin"][0], want)
