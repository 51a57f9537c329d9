"""Pins for the oracle: checks against what the pages and mathematics fix.

None of these re-types the oracle's own formulas.  Each pin comes from a
library routine (numpy's Philox, torch/scipy softmax, numpy argmax/lexsort), a
closed form the pages state (acceptance = 1 - TVD, Theorem 3.5; expected
tokens per iteration, Theorem 3.8 with c = 0; alpha^K all-accept rate; the
geometric fan-out), an exactness property (the emitted token is distributed as
the target p), or a special case the pages name (p >= q always accepts,
identical models accept everything, p(x) = 0 always rejects).
"""
import os

import numpy as np
import pytest
import torch
from scipy import stats
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG_SEED = 12345


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _chi2_ok(counts, probs, min_p=1e-6):
    """Chi-square goodness of fit; merges cells with expected count < 5."""
    counts = np.asarray(counts, float)
    n = counts.sum()
    exp = np.asarray(probs, float) * n
    keep = exp >= 5
    obs_k, exp_k = counts[keep], exp[keep]
    obs_rest, exp_rest = counts[~keep].sum(), exp[~keep].sum()
    if exp_rest > 0:
        obs_k = np.append(obs_k, obs_rest)
        exp_k = np.append(exp_k, exp_rest)
    exp_k = exp_k * obs_k.sum() / exp_k.sum()
    p = stats.chisquare(obs_k, exp_k).pvalue
    return p > min_p, p


# ----------------------------------------------------------------- Philox
def test_philox_known_answer_vectors():
    """Philox4x32-10 against the known-answer vectors published with its
    reference implementation."""
    rows = _read_golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        words = [int(x, 16) for x in r]
        ctr, key, ref = words[:4], words[4:6], words[6:10]
        assert list(oracle.philox4x32_10(ctr, key)) == ref


def test_uniform_word_mapping():
    """uniform(n) = ((w >> 8) + 1) * 2^-24 for word n % 4 of the block at
    counter (n / 4, stream, trial, pos) and key (low, high half of the key)."""
    key = 0x1234_5678_9ABC_DEF0
    seen = set()
    for n in range(12):
        w = oracle.philox4x32_10([n >> 2, 3, 7, 2], [key & 0xFFFFFFFF, key >> 32])[n & 3]
        u = oracle.uniform(key, 3, 7, 2, n)
        assert u == ((int(w) >> 8) + 1) * 2.0 ** -24
        assert 0 < u <= 1
        seen.add(u)
    assert len(seen) == 12


# ----------------------------------------------------------------- softmax
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_stats_vs_torch(T):
    rng = np.random.default_rng(RNG_SEED)
    z = (rng.normal(0, 3, 5000)).astype(np.float32)
    z[17] = -np.inf
    M, S = oracle.softmax_stats(z, T)
    p = np.exp(z.astype(np.float64) / T - M) / S
    ref = torch.softmax(torch.from_numpy(z.astype(np.float64)) / T, dim=0).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)
    assert abs(p.sum() - 1.0) < 1e-12
    assert p[17] == 0.0


def test_softmax_bad_rows():
    z = np.zeros(10, np.float32)
    for bad in (np.nan, np.inf):
        zz = z.copy()
        zz[3] = bad
        assert oracle.softmax_stats(zz, 1.0) is None
    assert oracle.softmax_stats(np.full(10, -np.inf, np.float32), 1.0) is None


# ----------------------------------------------------------------- helpers
def _chain(p_logits_rows, q_logits_rows, tokens, r, keys, T=1.0, want_Z=False):
    return oracle.verify_chain(np.asarray(p_logits_rows, np.float32), np.asarray(q_logits_rows, np.float32),
                               tokens, r, keys, T, want_Z=want_Z)


def _logits_from_probs(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _probs(logits, T=1.0):
    return softmax(np.asarray(logits, np.float64) / T)


def _keys(n, seed=RNG_SEED):
    return np.random.default_rng(seed).integers(0, 2 ** 63, n, dtype=np.int64).astype(np.uint64)


# ----------------------------------------------------------------- special cases
def test_identical_models_accept_everything():
    """q == p: every draft token accepted, for any r in (0, 1] (TVD = 0, alpha = 1)."""
    rng = np.random.default_rng(1)
    B, g, V = 64, 4, 300
    z = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    d = z[:, :g].copy()
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    r = np.ones((B, g), np.float32)
    r[::2] = rng.random((B // 2, g)).astype(np.float32) + np.float32(1e-6)
    out = _chain(z, d, tok, np.minimum(r, 1), _keys(B))
    assert (out["status"] == 0).all()
    assert (out["accept_count"] == g).all()
    assert (out["out_tokens"][:, :g] == tok).all()


def test_zero_target_prob_always_rejects():
    """p_i(x_i) = 0 rejects even with the smallest r."""
    rng = np.random.default_rng(2)
    B, g, V = 32, 3, 200
    z = rng.normal(0, 1, (B, g + 1, V)).astype(np.float32)
    d = z[:, :g].copy()
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    z[np.arange(B), 1, tok[:, 1]] = -np.inf
    r = np.full((B, g), 2.0 ** -24, np.float32)
    out = _chain(z, d, tok, r, _keys(B))
    assert (out["accept_count"] == 1).all()
    assert (out["out_tokens"][:, 1] != tok[:, 1]).all()
    assert (out["pq"][:, 1, 0] == 0).all()


def test_target_above_draft_always_accepts():
    """p(x) >= q(x): always accept (the pages' first case), even with r = 1."""
    rng = np.random.default_rng(3)
    B, g, V = 40, 2, 100
    z = rng.normal(0, 1, (B, g + 1, V)).astype(np.float32)
    d = rng.normal(0, 1, (B, g, V)).astype(np.float32)
    tok = np.zeros((B, g), np.int32)
    for b in range(B):
        for i in range(g):
            p, q = _probs(z[b, i]), _probs(d[b, i])
            tok[b, i] = int(np.argmax(p - q))  # a token with p > q
    r = np.ones((B, g), np.float32)
    out = _chain(z, d, tok, r, _keys(B))
    assert (out["accept_count"] == g).all()


def test_output_length_and_padding():
    rng = np.random.default_rng(4)
    B, g, V = 200, 5, 64
    z = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    d = (z[:, :g] + rng.normal(0, 1.5, (B, g, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    out = _chain(z, d, tok, r, _keys(B))
    k = out["accept_count"]
    assert ((k >= 0) & (k <= g)).all()
    for b in range(B):
        row = out["out_tokens"][b]
        assert (row[: k[b] + 1] >= 0).all() and (row[: k[b] + 1] < V).all()
        assert (row[k[b] + 1:] == -1).all()
        assert (row[: k[b]] == tok[b, : k[b]]).all()
        # the rejected token is never re-emitted: its residual mass is zero
        if k[b] < g:
            assert row[k[b]] != tok[b, k[b]]
    assert (k < g).any() and (k == g).any()


def test_bad_rows():
    rng = np.random.default_rng(5)
    B, g, V = 4, 2, 50
    z = rng.normal(0, 1, (B, g + 1, V)).astype(np.float32)
    d = z[:, :g].copy()
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    tok[0, 1] = V          # out of range
    z[1, 2, 7] = np.nan    # NaN in the bonus row
    d[2, 0, 3] = np.inf    # +inf in a draft row
    out = _chain(z, d, tok, np.ones((B, g), np.float32), _keys(B))
    assert list(out["status"]) == [4, 4, 4, 0]
    assert (out["accept_count"][:3] == -1).all() and (out["out_tokens"][:3] == -1).all()


# ----------------------------------------------------------------- statistics
def _iid_case(rng, V, g, B, T=1.0, z_std=1.5, noise=1.0):
    z1 = rng.normal(0, z_std, V).astype(np.float32)
    d1 = (z1 + rng.normal(0, noise, V)).astype(np.float32)
    z = np.broadcast_to(z1, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(d1, (B, g, V)).astype(np.float32)
    q = _probs(d1, T)
    tok = rng.choice(V, size=(B, g), p=q).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    return z, d, tok, r, _probs(z1, T), q


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_acceptance_rate_is_one_minus_tvd(T):
    """Theorem 3.5: alpha = sum_x min(p, q) = 1 - TVD(p, q)."""
    rng = np.random.default_rng(6)
    B, V = 30000, 40
    z, d, tok, r, p, q = _iid_case(rng, V, 1, B, T)
    out = _chain(z, d, tok, r, _keys(B), T=T)
    alpha = np.minimum(p, q).sum()
    assert abs(alpha - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    emp = (out["accept_count"] == 1).mean()
    sigma = np.sqrt(alpha * (1 - alpha) / B)
    assert abs(emp - alpha) < 5 * sigma, (emp, alpha, sigma)


def test_expected_tokens_per_iteration():
    """Theorem 3.8 with c = 0: E[tokens] = (1 - alpha^(g+1)) / (1 - alpha)."""
    rng = np.random.default_rng(7)
    B, V, g = 30000, 30, 4
    z, d, tok, r, p, q = _iid_case(rng, V, g, B)
    out = _chain(z, d, tok, r, _keys(B))
    alpha = np.minimum(p, q).sum()
    n = out["accept_count"] + 1
    expect = (1 - alpha ** (g + 1)) / (1 - alpha)
    assert abs(n.mean() - expect) < 5 * n.std() / np.sqrt(B), (n.mean(), expect)
    assert n.max() <= g + 1 and n.min() >= 1


def test_all_accept_rate_alpha_pow_K():
    """alpha^K all-accept rate with K = 5, alpha = 0.8 (the SSD review's 33%)."""
    gold = dict((r[0], float(r[1])) for r in _read_golden("all_accept_ssd.txt"))
    K, a = int(gold["K"]), gold["alpha"]
    assert abs(a ** K - gold["p_all_accept"]) < 1e-12 and round(a ** K, 2) == gold["page_rounded"]
    # p uniform on 5 tokens, q puts 0.16 on each of them and 0.2 on a sixth: sum min = 0.8
    V = 10
    p = np.zeros(V); p[:5] = 0.2
    q = np.zeros(V); q[:5] = 0.16; q[5] = 0.2
    zl, dl = _logits_from_probs(p), _logits_from_probs(q)
    pp, qq = _probs(zl), _probs(dl)
    alpha = np.minimum(pp, qq).sum()
    assert abs(alpha - a) < 1e-6
    rng = np.random.default_rng(8)
    B = 40000
    z = np.broadcast_to(zl, (B, K + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl, (B, K, V)).astype(np.float32)
    tok = rng.choice(V, size=(B, K), p=qq).astype(np.int32)
    r = (1 - rng.random((B, K))).astype(np.float32)
    out = _chain(z, d, tok, r, _keys(B))
    emp = (out["accept_count"] == K).mean()
    target = alpha ** K
    assert abs(emp - target) < 5 * np.sqrt(target * (1 - target) / B), (emp, target)


def _sparse_multiblock_case(rng, V=2100, n_support=12):
    """p and q with a few tokens of mass spread over several 1024-id blocks."""
    ids = np.sort(rng.choice(V, n_support, replace=False))
    zl = np.full(V, -np.inf, np.float32)
    dl = np.full(V, -np.inf, np.float32)
    zl[ids] = rng.normal(0, 1.0, n_support)
    dl[ids] = zl[ids] + rng.normal(0, 1.0, n_support)
    return ids, zl.astype(np.float32), dl.astype(np.float32)


def test_first_token_is_distributed_as_target():
    """Exactness: P(emitted first token = x) = p_1(x) for any p, q (the pages' proof)."""
    rng = np.random.default_rng(9)
    ids, zl, dl = _sparse_multiblock_case(rng)
    V, B = zl.size, 24000
    z = np.broadcast_to(np.stack([zl, zl]), (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(dl, (B, 1, V)).astype(np.float32)
    q = _probs(dl)
    tok = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
    r = (1 - rng.random((B, 1))).astype(np.float32)
    out = _chain(z, d, tok, r, _keys(B, 99))
    first = out["out_tokens"][:, 0]
    p = _probs(zl)
    counts = np.bincount(first, minlength=V)[ids]
    ok, pv = _chi2_ok(counts, p[ids])
    assert counts.sum() == B and ok, pv
    assert (out["accept_count"] == 0).any() and (out["accept_count"] == 1).any()


def test_residual_distribution_on_forced_rejection():
    """A rejected position emits from norm(max(0, p - q)); Z = TVD(p, q)."""
    rng = np.random.default_rng(10)
    ids, zl, dl = _sparse_multiblock_case(rng)
    V, B = zl.size, 20000
    p, q = _probs(zl), _probs(dl)
    x_rej = int(ids[np.argmax(q[ids] - p[ids])])
    assert q[x_rej] > p[x_rej]
    z = np.broadcast_to(np.stack([zl, zl]), (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(dl, (B, 1, V)).astype(np.float32)
    tok = np.full((B, 1), x_rej, np.int32)
    r = np.ones((B, 1), np.float32)          # r * q = q > p: always rejected
    out = _chain(z, d, tok, r, _keys(B, 7), want_Z=True)
    assert (out["accept_count"] == 0).all()
    w = np.maximum(0, p - q)
    np.testing.assert_allclose(out["Z"], 0.5 * np.abs(p - q).sum(), rtol=1e-12)
    counts = np.bincount(out["out_tokens"][:, 0], minlength=V)[ids]
    ok, pv = _chi2_ok(counts, w[ids] / w.sum())
    assert counts.sum() == B and ok, pv
    assert counts[w[ids] == 0].sum() == 0


def test_residual_fallback_is_exact():
    """Nearly identical p and q (small Z) exhaust the rejection trials; the
    direct fallback must still draw from norm(max(0, p - q))."""
    rng = np.random.default_rng(11)
    V, B = 1500, 10000
    zl = rng.normal(0, 1, V).astype(np.float32)
    dl = zl.copy()
    hot = rng.choice(V, 6, replace=False)
    dl[hot[:3]] += np.float32(0.05)
    dl[hot[3:]] -= np.float32(0.05)
    p, q = _probs(zl), _probs(dl)
    x_rej = int(np.argmax(q - p))
    z = np.broadcast_to(np.stack([zl, zl]), (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(dl, (B, 1, V)).astype(np.float32)
    tok = np.full((B, 1), x_rej, np.int32)
    out = _chain(z, d, tok, np.ones((B, 1), np.float32), _keys(B, 3), want_Z=True)
    Z = 0.5 * np.abs(p - q).sum()
    frac_fb = (out["trials"] == oracle.MAX_TRIALS + 1).mean()
    assert abs(frac_fb - (1 - Z) ** oracle.MAX_TRIALS) < 5 * np.sqrt(frac_fb * (1 - frac_fb) / B) + 1e-3
    assert frac_fb > 0.5
    w = np.maximum(0, p - q)
    counts = np.bincount(out["out_tokens"][:, 0], minlength=V)
    ok, pv = _chi2_ok(counts, w / w.sum())
    assert ok, pv
    assert counts[w == 0].sum() == 0


def test_bonus_is_distributed_as_last_target_row():
    """All accepted (q == p): the bonus token ~ p_{gamma+1}."""
    rng = np.random.default_rng(12)
    ids, zl, _ = _sparse_multiblock_case(rng)
    zb = np.full_like(zl, -np.inf)
    zb[ids] = rng.normal(0, 1, ids.size)
    V, B = zl.size, 20000
    z = np.broadcast_to(np.stack([zl, zb.astype(np.float32)]), (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(zl, (B, 1, V)).astype(np.float32)
    tok = np.full((B, 1), ids[0], np.int32)
    out = _chain(z, d, tok, np.ones((B, 1), np.float32), _keys(B, 5), want_Z=True)
    assert (out["accept_count"] == 1).all() and (out["Z"] == 1).all()
    pb = _probs(zb)
    counts = np.bincount(out["out_tokens"][:, 1], minlength=V)[ids]
    ok, pv = _chi2_ok(counts, pb[ids])
    assert ok, pv


def test_dense_support_draw_over_sub_blocks():
    """Every id of a 1500-id vocabulary (two blocks, 47 sub-blocks) carries
    mass: the bonus draw matches p over all ids."""
    rng = np.random.default_rng(16)
    V, B = 1500, 60000
    zb = rng.normal(0, 0.7, V).astype(np.float32)
    zl = rng.normal(0, 1, V).astype(np.float32)
    z = np.broadcast_to(np.stack([zl, zb]), (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(zl, (B, 1, V)).astype(np.float32)
    tok = np.zeros((B, 1), np.int32)
    out = _chain(z, d, tok, np.ones((B, 1), np.float32), _keys(B, 17))
    assert (out["accept_count"] == 1).all()
    counts = np.bincount(out["out_tokens"][:, 1], minlength=V)
    pb = _probs(zb)
    ok, pv = _chi2_ok(counts, pb)
    assert ok, pv
    # coarser check per sub-block of 32 ids
    sub = np.add.reduceat(counts, np.arange(0, V, 32))
    psub = np.add.reduceat(pb, np.arange(0, V, 32))
    ok, pv = _chi2_ok(sub, psub)
    assert ok, pv


def test_race_keys_are_independent_and_deterministic():
    rng = np.random.default_rng(13)
    B, g, V = 16, 3, 3000
    z = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    d = (z[:, :g] + rng.normal(0, 1, (B, g, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    a = _chain(z, d, tok, r, _keys(B))
    b = _chain(z, d, tok, r, _keys(B))
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    c = _chain(z, d, tok, r, _keys(B, 4242))
    assert not np.array_equal(a["out_tokens"], c["out_tokens"])


# ----------------------------------------------------------------- greedy
def test_greedy_matches_numpy_argmax():
    """T = 0: a draft token stands only if it is the target argmax (first occurrence on ties, as numpy.argmax)."""
    rng = np.random.default_rng(14)
    B, g, V = 50, 4, 777
    z = rng.integers(-4, 4, (B, g + 1, V)).astype(np.float32)  # many ties
    a = z.argmax(axis=2)
    tok = a[:, :g].astype(np.int32).copy()
    flip = rng.random((B, g)) < 0.3
    tok[flip] = rng.integers(0, V, flip.sum())
    out = oracle.verify_greedy(z, tok)
    for b in range(B):
        k = 0
        while k < g and tok[b, k] == a[b, k]:
            k += 1
        assert out["accept_count"][b] == k
        assert list(out["out_tokens"][b, :k + 1]) == list(tok[b, :k]) + [a[b, k]]
        assert (out["out_tokens"][b, k + 1:] == -1).all()
    # chain entry at T = 0 routes to greedy
    out2 = oracle.verify_chain(z, z[:, :g], tok, np.ones((B, g), np.float32), _keys(B), 0.0)
    assert np.array_equal(out2["out_tokens"], out["out_tokens"])


def test_greedy_negative_zero_ties_and_bad_rows():
    z = np.zeros((4, 2, 8), np.float32)
    z[0, 0, 2] = -0.0
    z[0, 0, 5] = 1.0
    z[0, 0, 6] = 1.0
    z[0, 1, :] = -0.0
    z[1, 0, 3] = np.nan
    z[2, 1, 4] = np.inf
    z[3, 1, :] = -np.inf
    tok = np.array([[5], [0], [0], [0]], np.int32)
    out = oracle.verify_greedy(z, tok)
    assert list(out["status"]) == [0, 4, 4, 4]
    assert list(out["out_tokens"][0]) == [5, 0]


# ----------------------------------------------------------------- fan-out
def test_fanout_sizes_golden():
    rows = _read_golden("fanout_sizes_ssd.txt")
    vals = [(int(r[0]), float(r[1]), int(r[2])) for r in rows if r[0] != "sum"]
    total = [int(r[1]) for r in rows if r[0] == "sum"][0]
    for k, f, fr in vals:
        assert abs(oracle.fanout_size(8, 0.8, 0.5, k) - f) < 5e-6
    sizes = oracle.fanout_sizes(8, 0.8, 0.5, 4, 128256)
    assert sizes == [v[2] for v in vals] and sum(sizes) == total
    # the fan-out shrinks geometrically: ratio a^(1/(1+r)) between neighbours
    for k in range(4):
        ratio = oracle.fanout_size(8, 0.8, 0.5, k + 1) / oracle.fanout_size(8, 0.8, 0.5, k)
        assert abs(ratio - 0.8 ** (1 / 1.5)) < 1e-12


@pytest.mark.parametrize("levels", [None, 8])
def test_fanout_vs_numpy_lexsort(levels):
    rng = np.random.default_rng(15)
    B, K1, V = 3, 5, 3000
    d = rng.normal(0, 2, (B, K1, V)).astype(np.float32)
    if levels:
        d = np.round(d * levels / 4).astype(np.float32)  # heavy ties
        d[d == 0] = np.where(rng.random((d == 0).sum()) < 0.5, -0.0, 0.0)
    ex = rng.integers(-1, V, (B, K1)).astype(np.int32)
    F = [8, 7, 6, 5, 64]
    out = oracle.fanout_topk(d, ex, F)
    offs = np.concatenate([[0], np.cumsum(F)])
    for b in range(B):
        for k in range(K1):
            v = d[b, k].astype(np.float64) + 0.0
            ids = np.arange(V)
            keep = ids != ex[b, k]
            order = np.lexsort((ids[keep], -v[keep]))
            ref = ids[keep][order][: F[k]]
            assert list(out["ids"][b, offs[k]:offs[k + 1]]) == list(ref)
    d[1, 2, 9] = np.nan
    out = oracle.fanout_topk(d, ex, F)
    assert out["status"][1, 2] == 4 and (out["status"].sum() == 4)


# ----------------------------------------------------------------- speculation cache
def _cache_case(rng, B, g, V, z_std=1.5, noise=1.0):
    """Distinct p_i / q_i per position, shared by all sequences (q also at the
    bonus position g); draft tokens x_i ~ q_i drawn per sequence."""
    zl = rng.normal(0, z_std, (g + 1, V)).astype(np.float32)
    dl = (zl + rng.normal(0, noise, (g + 1, V))).astype(np.float32)
    p = np.stack([_probs(zl[i]) for i in range(g + 1)])
    q = np.stack([_probs(dl[i]) for i in range(g + 1)])
    tok = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(g)], axis=1).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    z = np.broadcast_to(zl, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl[:g], (B, g, V)).astype(np.float32)
    dfan = np.broadcast_to(dl, (B, g + 1, V)).astype(np.float32)
    exclude = np.concatenate([tok, np.full((B, 1), -1, np.int32)], axis=1)
    return z, d, dfan, tok, r, exclude, p, q


def test_cache_full_fanout_always_hits():
    """[SSD] Figure 2 cache with every candidate listed: F_k = V - 1 with the
    verified token excluded (k < gamma), F_gamma = V.  A rejected token has
    max(0, p - q) = 0 and is never re-emitted, so every outcome hits, at an
    entry of its own position k holding the emitted token."""
    rng = np.random.default_rng(21)
    B, g, V = 3000, 3, 7
    z, d, dfan, tok, r, exclude, p, q = _cache_case(rng, B, g, V, z_std=1.0, noise=1.2)
    F = [V - 1] * g + [V]
    lists = oracle.fanout_topk(dfan, exclude, F)["ids"]
    out = _chain(z, d, tok, r, _keys(B, 31))
    slot = oracle.cache_slots(out["accept_count"], out["out_tokens"], lists, F)
    offs = np.concatenate([[0], np.cumsum(F)])
    k = out["accept_count"]
    t = out["out_tokens"][np.arange(B), k]
    assert (slot >= 0).all()
    assert (slot >= offs[k]).all() and (slot < offs[k + 1]).all()
    assert (lists[np.arange(B), slot] == t).all()
    assert len(np.unique(k)) == g + 1  # every position reached
    # a bad row never hits
    bad = out["accept_count"].copy()
    bad[:5] = -1
    assert (oracle.cache_slots(bad, out["out_tokens"], lists, F)[:5] == -1).all()


def test_cache_hit_rate_closed_form():
    """Hit rate of the fan-out cache against the closed form.  With the draft
    tokens fixed, position i accepts with probability a_i = min(1, p_i/q_i)
    at x_i ([SD] acceptance criterion), the first rejection at j emits from
    norm(max(0, p_j - q_j)) and full acceptance emits from p_gamma, so
      P(hit) = sum_j (prod_{i<j} a_i)(1 - a_j) R_j(C_j) + (prod_i a_i) p_gamma(C_gamma)
    with C_k position k's candidates and R_j the residual distribution."""
    rng = np.random.default_rng(22)
    B, g, V = 30000, 3, 40
    z, d, dfan, tok, r, exclude, p, q = _cache_case(rng, B, g, V)
    F = [6, 4, 3, 3]
    lists = oracle.fanout_topk(dfan, exclude, F)["ids"]
    out = _chain(z, d, tok, r, _keys(B, 32))
    slot = oracle.cache_slots(out["accept_count"], out["out_tokens"], lists, F)
    offs = np.concatenate([[0], np.cumsum(F)])
    resid = np.maximum(p[:g] - q[:g], 0.0)
    resid /= resid.sum(axis=1, keepdims=True)
    a = np.minimum(1.0, p[np.arange(g), tok] / q[np.arange(g), tok])  # [B, g]
    h = np.zeros(B)
    reach = np.ones(B)
    for j in range(g):
        c = lists[:, offs[j]:offs[j + 1]]
        h += reach * (1 - a[:, j]) * resid[j][c].sum(axis=1)
        reach = reach * a[:, j]
    h += reach * p[g][lists[:, offs[g]:offs[g + 1]]].sum(axis=1)
    hits = (slot >= 0).sum()
    sigma = np.sqrt((h * (1 - h)).sum())
    assert 0.05 < h.mean() < 0.95
    assert abs(hits - h.sum()) < 5 * sigma, (hits, h.sum(), sigma)


def test_cache_slot_first_entry_of_the_outcome_position():
    """The slot is the first entry of position k equal to t*; the same token
    listed under another position does not count."""
    F = [3, 2, 0, 2]
    ids = np.array([[4, 5, 6, 5, 9, 5, 5]], np.int32)
    cases = [(0, 5, 1), (1, 5, 3), (1, 6, -1), (2, 5, -1), (3, 5, 5), (0, 9, -1), (1, 9, 4), (-1, 5, -1)]
    for k, t, want in cases:
        toks = np.full((1, 4), -1, np.int32)
        if k >= 0:
            toks[0, k] = t
        assert oracle.cache_slots([k], toks, ids, F)[0] == want, (k, t)


# ----------------------------------------------------------------- top-k / top-p filtered verify
def _torch_filtered_probs(z, T, top_k):
    """p' from library routines: torch.topk then torch.softmax over the kept
    logits (rows without ties), scattered back to a length-V vector."""
    zt = torch.from_numpy(np.asarray(z, np.float64))
    v, i = torch.topk(zt, top_k)
    p = torch.zeros_like(zt)
    p[i] = torch.softmax(v / T, dim=0)
    return p.numpy()


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_filter_row_vs_torch_topk_softmax(T):
    rng = np.random.default_rng(30)
    for V, k in [(1000, 50), (300, 1), (64, 64), (5000, 7)]:
        z = rng.normal(0, 2, V).astype(np.float32)
        ids, probs, margin = oracle.filter_row(z, T, k)
        ref = _torch_filtered_probs(z, T, k)
        order = np.argsort(-z.astype(np.float64), kind="stable")[:k]
        assert list(ids) == list(order)
        np.testing.assert_allclose(probs, ref[ids], rtol=1e-12, atol=0)
        assert abs(probs.sum() - 1) < 1e-12 and margin == np.inf


def test_filter_top_p_closed_form():
    """Nucleus cut on p = (0.5, 0.3, 0.15, 0.05): the shortest prefix whose
    mass reaches top_p, renormalised; applied after the top-k cut."""
    z = np.log(np.array([0.5, 0.3, 0.15, 0.05]))[[2, 0, 3, 1]].astype(np.float32)  # ids 1, 3, 0, 2 by rank
    cases = [(4, 0.4, [1], [1.0]),
             (4, 0.75, [1, 3], [0.625, 0.375]),
             (4, 0.9, [1, 3, 0], [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95]),
             (4, 1.0, [1, 3, 0, 2], [0.5, 0.3, 0.15, 0.05]),
             (3, 0.9, [1, 3, 0], [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95]),  # top-3 mass (0.526, 0.842, 1.0)
             (2, 0.6, [1], [1.0]),                                          # top-2 mass (0.625, 1.0)
             (2, 0.7, [1, 3], [0.625, 0.375])]
    for k, top_p, want_ids, want_p in cases:
        ids, probs, _ = oracle.filter_row(z, 1.0, k, top_p)
        assert list(ids) == want_ids, (k, top_p)
        np.testing.assert_allclose(probs, want_p, rtol=1e-6)


def test_filter_ties_and_bad_rows():
    z = np.array([1.0, 3.0, 3.0, -0.0, 0.0, 3.0], np.float32)
    ids, probs, _ = oracle.filter_row(z, 1.0, 2)
    assert list(ids) == [1, 2]   # ties to the lower id
    ids, probs, _ = oracle.filter_row(z, 1.0, 6)
    assert list(ids) == [1, 2, 5, 0, 3, 4]   # -0.0 ranks equal to +0.0
    for bad in (np.nan, np.inf):
        zz = z.copy()
        zz[4] = bad
        assert oracle.filter_row(zz, 1.0, 2) is None
    assert oracle.filter_row(np.full(10, -np.inf, np.float32), 1.0, 3) is None
    ids, probs, _ = oracle.filter_row(np.array([-np.inf, 0.5, -np.inf], np.float32), 1.0, 3)
    assert list(ids) == [1, 0, 2] and list(probs) == [1.0, 0.0, 0.0]


def _filtered_case(rng, B, g, V, top_k, z_std=1.5, noise=1.0, T=1.0):
    zl = rng.normal(0, z_std, (g + 1, V)).astype(np.float32)
    dl = (zl[:g] + rng.normal(0, noise, (g, V))).astype(np.float32)
    p = np.stack([_torch_filtered_probs(zl[i], T, top_k) for i in range(g + 1)])
    q = np.stack([_torch_filtered_probs(dl[i], T, top_k) for i in range(g)])
    tok = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(g)], axis=1).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    z = np.broadcast_to(zl, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl, (B, g, V)).astype(np.float32)
    return z, d, tok, r, p, q


def test_filtered_top1_is_greedy():
    """top_k = 1 makes p' and q' point masses on the argmaxes: a draft token
    stands iff it is the target argmax, and the emitted token at the first
    mismatch (or the bonus) is the target argmax -- the T = 0 rule."""
    rng = np.random.default_rng(31)
    B, g, V = 400, 3, 50
    z = rng.integers(-3, 4, (B, g + 1, V)).astype(np.float32)   # ties: the lowest id is the argmax
    a = np.argmax(z, axis=2)
    d = rng.integers(-3, 4, (B, g, V)).astype(np.float32)
    agree = rng.random((B, g)) < 0.7
    bb, ii = np.nonzero(agree)
    d[bb, ii, a[bb, ii]] = 9.0                                    # the draft argmax is the target's
    tok = np.argmax(d, axis=2).astype(np.int32)                   # drawn from q' = point mass
    r = (1 - rng.random((B, g))).astype(np.float32)
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 41), 1.0, 1)
    for b in range(B):
        k = 0
        while k < g and tok[b, k] == a[b, k]:
            k += 1
        assert out["accept_count"][b] == k
        assert list(out["out_tokens"][b, :k]) == list(tok[b, :k]) and out["out_tokens"][b, k] == a[b, k]


@pytest.mark.parametrize("top_k", [10, 40])
def test_filtered_acceptance_rate_is_one_minus_tvd(top_k):
    """Theorem 3.5 on the filtered distributions: P(accept) = sum min(p', q')."""
    rng = np.random.default_rng(32)
    B, V = 30000, 200
    z, d, tok, r, p, q = _filtered_case(rng, B, 1, V, top_k)
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 42), 1.0, top_k)
    np.testing.assert_allclose(out["pq"][:, 0, 0], p[0][tok[:, 0]], rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out["pq"][:, 0, 1], q[0][tok[:, 0]], rtol=1e-12, atol=1e-300)
    alpha = np.minimum(p[0], q[0]).sum()
    emp = (out["accept_count"] == 1).mean()
    assert abs(emp - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / B), (emp, alpha)


def test_filtered_first_token_and_bonus_are_exact():
    """Exactness on the filtered distributions: the first emitted token ~ p'_1
    and the bonus ~ p'_2 (chi-square)."""
    rng = np.random.default_rng(33)
    B, V, k = 30000, 300, 12
    z, d, tok, r, p, q = _filtered_case(rng, B, 1, V, k, noise=0.7)
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 43), 1.0, k)
    first = out["out_tokens"][:, 0]
    ok, pv = _chi2_ok(np.bincount(first, minlength=V), p[0])
    assert ok, pv
    full = out["accept_count"] == 1
    ok, pv = _chi2_ok(np.bincount(out["out_tokens"][full, 1], minlength=V), p[1])
    assert ok and full.sum() > 5000, pv


def test_filtered_residual_on_forced_rejection():
    """A rejected position emits from norm(max(0, p' - q')); Z = TVD(p', q')."""
    rng = np.random.default_rng(34)
    B, V, k = 20000, 400, 16
    z, d, tok, r, p, q = _filtered_case(rng, B, 1, V, k, noise=1.5)
    x_rej = int(np.argmax(q[0] - p[0]))
    tok[:] = x_rej
    r[:] = 1.0
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 44), 1.0, k, want_Z=True)
    assert (out["accept_count"] == 0).all()
    w = np.maximum(p[0] - q[0], 0)
    np.testing.assert_allclose(out["Z"], 0.5 * np.abs(p[0] - q[0]).sum(), rtol=1e-10)
    ok, pv = _chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), w / w.sum())
    assert ok and (out["out_tokens"][:, 0] != x_rej).all(), pv


def test_filtered_nucleus_first_token():
    """With top_p < 1 the first emitted token follows the nucleus-restricted,
    renormalised target distribution (chi-square)."""
    rng = np.random.default_rng(35)
    B, V, k, top_p = 30000, 200, 30, 0.8
    z, d, tok, r, _, _ = _filtered_case(rng, B, 1, V, k)
    ids, probs, _ = oracle.filter_row(z[0, 0], 1.0, k, top_p)
    # independent nucleus: sort the torch top-k probabilities, cut where the cumulative sum reaches top_p
    pk = _torch_filtered_probs(z[0, 0], 1.0, k)
    srt = np.argsort(-pk, kind="stable")
    n = int(np.searchsorted(np.cumsum(pk[srt]), top_p) + 1)
    nucleus = np.zeros(V)
    nucleus[srt[:n]] = pk[srt[:n]] / pk[srt[:n]].sum()
    assert sorted(ids) == sorted(srt[:n])
    q_ids, q_probs, _ = oracle.filter_row(d[0, 0], 1.0, k, top_p)
    qv = np.zeros(V)
    qv[q_ids] = q_probs
    tok = rng.choice(V, size=(B, 1), p=qv).astype(np.int32)
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 45), 1.0, k, top_p)
    ok, pv = _chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), nucleus)
    assert ok, pv


def test_filtered_without_cut_is_the_softmax():
    """top_k >= V and top_p = 1: p', q' are the plain temperature softmax."""
    rng = np.random.default_rng(36)
    B, g, V = 50, 2, 60
    z = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    d = rng.normal(0, 2, (B, g, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    out = oracle.verify_filtered(z, d, tok, r, _keys(B, 46), 0.8, 64)
    bb = np.arange(B)[:, None]
    gg = np.arange(g)[None, :]
    np.testing.assert_allclose(out["pq"][..., 0], softmax(z[:, :g].astype(np.float64) / 0.8, axis=2)[bb, gg, tok],
                               rtol=1e-12)
    np.testing.assert_allclose(out["pq"][..., 1], softmax(d.astype(np.float64) / 0.8, axis=2)[bb, gg, tok],
                               rtol=1e-12)


def test_zero_residual_mass_is_a_bad_row():
    """A draft token outside q's support (q(x) = 0) with p(x) = 0 is rejected,
    and when p = q everywhere else the residual max(0, p - q) has no mass:
    nothing can be drawn, so the sequence is a bad row (chain and filtered)."""
    V = 40
    rng = np.random.default_rng(37)
    zl = rng.normal(0, 1, V).astype(np.float32)
    zl[7] = -np.inf
    z = np.stack([zl, zl])[None]
    d = zl[None, None].copy()
    out = oracle.verify_chain(z, d, np.array([[7]], np.int32), np.ones((1, 1), np.float32), _keys(1), 1.0)
    assert out["status"][0] == 4 and out["accept_count"][0] == -1 and (out["out_tokens"] == -1).all()
    out = oracle.verify_filtered(z, d, np.array([[7]], np.int32), np.ones((1, 1), np.float32), _keys(1), 1.0, 64)
    assert out["status"][0] == 4 and out["accept_count"][0] == -1
    # the same row with a token inside the support is fine
    out = oracle.verify_chain(z, d, np.array([[3]], np.int32), np.ones((1, 1), np.float32), _keys(1), 1.0)
    assert out["status"][0] == 0 and out["accept_count"][0] == 1


# ----------------------------------------------------------------- Saguaro sampling
def _saguaro_case(rng, B, g, V, F, z_std=1.5, noise=1.0):
    """Per-position p_i, q_i shared by all sequences; cached candidates S_i =
    the top-F_i draft ids (no exclusion); q_C and tokens drawn from it are
    built per C by the caller."""
    zl = rng.normal(0, z_std, (g + 1, V)).astype(np.float32)
    dl = (zl + rng.normal(0, noise, (g + 1, V))).astype(np.float32)
    p = np.stack([_probs(zl[i]) for i in range(g + 1)])
    q = np.stack([_probs(dl[i]) for i in range(g + 1)])
    lists = [np.argsort(-dl[i].astype(np.float64), kind="stable")[:F[i]] for i in range(g + 1)]
    ids = np.concatenate(lists).astype(np.int32)
    return zl, dl, p, q, lists, np.broadcast_to(ids, (B, ids.size)).copy()


def _q_C(q, S, C):
    w = np.ones_like(q)
    w[S] = 1.0 / C
    qc = q * w
    return qc / qc.sum()


def test_saguaro_C1_is_plain_chain():
    """C = 1 leaves the draft distribution as it is: identical outputs."""
    rng = np.random.default_rng(40)
    B, g, V = 300, 3, 500
    F = [6, 5, 4, 3]
    zl, dl, p, q, lists, ids = _saguaro_case(rng, B, g, V, F)
    z = np.broadcast_to(zl, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl[:g], (B, g, V)).astype(np.float32)
    tok = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(g)], axis=1).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    a = oracle.verify_saguaro(z, d, tok, r, _keys(B, 50), 1.0, ids, F, 1.0, want_Z=True)
    b = oracle.verify_chain(z, d, tok, r, _keys(B, 50), 1.0, want_Z=True)
    for key in ("accept_count", "out_tokens", "status", "trials"):
        assert np.array_equal(a[key], b[key]), key
    np.testing.assert_allclose(a["pq"], b["pq"], rtol=1e-13)
    np.testing.assert_allclose(a["Z"], b["Z"], rtol=1e-12)


@pytest.mark.parametrize("C", [2.0, 8.0, 0.5])
def test_saguaro_draft_probabilities(C):
    """q_C(x) = q(x) w(x) / sum q w with w = 1/C on the cached candidates,
    computed here from the softmax probabilities (scipy)."""
    rng = np.random.default_rng(41)
    B, g, V = 40, 2, 300
    F = [9, 4, 2]
    zl, dl, p, q, lists, ids = _saguaro_case(rng, B, g, V, F)
    z = np.broadcast_to(zl, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl[:g], (B, g, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    tok[:, 0] = lists[0][rng.integers(0, F[0], B)]          # many cached tokens
    r = (1 - rng.random((B, g))).astype(np.float32)
    out = oracle.verify_saguaro(z, d, tok, r, _keys(B, 51), 1.0, ids, F, C)
    for i in range(g):
        qc = _q_C(q[i], lists[i], C)
        np.testing.assert_allclose(out["pq"][:, i, 1], qc[tok[:, i]], rtol=1e-12)
        np.testing.assert_allclose(out["pq"][:, i, 0], p[i][tok[:, i]], rtol=1e-12)


def test_saguaro_preserves_the_target_distribution():
    """With tokens drawn from q_C the first emitted token is still
    distributed as p_1 (the [SD] exactness argument with q_C as the draft)."""
    rng = np.random.default_rng(42)
    B, V, C = 30000, 200, 4.0
    F = [12, 12]
    zl, dl, p, q, lists, ids = _saguaro_case(rng, B, 1, V, F, noise=0.8)
    qc = _q_C(q[0], lists[0], C)
    z = np.broadcast_to(zl, (B, 2, V)).astype(np.float32)
    d = np.broadcast_to(dl[:1], (B, 1, V)).astype(np.float32)
    tok = rng.choice(V, size=(B, 1), p=qc).astype(np.int32)
    r = (1 - rng.random((B, 1))).astype(np.float32)
    out = oracle.verify_saguaro(z, d, tok, r, _keys(B, 52), 1.0, ids, F, C)
    ok, pv = _chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), p[0])
    assert ok, pv
    alpha = np.minimum(p[0], qc).sum()
    emp = (out["accept_count"] == 1).mean()
    assert abs(emp - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / B), (emp, alpha)


def _saguaro_hit_closed_form(p, q, lists, C, g):
    reach, h = 1.0, 0.0
    for j in range(g):
        qc = _q_C(q[j], lists[j], C)
        a = np.minimum(p[j], qc).sum()
        res = np.maximum(p[j] - qc, 0.0)
        h += reach * (1 - a) * res[lists[j]].sum() / res.sum()
        reach *= a
    return h + reach * p[g][lists[g]].sum()


def test_saguaro_hit_rate_grows_with_C():
    """Theorem 15: the cache hit rate increases with C (closed form over
    C = 1, 2, 4, 8), and the oracle's hit frequency matches the closed form
    at C = 1 and C = 4 (5 sigma)."""
    rng = np.random.default_rng(43)
    B, g, V = 20000, 3, 60
    F = [6, 5, 4, 3]
    zl, dl, p, q, lists, ids = _saguaro_case(rng, B, g, V, F)
    h = [_saguaro_hit_closed_form(p, q, lists, C, g) for C in (1.0, 2.0, 4.0, 8.0)]
    assert all(b > a for a, b in zip(h, h[1:])), h
    z = np.broadcast_to(zl, (B, g + 1, V)).astype(np.float32)
    d = np.broadcast_to(dl[:g], (B, g, V)).astype(np.float32)
    for C, want in ((1.0, h[0]), (4.0, h[2])):
        tok = np.stack([rng.choice(V, size=B, p=_q_C(q[i], lists[i], C)) for i in range(g)], axis=1).astype(np.int32)
        r = (1 - rng.random((B, g))).astype(np.float32)
        out = oracle.verify_saguaro(z, d, tok, r, _keys(B, 53 + int(C)), 1.0, ids, F, C)
        hits = (oracle.cache_slots(out["accept_count"], out["out_tokens"], ids, F) >= 0).mean()
        assert abs(hits - want) < 5 * np.sqrt(want * (1 - want) / B), (C, hits, want)


# ----------------------------------------------------------------- tree verify
def _tree_star(B, W, V, rng, z_std=1.5, noise=1.0, depth2=0):
    """Root with W children drawn i.i.d. from q_root; with depth2 > 0 each
    child gets that many children drawn from its own q."""
    zl = rng.normal(0, z_std, V).astype(np.float32)
    dl = (zl + rng.normal(0, noise, V)).astype(np.float32)
    N = 1 + W + W * depth2
    z = np.zeros((B, N, V), np.float32)
    d = np.zeros((B, N, V), np.float32)
    parent = np.full((B, N), -1, np.int32)
    tok = np.zeros((B, N), np.int32)
    q0 = _probs(dl)
    for b in range(B):
        z[b, 0], d[b, 0] = zl, dl
    for j in range(W):
        v = 1 + j
        parent[:, v] = 0
        tok[:, v] = rng.choice(V, size=B, p=q0)
        cz = rng.normal(0, z_std, V).astype(np.float32)
        cd = (cz + rng.normal(0, noise, V)).astype(np.float32)
        z[:, v], d[:, v] = cz, cd
        for h in range(depth2):
            w2 = 1 + W + j * depth2 + h
            parent[:, w2] = v
            tok[:, w2] = rng.choice(V, size=B, p=_probs(cd))
            z[:, w2] = rng.normal(0, z_std, V).astype(np.float32)
            d[:, w2] = z[:, w2]
    r = (1 - rng.random((B, N))).astype(np.float32)
    return z, d, parent, tok, r


def test_tree_path_is_the_chain():
    """A tree that is a single path is the chain: identical outputs."""
    rng = np.random.default_rng(70)
    B, g, V = 400, 4, 300
    z = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    d = (z[:, :g] + rng.normal(0, 1, (B, g, V))).astype(np.float32)
    tok = np.stack([np.array([rng.choice(V, p=_probs(d[b, i])) for b in range(B)]) for i in range(g)], 1).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    keys = _keys(B, 71)
    ref = oracle.verify_chain(z, d, tok, r, keys, 1.0)
    dt = np.concatenate([d, np.zeros((B, 1, V), np.float32)], axis=1)
    parent = np.tile(np.arange(-1, g, dtype=np.int32), (B, 1))
    ttok = np.concatenate([np.zeros((B, 1), np.int32), tok], axis=1)
    tr = np.concatenate([np.ones((B, 1), np.float32), r], axis=1)
    out = oracle.verify_tree(z, dt, parent, ttok, tr, keys, 1.0)
    assert np.array_equal(out["accept_count"], ref["accept_count"])
    assert np.array_equal(out["out_tokens"], ref["out_tokens"])
    assert np.array_equal(out["trials"], ref["trials"])
    k = out["accept_count"]
    assert all(list(out["out_nodes"][b, :k[b]]) == list(range(1, k[b] + 1)) for b in range(B))


@pytest.mark.parametrize("W", [2, 4])
def test_tree_root_acceptance_closed_form(W):
    """Children drawn i.i.d. from q: child m is accepted with probability
    sum min(P_m, q), P_0 = p, P_{m+1} = norm(max(0, P_m - q)) (normalising
    after every step), so P(no child accepted) = prod_m (1 - alpha_m)."""
    rng = np.random.default_rng(72)
    B, V = 30000, 80
    z, d, parent, tok, r = _tree_star(B, W, V, rng)
    p, q = _probs(z[0, 0]), _probs(d[0, 0])
    none, P = 1.0, p.copy()
    for m in range(W):
        alpha = np.minimum(P, q).sum()
        none *= 1 - alpha
        P = np.maximum(P - q, 0)
        P /= P.sum()
    out = oracle.verify_tree(z, d, parent, tok, r, _keys(B, 73), 1.0)
    emp = (out["accept_count"] == 0).mean()
    assert abs(emp - none) < 5 * np.sqrt(none * (1 - none) / B), (emp, none)


@pytest.mark.parametrize("W", [3, 4])
def test_tree_first_token_is_exact(W):
    """With W children drawn i.i.d. from q_root the first emitted token is
    distributed as p_root (chi-square)."""
    rng = np.random.default_rng(74 + W)
    B, V = 30000, 120
    z, d, parent, tok, r = _tree_star(B, W, V, rng, noise=1.3)
    out = oracle.verify_tree(z, d, parent, tok, r, _keys(B, 75), 1.0)
    ok, pv = _chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), _probs(z[0, 0]))
    assert ok, pv


def test_tree_second_token_given_first_child():
    """Two levels: given that root child c was accepted, the next emitted
    token is distributed as p_c (chi-square over the sequences that took
    child 1)."""
    rng = np.random.default_rng(77)
    B, V, W = 40000, 60, 3
    z, d, parent, tok, r = _tree_star(B, W, V, rng, noise=0.9, depth2=2)
    out = oracle.verify_tree(z, d, parent, tok, r, _keys(B, 78), 1.0)
    took1 = (out["accept_count"] >= 1) & (out["out_nodes"][:, 0] == 1)
    second = out["out_tokens"][took1, 1]
    ok, pv = _chi2_ok(np.bincount(second, minlength=V), _probs(z[0, 1]))
    assert ok and took1.sum() > 3000, (pv, took1.sum())


def test_tree_greedy_walk():
    """T = 0: descend into the first child whose token is the argmax
    (numpy argmax, first occurrence); emit the last node's argmax."""
    rng = np.random.default_rng(79)
    B, N, V = 200, 9, 40
    z = rng.integers(-3, 4, (B, N, V)).astype(np.float32)
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 4, 4], np.int32)
    P_ = np.tile(parent, (B, 1))
    a = np.argmax(z, axis=2)
    tok = np.where(rng.random((B, N)) < 0.6, a[:, np.maximum(parent, 0)], rng.integers(0, V, (B, N))).astype(np.int32)
    out = oracle.verify_tree(z, None, P_, tok, None, None, 0.0)
    for b in range(B):
        u, k, path = 0, 0, []
        while True:
            nxt = [c for c in range(u + 1, N) if parent[c] == u and tok[b, c] == a[b, u]]
            if not nxt:
                break
            path.append(nxt[0])
            u = nxt[0]
        assert out["accept_count"][b] == len(path)
        assert list(out["out_nodes"][b, :len(path)]) == path
        assert list(out["out_tokens"][b, :len(path)]) == [tok[b, c] for c in path]
        assert out["out_tokens"][b, len(path)] == a[b, u]


def test_tree_bad_rows_anywhere():
    """A bad target row, or a bad draft row of a node with children, makes the
    sequence bad wherever it sits, reached by the walk or not; the draft row
    of a leaf is never read."""
    rng = np.random.default_rng(76)
    B, V = 6, 50
    parent = np.tile(np.array([-1, 0, 0, 1, 2], np.int32), (B, 1))
    N = parent.shape[1]
    z = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    d = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    r = np.ones((B, N), np.float32)
    keys = _keys(B, 77)
    z[1, 4, 3] = np.nan          # target row of a leaf
    d[2, 2, 0] = np.inf          # draft row of an internal node
    d[3, 3, :] = np.nan          # draft row of a leaf: not read
    d[3, 4, :] = -np.inf
    tok[4, 2] = V                # token out of range
    parent[5, 3] = 3             # parent not before the node
    out = oracle.verify_tree(z, d, parent, tok, r, keys, 1.0)
    assert list(np.nonzero(out["status"])[0]) == [1, 2, 4, 5]
    assert (out["accept_count"][[1, 2, 4, 5]] == -1).all()
    assert (out["out_tokens"][[1, 2, 4, 5]] == -1).all()
    g = oracle.verify_tree(z, None, parent, tok, None, None, 0.0)
    assert list(np.nonzero(g["status"])[0]) == [1, 4, 5]
