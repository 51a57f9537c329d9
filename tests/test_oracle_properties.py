"""Property tests of the oracle's output structure on random small inputs
(hypothesis; CPU only).  These hold for any sampling rule that follows the
method: the accepted prefix is the draft prefix, exactly one token is drawn
after it, padding is -1, every id is in range, a rejected draft token is
never the drawn one, and a tree outcome is a path from the root."""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


def _keys(B, seed):
    return np.random.default_rng(seed).integers(0, 2 ** 63, B, dtype=np.int64).view(np.uint64)


@st.composite
def chain_case(draw):
    B = draw(st.integers(1, 6))
    g = draw(st.integers(1, 6))
    V = draw(st.integers(2, 60))
    seed = draw(st.integers(0, 2 ** 31))
    T = draw(st.sampled_from([0.3, 1.0, 2.0]))
    rng = np.random.default_rng(seed)
    z = (rng.normal(0, 2, (B, g + 1, V))).astype(np.float32)
    d = (z[:, :g] + rng.normal(0, draw(st.sampled_from([0.0, 0.5, 2.0])), (B, g, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    r = (1 - rng.random((B, g))).astype(np.float32)
    return z, d, tok, r, _keys(B, seed), T


@settings(max_examples=60, deadline=None)
@given(chain_case())
def test_chain_output_structure(case):
    z, d, tok, r, keys, T = case
    B, g1, V = z.shape
    g = g1 - 1
    out = oracle.verify_chain(z, d, tok, r, keys, T)
    for b in range(B):
        k = out["accept_count"][b]
        assert 0 <= k <= g
        row = out["out_tokens"][b]
        assert list(row[:k]) == list(tok[b, :k])
        assert 0 <= row[k] < V
        assert (row[k + 1:] == -1).all()
        if k < g:  # rejected means p(x) < q(x): the residual max(0, p - q) is 0 there
            assert row[k] != tok[b, k]
            assert 0 <= out["trials"][b] <= 65


@settings(max_examples=40, deadline=None)
@given(chain_case())
def test_greedy_output_structure(case):
    z, _, tok, _, _, _ = case
    B, g1, V = z.shape
    g = g1 - 1
    a = np.argmax(z, axis=2)
    tok = np.where(np.random.default_rng(1).random(tok.shape) < 0.7, a[:, :g], tok).astype(np.int32)
    out = oracle.verify_greedy(z, tok)
    for b in range(B):
        k = out["accept_count"][b]
        assert list(out["out_tokens"][b, :k]) == list(tok[b, :k]) == list(a[b, :k])
        assert k == g or tok[b, k] != a[b, k]
        assert out["out_tokens"][b, k] == a[b, k]


@settings(max_examples=40, deadline=None)
@given(chain_case(), st.integers(1, 64), st.sampled_from([1.0, 0.9, 0.5]))
def test_filtered_output_structure(case, top_k, top_p):
    z, d, tok, r, keys, T = case
    B, g1, V = z.shape
    g = g1 - 1
    out = oracle.verify_filtered(z, d, tok, r, keys, T, top_k, top_p)
    for b in range(B):
        if out["status"][b] != 0:  # a draft token outside both kept sets can leave no residual
            assert out["accept_count"][b] == -1
            continue
        k = out["accept_count"][b]
        assert list(out["out_tokens"][b, :k]) == list(tok[b, :k])
        x = out["out_tokens"][b, k]
        assert 0 <= x < V
        if k < g:
            assert x != tok[b, k]
        kept = oracle.filter_row(z[b, k], T, top_k, top_p)[0]
        assert x in set(np.asarray(kept).tolist())   # every emitted token lies in the filtered target support


@st.composite
def tree_case(draw):
    B = draw(st.integers(1, 5))
    N = draw(st.integers(1, 12))
    V = draw(st.integers(2, 40))
    seed = draw(st.integers(0, 2 ** 31))
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, np.int32)
    for v in range(1, N):
        parent[:, v] = rng.integers(0, v, B)
    z = rng.normal(0, 2, (B, N, V)).astype(np.float32)
    d = (z + rng.normal(0, 1, (B, N, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    r = (1 - rng.random((B, N))).astype(np.float32)
    return z, d, parent, tok, r, _keys(B, seed), draw(st.sampled_from([0.0, 1.0]))


@settings(max_examples=60, deadline=None)
@given(tree_case())
def test_tree_outcome_is_a_path(case):
    z, d, parent, tok, r, keys, T = case
    B, N, V = z.shape
    out = oracle.verify_tree(z, d if T > 0 else None, parent, tok, r if T > 0 else None, keys if T > 0 else None, T)
    for b in range(B):
        assert out["status"][b] == 0
        k = out["accept_count"][b]
        nodes = out["out_nodes"][b]
        u = 0
        for j in range(k):  # each accepted node is a child of the previous one
            v = nodes[j]
            assert parent[b, v] == u
            assert out["out_tokens"][b, j] == tok[b, v]
            u = v
        assert 0 <= out["out_tokens"][b, k] < V
        assert (out["out_tokens"][b, k + 1:] == -1).all() and (nodes[k:] == -1).all()
        if T == 0:
            assert out["out_tokens"][b, k] == np.argmax(z[b, u])
