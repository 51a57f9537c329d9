"""GPU parity of the tree verify (spv_verify_tree) against the oracle
(oracle.verify_tree), element by element.

Draft trees: the 21-node tree (root, 4, 8, 8) of tree-style verification and
the width-4 tree of [SPD]'s tree drafting, on the spd distributions; the
children of a node are drawn i.i.d. from its draft distribution (T > 0) or
are its top draft ids (T = 0).  Verification by multi-round speculative
sampling (SpecInfer, stochastic verification).  Same rule as the chain
parity tests: accept counts, emitted ids and accepted nodes bit-exact except
for sequences whose oracle decision margin is below 1e-6, counted and kept
under 1e-4 of the nodes checked.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_token_spv_gb300 import workloads
from test_gpu_parity import MARGIN, _np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def _oracle_tree(w):
    T = w.temperature
    return oracle.verify_tree(_np(w.target), _np(w.draft) if T > 0 else None, _np(w.parent), _np(w.tokens),
                              _np(w.r) if T > 0 else None,
                              w.keys.cpu().numpy().view(np.uint64) if T > 0 else None, T)


def check_tree(spv, w, expect_bad=None):
    got = spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, w.temperature)
    torch.cuda.synchronize()
    ref = _oracle_tree(w)
    st = _np(got["row_status"])
    assert np.array_equal(st, ref["status"]), (st, ref["status"])
    if expect_bad is not None:
        assert list(np.nonzero(ref["status"])[0]) == list(expect_bad)
    near = ref["margin"] < MARGIN
    same = ((_np(got["accept_count"]) == ref["accept_count"]) & (_np(got["out_tokens"]) == ref["out_tokens"]).all(1)
            & (_np(got["out_nodes"]) == ref["out_nodes"]).all(1))
    bad_far = ~same & ~near
    assert not bad_far.any(), (f"{w.name}: {bad_far.sum()} sequences differ: {np.nonzero(bad_far)[0][:10]}",
                               _np(got["accept_count"])[bad_far][:5], ref["accept_count"][bad_far][:5],
                               _np(got["out_tokens"])[bad_far][:3], ref["out_tokens"][bad_far][:3])
    assert near.sum() <= 1e-4 * w.B * w.N, f"{near.sum()} near-tie sequences"
    return got, ref


def _chain_as_tree(w):
    """The chain inputs as a path tree: node v = position v; the leaf's draft
    row is a copy of the last one (never read)."""
    B, g = w.B, w.gamma
    draft = torch.cat([w.draft, w.draft[:, -1:]], dim=1)
    parent = torch.arange(-1, g, dtype=torch.int32, device=w.target.device).repeat(B, 1)
    tok = torch.cat([torch.zeros(B, 1, dtype=torch.int32, device=w.target.device), w.tokens], dim=1)
    r = torch.cat([torch.ones(B, 1, device=w.target.device), w.r], dim=1)
    return workloads.TreeInputs("path_" + w.name, w.target, draft.contiguous(), parent, tok.contiguous(),
                                r.contiguous(), w.keys, w.temperature)


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_path_tree_is_the_chain(spv, dtype, T):
    """A single path: the same outcome as spv_verify_chain on the chain."""
    w = workloads.sweep(B=64, dtype=dtype, device="cuda", temperature=T)
    t = _chain_as_tree(w)
    got, ref = check_tree(spv, t)
    ch = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, T)
    torch.cuda.synchronize()
    near = ref["margin"] < MARGIN
    k = _np(got["accept_count"])
    assert np.array_equal(k[~near], _np(ch["accept_count"])[~near])
    assert np.array_equal(_np(got["out_tokens"])[~near], _np(ch["out_tokens"])[~near])
    nodes = _np(got["out_nodes"])
    assert all(list(nodes[b, :k[b]]) == list(range(1, k[b] + 1)) for b in range(w.B))


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("shape", ["k21", "w4"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_trees_spd(spv, dtype, shape, T):
    """B = 32 trees over V = 151,936."""
    w = workloads.tree(B=32, shape=shape, dtype=dtype, temperature=T, device="cuda")
    got, ref = check_tree(spv, w)
    k = ref["accept_count"]
    assert (k >= 1).any()
    if T > 0:
        assert (k == 0).any() or shape == "w4"


def test_many_children_and_ragged_vocab(spv):
    """A root with 31 children (the maximum node count), V not a multiple of
    the block or of 4 ids (plain loads); a star with low acceptance walks
    through many residuals."""
    for V in (1001, 20000):
        gen = torch.Generator(device="cpu").manual_seed(80 + V)
        B, N = 24, 32
        z = torch.randn(B, N, V, generator=gen) * 2.0
        d = torch.randn(B, N, V, generator=gen) * 2.0    # unrelated: low acceptance
        parent = torch.zeros(B, N, dtype=torch.int32)
        parent[:, 0] = -1
        q0 = torch.softmax(d[:, 0], dim=1)
        tok = torch.zeros(B, N, dtype=torch.int32)
        tok[:, 1:] = torch.multinomial(q0, N - 1, replacement=True, generator=gen).int()
        r = 1.0 - torch.rand(B, N, generator=gen)
        keys = torch.randint(-(2 ** 62), 2 ** 62, (B,), generator=gen, dtype=torch.int64)
        w = workloads.TreeInputs("star31", z.cuda(), d.cuda(), parent.cuda(), tok.cuda(), r.cuda(), keys.cuda(), 1.0)
        got, ref = check_tree(spv, w)
        assert (ref["accept_count"] == 0).any()


def test_single_node_and_deep_path(spv):
    """N = 1: the bonus token from the root; N = 32 and N = 64 (the node
    limit) as one path."""
    gen = torch.Generator(device="cpu").manual_seed(83)
    for N in (1, 32, 64):
        B, V = 8, 5000
        z = torch.randn(B, N, V, generator=gen)
        d = z + 0.3 * torch.randn(B, N, V, generator=gen)
        parent = torch.arange(-1, N - 1, dtype=torch.int32).repeat(B, 1)
        tok = torch.zeros(B, N, dtype=torch.int32)
        for v in range(1, N):
            tok[:, v] = torch.multinomial(torch.softmax(d[:, v - 1], dim=1), 1, generator=gen)[:, 0].int()
        r = 1.0 - torch.rand(B, N, generator=gen)
        keys = torch.arange(B, dtype=torch.int64) * 1000003
        w = workloads.TreeInputs(f"path{N}", z.cuda(), d.cuda(), parent.cuda(), tok.cuda(), r.cuda(), keys.cuda(), 1.0)
        check_tree(spv, w)
        w0 = workloads.TreeInputs(w.name, w.target, w.draft, w.parent, w.tokens, w.r, w.keys, 0.0)
        check_tree(spv, w0)


def test_direct_residual_draw(spv):
    """p close to q at the root and two children: after two rejections the
    residual max(0, p - 2q) holds little mass, the rejection trials fail and
    the direct residual race runs."""
    gen = torch.Generator(device="cpu").manual_seed(84)
    B, V = 16, 9000
    d = torch.randn(B, 3, V, generator=gen) * 2.0
    z = d + torch.randn(B, 3, V, generator=gen) * 1e-2
    parent = torch.tensor([-1, 0, 0], dtype=torch.int32).repeat(B, 1)
    # children: two ids whose draft probability is raised above p, so both
    # are rejected at r = 1
    low = torch.argsort(z[:, 0], dim=1)[:, :2]
    d[:, 0].scatter_add_(1, low, torch.ones(B, 2))
    tok = torch.cat([torch.zeros(B, 1, dtype=torch.int32), low.int()], dim=1)
    r = torch.ones(B, 3)
    keys = torch.arange(B, dtype=torch.int64) * 7919
    w = workloads.TreeInputs("near_q", z.cuda(), d.cuda(), parent.cuda(), tok.cuda(), r.cuda(), keys.cuda(), 1.0)
    got, ref = check_tree(spv, w)
    assert (ref["trials"] > 64).any()


def test_bad_rows(spv):
    w = workloads.tree(B=8, shape="k21", V=3000, dtype=torch.float32, device="cpu")
    w.target[1, 20, 3] = float("nan")     # target row of a leaf
    w.draft[2, 4, 0] = float("inf")       # draft row of an internal node
    w.draft[3, 20] = float("nan")         # draft row of a leaf: never read
    w.tokens[4, 7] = 3000                 # out of range
    w.parent[5, 9] = 9                    # not before the node
    w.target[6, 0] = float("-inf")        # no finite logit at the root
    w = workloads.TreeInputs(w.name, w.target.cuda(), w.draft.cuda(), w.parent.cuda(), w.tokens.cuda(), w.r.cuda(),
                             w.keys.cuda(), 1.0)
    check_tree(spv, w, expect_bad=[1, 2, 4, 5, 6])
    w0 = workloads.TreeInputs(w.name, w.target, w.draft, w.parent, w.tokens, w.r, w.keys, 0.0)
    check_tree(spv, w0, expect_bad=[1, 4, 5, 6])


def test_invalid_arguments(spv):
    w = workloads.tree(B=2, shape="w4", V=500, dtype=torch.float32, device="cuda")
    with pytest.raises(spv.SpvError):
        spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, -1.0)
    with pytest.raises(spv.SpvError):
        spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, float("nan"))
    big = torch.zeros(1, 65, 64, device="cuda")
    par = torch.arange(-1, 64, dtype=torch.int32, device="cuda")[None]
    with pytest.raises(spv.SpvError):
        spv.spv_verify_tree(big, big, par, torch.zeros_like(par), torch.ones(1, 65, device="cuda"),
                            torch.zeros(1, dtype=torch.int64, device="cuda"), 1.0)


@pytest.mark.parametrize("B", [8, 40, 80, 200])
def test_finalize_split_over_clusters(spv, B):
    """The walk's residual passes run on a cluster of CTAs per sequence, as
    many as the idle SMs allow (8 at B = 8, 2 at B = 40, 1 at B = 80, and
    the narrow finalize at B = 200): the same outcomes as the oracle."""
    w = workloads.tree(B=B, shape="w4", V=30000, dtype=torch.float32, device="cuda", d_std=2.0)
    got, ref = check_tree(spv, w)
    assert (ref["accept_count"] == 0).any()


def test_statistics_not_staged(spv):
    """A 32-node path at V = 151,936: 32 target rows x 149 blocks exceed the
    shared-memory staging of block statistics (the workspace path)."""
    gen = torch.Generator(device="cpu").manual_seed(90)
    B, N, V = 2, 32, 151936
    z = torch.randn(B, N, V, generator=gen) * 2.0
    d = z + 0.4 * torch.randn(B, N, V, generator=gen)
    parent = torch.arange(-1, N - 1, dtype=torch.int32).repeat(B, 1)
    parent[:, 5] = 0   # a second child of the root
    tok = torch.zeros(B, N, dtype=torch.int32)
    for v in range(1, N):
        pv = parent[0, v].item()
        tok[:, v] = torch.multinomial(torch.softmax(d[:, pv], dim=1), 1, generator=gen)[:, 0].int()
    r = 1.0 - torch.rand(B, N, generator=gen)
    keys = torch.arange(B, dtype=torch.int64) * 31337 + 5
    w = workloads.TreeInputs("unstaged", z.cuda(), d.cuda(), parent.cuda(), tok.cuda(), r.cuda(), keys.cuda(), 1.0)
    check_tree(spv, w)


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_binary_tree_63_nodes(spv, dtype, T):
    """A depth-5 binary tree (63 nodes): children masks past 32 nodes, the
    parents of nodes 32..62 in the leaf-row skip."""
    w = workloads.tree(B=16, shape="b63", V=20000, dtype=dtype, temperature=T, device="cuda")
    got, ref = check_tree(spv, w)
    assert (ref["accept_count"] >= 3).any()


def _random_trees(B, N, V, dtype, seed, T=1.0):
    """A different random recursive tree per sequence (parent of node v
    uniform over 0 .. v-1), so the sequences read different numbers of draft
    rows; children's tokens drawn from their parent's draft distribution."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    z = torch.randn(B, N, V, generator=gen) * 2.0
    d = z + torch.randn(B, N, V, generator=gen)
    parent = torch.full((B, N), -1, dtype=torch.int32)
    for v in range(1, N):
        parent[:, v] = torch.randint(0, v, (B,), generator=gen, dtype=torch.int32)
    tok = torch.zeros(B, N, dtype=torch.int32)
    for v in range(1, N):
        q = torch.softmax(d[torch.arange(B), parent[:, v].long()], dim=1)
        tok[:, v] = torch.multinomial(q, 1, generator=gen)[:, 0].int()
    r = 1.0 - torch.rand(B, N, generator=gen)
    keys = torch.randint(-(2 ** 62), 2 ** 62, (B,), generator=gen, dtype=torch.int64)
    return workloads.TreeInputs(f"random{N}_B{B}", z.to(dtype).cuda(), d.to(dtype).cuda(), parent.cuda(), tok.cuda(),
                                r.cuda(), keys.cuda(), T)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_random_tree_per_sequence(spv, dtype):
    """Every sequence its own tree (different rows read per sequence, the
    streaming pass numbering only the rows it reads), at T = 1 and T = 0."""
    w = _random_trees(B=48, N=24, V=12288, dtype=dtype, seed=91)
    check_tree(spv, w)
    check_tree(spv, workloads.TreeInputs(w.name, w.target, w.draft, w.parent, w.tokens, w.r, w.keys, 0.0))


def test_more_sequences_than_the_skip_table(spv):
    """B = 1100 bf16 sequences, above the 1024 the streaming pass's
    shared-memory table of rows read holds: the rows are taken on the static
    stride with a vote per row instead; same outputs as the oracle."""
    w = _random_trees(B=1100, N=9, V=2048, dtype=torch.bfloat16, seed=92)
    check_tree(spv, w)


def test_bf16_rows_not_16_byte_aligned(spv):
    """bf16 rows of V = 12,289 logits (not a multiple of 8 ids, so not
    16-byte aligned): the streaming pass loads the rows without TMA and
    votes on the skipped rows, the residual passes use plain loads; same
    outputs as the oracle at T = 1 and T = 0."""
    w = _random_trees(B=24, N=12, V=12289, dtype=torch.bfloat16, seed=93)
    check_tree(spv, w)
    check_tree(spv, workloads.TreeInputs(w.name, w.target, w.draft, w.parent, w.tokens, w.r, w.keys, 0.0))
