"""GPU parity of the top-k / top-p filtered verify (spv_verify_chain_filtered)
against the oracle (oracle.verify_filtered), element by element.

The filtered distributions are those of the sampled runs in "Speculative
Pipeline Decoding", section "Evaluation" (top-k = 50, top-p = 1.0 at T = 1).
Same rule as the unfiltered parity tests: accept counts and emitted ids
bit-exact except for sequences whose oracle decision margin (accept test,
race log-gap, top-p cut) is below 1e-6, counted and kept under 1e-4 of the
positions; p'(x_i), q'(x_i) and the residual normaliser within 1e-5
relative.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_token_spv_gb300 import workloads
from test_gpu_parity import MARGIN, RTOL, _np, _to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def check_filtered(spv, w, top_k, top_p=1.0, want_Z=True, expect_bad=None, z_atol=0.0, near_budget=1e-4):
    got = spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, top_k, top_p,
                                        want_resid_norm=want_Z)
    torch.cuda.synchronize()
    ref = oracle.verify_filtered(_np(w.target), _np(w.draft), _np(w.tokens), _np(w.r),
                                 w.keys.cpu().numpy().view(np.uint64), w.temperature, top_k, top_p,
                                 want_Z=want_Z and w.temperature > 0)
    B, g = w.B, w.gamma
    st = _np(got["row_status"])
    assert np.array_equal(st, ref["status"]), (st, ref["status"])
    if expect_bad is not None:
        assert list(np.nonzero(ref["status"])[0]) == list(expect_bad)
    margin = ref.get("margin", np.full(B, np.inf))
    near = margin < MARGIN
    same = (_np(got["accept_count"]) == ref["accept_count"]) & (_np(got["out_tokens"]) == ref["out_tokens"]).all(1)
    bad_far = ~same & ~near
    assert not bad_far.any(), (f"{w.name}: {bad_far.sum()} sequences differ: {np.nonzero(bad_far)[0][:10]}",
                               _np(got["accept_count"])[bad_far][:5], ref["accept_count"][bad_far][:5],
                               _np(got["out_tokens"])[bad_far][:3], ref["out_tokens"][bad_far][:3])
    assert near.sum() <= max(near_budget * B * (g + 1), 0), f"{near.sum()} near-tie sequences"
    if w.temperature > 0:
        ok = ref["status"] == 0
        np.testing.assert_allclose(_np(got["pq"])[ok], ref["pq"][ok], rtol=RTOL, atol=1e-30)
        if want_Z:
            np.testing.assert_allclose(_np(got["resid_norm"])[ok], ref["Z"][ok], rtol=RTOL, atol=z_atol)
    return got, ref


@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (1, 1.0), (64, 1.0), (20, 0.8), (7, 0.3)])
def test_tiny(spv, top_k, top_p):
    w = _to(workloads.tiny(device="cpu", top_k=top_k, top_p=top_p), "cuda")
    check_filtered(spv, w, top_k, top_p)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_spd_top50(spv, T):
    """The SPD sampling setup: B = 64, gamma = 1, V = 151,936, bf16, top-k 50."""
    w = workloads.spd(device="cuda", temperature=T, top_k=50)
    got, ref = check_filtered(spv, w, 50)
    k = ref["accept_count"]
    assert (k == 0).any() and (k == 1).any()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B", [1, 8, 64])
def test_sweep_top50(spv, dtype, B):
    """B = 1 (a few rows, many streaming CTAs per row) to B = 64."""
    w = workloads.sweep(B=B, dtype=dtype, device="cuda", top_k=50)
    check_filtered(spv, w, 50)


def test_eagle_nucleus(spv):
    w = workloads.eagle(gamma=7, device="cuda", top_k=40, top_p=0.9)
    check_filtered(spv, w, 40, 0.9)


@pytest.mark.parametrize("gamma", [8, 15])
def test_more_rows_than_sixteen(spv, gamma):
    """2 gamma + 1 > 16 rows per sequence (the finalize selects every row's
    top k at once with one warp per row): the EAGLE gamma = 15 workload with
    top-k 50 and top-p 0.9, and gamma = 8 on a smaller vocabulary."""
    if gamma == 15:
        w = workloads.eagle(gamma=15, device="cuda", top_k=50, top_p=0.9)
        check_filtered(spv, w, 50, 0.9)
    else:
        w = workloads.sweep(B=24, dtype=torch.float32, device="cuda", V=30000, gamma=8, top_k=50)
        check_filtered(spv, w, 50)
        check_filtered(spv, w, 64, 0.9)


@pytest.mark.parametrize("V", [20, 1001, 1025, 8193, 50000])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_vocab_and_plain_loads(spv, V, dtype):
    """Ragged tails, V < top_k, and vocabularies whose rows are not 16-byte
    multiples (plain-load path)."""
    w = workloads.sweep(B=6, dtype=dtype, device="cuda", V=V, gamma=3, top_k=33)
    check_filtered(spv, w, 33)
    check_filtered(spv, w, 64, 0.95)


@pytest.mark.parametrize("levels", [3, 8])
def test_heavy_ties(spv, levels):
    """Quantised logits: the top-k cut falls inside a run of equal logits, which
    goes to the lower ids; -0.0 ranks with +0.0.  A constant row makes every
    logit reach the sampled threshold (more candidates than the buffers hold:
    the exact re-scan)."""
    gen = torch.Generator(device="cuda").manual_seed(50 + levels)
    B, g, V = 8, 3, 9000
    z = torch.round(torch.randn(B, g + 1, V, generator=gen, device="cuda") * levels / 3)
    d = torch.round(z[:, :g] + torch.randn(B, g, V, generator=gen, device="cuda") * 0.7)
    z[z == 0] = -0.0
    z[2] = 1.5   # constant rows
    d[2] = 1.5
    tok = workloads._draft_tokens(d, 1.0, 5, "cuda", 50)
    r = 1.0 - torch.rand(B, g, generator=gen, device="cuda")
    keys = torch.randint(-(2 ** 62), 2 ** 62, (B,), generator=gen, device="cuda", dtype=torch.int64)
    w = workloads.ChainInputs("ties", z, d, tok, r, keys, 1.0, {})
    check_filtered(spv, w, 50)


def test_bad_rows(spv):
    w = _to(workloads.sweep(B=6, V=3000, gamma=2, device="cpu", top_k=20), "cuda")
    w.target[1, 0, 17] = float("nan")
    w.draft[2, 1, 2999] = float("inf")
    w.target[3, 2] = float("-inf")          # no finite logit in the bonus row
    w.tokens[4, 1] = 3000                   # out of range
    # sequence 5: a draft token outside both kept sets with p' = q' elsewhere
    w.draft[5, 0] = w.target[5, 0]
    w.target[5, 0, 11] = float("-inf")
    w.draft[5, 0, 11] = float("-inf")
    w.tokens[5, 0] = 11
    check_filtered(spv, w, 20, expect_bad=[1, 2, 3, 4, 5])


def test_repeat_calls_and_workspace_reuse(spv):
    """Two shapes through one workspace, then the first again: same results."""
    a = workloads.sweep(B=8, V=20000, gamma=4, device="cuda", top_k=50)
    b = workloads.sweep(B=3, V=151936, gamma=2, device="cuda", top_k=10)
    ws = spv.new_workspace(max(spv.spv_filtered_workspace_bytes(8, 4, 151936),
                               spv.spv_filtered_workspace_bytes(3, 2, 151936)), "cuda")
    o1 = spv.spv_verify_chain_filtered(a.target, a.draft, a.tokens, a.r, a.keys, 1.0, 50, workspace=ws)
    o1 = {k: v.clone() for k, v in o1.items()}
    spv.spv_verify_chain_filtered(b.target, b.draft, b.tokens, b.r, b.keys, 1.0, 10, workspace=ws)
    o3 = spv.spv_verify_chain_filtered(a.target, a.draft, a.tokens, a.r, a.keys, 1.0, 50, workspace=ws)
    torch.cuda.synchronize()
    for k in o1:
        assert torch.equal(o1[k], o3[k]), k
    assert spv.spv_workspace_status(ws) == spv.SPV_OK


def test_invalid_arguments(spv):
    w = _to(workloads.tiny(device="cpu", top_k=5), "cuda")
    for k, p in [(0, 1.0), (65, 1.0), (5, 0.0), (5, 1.5), (5, float("nan"))]:
        with pytest.raises(spv.SpvError):
            spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, k, p)


def test_max_gamma(spv):
    """gamma = 32 at B = 1: 65 rows, five row groups in the finalize."""
    w = workloads.sweep(B=1, gamma=32, device="cuda", top_k=64, top_p=0.9)
    check_filtered(spv, w, 64, 0.9)


def test_many_sequences_narrow_finalize(spv):
    """B = 200 > the SM count: the 8-warp finalize, two CTAs per SM."""
    w = workloads.sweep(B=200, V=20000, gamma=2, device="cuda", top_k=40, top_p=0.95)
    check_filtered(spv, w, 40, 0.95)
    wb = workloads.sweep(B=200, V=20000, gamma=2, dtype=torch.bfloat16, device="cuda", top_k=8)
    check_filtered(spv, wb, 8)
