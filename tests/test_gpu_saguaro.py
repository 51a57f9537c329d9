"""GPU parity of the verify step for Saguaro-sampled drafts
(spv_verify_chain_saguaro) against the oracle (oracle.verify_saguaro).

Saguaro sampling ("Speculative Speculative Decoding", Key Innovations /
Table 7b, logit bonus C): the draft draws position i from q_C, its
distribution with the probability of the position's cached candidates
divided by C.  The cache lists are the top-F_k ids of the draft rows of
positions 0..gamma (the oracle's fan-out, no exclusion); the draft tokens are
drawn from q_C.  Same bit-exact-or-near-tie rule as the other parity tests;
the cache slot is compared too.
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


def _lists(w, F):
    d, _ = workloads.cache_fanout_inputs(w)
    ex = np.full((w.B, w.gamma + 1), -1, np.int32)
    return oracle.fanout_topk(_np(d), ex, F)["ids"]


def _with_tokens(w, tok):
    return workloads.ChainInputs(w.name, w.target, w.draft, tok, w.r, w.keys, w.temperature, w.meta, w.draft_bonus)


def check_saguaro(spv, w, F, lists, C, want_Z=True, expect_bad=None, z_atol=0.0):
    ids = torch.from_numpy(np.ascontiguousarray(lists)).to(w.target.device)
    got = spv.spv_verify_chain_saguaro(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, ids, F, C,
                                       want_resid_norm=want_Z and w.temperature > 0)
    torch.cuda.synchronize()
    ref = oracle.verify_saguaro(_np(w.target), _np(w.draft), _np(w.tokens), _np(w.r),
                                w.keys.cpu().numpy().view(np.uint64), w.temperature, lists, F, C,
                                want_Z=want_Z and w.temperature > 0)
    B, g = w.B, w.gamma
    st = _np(got["row_status"])
    assert np.array_equal(st, ref["status"]), (st, ref["status"])
    if expect_bad is not None:
        assert list(np.nonzero(ref["status"])[0]) == list(expect_bad)
    margin = ref.get("margin", np.full(B, np.inf))
    near = margin < MARGIN
    same = (_np(got["accept_count"]) == ref["accept_count"]) & (_np(got["out_tokens"]) == ref["out_tokens"]).all(1)
    assert not (~same & ~near).any(), np.nonzero(~same & ~near)[0][:10]
    assert near.sum() <= 1e-4 * B * (g + 1)
    want = oracle.cache_slots(ref["accept_count"], ref["out_tokens"], lists, F)
    far = ~near
    assert np.array_equal(_np(got["cache_slot"])[far], want[far])
    if w.temperature > 0:
        ok = ref["status"] == 0
        np.testing.assert_allclose(_np(got["pq"])[ok], ref["pq"][ok], rtol=RTOL, atol=1e-30)
        if want_Z:
            np.testing.assert_allclose(_np(got["resid_norm"])[ok], ref["Z"][ok], rtol=RTOL, atol=z_atol)
    return got, ref


@pytest.mark.parametrize("C", [1.0, 4.0, 16.0])
def test_sweep_B64(spv, C):
    w = workloads.sweep(B=64, device="cuda", bonus_draft=True)
    F = [8, 7, 6, 5, 4]
    lists = _lists(w, F)
    w = _with_tokens(w, workloads.saguaro_tokens(w, torch.from_numpy(lists).cuda(), F, C))
    got, ref = check_saguaro(spv, w, F, lists, C)
    if C == 1.0:  # the same kernels as the plain cached verify
        plain = spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, w.r, w.keys, 1.0,
                                            torch.from_numpy(lists).cuda(), F)
        torch.cuda.synchronize()
        for key in ("accept_count", "out_tokens", "cache_slot", "pq"):
            assert torch.equal(got[key], plain[key]), key


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_spd_and_tiny(spv, T):
    for w, C in ((workloads.spd(device="cuda", temperature=T, bonus_draft=True), 2.0),
                 (_to(workloads.tiny(device="cpu", temperature=T, bonus_draft=True), "cuda"), 8.0)):
        F = [16] * (w.gamma + 1)
        lists = _lists(w, F)
        if T > 0:
            w = _with_tokens(w, workloads.saguaro_tokens(w, torch.from_numpy(lists).cuda(), F, C))
        check_saguaro(spv, w, F, lists, C)


def test_eagle_bf16_wide_lists(spv):
    w = workloads.eagle(gamma=7, device="cuda", bonus_draft=True)
    F = [64, 40, 33, 20, 9, 5, 1, 0]
    lists = _lists(w, F)
    w = _with_tokens(w, workloads.saguaro_tokens(w, torch.from_numpy(lists).cuda(), F, 3.0))
    check_saguaro(spv, w, F, lists, 3.0)


def test_direct_residual_draw(spv):
    """Targets equal to q_C up to a small perturbation: the residual has
    little mass, the rejection trials fail and the direct residual race runs,
    with the cached ids' masses corrected in their blocks."""
    gen = torch.Generator(device="cpu").manual_seed(61)
    B, g, V, C = 16, 2, 9000, 5.0
    d = torch.randn(B, g + 1, V, generator=gen) * 2.0
    F = [40, 40, 40]
    lists = np.stack([np.concatenate([np.argsort(-d[b, i].numpy(), kind="stable")[:40] for i in range(g + 1)])
                      for b in range(B)]).astype(np.int32)
    z = d.clone()
    for b in range(B):
        for i in range(g + 1):
            z[b, i, lists[b, 40 * i:40 * (i + 1)]] -= float(np.log(C))   # p proportional to q_C
    z += torch.randn(B, g + 1, V, generator=gen) * 1e-3
    tok = torch.stack([torch.from_numpy(lists[:, 40 * i]) for i in range(g)], dim=1).int()
    r = torch.ones(B, g)
    keys = torch.arange(B, dtype=torch.int64) * 7919
    w = workloads.ChainInputs("near_qc", z, d[:, :g].contiguous(), tok, r, keys, 1.0, {})
    w = _to(w, "cuda")
    got, ref = check_saguaro(spv, w, F, lists, C, z_atol=1e-6)
    assert (ref["trials"] > 64).any()


def test_bad_rows_and_arguments(spv):
    w = _to(workloads.sweep(B=4, V=3000, gamma=2, device="cpu", bonus_draft=True), "cuda")
    F = [10, 10, 10]
    lists = _lists(w, F)
    w.target[1, 0, 5] = float("nan")
    w.tokens[2, 1] = -3
    check_saguaro(spv, w, F, lists, 2.0, expect_bad=[1, 2])
    ids = torch.from_numpy(lists).cuda()
    for C in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(spv.SpvError):
            spv.spv_verify_chain_saguaro(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, ids, F, C)


def test_many_sequences_narrow_finalize(spv):
    """B = 200 > the SM count: the 8-warp finalize with Saguaro weights."""
    w = workloads.sweep(B=200, V=20000, gamma=3, device="cuda", bonus_draft=True)
    F = [12, 10, 8, 6]
    lists = _lists(w, F)
    w = _with_tokens(w, workloads.saguaro_tokens(w, torch.from_numpy(lists).cuda(), F, 4.0))
    check_saguaro(spv, w, F, lists, 4.0)
