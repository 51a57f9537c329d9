"""GPU parity of the fused verify -> speculation-cache lookup
(spv_verify_chain_cached) against the oracle.

The cache of each sequence is the fan-out of "Speculative Speculative
Decoding" (Figure 2): at each position k = 0..gamma the F_k top-ranked draft
tokens, skipping the token verified there.  The candidate lists fed to the GPU
come from the oracle's fan-out of the same draft rows; the expected slot is the
oracle's lookup of the oracle's verify outcome.  Slots are compared bit-exactly
on every sequence whose verify outcome is outside the near-tie exemption.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_token_spv_gb300 import workloads
from test_gpu_parity import MARGIN, _np, _oracle_chain, _to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def _oracle_lists(w, F):
    d, ex = workloads.cache_fanout_inputs(w)
    return oracle.fanout_topk(_np(d), _np(ex), F)["ids"]


def check_cached(spv, w, F, lists):
    ids = torch.from_numpy(np.ascontiguousarray(lists)).to(w.target.device)
    got = spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, ids, F)
    plain = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature)
    torch.cuda.synchronize()
    ref = _oracle_chain(w)
    # the lookup changes none of the verify outputs
    for key in ("accept_count", "out_tokens", "row_status"):
        assert torch.equal(got[key], plain[key]), key
    if "pq" in plain:
        assert torch.equal(got["pq"], plain["pq"])
    margin = ref.get("margin", np.full(w.B, np.inf))
    far = margin >= MARGIN
    same = (_np(got["accept_count"]) == ref["accept_count"]) & (_np(got["out_tokens"]) == ref["out_tokens"]).all(1)
    assert same[far].all()
    want = oracle.cache_slots(ref["accept_count"], ref["out_tokens"], lists, F)
    slot = _np(got["cache_slot"])
    assert np.array_equal(slot[far], want[far]), np.nonzero(slot != want)[0][:10]
    # the slot's entry is the emitted token, at the outcome's position
    k = _np(got["accept_count"])
    t = _np(got["out_tokens"])[np.arange(w.B), np.maximum(k, 0)]
    offs = np.concatenate([[0], np.cumsum(F)])
    hit = slot >= 0
    assert (lists[hit, slot[hit]] == t[hit]).all()
    assert (slot[hit] >= offs[k[hit]]).all() and (slot[hit] < offs[k[hit] + 1]).all()
    return got, ref, slot


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_cached_sweep_B64(spv, T):
    w = workloads.sweep(B=64, device="cuda", temperature=T, bonus_draft=True)
    F = spv.fanout_sizes(8, 0.8, 0.5, w.gamma, w.V)
    assert F == [8, 7, 6, 5, 4]
    lists = _oracle_lists(w, F)
    _, _, slot = check_cached(spv, w, F, lists)
    assert (slot >= 0).any()


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_cached_spd_and_tiny(spv, T):
    for w in (workloads.spd(device="cuda", temperature=T, bonus_draft=True),
              _to(workloads.tiny(device="cpu", temperature=T, bonus_draft=True), "cuda")):
        F = spv.fanout_sizes(8, 0.8, 0.5, w.gamma, w.V)
        check_cached(spv, w, F, _oracle_lists(w, F))


def test_cached_eagle_bf16(spv):
    w = workloads.eagle(gamma=7, device="cuda", bonus_draft=True)
    F = spv.fanout_sizes(8, 0.8, 0.5, w.gamma, w.V)
    check_cached(spv, w, F, _oracle_lists(w, F))


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_cached_planted_hits_and_misses(spv, T):
    """Lists built from the oracle's outcome: a third of the sequences carry t*
    at a random rank of position k (hit), a third carry it under another
    position only (miss), the rest not at all; F up to 64 and an empty
    position exercise the multi-pass and zero-length lookups."""
    w = workloads.sweep(B=96, V=20000, gamma=5, device="cuda", temperature=T, bonus_draft=True)
    F = [64, 33, 0, 7, 1, 40]
    ref = _oracle_chain(w)
    rng = np.random.default_rng(5)
    offs = np.concatenate([[0], np.cumsum(F)])
    lists = rng.integers(0, w.V, (w.B, offs[-1])).astype(np.int32)
    for b in range(w.B):
        k = ref["accept_count"][b]
        t = ref["out_tokens"][b, k]
        lists[b][lists[b] == t] = (t + 1) % w.V
        mode = b % 3
        if mode == 0 and F[k] > 0:
            lists[b, offs[k] + rng.integers(F[k])] = t
        elif mode == 1:
            others = [j for j in range(len(F)) if j != k and F[j] > 0]
            j = others[rng.integers(len(others))]
            lists[b, offs[j] + rng.integers(F[j])] = t
    _, _, slot = check_cached(spv, w, F, lists)
    modes = np.arange(w.B) % 3
    k = ref["accept_count"]
    assert ((slot >= 0) == ((modes == 0) & (np.array(F)[k] > 0))).all()


def test_cached_bad_rows_miss(spv):
    w = _to(workloads.tiny(device="cpu", bonus_draft=True), "cuda")
    w = workloads.ChainInputs(w.name, w.target.repeat(4, 1, 1), w.draft.repeat(4, 1, 1), w.tokens.repeat(4, 1),
                              w.r.repeat(4, 1), w.keys.repeat(4), w.temperature, w.meta, w.draft_bonus.repeat(4, 1, 1))
    w.target[1, 2, 17] = float("nan")
    w.tokens[2, 0] = w.V + 3
    F = [4, 3, 3, 2, 2]
    lists = np.tile(np.arange(sum(F), dtype=np.int32), (4, 1))
    got = spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, w.r, w.keys, 1.0,
                                      torch.from_numpy(lists).cuda(), F)
    torch.cuda.synchronize()
    st = _np(got["row_status"])
    assert st[1] == 4 and st[2] == 4 and st[0] == 0 and st[3] == 0
    assert _np(got["cache_slot"])[1] == -1 and _np(got["cache_slot"])[2] == -1


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_cached_many_sequences(spv, T):
    """B = 200 > the SM count: the 8-warp finalize (T > 0) with the lookup."""
    w = workloads.sweep(B=200, V=20000, gamma=3, device="cuda", temperature=T, bonus_draft=True)
    F = [9, 7, 5, 3]
    check_cached(spv, w, F, _oracle_lists(w, F))
