"""GPU parity: libspv (through the C ABI) against the oracle, element by element.

Rule (the acceptance criterion): accept counts, emitted ids and
fan-out ids are bit-exact, except for sequences whose oracle decision margin
(|r - p/q| of an accept test, the log-gap of a race, |(1-v) - q/p| of a
residual trial) is below 1e-6; such near-tie sequences are counted and must
stay under 1e-4 of the positions checked.  p_i(x_i), q_i(x_i) and the
residual normaliser agree within 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_token_spv_gb300 import workloads

pytestmark = pytest.mark.gpu

MARGIN = 1e-6
RTOL = 1e-5
# Z = sum max(0, p - q) from fp32 p and q: each of p, q carries a relative
# error of a few 1e-7 (fp32 exp and row sums) and sums to 1, so |dZ| is at
# most about 1e-6 whatever Z is.  Where p and q nearly coincide Z is tiny and
# cancellation makes 1e-5 relative unreachable in fp32; only that case uses
# this absolute bound (every workload run checks Z at 1e-5 relative, atol 0).
Z_ATOL_ILL_CONDITIONED = 1e-6


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float32) else t.detach().cpu().numpy()


def _oracle_chain(w, want_Z=False):
    if w.temperature == 0:
        return oracle.verify_greedy(_np(w.target), _np(w.tokens))
    return oracle.verify_chain(_np(w.target), _np(w.draft), _np(w.tokens), _np(w.r),
                               w.keys.cpu().numpy().view(np.uint64), w.temperature, want_Z=want_Z)


def _to(w, dev):
    return workloads.ChainInputs(w.name, w.target.to(dev), w.draft.to(dev), w.tokens.to(dev), w.r.to(dev),
                                 w.keys.to(dev), w.temperature, w.meta,
                                 None if w.draft_bonus is None else w.draft_bonus.to(dev))


def check_chain(spv, w, want_Z=False, expect_bad=None, z_atol=0.0):
    got = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature,
                               want_resid_norm=want_Z)
    torch.cuda.synchronize()
    ref = _oracle_chain(w, want_Z=want_Z and w.temperature > 0)
    B, g = w.B, w.gamma
    k_got, k_ref = _np(got["accept_count"]), ref["accept_count"]
    t_got, t_ref = _np(got["out_tokens"]), ref["out_tokens"]
    st_got = _np(got["row_status"])
    assert np.array_equal(st_got, ref["status"]), "row status"
    if expect_bad is not None:
        assert list(np.nonzero(ref["status"])[0]) == list(expect_bad)
    margin = ref.get("margin", np.full(B, np.inf))
    near = margin < MARGIN
    same = (k_got == k_ref) & (t_got == t_ref).all(axis=1)
    bad_far = ~same & ~near
    assert not bad_far.any(), (f"{w.name}: {bad_far.sum()} sequences differ with margin >= {MARGIN}: "
                               f"{np.nonzero(bad_far)[0][:10]}")
    positions = B * (g + 1)
    assert near.sum() <= 1e-4 * positions, f"{w.name}: {near.sum()} near-tie sequences of {positions} positions"
    if w.temperature > 0:
        ok = ref["status"] == 0
        np.testing.assert_allclose(_np(got["pq"])[ok], ref["pq"][ok], rtol=RTOL, atol=1e-30)
        if want_Z:
            np.testing.assert_allclose(_np(got["resid_norm"])[ok], ref["Z"][ok], rtol=RTOL, atol=z_atol)
    return got, ref


# ----------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tiny(spv, T):
    w = _to(workloads.tiny(device="cpu", temperature=T), "cuda")
    check_chain(spv, w, want_Z=True)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_spd_gamma1(spv, T):
    w = workloads.spd(device="cuda", temperature=T)
    got, ref = check_chain(spv, w, want_Z=True)
    k = ref["accept_count"]
    assert (k == 0).any() and (k == 1).any()


@pytest.mark.parametrize("gamma", [7, 15])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_eagle(spv, gamma, T):
    w = workloads.eagle(gamma=gamma, device="cuda", temperature=T)
    check_chain(spv, w)


@pytest.mark.parametrize("case", ["spd_B64_bf16", "sweep_B256_fp32"])
def test_greedy_entry_point(spv, case):
    """spv_verify_greedy itself (its own argument checks and greedy-sized
    workspace), bit-exact against the oracle's argmax rule: the SPD gamma = 1
    workload (B = 64, V = 151,936, bf16) and the batch sweep's largest point
    (B = 256, gamma = 4, fp32)."""
    if case == "spd_B64_bf16":
        w = workloads.spd(device="cuda", temperature=0.0)
    else:
        w = workloads.sweep(B=256, dtype=torch.float32, device="cuda", temperature=0.0)
    ws = spv.new_workspace(spv.spv_greedy_workspace_bytes(w.B, w.gamma, w.V), "cuda")
    got = spv.spv_verify_greedy(w.target, w.tokens, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(_np(w.target), _np(w.tokens))
    assert np.array_equal(_np(got["accept_count"]), ref["accept_count"])
    assert np.array_equal(_np(got["out_tokens"]), ref["out_tokens"])
    assert np.array_equal(_np(got["row_status"]), ref["status"])
    k = ref["accept_count"]
    assert (k == 0).any() and (k > 0).any()  # both a mismatch and an accepted draft token occur


def test_fanout_config(spv):
    fw = workloads.fanout(device="cuda")
    sizes = spv.fanout_sizes(8, 0.8, 0.5, 4, fw.draft.shape[2])
    assert sizes == fw.fanout == [8, 7, 6, 5, 4]
    got = spv.spv_fanout_topk(fw.draft, fw.exclude, fw.fanout)
    torch.cuda.synchronize()
    ref = oracle.fanout_topk(_np(fw.draft), _np(fw.exclude), fw.fanout)
    assert np.array_equal(_np(got["ids"]), ref["ids"])
    assert (_np(got["row_status"]) == 0).all()
    # the excluded draft token never appears among its position's candidates
    ids, ex = _np(got["ids"]), _np(fw.exclude)
    offs = np.concatenate([[0], np.cumsum(fw.fanout)])
    for k in range(4):
        assert not (ids[:, offs[k]:offs[k + 1]] == ex[:, k:k + 1]).any()


@pytest.mark.parametrize("V", [7, 1000, 1025, 8193, 50000])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("levels", [None, 6])
def test_fanout_ties_ragged_and_wide(spv, V, dtype, levels):
    """Top-F over ragged vocabularies, F up to 64 (the unpruned path), heavy
    ties from quantised logits (lowest id first, -0.0 equal to +0.0),
    exclusions and a NaN row."""
    gen = torch.Generator(device="cuda").manual_seed(V + (levels or 0))
    B, K1 = 3, 6
    d = torch.randn(B, K1, V, generator=gen, device="cuda") * 2.0
    if levels:
        d = torch.round(d * levels / 4)
        d[d == 0] = -0.0
    d = d.to(dtype)
    F = [min(f, V - 1) for f in (8, 1, 0, 33, 64, 5)]
    ex = torch.randint(-1, V, (B, K1), generator=gen, device="cuda", dtype=torch.int32)
    got = spv.spv_fanout_topk(d, ex, F)
    torch.cuda.synchronize()
    ref = oracle.fanout_topk(_np(d), _np(ex), F)
    assert np.array_equal(_np(got["ids"]), ref["ids"])
    assert np.array_equal(_np(got["row_status"]), ref["status"])
    d2 = d.clone()
    d2[1, 3, V // 2] = float("nan")
    got = spv.spv_fanout_topk(d2, ex, F)
    torch.cuda.synchronize()
    ref = oracle.fanout_topk(_np(d2), _np(ex), F)
    assert np.array_equal(_np(got["ids"]), ref["ids"])
    assert np.array_equal(_np(got["row_status"]), ref["status"])
    assert ref["status"][1, 3] == 4


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B", [1, 8, 64, 128, 256])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_sweep(spv, B, dtype, T):
    w = workloads.sweep(B=B, dtype=dtype, device="cuda", temperature=T)
    check_chain(spv, w)


# ----------------------------------------------------------------- edge cases
def _random_case(B, g, V, dtype, T, seed, dev="cuda", z_std=2.0, noise=1.0):
    return workloads.chain_from_params(f"edge_B{B}_g{g}_V{V}", B, g, V, dtype, T, z_std, 1.0, noise, 0,
                                       (seed, seed + 1, seed + 2, seed + 3), dev)


@pytest.mark.parametrize("V", [2, 7, 1000, 1001, 1024, 1025, 8191, 8192, 8193, 20000])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_vocab(spv, V, dtype):
    for T in (1.0, 0.0):
        w = _random_case(24, 3, V, dtype, T, 500 + V)
        check_chain(spv, w, want_Z=T > 0)


def test_max_gamma_and_temperature(spv):
    w = _random_case(16, 32, 3000, torch.float32, 0.7, 901, noise=0.3)
    check_chain(spv, w, want_Z=True)
    w = _random_case(16, 32, 3000, torch.bfloat16, 0.0, 902)
    check_chain(spv, w)


def test_unaligned_rows_use_plain_loads(spv):
    """Rows not 16-byte aligned (a view at an odd offset) take the non-TMA path."""
    w = _random_case(8, 2, 4000, torch.float32, 1.0, 777)
    flat = torch.empty(w.target.numel() + 1, dtype=torch.float32, device="cuda")
    flat[1:] = w.target.reshape(-1)
    t_off = flat[1:].view(w.target.shape)
    assert t_off.data_ptr() % 16 != 0
    w2 = workloads.ChainInputs(w.name, t_off, w.draft, w.tokens, w.r, w.keys, 1.0, w.meta)
    check_chain(spv, w2, want_Z=True)


def test_bad_rows(spv):
    w = _random_case(6, 2, 3000, torch.float32, 1.0, 31)
    t, d, tok = w.target.clone(), w.draft.clone(), w.tokens.clone()
    t[0, 1, 5] = float("nan")
    d[1, 0, 7] = float("inf")
    t[2, 2, :] = float("-inf")
    tok[3, 1] = 3000
    t[4, 0, 11] = float("-inf")   # allowed: probability 0
    w2 = workloads.ChainInputs(w.name, t, d, tok, w.r, w.keys, 1.0, w.meta)
    got, ref = check_chain(spv, w2, want_Z=True, expect_bad=[0, 1, 2, 3])
    assert (_np(got["accept_count"])[:4] == -1).all()
    assert (_np(got["out_tokens"])[:4] == -1).all()
    wg = workloads.ChainInputs(w.name, t, d, tok, w.r, w.keys, 0.0, w.meta)
    check_chain(spv, wg, expect_bad=[0, 2, 3])


def test_greedy_ties(spv):
    """Quantised logits: many exact ties, lowest id wins; -0.0 ties +0.0."""
    gen = torch.Generator(device="cuda").manual_seed(5)
    B, g, V = 32, 4, 5000
    z = torch.randint(-3, 3, (B, g + 1, V), generator=gen, device="cuda").float()
    z[z == 0] = -0.0
    a = z.argmax(dim=2)
    tok = a[:, :g].to(torch.int32).clone()
    tok[::3, 1] = 0
    for dtype in (torch.float32, torch.bfloat16):
        w = workloads.ChainInputs("ties", z.to(dtype), z[:, :g].to(dtype), tok, None, None, 0.0)
        check_chain(spv, w)


def test_residual_fallback_path(spv):
    """q nearly equal to p with a forced rejection: the 64 rejection trials
    mostly fail and the direct residual race decides."""
    gen = torch.Generator(device="cpu").manual_seed(8)
    B, V = 48, 2500
    z1 = torch.randn(V, generator=gen) * 1.0
    d1 = z1.clone()
    hot = torch.randperm(V, generator=gen)[:6]
    d1[hot[:3]] += 0.05
    d1[hot[3:]] -= 0.05
    p, q = torch.softmax(z1.double(), 0), torch.softmax(d1.double(), 0)
    x_rej = int(torch.argmax(q - p))
    t = torch.stack([z1, z1]).expand(B, 2, V).contiguous()
    d = d1.expand(B, 1, V).contiguous()
    tok = torch.full((B, 1), x_rej, dtype=torch.int32)
    r = torch.ones(B, 1)
    keys = torch.randint(-(2 ** 62), 2 ** 62, (B,), generator=gen, dtype=torch.int64)
    w = workloads.ChainInputs("fallback", t.cuda(), d.cuda(), tok.cuda(), r.cuda(), keys.cuda(), 1.0)
    got, ref = check_chain(spv, w, want_Z=True, z_atol=Z_ATOL_ILL_CONDITIONED)
    assert (ref["trials"] == oracle.MAX_TRIALS + 1).sum() > B // 2
    assert (ref["accept_count"] == 0).all()


def test_repeat_calls_reuse_workspace(spv):
    """The same workspace serves consecutive calls with identical results."""
    w = _random_case(40, 4, 30000, torch.bfloat16, 1.0, 44)
    ws = spv.new_workspace(spv.spv_chain_workspace_bytes(40, 4, 30000), "cuda")
    outs = [spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o["out_tokens"], outs[0]["out_tokens"])
        assert torch.equal(o["pq"], outs[0]["pq"])
    assert spv.spv_workspace_status(ws) == spv.SPV_OK


def test_work_item_counter_returns_to_zero(spv):
    """The streaming pass hands its later work items out through a counter in
    the workspace header (bytes 8..15); every call leaves it at zero, so one
    workspace serves calls of different kinds and shapes in any order, each
    matching a call on a fresh workspace."""
    w = _random_case(24, 4, 70000, torch.float32, 1.0, 45)
    wg = _random_case(9, 3, 100000, torch.bfloat16, 0.0, 46)
    fw = workloads.fanout(device="cuda", B=2, V=50000)
    n = max(spv.spv_chain_workspace_bytes(24, 4, 70000), spv.spv_greedy_workspace_bytes(9, 3, 100000),
            spv.spv_fanout_workspace_bytes(2, 4, 50000, 8), spv.spv_filtered_workspace_bytes(24, 4, 70000))
    ws = spv.new_workspace(n, "cuda")
    calls = [
        lambda ws: spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, workspace=ws),
        lambda ws: spv.spv_verify_chain(wg.target, wg.draft, wg.tokens, wg.r, wg.keys, 0.0, workspace=ws),
        lambda ws: spv.spv_fanout_topk(fw.draft, fw.exclude, fw.fanout, workspace=ws),
        lambda ws: spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, 50, 0.9,
                                                 workspace=ws),
    ]
    for call in calls + calls[::-1]:
        got = call(ws)
        torch.cuda.synchronize()
        assert int(ws[8:16].count_nonzero()) == 0
        ref = call(spv.new_workspace(n, "cuda"))
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), k
    assert spv.spv_workspace_status(ws) == spv.SPV_OK


def test_invalid_arguments_raise(spv):
    w = _random_case(2, 2, 100, torch.float32, 1.0, 3)
    with pytest.raises(spv.SpvError):
        spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, -1.0)
    with pytest.raises(spv.SpvError):
        spv.spv_fanout_topk(w.draft, torch.zeros(2, 2, dtype=torch.int32, device="cuda"), [1, 100])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_residual_mass_is_a_bad_row(spv, dtype):
    """A draft token with p = q = 0 is rejected and, with p = q elsewhere, the
    residual has no mass: every trial fails, the direct draw finds no block
    with mass, and the sequence is reported as a bad row (as by the oracle)."""
    gen = torch.Generator(device="cpu").manual_seed(11)
    V = 5000
    zl = torch.randn(V, generator=gen)
    zl[7] = float("-inf")
    B, g = 3, 2
    tgt = zl.repeat(B, g + 1, 1).to(dtype)
    drf = zl.repeat(B, g, 1).to(dtype)
    tok = torch.tensor([[7, 3], [3, 7], [3, 4]], dtype=torch.int32)
    r = torch.full((B, g), 0.5)   # p = q: accepted with margin 0.5
    keys = torch.tensor([5, 6, 7], dtype=torch.int64)
    w = workloads.ChainInputs("zero_resid", tgt, drf, tok, r, keys, 1.0, {})
    w = _to(w, "cuda")
    got, ref = check_chain(spv, w, want_Z=True, expect_bad=[0, 1])
    assert list(_np(got["accept_count"])) == [-1, -1, 2]


@pytest.mark.parametrize("V", [1032, 5000, 1001])
def test_greedy_bf16_edges(spv, V):
    """Greedy on bf16 rows (packed max with NaN propagation, then the first id
    holding it): a maximum of zero reached by -0.0 before +0.0, NaN, +inf, an
    all -inf row, a single finite logit, the maximum in the ragged tail, and
    the maximum tied across blocks.  V = 1001 takes the plain-load path."""
    gen = torch.Generator(device="cpu").manual_seed(61 + V)
    B, g = 8, 2
    z = torch.randint(-3, 3, (B, g + 1, V), generator=gen).float()
    z[0] = -torch.randint(0, 3, (g + 1, V), generator=gen).float()   # max 0
    z[0, :, 3] = -0.0
    z[0, :, 9] = 0.0
    z[1, 1, V // 2] = float("nan")
    z[2, 0, 17] = float("inf")
    z[3, 2] = float("-inf")
    z[4] = float("-inf")
    z[4, :, V - 5] = -1.0
    z[5, :, V - 1] = 9.0
    z[6, :, 40] = 7.0
    z[6, :, min(V - 1, 3 * 1024 + 5)] = 7.0
    a = z.nan_to_num(nan=0.0).argmax(dim=2)
    tok = a[:, :g].to(torch.int32).clone()
    w = workloads.ChainInputs("bf16_edges", z.to(torch.bfloat16).cuda(), z[:, :g].to(torch.bfloat16).cuda(),
                              tok.cuda(), None, None, 0.0)
    got, ref = check_chain(spv, w, expect_bad=[1, 2, 3])
    ok = ref["status"] == 0
    assert (ref["accept_count"][ok] == g).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_statistics_not_staged(spv, dtype):
    """gamma = 32 at V = 151,936: 33 target rows x 149 blocks exceed the
    finalize's shared-memory staging of block statistics, so the draws read
    them from the workspace (the other path of the block race)."""
    w = _random_case(3, 32, 151936, dtype, 1.0, 4242, noise=0.4)
    check_chain(spv, w, want_Z=True)
