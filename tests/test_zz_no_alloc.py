"""spv_verify_chain_noalloc: the entry point for callers that cannot allocate
device memory (their memory is pre-reserved by their own pool, they manage no
device memory, or cudaMalloc is not allowed or would stall where they call).

Called through the C ABI with ctypes; its outputs must equal those of
spv_verify_chain (which takes a caller workspace) on the same inputs, on two
calls in a row -- the second call reuses the library's scratch array with the
first call's contents still in it.  Collected last, so a run that stops at
the first failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_token_spv_gb300 import workloads

pytestmark = pytest.mark.gpu

RTOL = 1e-5  # the tolerance the parity tests use for p_i(x_i), q_i(x_i)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as spv
    L = spv.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    L.spv_verify_chain_noalloc.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, P, P, P, P, P, P]
    L.spv_verify_chain_noalloc.restype = I
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(L, w):
    B, g = w.B, w.gamma
    dev = w.target.device
    out = dict(accept_count=torch.full((B,), -7, dtype=torch.int32, device=dev),
               out_tokens=torch.full((B, g + 1), -7, dtype=torch.int32, device=dev),
               pq=torch.full((B, g, 2), -7.0, device=dev),
               row_status=torch.full((B,), -7, dtype=torch.int32, device=dev))
    dt = 0 if w.target.dtype == torch.float32 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.spv_verify_chain_noalloc(_p(w.target), _p(w.draft), dt, _p(w.tokens), _p(w.r), _p(w.keys), B, g, w.V,
                                    ctypes.c_float(w.temperature), _p(out["accept_count"]), _p(out["out_tokens"]),
                                    _p(out["pq"]) if w.temperature > 0 else None, None, _p(out["row_status"]),
                                    stream)
    assert st == 0, f"spv_verify_chain_noalloc returned {st}"
    return out


@pytest.mark.parametrize("case", ["sweep_B64_fp32_T1", "tiny_T1", "spd_T0"])
def test_noalloc_matches_workspace_entry_point(lib, case):
    import speculative_decoding_token_spv_gb300 as spv
    if case == "sweep_B64_fp32_T1":
        w = workloads.sweep(B=64, dtype=torch.float32, device="cuda", temperature=1.0)
    elif case == "tiny_T1":
        w = workloads.tiny(device="cuda", temperature=1.0)
    else:
        w = workloads.spd(device="cuda", temperature=0.0)
    ref = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share the scratch array
        got = _noalloc(lib, w)
        torch.cuda.synchronize()
        assert torch.equal(got["accept_count"], ref["accept_count"])
        assert torch.equal(got["out_tokens"], ref["out_tokens"])
        assert torch.equal(got["row_status"], ref["row_status"])
        if w.temperature > 0:
            np.testing.assert_allclose(got["pq"].cpu().numpy(), ref["pq"].cpu().numpy(), rtol=RTOL)


def test_noalloc_starts_from_a_clear_header(lib):
    """A work-item counter left nonzero in the scratch array (what a call that
    failed between its two launches leaves) changes nothing: every call clears
    the array's header before its kernels run."""
    import speculative_decoding_token_spv_gb300 as spv
    lib.spv_internal_noalloc_set_item_counter.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    lib.spv_internal_noalloc_set_item_counter.restype = ctypes.c_int
    w = workloads.sweep(B=64, dtype=torch.float32, device="cuda", temperature=1.0)
    ref = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for planted in (1000, 1 << 40):
        assert lib.spv_internal_noalloc_set_item_counter(planted, stream) == 0
        got = _noalloc(lib, w)
        torch.cuda.synchronize()
        assert torch.equal(got["accept_count"], ref["accept_count"])
        assert torch.equal(got["out_tokens"], ref["out_tokens"])
        assert torch.equal(got["row_status"], ref["row_status"])
        np.testing.assert_allclose(got["pq"].cpu().numpy(), ref["pq"].cpu().numpy(), rtol=RTOL)


def test_noalloc_greedy_uses_the_greedy_scratch_bound(lib):
    """At T = 0 the call needs only the greedy layout: B = 600, gamma = 4,
    V = 151,936 fits the array at T = 0 (about 3.6 MB) although the chain
    layout would not, and matches spv_verify_greedy."""
    import speculative_decoding_token_spv_gb300 as spv
    B, g, V = 600, 4, 151936
    assert spv.spv_greedy_workspace_bytes(B, g, V) <= spv.SPV_NOALLOC_SCRATCH_BYTES
    assert spv.spv_chain_workspace_bytes(B, g, V) > spv.SPV_NOALLOC_SCRATCH_BYTES
    w = workloads.sweep(B=B, dtype=torch.bfloat16, device="cuda", temperature=0.0)
    ref = spv.spv_verify_greedy(w.target, w.tokens)
    torch.cuda.synchronize()
    got = _noalloc(lib, w)
    torch.cuda.synchronize()
    assert torch.equal(got["accept_count"], ref["accept_count"])
    assert torch.equal(got["out_tokens"], ref["out_tokens"])
    assert torch.equal(got["row_status"], ref["row_status"])
