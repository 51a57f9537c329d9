"""Failure detection on the GPU without a fault: the library's bounded wait
is run on a flag that nothing sets (spv_selftest_timeout); it must give up,
report SPV_ERR_TIMEOUT through the workspace's error word, and leave the
CUDA context usable for the next verify call."""
import pytest
import torch

from speculative_decoding_token_spv_gb300 import workloads
from test_gpu_parity import _to, check_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def test_bounded_wait_gives_up_and_reports(spv):
    ws = spv.new_workspace(4096, "cuda")
    assert spv.spv_workspace_status(ws) == spv.SPV_OK
    spv.spv_selftest_timeout(ws, polls=20000)
    torch.cuda.synchronize()
    assert spv.spv_workspace_status(ws) == spv.SPV_ERR_TIMEOUT
    # the error word is sticky until the workspace is zero-filled again
    assert spv.spv_workspace_status(ws) == spv.SPV_ERR_TIMEOUT
    ws.zero_()
    assert spv.spv_workspace_status(ws) == spv.SPV_OK


def test_context_usable_after_timeout(spv):
    ws = spv.new_workspace(4096, "cuda")
    spv.spv_selftest_timeout(ws, polls=5000)
    torch.cuda.synchronize()
    assert spv.spv_workspace_status(ws) == spv.SPV_ERR_TIMEOUT
    for T in (1.0, 0.0):
        check_chain(spv, _to(workloads.tiny(device="cpu", temperature=T), "cuda"))


def test_timeout_is_reported_in_row_status(spv):
    """A verify call on a workspace whose error word records a wait that gave
    up reports every sequence as SPV_ERR_TIMEOUT (accept_count and out_tokens
    -1) at T = 1 and T = 0; once the workspace is zero-filled the same call
    matches the oracle again."""
    w = _to(workloads.tiny(device="cpu", temperature=1.0), "cuda")
    ws = spv.new_workspace(spv.spv_chain_workspace_bytes(w.B, w.gamma, w.V), "cuda")
    for T in (1.0, 0.0):
        spv.spv_selftest_timeout(ws, polls=2000)
        torch.cuda.synchronize()
        assert spv.spv_workspace_status(ws) == spv.SPV_ERR_TIMEOUT
        out = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, T, workspace=ws)
        torch.cuda.synchronize()
        assert (out["row_status"] == spv.SPV_ERR_TIMEOUT).all()
        assert (out["accept_count"] == -1).all()
        assert (out["out_tokens"] == -1).all()
        ws.zero_()
        check_chain(spv, _to(workloads.tiny(device="cpu", temperature=T), "cuda"))


def test_invalid_arguments(spv):
    ws = spv.new_workspace(4096, "cuda")
    for polls in (0, (1 << 24) + 1):
        with pytest.raises(spv.SpvError):
            spv.spv_selftest_timeout(ws, polls=polls)
