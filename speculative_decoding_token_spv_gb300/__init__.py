"""Speculative-sampling verify step on GB300: Python binding of libspv.

Thin ctypes marshalling over the C ABI in ``include/spv.h`` -- the functions
keep the C names.  Tensors are torch CUDA tensors (contiguous, row-major);
outputs and the zero-filled workspace are allocated with torch when the caller
does not pass them.  Every step of the verify step runs in libspv's kernels on
the tensors' device, on torch's current CUDA stream (or ``stream``).  There is
no CPU fallback: calls fail loudly if libspv.so is missing or the tensors are
not on a CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspv.so")

SPV_OK, SPV_ERR_INVALID_ARG, SPV_ERR_CUDA, SPV_ERR_UNSUPPORTED, SPV_ERR_BAD_ROW, SPV_ERR_TIMEOUT = range(6)
SPV_F32, SPV_BF16 = 0, 1
SPV_MAX_GAMMA = 32
SPV_MAX_FANOUT = 64
SPV_MAX_FANOUT_ROWS = 64
SPV_SAMPLER_BLOCK = 1024
SPV_SAMPLER_SUB = 32
SPV_MAX_TRIALS = 64
SPV_MAX_TOP_K = 64
SPV_MAX_TREE_NODES = 64
SPV_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024

_lib = None


class SpvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {spv_status_string(status)} ({status})")
        self.status = status


def load_library():
    """Load libspv.so (built by ``speculative_decoding_token_spv_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libspv.so not found at {LIB_PATH}: run speculative_decoding_token_spv_gb300.build "
                           "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.spv_verify_chain.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, P, P, P, P, P, P, S, P]
    lib.spv_verify_chain.restype = I
    lib.spv_verify_chain_cached.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, P, P, P, P, P, P, P, P, P,
                                            S, P]
    lib.spv_verify_chain_cached.restype = I
    lib.spv_verify_chain_saguaro.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, P, P, ctypes.c_float, P, P,
                                             P, P, P, P, P, S, P]
    lib.spv_verify_chain_saguaro.restype = I
    lib.spv_verify_tree.argtypes = [P, P, I, P, P, P, P, I, I, I, ctypes.c_float, P, P, P, P, P, S, P]
    lib.spv_verify_tree.restype = I
    lib.spv_tree_workspace_bytes.argtypes = [I, I, I]
    lib.spv_tree_workspace_bytes.restype = S
    lib.spv_verify_chain_filtered.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, I, ctypes.c_float, P, P, P,
                                              P, P, P, S, P]
    lib.spv_verify_chain_filtered.restype = I
    lib.spv_filtered_workspace_bytes.argtypes = [I, I, I]
    lib.spv_filtered_workspace_bytes.restype = S
    lib.spv_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, P, S, P]
    lib.spv_verify_greedy.restype = I
    lib.spv_fanout_topk.argtypes = [P, I, P, P, I, I, I, P, P, P, S, P]
    lib.spv_fanout_topk.restype = I
    lib.spv_chain_workspace_bytes.argtypes = [I, I, I]
    lib.spv_chain_workspace_bytes.restype = S
    lib.spv_greedy_workspace_bytes.argtypes = [I, I, I]
    lib.spv_greedy_workspace_bytes.restype = S
    lib.spv_fanout_workspace_bytes.argtypes = [I, I, I, I]
    lib.spv_fanout_workspace_bytes.restype = S
    lib.spv_fanout_size.argtypes = [I, ctypes.c_double, ctypes.c_double, I]
    lib.spv_fanout_size.restype = ctypes.c_double
    lib.spv_fanout_sizes.argtypes = [I, ctypes.c_double, ctypes.c_double, I, I, P]
    lib.spv_fanout_sizes.restype = I
    lib.spv_workspace_status.argtypes = [P, P]
    lib.spv_selftest_timeout.argtypes = [P, S, ctypes.c_uint, P]
    lib.spv_selftest_timeout.restype = I
    lib.spv_workspace_status.restype = I
    lib.spv_status_string.argtypes = [I]
    lib.spv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def spv_status_string(status: int) -> str:
    return load_library().spv_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPV_F32
    if t.dtype == torch.bfloat16:
        return SPV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _cuda(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != SPV_OK:
        raise SpvError(status, what)


def spv_chain_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return load_library().spv_chain_workspace_bytes(B, gamma, V)


def spv_greedy_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return load_library().spv_greedy_workspace_bytes(B, gamma, V)


def spv_fanout_workspace_bytes(B: int, K: int, V: int, max_fanout: int) -> int:
    return load_library().spv_fanout_workspace_bytes(B, K, V, max_fanout)


def spv_fanout_size(F0: int, a: float, r: float, k: int) -> float:
    return load_library().spv_fanout_size(int(F0), float(a), float(r), int(k))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled byte workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def spv_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Device error word of a workspace (synchronises the stream)."""
    return load_library().spv_workspace_status(_ptr(workspace), _stream(stream, workspace.device))


def spv_selftest_timeout(workspace: torch.Tensor, polls: int = 20000, stream=None) -> None:
    """Run the library's bounded wait on a flag nothing sets (see
    spv_selftest_timeout in spv.h): it gives up after `polls` polls and
    records SPV_ERR_TIMEOUT in the workspace's error word."""
    workspace = _cuda(workspace, "workspace")
    st = load_library().spv_selftest_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                             int(polls), _stream(stream, workspace.device))
    _check(st, "spv_selftest_timeout")


def spv_verify_chain(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature: float, *,
                     workspace=None, out=None, want_pq: bool = True, want_resid_norm: bool = False,
                     want_status: bool = True, stream=None) -> dict:
    """Chain verify (T > 0) or greedy (T == 0).  See spv_verify_chain in spv.h.

    target_logits [B, g+1, V] and draft_logits [B, g, V] (fp32 or bf16, same
    dtype), draft_tokens [B, g] int32, r [B, g] float32, sample_keys [B] int64
    holding uint64 bit patterns.  Returns dict(accept_count, out_tokens, and
    pq / resid_norm / row_status when requested)."""
    return _verify_chain(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature, None, None,
                         workspace, out, want_pq, want_resid_norm, want_status, stream)


def spv_verify_chain_cached(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature: float,
                            cache_ids, fanout, *, workspace=None, out=None, want_pq: bool = True,
                            want_resid_norm: bool = False, want_status: bool = True, stream=None) -> dict:
    """spv_verify_chain plus the speculation-cache lookup of the outcome
    (see spv_verify_chain_cached in spv.h).  cache_ids [B, sum F] int32 (the
    k-major candidate lists spv_fanout_topk writes), fanout: gamma+1 ints.
    The result adds cache_slot [B] int32 (-1 = miss)."""
    return _verify_chain(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature, cache_ids,
                         fanout, workspace, out, want_pq, want_resid_norm, want_status, stream)


def spv_verify_chain_saguaro(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature: float,
                             cache_ids, fanout, C: float, *, workspace=None, out=None, want_pq: bool = True,
                             want_resid_norm: bool = False, want_status: bool = True, stream=None) -> dict:
    """Verify of Saguaro-sampled drafts (the draft probability of each
    position's cached candidates divided by C) with the cache lookup; see
    spv_verify_chain_saguaro in spv.h.  Arguments and outputs as
    :func:`spv_verify_chain_cached` plus C."""
    return _verify_chain(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature, cache_ids,
                         fanout, workspace, out, want_pq, want_resid_norm, want_status, stream, sag_C=float(C))


def _verify_chain(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature, cache_ids, fanout,
                  workspace, out, want_pq, want_resid_norm, want_status, stream, sag_C=None) -> dict:
    target_logits = _cuda(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, gamma+1, V]")
    B, g1, V = target_logits.shape
    g = g1 - 1
    greedy = float(temperature) == 0.0
    dt = _dtype_code(target_logits)
    draft_tokens = _cuda(draft_tokens, "draft_tokens", torch.int32)
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    if not greedy:
        draft_logits = _cuda(draft_logits, "draft_logits", target_logits.dtype)
        r = _cuda(r, "r", torch.float32)
        sample_keys = _cuda(sample_keys, "sample_keys", torch.int64)
        if tuple(draft_logits.shape) != (B, g, V) or tuple(r.shape) != (B, g) or tuple(sample_keys.shape) != (B,):
            raise ValueError("draft_logits [B,g,V], r [B,g], sample_keys [B] expected")
    else:
        draft_logits = r = sample_keys = None
    cached = cache_ids is not None
    if cached:
        F = [int(f) for f in fanout]
        cache_ids = _cuda(cache_ids, "cache_ids", torch.int32)
        if len(F) != g + 1 or tuple(cache_ids.shape) != (B, sum(F)):
            raise ValueError("fanout needs gamma+1 entries and cache_ids [B, sum(fanout)]")
    lib = load_library()
    need = lib.spv_chain_workspace_bytes(B, g, V)
    if workspace is None:
        workspace = new_workspace(need, dev)
    out = dict(out) if out else {}
    if "accept_count" not in out:
        out["accept_count"] = torch.empty(B, dtype=torch.int32, device=dev)
    if "out_tokens" not in out:
        out["out_tokens"] = torch.empty(B, g + 1, dtype=torch.int32, device=dev)
    if want_pq and not greedy and "pq" not in out:
        out["pq"] = torch.empty(B, g, 2, dtype=torch.float32, device=dev)
    if want_resid_norm and not greedy and "resid_norm" not in out:
        out["resid_norm"] = torch.empty(B, dtype=torch.float32, device=dev)
    if want_status and "row_status" not in out:
        out["row_status"] = torch.empty(B, dtype=torch.int32, device=dev)
    args = (_ptr(target_logits), _ptr(draft_logits), dt, _ptr(draft_tokens), _ptr(r), _ptr(sample_keys), B, g, V,
            float(temperature), _ptr(out["accept_count"]), _ptr(out["out_tokens"]), _ptr(out.get("pq")),
            _ptr(out.get("resid_norm")), _ptr(out.get("row_status")))
    tail = (_ptr(workspace), workspace.numel(), _stream(stream, dev))
    if cached:
        if "cache_slot" not in out:
            out["cache_slot"] = torch.empty(B, dtype=torch.int32, device=dev)
        f_host = (ctypes.c_int32 * (g + 1))(*F)
        if sag_C is None:
            st = lib.spv_verify_chain_cached(*args, _ptr(cache_ids), ctypes.addressof(f_host),
                                             _ptr(out["cache_slot"]), *tail)
            _check(st, "spv_verify_chain_cached")
        else:
            st = lib.spv_verify_chain_saguaro(*args[:10], _ptr(cache_ids), ctypes.addressof(f_host), sag_C, *args[10:],
                                              _ptr(out["cache_slot"]), *tail)
            _check(st, "spv_verify_chain_saguaro")
    else:
        st = lib.spv_verify_chain(*args, *tail)
        _check(st, "spv_verify_chain")
    return out


def spv_filtered_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return load_library().spv_filtered_workspace_bytes(B, gamma, V)


def spv_verify_chain_filtered(target_logits, draft_logits, draft_tokens, r, sample_keys, temperature: float,
                              top_k: int, top_p: float = 1.0, *, workspace=None, out=None, want_pq: bool = True,
                              want_resid_norm: bool = False, want_status: bool = True, stream=None) -> dict:
    """Chain verify on top-k / top-p filtered target and draft distributions
    (see spv_verify_chain_filtered in spv.h); arguments and outputs as
    :func:`spv_verify_chain`."""
    target_logits = _cuda(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, gamma+1, V]")
    B, g1, V = target_logits.shape
    g = g1 - 1
    greedy = float(temperature) == 0.0
    draft_tokens = _cuda(draft_tokens, "draft_tokens", torch.int32)
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    if not greedy:
        draft_logits = _cuda(draft_logits, "draft_logits", target_logits.dtype)
        r = _cuda(r, "r", torch.float32)
        sample_keys = _cuda(sample_keys, "sample_keys", torch.int64)
        if tuple(draft_logits.shape) != (B, g, V) or tuple(r.shape) != (B, g) or tuple(sample_keys.shape) != (B,):
            raise ValueError("draft_logits [B,g,V], r [B,g], sample_keys [B] expected")
    else:
        draft_logits = r = sample_keys = None
    lib = load_library()
    if workspace is None:
        workspace = new_workspace(lib.spv_filtered_workspace_bytes(B, g, V), dev)
    out = dict(out) if out else {}
    if "accept_count" not in out:
        out["accept_count"] = torch.empty(B, dtype=torch.int32, device=dev)
    if "out_tokens" not in out:
        out["out_tokens"] = torch.empty(B, g + 1, dtype=torch.int32, device=dev)
    if want_pq and not greedy and "pq" not in out:
        out["pq"] = torch.empty(B, g, 2, dtype=torch.float32, device=dev)
    if want_resid_norm and not greedy and "resid_norm" not in out:
        out["resid_norm"] = torch.empty(B, dtype=torch.float32, device=dev)
    if want_status and "row_status" not in out:
        out["row_status"] = torch.empty(B, dtype=torch.int32, device=dev)
    st = lib.spv_verify_chain_filtered(_ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits),
                                       _ptr(draft_tokens), _ptr(r), _ptr(sample_keys), B, g, V, float(temperature),
                                       int(top_k), float(top_p), _ptr(out["accept_count"]), _ptr(out["out_tokens"]),
                                       _ptr(out.get("pq")), _ptr(out.get("resid_norm")), _ptr(out.get("row_status")),
                                       _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "spv_verify_chain_filtered")
    return out


def spv_tree_workspace_bytes(B: int, N: int, V: int) -> int:
    return load_library().spv_tree_workspace_bytes(B, N, V)


def spv_verify_tree(target_logits, draft_logits, parent, tokens, r, sample_keys, temperature: float, *,
                    workspace=None, out=None, want_nodes: bool = True, want_status: bool = True, stream=None) -> dict:
    """Verify of a draft token tree per sequence (see spv_verify_tree in
    spv.h).  target_logits, draft_logits [B, N, V]; parent, tokens [B, N]
    int32; r [B, N] float32; sample_keys [B] int64.  Returns accept_count,
    out_tokens [B, N], out_nodes [B, N] and row_status."""
    target_logits = _cuda(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = target_logits.shape
    greedy = float(temperature) == 0.0
    parent = _cuda(parent, "parent", torch.int32)
    tokens = _cuda(tokens, "tokens", torch.int32)
    if tuple(parent.shape) != (B, N) or tuple(tokens.shape) != (B, N):
        raise ValueError("parent and tokens must be [B, N]")
    if not greedy:
        draft_logits = _cuda(draft_logits, "draft_logits", target_logits.dtype)
        r = _cuda(r, "r", torch.float32)
        sample_keys = _cuda(sample_keys, "sample_keys", torch.int64)
        if tuple(draft_logits.shape) != (B, N, V) or tuple(r.shape) != (B, N) or tuple(sample_keys.shape) != (B,):
            raise ValueError("draft_logits [B,N,V], r [B,N], sample_keys [B] expected")
    else:
        draft_logits = r = sample_keys = None
    lib = load_library()
    if workspace is None:
        workspace = new_workspace(lib.spv_tree_workspace_bytes(B, N, V), dev)
    out = dict(out) if out else {}
    if "accept_count" not in out:
        out["accept_count"] = torch.empty(B, dtype=torch.int32, device=dev)
    if "out_tokens" not in out:
        out["out_tokens"] = torch.empty(B, N, dtype=torch.int32, device=dev)
    if want_nodes and "out_nodes" not in out:
        out["out_nodes"] = torch.empty(B, N, dtype=torch.int32, device=dev)
    if want_status and "row_status" not in out:
        out["row_status"] = torch.empty(B, dtype=torch.int32, device=dev)
    st = lib.spv_verify_tree(_ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(parent),
                             _ptr(tokens), _ptr(r), _ptr(sample_keys), B, N, V, float(temperature),
                             _ptr(out["accept_count"]), _ptr(out["out_tokens"]), _ptr(out.get("out_nodes")),
                             _ptr(out.get("row_status")), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "spv_verify_tree")
    return out


def spv_verify_greedy(target_logits, draft_tokens, *, workspace=None, out=None, want_status: bool = True,
                      stream=None) -> dict:
    """Greedy (T = 0) verify: argmax agreement.  target_logits [B, g+1, V]."""
    target_logits = _cuda(target_logits, "target_logits")
    dev = target_logits.device
    B, g1, V = target_logits.shape
    g = g1 - 1
    draft_tokens = _cuda(draft_tokens, "draft_tokens", torch.int32)
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    lib = load_library()
    if workspace is None:
        workspace = new_workspace(lib.spv_greedy_workspace_bytes(B, g, V), dev)
    out = dict(out) if out else {}
    if "accept_count" not in out:
        out["accept_count"] = torch.empty(B, dtype=torch.int32, device=dev)
    if "out_tokens" not in out:
        out["out_tokens"] = torch.empty(B, g + 1, dtype=torch.int32, device=dev)
    if want_status and "row_status" not in out:
        out["row_status"] = torch.empty(B, dtype=torch.int32, device=dev)
    st = lib.spv_verify_greedy(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), B, g, V,
                               _ptr(out["accept_count"]), _ptr(out["out_tokens"]), _ptr(out.get("row_status")),
                               _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "spv_verify_greedy")
    return out


def spv_fanout_topk(draft_logits, exclude, fanout, *, workspace=None, out=None, want_status: bool = True,
                    stream=None) -> dict:
    """Top-F_k ids per (b, k) of draft_logits [B, K+1, V], skipping exclude[b, k]."""
    draft_logits = _cuda(draft_logits, "draft_logits")
    dev = draft_logits.device
    B, K1, V = draft_logits.shape
    exclude = _cuda(exclude, "exclude", torch.int32)
    F = [int(f) for f in fanout]
    if len(F) != K1 or tuple(exclude.shape) != (B, K1):
        raise ValueError("fanout needs K+1 entries and exclude [B, K+1]")
    lib = load_library()
    Fmax = max(F) if F else 0
    if workspace is None:
        workspace = new_workspace(lib.spv_fanout_workspace_bytes(B, K1 - 1, V, Fmax), dev)
    out = dict(out) if out else {}
    if "ids" not in out:
        out["ids"] = torch.empty(B, sum(F), dtype=torch.int32, device=dev)
    if want_status and "row_status" not in out:
        out["row_status"] = torch.empty(B, K1, dtype=torch.int32, device=dev)
    f_host = (ctypes.c_int32 * max(K1, 1))(*F)
    st = lib.spv_fanout_topk(_ptr(draft_logits), _dtype_code(draft_logits), _ptr(exclude),
                             ctypes.addressof(f_host), B, K1 - 1, V, _ptr(out["ids"]),
                             _ptr(out.get("row_status")), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st, "spv_fanout_topk")
    return out


def spv_fanout_sizes(F0: int, a: float, r: float, K: int, V: int) -> list:
    """F_k for k = 0..K from the C library (rounded half away from zero,
    clamped to [0, V-1])."""
    out = (ctypes.c_int32 * (max(int(K), 0) + 1))()
    _check(load_library().spv_fanout_sizes(int(F0), float(a), float(r), int(K), int(V), ctypes.addressof(out)),
           "spv_fanout_sizes")
    return list(out)


fanout_sizes = spv_fanout_sizes
