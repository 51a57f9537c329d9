"""Oracle for the speculative-sampling verify step -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper over ``spv_oracle.c``: a plain, slow, double-precision CPU
restatement of the verify step (accept/reject, first-rejection stop, residual
resample, bonus token), the greedy argmax case and the top-F_k fan-out.  Only
the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use
it; the CUDA library never imports or calls it.

Inputs are numpy arrays.  Logits are passed as float32 (bf16 values convert to
float32 exactly), the oracle widens them to float64 itself.  Sequences are
independent, so a thread pool runs them in parallel (ctypes releases the GIL
around each call); the arithmetic of each sequence is the single-threaded C.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spv_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_spv.so")

BLOCK = 1024          # tokens per sampler block (must equal the C constant)
SUB = 32              # tokens per sampler sub-block
MAX_TRIALS = 64       # residual rejection trials before the direct fallback
(STREAM_BLOCK, STREAM_SUB, STREAM_TOKEN, STREAM_ACCEPT,
 STREAM_FB_BLOCK, STREAM_FB_SUB, STREAM_FB_TOKEN) = 1, 2, 3, 4, 5, 6, 7
OK, BAD_ROW = 0, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle_spv.so`` (gcc, -O2)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.spvo_philox4x32_10.argtypes = [P, P, P]
        lib.spvo_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                     ctypes.c_uint64]
        lib.spvo_uniform.restype = ctypes.c_double
        lib.spvo_softmax_stats.argtypes = [P, ctypes.c_int, ctypes.c_double, P, P]
        lib.spvo_verify_chain_seq.argtypes = [P, P, P, P, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, P, P, P, P, P, P]
        lib.spvo_verify_greedy_seq.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
        lib.spvo_fanout_row.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
        lib.spvo_fanout_size.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int]
        lib.spvo_fanout_size.restype = ctypes.c_double
        lib.spvo_cache_slot.argtypes = [ctypes.c_int, ctypes.c_int32, P, P, ctypes.c_int]
        lib.spvo_cache_slot.restype = ctypes.c_int
        lib.spvo_verify_chain_batch.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, P, P, P, P, P, P, P]
        lib.spvo_filter_row.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double, P, P, P]
        lib.spvo_filter_row.restype = ctypes.c_int
        lib.spvo_verify_filtered_batch.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double,
                                                   P, P, P, P, P, P]
        lib.spvo_verify_saguaro_batch.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_double, P, P, ctypes.c_int, ctypes.c_double,
                                                  P, P, P, P, P, P, P]
        lib.spvo_verify_tree_batch.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_double, P, P, P, P, P, P]
        lib.spvo_verify_greedy_batch.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 P, P, P]
        lib.spvo_set_uniform_override.argtypes = [P]
        lib.spvo_set_uniform_override.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _threads(threads):
    return threads or len(os.sched_getaffinity(0))


# ---------------------------------------------------------------- primitives
def philox4x32_10(counter, key) -> np.ndarray:
    """One Philox4x32-10 block: 4 uint32 words for a 4-word counter, 2-word key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().spvo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seq_key: int, stream: int, trial: int, pos: int, n: int) -> float:
    """The (0,1] uniform both sides derive for draw n of (stream, trial, pos)."""
    return _load().spvo_uniform(seq_key, stream, trial, pos, n)


UNIFORM_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                              ctypes.c_uint64)


@contextlib.contextmanager
def uniform_override(fn):
    """Within the block, every uniform the oracle's draws consume is
    ``fn(seq_key, stream, trial, pos, n)`` (a float in (0, 1]) instead of the
    Philox value -- for tests that enumerate a draw's variates on a grid or
    build a decision with a known margin.  Use with ``threads=1``."""
    lib = _load()
    cb = UNIFORM_FN(fn)
    lib.spvo_set_uniform_override(ctypes.cast(cb, ctypes.c_void_p))
    try:
        yield
    finally:
        lib.spvo_set_uniform_override(None)


def softmax_stats(z, T: float):
    """(M, S) of softmax(z / T) for one row, or None for a bad row."""
    z = _f32(z)
    M = np.zeros(1)
    S = np.zeros(1)
    st = _load().spvo_softmax_stats(_ptr(z), z.size, float(T), _ptr(M), _ptr(S))
    return None if st != OK else (float(M[0]), float(S[0]))


# ---------------------------------------------------------------- verify step
def verify_chain(target, draft, tokens, r, keys, temperature: float, want_Z: bool = False,
                 threads: int | None = None) -> dict:
    """Chain verify for B sequences (T > 0); T == 0 routes to :func:`verify_greedy`.

    target [B, g+1, V], draft [B, g, V] float32; tokens [B, g] int32; r [B, g]
    float32 in (0,1]; keys [B] uint64.  Returns a dict of numpy arrays:
    accept_count [B], out_tokens [B, g+1], pq [B, g, 2], Z [B] (if want_Z),
    margin [B], trials [B], status [B].
    """
    if temperature == 0:
        return verify_greedy(target, tokens, threads=threads)
    target, draft = _f32(target), _f32(draft)
    B, g1, V = target.shape
    g = g1 - 1
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).reshape(B, g)
    r = _f32(r).reshape(B, g)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64)).reshape(B)
    out = dict(accept_count=np.zeros(B, np.int32), out_tokens=np.zeros((B, g + 1), np.int32),
               pq=np.zeros((B, g, 2)), margin=np.zeros(B), trials=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    Z = np.zeros(B) if want_Z else None
    lib = _load()

    def run(b0, b1):
        lib.spvo_verify_chain_batch(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(r), _ptr(keys), b0, b1, g, V,
                                    float(temperature), _ptr(out["accept_count"]), _ptr(out["out_tokens"]),
                                    _ptr(out["pq"]), _ptr(Z) if want_Z else None, _ptr(out["margin"]),
                                    _ptr(out["trials"]), _ptr(out["status"]))

    _run_ranges(run, B, threads)
    if want_Z:
        out["Z"] = Z
    return out


MAX_TOP_K = 64
STREAM_FILTERED = 8


def filter_row(z, temperature: float, top_k: int, top_p: float = 1.0):
    """Top-k / top-p filter of one row: (ids, probs) of the kept ids in rank
    order (logit descending, ties to the lower id), probs renormalised; None
    for a bad row.  Also returns the top-p cut margin."""
    z = _f32(z).reshape(-1)
    if not 1 <= top_k <= MAX_TOP_K:
        raise ValueError("top_k out of range")
    K = min(top_k, z.size)
    ids = np.zeros(K, np.int32)
    probs = np.zeros(K)
    margin = np.full(1, np.inf)
    n = _load().spvo_filter_row(_ptr(z), z.size, float(temperature), int(top_k), float(top_p), _ptr(ids),
                                _ptr(probs), _ptr(margin))
    if n < 0:
        return None
    return ids[:n].copy(), probs[:n].copy(), float(margin[0])


def verify_filtered(target, draft, tokens, r, keys, temperature: float, top_k: int, top_p: float = 1.0,
                    want_Z: bool = False, threads: int | None = None) -> dict:
    """Chain verify on top-k / top-p filtered target and draft distributions
    (T > 0; T == 0 routes to :func:`verify_greedy`, which no top-k filter
    changes).  Arguments and outputs as :func:`verify_chain` (no trials)."""
    if temperature == 0:
        return verify_greedy(target, tokens, threads=threads)
    if not 1 <= top_k <= MAX_TOP_K or not 0.0 < top_p <= 1.0:
        raise ValueError("top_k in [1, 64] and top_p in (0, 1] expected")
    target, draft = _f32(target), _f32(draft)
    B, g1, V = target.shape
    g = g1 - 1
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).reshape(B, g)
    r = _f32(r).reshape(B, g)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64)).reshape(B)
    out = dict(accept_count=np.zeros(B, np.int32), out_tokens=np.zeros((B, g + 1), np.int32),
               pq=np.zeros((B, g, 2)), margin=np.zeros(B), status=np.zeros(B, np.int32))
    Z = np.zeros(B) if want_Z else None
    lib = _load()

    def run(b0, b1):
        lib.spvo_verify_filtered_batch(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(r), _ptr(keys), b0, b1, g, V,
                                       float(temperature), int(top_k), float(top_p), _ptr(out["accept_count"]),
                                       _ptr(out["out_tokens"]), _ptr(out["pq"]), _ptr(Z) if want_Z else None,
                                       _ptr(out["margin"]), _ptr(out["status"]))

    _run_ranges(run, B, threads)
    if want_Z:
        out["Z"] = Z
    return out


def verify_saguaro(target, draft, tokens, r, keys, temperature: float, cache_ids, fanout, C: float,
                   want_Z: bool = False, threads: int | None = None) -> dict:
    """Chain verify against Saguaro-sampled drafts: the draft distribution
    at position i divides the probability of that position's cached
    candidates (cache_ids [B, sum F], k-major, fanout: gamma+1 ints; the
    first gamma positions are used) by C and renormalises.  T == 0 routes to
    :func:`verify_greedy` (the argmax rule ignores the draft distribution).
    Outputs as :func:`verify_chain`."""
    if temperature == 0:
        return verify_greedy(target, tokens, threads=threads)
    target, draft = _f32(target), _f32(draft)
    B, g1, V = target.shape
    g = g1 - 1
    F = np.ascontiguousarray(np.asarray(fanout, dtype=np.int32))
    if F.shape[0] != g + 1:
        raise ValueError("fanout needs gamma+1 entries")
    sumF = int(F.sum())
    ids = np.ascontiguousarray(np.asarray(cache_ids, dtype=np.int32).reshape(B, sumF))
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).reshape(B, g)
    r = _f32(r).reshape(B, g)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64)).reshape(B)
    out = dict(accept_count=np.zeros(B, np.int32), out_tokens=np.zeros((B, g + 1), np.int32),
               pq=np.zeros((B, g, 2)), margin=np.zeros(B), trials=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    Z = np.zeros(B) if want_Z else None
    lib = _load()

    def run(b0, b1):
        lib.spvo_verify_saguaro_batch(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(r), _ptr(keys), b0, b1, g, V,
                                      float(temperature), _ptr(ids), _ptr(F), sumF, float(C),
                                      _ptr(out["accept_count"]), _ptr(out["out_tokens"]), _ptr(out["pq"]),
                                      _ptr(Z) if want_Z else None, _ptr(out["margin"]), _ptr(out["trials"]),
                                      _ptr(out["status"]))

    _run_ranges(run, B, threads)
    if want_Z:
        out["Z"] = Z
    return out


def verify_tree(target, draft, parent, tokens, r, keys, temperature: float, threads: int | None = None) -> dict:
    """Tree verify (multi-round speculative sampling; greedy at T == 0).
    target, draft [B, N, V] (row v: p, q at node v); parent [B, N] (-1 at the
    root, parent[v] < v); tokens [B, N] (node v's token); r [B, N]; keys [B].
    Returns accept_count [B], out_tokens [B, N], out_nodes [B, N], margin,
    trials, status."""
    target = _f32(target)
    B, N, V = target.shape
    draft = _f32(draft) if temperature > 0 else target
    parent = np.ascontiguousarray(np.asarray(parent, dtype=np.int32)).reshape(B, N)
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).reshape(B, N)
    r = _f32(r).reshape(B, N) if r is not None else np.ones((B, N), np.float32)
    keys = np.ascontiguousarray(np.asarray(keys if keys is not None else np.zeros(B), dtype=np.uint64)).reshape(B)
    out = dict(accept_count=np.zeros(B, np.int32), out_tokens=np.zeros((B, N), np.int32),
               out_nodes=np.zeros((B, N), np.int32), margin=np.zeros(B), trials=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    lib = _load()

    def run(b0, b1):
        lib.spvo_verify_tree_batch(_ptr(target), _ptr(draft), _ptr(parent), _ptr(tokens), _ptr(r), _ptr(keys), b0, b1,
                                   N, V, float(temperature), _ptr(out["accept_count"]), _ptr(out["out_tokens"]),
                                   _ptr(out["out_nodes"]), _ptr(out["margin"]), _ptr(out["trials"]),
                                   _ptr(out["status"]))

    _run_ranges(run, B, threads)
    return out


def verify_greedy(target, tokens, threads: int | None = None) -> dict:
    """Greedy (T = 0) verify: argmax agreement.  target [B, g+1, V]."""
    target = _f32(target)
    B, g1, V = target.shape
    g = g1 - 1
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).reshape(B, g)
    out = dict(accept_count=np.zeros(B, np.int32), out_tokens=np.zeros((B, g + 1), np.int32),
               status=np.zeros(B, np.int32))
    lib = _load()

    def run(b0, b1):
        lib.spvo_verify_greedy_batch(_ptr(target), _ptr(tokens), b0, b1, g, V, _ptr(out["accept_count"]),
                                     _ptr(out["out_tokens"]), _ptr(out["status"]))

    _run_ranges(run, B, threads)
    return out


def fanout_size(F0: int, a: float, r: float, k: int) -> float:
    """F_0 * a^(k/(1+r)) (unrounded)."""
    return _load().spvo_fanout_size(int(F0), float(a), float(r), int(k))


def fanout_sizes(F0: int, a: float, r: float, K: int, V: int) -> list[int]:
    """F_k for k = 0..K, rounded half away from zero and clamped to [0, V-1]."""
    out = []
    for k in range(K + 1):
        f = fanout_size(F0, a, r, k)
        n = int(np.floor(f + 0.5))
        out.append(max(0, min(V - 1, n)))
    return out


def fanout_topk(draft, exclude, fanout, threads: int | None = None) -> dict:
    """Top-F_k ids per (b, k).  draft [B, K+1, V]; exclude [B, K+1] (-1 none);
    fanout: K+1 ints.  Returns ids [B, sum F] (k-major, then rank), status [B, K+1]."""
    draft = _f32(draft)
    B, K1, V = draft.shape
    exclude = np.asarray(exclude, dtype=np.int64).reshape(B, K1)
    F = [int(f) for f in fanout]
    offs = np.concatenate([[0], np.cumsum(F)]).astype(int)
    ids = np.full((B, offs[-1]), -1, np.int32)
    status = np.zeros((B, K1), np.int32)
    lib = _load()

    def one(i):
        b, k = divmod(i, K1)
        o = np.zeros(max(F[k], 1), np.int32)
        st = lib.spvo_fanout_row(_ptr(draft[b, k]), V, int(exclude[b, k]), F[k], _ptr(o))
        ids[b, offs[k]:offs[k + 1]] = o[:F[k]]
        status[b, k] = st

    _run(one, B * K1, threads)
    return dict(ids=ids, status=status)


def cache_slots(accept_count, out_tokens, cache_ids, fanout) -> np.ndarray:
    """Speculation-cache lookup of each sequence's verify outcome (k, t*):
    the index of the entry (position k, token t*) in cache_ids[b] (k-major
    lists of fanout[k] candidates), or -1.  accept_count [B], out_tokens
    [B, gamma+1], cache_ids [B, sum F]; fanout: gamma+1 ints."""
    k = np.asarray(accept_count, dtype=np.int64).reshape(-1)
    toks = np.asarray(out_tokens, dtype=np.int64).reshape(k.shape[0], -1)
    F = np.ascontiguousarray(np.asarray(fanout, dtype=np.int32))
    ids = np.ascontiguousarray(np.asarray(cache_ids, dtype=np.int32).reshape(k.shape[0], int(F.sum())))
    K = F.shape[0] - 1
    lib = _load()
    out = np.full(k.shape[0], -1, np.int32)
    for b in range(k.shape[0]):
        t = int(toks[b, k[b]]) if k[b] >= 0 else -1
        out[b] = lib.spvo_cache_slot(int(k[b]), t, _ptr(ids[b]), _ptr(F), K)
    return out


def _run(fn, n, threads):
    t = min(_threads(threads), n)
    if t <= 1:
        for i in range(n):
            fn(i)
        return
    with ThreadPoolExecutor(max_workers=t) as ex:
        list(ex.map(fn, range(n)))


def _run_ranges(fn, n, threads):
    """Split [0, n) into contiguous ranges, one per thread (at most 4 ranges
    per thread so uneven sequences still balance)."""
    t = min(_threads(threads), n)
    if t <= 1:
        fn(0, n)
        return
    parts = min(n, 4 * t)
    bounds = [n * i // parts for i in range(parts + 1)]
    with ThreadPoolExecutor(max_workers=t) as ex:
        list(ex.map(lambda i: fn(bounds[i], bounds[i + 1]), range(parts)))
