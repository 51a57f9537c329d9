"""Host-side checks of libspv that need no GPU: it builds, loads, exports every
function spv.h declares, sizes workspaces, and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_token_spv_gb300 import build
    build.build_library()
    import speculative_decoding_token_spv_gb300 as spv
    return spv.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "spv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spv_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"spv_verify_chain", "spv_verify_greedy", "spv_fanout_topk"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(lib):
    import speculative_decoding_token_spv_gb300 as spv
    a = spv.spv_chain_workspace_bytes(64, 4, 151936)
    g = spv.spv_greedy_workspace_bytes(64, 4, 151936)
    f = spv.spv_fanout_workspace_bytes(8, 4, 128256, 8)
    assert a >= g > 0 and f > 0
    nb = (151936 + 1023) // 1024
    assert a >= 64 * 9 * nb * 8
    assert spv.spv_chain_workspace_bytes(0, 4, 100) == 0
    assert spv.spv_chain_workspace_bytes(1, 33, 100) == 0
    assert spv.spv_fanout_workspace_bytes(1, 64, 100, 1) == 0
    # every workspace holds the 256-byte header (error word, self-test flag,
    # work-item counter at bytes 8..15) even at the smallest shapes
    for n in (spv.spv_chain_workspace_bytes(1, 1, 2), spv.spv_greedy_workspace_bytes(1, 1, 2),
              spv.spv_fanout_workspace_bytes(1, 0, 2, 0), spv.spv_filtered_workspace_bytes(1, 1, 2),
              spv.spv_tree_workspace_bytes(1, 1, 2)):
        assert n >= 256


def test_binding_constants_match_header():
    """The binding's copies of the header's limits are the header's values."""
    import speculative_decoding_token_spv_gb300 as spv
    src = open(os.path.join(ROOT, "include", "spv.h")).read()
    defs = dict(re.findall(r"#define[ \t]+(SPV_[A-Z_]+)[ \t]+([^/\n]+?)[ \t]*(?:/\*.*)?$", src, flags=re.M))
    assert defs, "no limits found in spv.h"
    for name, val in defs.items():
        assert getattr(spv, name) == eval(val), name


def test_fanout_sizes_in_c(lib):
    """spv_fanout_sizes rounds F_0 a^(k/(1+r)) half away from zero and clamps to
    [0, V-1] in C; the golden fan-out of the SSD workload is [8, 7, 6, 5, 4]."""
    import speculative_decoding_token_spv_gb300 as spv
    assert spv.spv_fanout_sizes(8, 0.8, 0.5, 4, 128256) == [8, 7, 6, 5, 4]
    # half away from zero: 2.5 -> 3 (a^(k/(1+r)) = 0.5 at k = 1, r = 0 with F0 = 5)
    assert spv.spv_fanout_sizes(5, 0.5, 0.0, 2, 1000) == [5, 3, 1]
    assert spv.spv_fanout_sizes(100, 1.0, 0.0, 1, 40) == [39, 39]       # clamped to V - 1
    assert spv.spv_fanout_sizes(0, 0.8, 0.5, 3, 100) == [0, 0, 0, 0]
    out = (ctypes.c_int32 * 2)()
    for args in ((8, 0.8, 0.5, -1, 100), (8, 0.0, 0.5, 1, 100), (8, 0.8, -1.0, 1, 100), (-1, 0.8, 0.5, 1, 100),
                 (8, 0.8, 0.5, 1, 1), (8, float("inf"), 0.5, 1, 100), (8, 0.8, 0.5, 64, 100)):
        assert lib.spv_fanout_sizes(*args, ctypes.addressof(out)) == 1, args
    assert lib.spv_fanout_sizes(8, 0.8, 0.5, 1, 100, None) == 1


def test_fanout_size_and_status_strings(lib):
    import speculative_decoding_token_spv_gb300 as spv
    assert spv.fanout_sizes(8, 0.8, 0.5, 4, 128256) == [8, 7, 6, 5, 4]
    assert abs(spv.spv_fanout_size(8, 0.8, 0.5, 3) - 5.12) < 1e-12
    for code in range(6):
        assert spv.spv_status_string(code).startswith("SPV_")


def test_invalid_arguments_rejected_on_host(lib):
    """Each of these fails validation before the library touches CUDA."""
    P = ctypes.c_void_p
    fake = P(4096)   # never dereferenced: validation fails first
    ws = P(1 << 20)
    big = 1 << 40
    INV = 1
    chain = lib.spv_verify_chain
    ok_args = dict(t=fake, d=fake, dt=0, tok=fake, r=fake, keys=fake, B=4, g=4, V=1000, T=1.0, k=fake,
                   out=fake, pq=None, z=None, st=None, ws=ws, wsb=big, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return chain(a["t"], a["d"], a["dt"], a["tok"], a["r"], a["keys"], a["B"], a["g"], a["V"],
                     ctypes.c_float(a["T"]), a["k"], a["out"], a["pq"], a["z"], a["st"], a["ws"], a["wsb"],
                     a["stream"])

    assert call(t=None) == INV
    assert call(tok=None) == INV
    assert call(dt=7) == INV
    assert call(B=0) == INV
    assert call(g=0) == INV
    assert call(g=33) == INV
    assert call(V=1) == INV
    assert call(T=-1.0) == INV
    assert call(T=float("nan")) == INV
    assert call(T=float("inf")) == INV
    assert call(T=1e-45) == INV          # 1/T overflows
    assert call(d=None) == INV           # T > 0 needs draft logits, r and keys
    assert call(r=None) == INV
    assert call(keys=None) == INV
    assert call(wsb=16) == INV           # workspace too small
    assert call(ws=P((1 << 20) + 8)) == INV  # workspace not 256-byte aligned
    greedy = lib.spv_verify_greedy
    assert greedy(fake, 0, fake, 4, 0, 1000, fake, fake, None, ws, big, None) == INV
    assert greedy(fake, 0, None, 4, 2, 1000, fake, fake, None, ws, big, None) == INV
    fan = lib.spv_fanout_topk
    f_bad = (ctypes.c_int32 * 2)(3, 65)
    f_big = (ctypes.c_int32 * 2)(3, 10)
    assert fan(fake, 0, fake, ctypes.cast(f_bad, P), 2, 1, 1000, fake, None, ws, big, None) == INV
    assert fan(fake, 0, fake, ctypes.cast(f_big, P), 2, 1, 10, fake, None, ws, big, None) == INV   # F > V-1
    assert fan(fake, 0, fake, ctypes.cast(f_big, P), 2, 64, 1000, fake, None, ws, big, None) == INV
    assert fan(fake, 0, fake, ctypes.cast(f_big, P), 2, 1, 2_000_000, fake, None, ws, big, None) == 3


def test_cached_verify_arguments_rejected_on_host(lib):
    """spv_verify_chain_cached: the cache arguments are all required, F_k in
    [0, SPV_MAX_FANOUT]; the usual chain checks still apply."""
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(1 << 20)
    big = 1 << 40
    INV = 1
    f_ok = (ctypes.c_int32 * 5)(8, 7, 6, 5, 4)
    f_neg = (ctypes.c_int32 * 5)(8, 7, -1, 5, 4)
    f_big = (ctypes.c_int32 * 5)(8, 7, 65, 5, 4)
    ok_args = dict(t=fake, d=fake, dt=0, tok=fake, r=fake, keys=fake, B=4, g=4, V=1000, T=1.0, k=fake,
                   out=fake, pq=None, z=None, st=None, ids=fake, fan=ctypes.cast(f_ok, P), slot=fake, ws=ws,
                   wsb=big, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spv_verify_chain_cached(a["t"], a["d"], a["dt"], a["tok"], a["r"], a["keys"], a["B"], a["g"],
                                           a["V"], ctypes.c_float(a["T"]), a["k"], a["out"], a["pq"], a["z"],
                                           a["st"], a["ids"], a["fan"], a["slot"], a["ws"], a["wsb"], a["stream"])

    assert call(ids=None) == INV
    assert call(fan=None) == INV
    assert call(slot=None) == INV
    assert call(fan=ctypes.cast(f_neg, P)) == INV
    assert call(fan=ctypes.cast(f_big, P)) == INV
    assert call(g=0) == INV
    assert call(t=None) == INV
    assert call(T=0.0, wsb=16) == INV


def test_filtered_verify_arguments_rejected_on_host(lib):
    """spv_verify_chain_filtered: 1 <= top_k <= SPV_MAX_TOP_K, 0 < top_p <= 1,
    plus the chain checks; its workspace size covers the segment lists."""
    import speculative_decoding_token_spv_gb300 as spv
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(1 << 20)
    big = 1 << 40
    INV = 1
    ok_args = dict(t=fake, d=fake, dt=0, tok=fake, r=fake, keys=fake, B=4, g=4, V=1000, T=1.0, k=50, p=1.0,
                   acc=fake, out=fake, pq=None, z=None, st=None, ws=ws, wsb=big, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spv_verify_chain_filtered(a["t"], a["d"], a["dt"], a["tok"], a["r"], a["keys"], a["B"], a["g"],
                                             a["V"], ctypes.c_float(a["T"]), a["k"], ctypes.c_float(a["p"]),
                                             a["acc"], a["out"], a["pq"], a["z"], a["st"], a["ws"], a["wsb"],
                                             a["stream"])

    for kw in (dict(k=0), dict(k=65), dict(p=0.0), dict(p=-0.5), dict(p=1.0001), dict(p=float("nan")),
               dict(t=None), dict(g=33), dict(T=-1.0), dict(d=None), dict(wsb=16), dict(ws=P((1 << 20) + 8))):
        assert call(**kw) == INV, kw
    n = spv.spv_filtered_workspace_bytes(64, 4, 151936)
    assert n >= 64 * 9 * 19 * 64 * 8 and n >= spv.spv_greedy_workspace_bytes(64, 4, 151936)
    assert spv.spv_filtered_workspace_bytes(0, 4, 100) == 0


def test_saguaro_arguments_rejected_on_host(lib):
    """spv_verify_chain_saguaro: C > 0 finite, cache arguments required,
    vocabularies up to 1,048,576."""
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(1 << 20)
    big = 1 << 40
    f_ok = (ctypes.c_int32 * 5)(8, 7, 6, 5, 4)
    ok_args = dict(t=fake, d=fake, dt=0, tok=fake, r=fake, keys=fake, B=4, g=4, V=1000, T=1.0, ids=fake,
                   fan=ctypes.cast(f_ok, P), C=2.0, acc=fake, out=fake, pq=None, z=None, st=None, slot=fake, ws=ws,
                   wsb=big, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spv_verify_chain_saguaro(a["t"], a["d"], a["dt"], a["tok"], a["r"], a["keys"], a["B"], a["g"],
                                            a["V"], ctypes.c_float(a["T"]), a["ids"], a["fan"], ctypes.c_float(a["C"]),
                                            a["acc"], a["out"], a["pq"], a["z"], a["st"], a["slot"], a["ws"], a["wsb"],
                                            a["stream"])

    for kw in (dict(C=0.0), dict(C=-2.0), dict(C=float("inf")), dict(C=float("nan")), dict(C=1e-45), dict(ids=None),
               dict(fan=None), dict(slot=None), dict(t=None), dict(g=0)):
        assert call(**kw) == 1, kw
    assert call(V=2_000_000) == 3


def test_tree_arguments_rejected_on_host(lib):
    """spv_verify_tree: 1 <= N <= 64 nodes, T >= 0 finite, draft rows,
    uniforms and keys required when T > 0, a large enough workspace."""
    import speculative_decoding_token_spv_gb300 as spv
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(1 << 20)
    big = 1 << 40
    ok_args = dict(t=fake, d=fake, dt=0, par=fake, tok=fake, r=fake, keys=fake, B=4, N=21, V=1000, T=1.0, acc=fake,
                   out=fake, nodes=None, st=None, ws=ws, wsb=big, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.spv_verify_tree(a["t"], a["d"], a["dt"], a["par"], a["tok"], a["r"], a["keys"], a["B"], a["N"],
                                   a["V"], ctypes.c_float(a["T"]), a["acc"], a["out"], a["nodes"], a["st"], a["ws"],
                                   a["wsb"], a["stream"])

    for kw in (dict(N=0), dict(N=65), dict(B=0), dict(T=-1.0), dict(T=float("inf")), dict(T=float("nan")),
               dict(T=1e-45), dict(d=None), dict(r=None), dict(keys=None), dict(par=None), dict(tok=None),
               dict(t=None), dict(acc=None), dict(out=None), dict(wsb=16), dict(ws=P((1 << 20) + 8)), dict(dt=7)):
        assert call(**kw) == 1, kw
    n = spv.spv_tree_workspace_bytes(64, 21, 151936)
    assert n > 0 and spv.spv_tree_workspace_bytes(64, 65, 151936) == 0 and spv.spv_tree_workspace_bytes(0, 4, 10) == 0


def test_selftest_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    ws = P(1 << 20)
    assert lib.spv_selftest_timeout(None, 4096, 10, None) == 1
    assert lib.spv_selftest_timeout(ws, 4096, 0, None) == 1
    assert lib.spv_selftest_timeout(ws, 4096, (1 << 24) + 1, None) == 1
    assert lib.spv_selftest_timeout(ws, 128, 10, None) == 1
    assert lib.spv_selftest_timeout(P((1 << 20) + 64), 4096, 10, None) == 1


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    """spv_verify_chain_noalloc refuses, before any CUDA call, a call whose
    scratch would not fit its fixed array: the chain layout at T > 0, the
    (smaller) greedy layout at T = 0; other argument errors as
    spv_verify_chain."""
    import speculative_decoding_token_spv_gb300 as spv
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.spv_verify_chain_noalloc
    f.argtypes = [P, P, I, P, P, P, I, I, I, ctypes.c_float, P, P, P, P, P, P]
    f.restype = I
    lim = spv.SPV_NOALLOC_SCRATCH_BYTES
    fake = P(256)  # never dereferenced: the checks come first
    g, V = 4, 151936

    def call(B, T, **kw):
        a = dict(t=fake, tok=fake, k=fake)
        a.update(kw)
        return f(a["t"], fake, 0, a["tok"], fake, fake, B, g, V, ctypes.c_float(T), a["k"], fake, None, None, None,
                 None)

    assert spv.spv_chain_workspace_bytes(600, g, V) > lim >= spv.spv_greedy_workspace_bytes(600, g, V)
    assert call(600, 1.0) == spv.SPV_ERR_UNSUPPORTED      # chain layout too large
    assert spv.spv_greedy_workspace_bytes(1024, g, V) > lim
    assert call(1024, 0.0) == spv.SPV_ERR_UNSUPPORTED     # greedy layout too large
    assert call(2048, 1.0) == spv.SPV_ERR_UNSUPPORTED
    assert call(4, 1.0, t=None) == spv.SPV_ERR_INVALID_ARG
    assert call(4, 1.0, tok=None) == spv.SPV_ERR_INVALID_ARG
    assert call(4, -1.0) == spv.SPV_ERR_INVALID_ARG
    assert call(4, float("nan")) == spv.SPV_ERR_INVALID_ARG
    assert call(0, 1.0) == spv.SPV_ERR_INVALID_ARG
