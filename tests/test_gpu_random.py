"""Seeded random configurations through every entry point, against the
oracle: batch sizes, draft lengths, vocabularies (odd sizes take the
plain-load path), dtypes, temperatures, top-k / top-p and random tree
shapes.  Same acceptance rule as the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_token_spv_gb300 import workloads
from test_gpu_parity import MARGIN, _np, check_chain
from test_gpu_filtered import check_filtered
from test_gpu_tree import check_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_token_spv_gb300 as m
    return m


def _configs(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 41))
        g = int(rng.integers(1, 13))
        V = int(rng.choice([int(rng.integers(2, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 40000))]))
        while B * (2 * g + 1) * V > 3_000_000:
            V = max(2, V // 2)
        dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
        T = float(rng.choice([0.0, 0.5, 1.0, 1.7]))
        out.append((i, B, g, V, dtype, T, int(rng.integers(1, 1 << 30))))
    return out


@pytest.mark.parametrize("cfg", _configs(2024, 16), ids=lambda c: f"B{c[1]}_g{c[2]}_V{c[3]}_{str(c[4])[6:]}_T{c[5]}")
def test_chain_random(spv, cfg):
    _, B, g, V, dtype, T, seed = cfg
    w = workloads.chain_from_params("rand", B, g, V, dtype, T, 2.5, 1.0, 0.8, 0, (seed, seed + 1, seed + 2, seed + 3),
                                    "cuda")
    check_chain(spv, w, want_Z=T > 0)


@pytest.mark.parametrize("cfg", _configs(2025, 10), ids=lambda c: f"B{c[1]}_g{c[2]}_V{c[3]}_{str(c[4])[6:]}")
def test_filtered_random(spv, cfg):
    i, B, g, V, dtype, _, seed = cfg
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 65))
    p = float(rng.choice([1.0, 0.95, 0.7, 0.3]))
    w = workloads.chain_from_params("rand_f", B, g, V, dtype, 1.0, 2.5, 1.0, 0.8, 0,
                                    (seed, seed + 1, seed + 2, seed + 3), "cuda", False, k, p)
    check_filtered(spv, w, k, p)


def _random_tree(B, N, V, dtype, T, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    rng = np.random.default_rng(seed)
    z = torch.randn(B, N, V, generator=gen) * 2.5
    d = z + torch.randn(B, N, V, generator=gen)
    parent = np.full((B, N), -1, np.int32)
    for v in range(1, N):
        parent[:, v] = rng.integers(0, v, B)
    z, d = z.to(dtype), d.to(dtype)
    tok = torch.zeros(B, N, dtype=torch.int32)
    for v in range(1, N):
        du = d[torch.arange(B), torch.from_numpy(parent[:, v]).long()].float()
        if T > 0:
            tok[:, v] = torch.multinomial(torch.softmax(du / T, dim=1), 1, generator=gen)[:, 0].int()
        else:
            tok[:, v] = du.argmax(dim=1).int()
    r = 1.0 - torch.rand(B, N, generator=gen)
    keys = torch.randint(-(2 ** 62), 2 ** 62, (B,), generator=gen, dtype=torch.int64)
    return workloads.TreeInputs("rand_tree", z.cuda(), d.cuda(), torch.from_numpy(parent).cuda(), tok.cuda(), r.cuda(),
                                keys.cuda(), T)


@pytest.mark.parametrize("seed", range(8))
def test_tree_random(spv, seed):
    rng = np.random.default_rng(700 + seed)
    B = int(rng.integers(1, 48))
    N = int(rng.integers(1, 65))
    V = int(rng.choice([int(rng.integers(2, 200)), int(rng.integers(200, 20000))]))
    while B * 2 * N * V > 3_000_000:
        V = max(2, V // 2)
    dtype = torch.float32 if seed % 2 == 0 else torch.bfloat16
    T = float(rng.choice([0.0, 0.8, 1.0]))
    check_tree(spv, _random_tree(B, N, V, dtype, T, 900 + seed))
