"""The benchmark's same-run parity check (CPU): far mismatches, near-tie
counts and the p / q error are computed from the timed outputs and the
oracle's on the same inputs."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _case():
    B, g = 4, 2
    ref = {"accept_count": np.array([2, 0, 1, -1], np.int32),
           "out_tokens": np.array([[5, 6, 7], [3, -1, -1], [5, 9, -1], [-1, -1, -1]], np.int32),
           "status": np.array([0, 0, 0, 4], np.int32),
           "margin": np.array([0.3, 5e-7, 0.2, np.inf]),
           "pq": np.array([[[0.1, 0.2], [0.3, 0.4]]] * 4)}
    got = {"accept_count": torch.tensor(ref["accept_count"]), "out_tokens": torch.tensor(ref["out_tokens"]),
           "row_status": torch.tensor(ref["status"]), "pq": torch.tensor(ref["pq"], dtype=torch.float32)}
    return got, ref, B, g


def test_parity_counts_agreeing_outputs():
    got, ref, B, g = _case()
    p = bench.parity_against_oracle(got, ref, B, g)
    assert p["far_mismatches"] == 0 and p["near_tie_mismatches"] == 0
    assert p["near_ties"] == 1 and p["positions"] == B * (g + 1)
    assert p["pq_max_rel_err"] < 1e-6


def test_parity_flags_a_far_mismatch_and_forgives_a_near_tie():
    got, ref, B, g = _case()
    got["out_tokens"][0, 2] = 8      # sequence 0: margin 0.3, a real mismatch
    got["accept_count"][1] = 1       # sequence 1: margin 5e-7, a near tie
    got["out_tokens"][1, :2] = torch.tensor([3, 4], dtype=torch.int32)
    p = bench.parity_against_oracle(got, ref, B, g)
    assert p["far_mismatches"] == 1 and p["near_tie_mismatches"] == 1
