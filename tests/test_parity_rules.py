"""The comparison rules the GPU tests and the benchmark's parity record apply,
checked on the CPU with oracle outputs and planted differences: a label that
differs where the oracle's winner is clear fails, a near-tie flip is counted
and accepted only if it is itself within the distance tolerance, and a
distance outside the tolerance fails."""
import os
import sys

import numpy as np
import pytest

import oracle
import synth
from parity import check_assign_every_row

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _case():
    # blobs plus three samples exactly halfway between centroids 0 and 1
    # (small integers: the two distances are equal in any precision)
    X, _, _ = synth.planted_blobs(600, 8, 6, seed=4)
    C = np.ascontiguousarray(X[synth.init_rows(600, 6, seed=5)])
    C[0] = 0.0
    C[1] = 0.0
    C[1, 0] = 2.0
    X[:3] = 0.0
    X[:3, 0] = 1.0
    o_l, o_b, o_s, o_in = oracle.assign(X, C)
    xn = (X.astype(np.float64) ** 2).sum(1)
    cn = (C.astype(np.float64) ** 2).sum(1)
    near = np.flatnonzero((o_s - o_b) <= 1e-3 * (xn + cn[o_l]))
    return X, C, o_l, o_b, o_s, o_in, near


def test_oracle_outputs_pass_with_no_flips():
    X, C, o_l, o_b, o_s, _, near = _case()
    flips, worst, n_near = check_assign_every_row(X, C, o_l, o_b.astype(np.float32), o_l, near, o_b[near],
                                                  o_s[near])
    assert flips == 0 and worst < 1e-6 and n_near >= 1


def test_near_tie_flip_is_counted_and_clear_mismatch_fails():
    X, C, o_l, o_b, o_s, _, near = _case()
    tie = [i for i in near if (o_s[i] - o_b[i]) == 0.0]
    assert tie, "the halfway samples are exact ties"
    i = tie[0]
    other = [j for j in range(C.shape[0]) if j != o_l[i] and oracle.sqdist(X[i], C[j]) == o_b[i]][0]
    lab = o_l.copy()
    lab[i] = other
    flips, _, _ = check_assign_every_row(X, C, lab, o_b.astype(np.float32), o_l, near, o_b[near], o_s[near])
    assert flips == 1
    clear = int(np.setdiff1d(np.arange(len(X)), near)[0])
    lab[clear] = (o_l[clear] + 1) % C.shape[0]
    with pytest.raises(AssertionError, match="winner is clear"):
        check_assign_every_row(X, C, lab, o_b.astype(np.float32), o_l, near, o_b[near], o_s[near])


def test_distance_outside_tolerance_fails():
    X, C, o_l, o_b, o_s, _, near = _case()
    best = o_b.copy()
    scale = (X.astype(np.float64) ** 2).sum(1) + (C.astype(np.float64) ** 2).sum(1)[o_l]
    best[10] += 2e-4 * scale[10]
    with pytest.raises(AssertionError, match="outside tolerance"):
        check_assign_every_row(X, C, o_l, best, o_l, near, o_b[near], o_s[near])


def test_bench_parity_record():
    sys.path.insert(0, ROOT)
    import bench
    X, C, o_l, o_b, o_s, _, near = _case()
    rows = np.arange(0, len(X), 2)
    tie = [i for i in rows if (o_s[i] - o_b[i]) == 0.0][0]
    lab = o_l.copy()
    lab[tie] = [j for j in range(C.shape[0]) if j != o_l[tie] and oracle.sqdist(X[tie], C[j]) == o_b[tie]][0]
    lab[rows[-1]] = (o_l[rows[-1]] + 1) % C.shape[0]  # a clear mismatch
    rec = bench.assign_parity(X, C, rows, lab, o_b.astype(np.float32), o_l[rows], o_b[rows], o_s[rows])
    assert rec["rows_checked"] == len(rows)
    assert rec["near_tie_flips"] == 1 and rec["clear_label_mismatches"] == 1
    assert rec["distances_within_tolerance"] and rec["worst_rel_distance_error"] < 1e-6
    o_C, o_cnt = oracle.update(X, o_l, C)
    C_bad = o_C.copy()
    C_bad[2, 3] += 1e-3 * np.abs(o_C[2]).max()
    rec = bench.centroid_parity(C_bad, o_cnt.astype(np.int32), o_C, o_cnt)
    assert not rec["centroids_within_tolerance"] and rec["counts_equal"]
    assert rec["worst_centroid_row_error"] == pytest.approx(1e-3, rel=1e-3)
