"""Pins for the CPU oracle: each test ties it to something other than itself.

The pages print no labels or centroids for a worked example, so the oracle is
pinned by exact arithmetic on tiny inputs, independent library routines,
closed forms, invariants and planted structure.  Each test names the plausible
mistake it would catch.
"""
import math
import os

import numpy as np
import pytest
from scipy import stats
from scipy.spatial.distance import cdist

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# Philox4x32-10 (the k-means++ draws)
# --------------------------------------------------------------------------
def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,want", _kat_rows())
def test_philox_known_answers(ctr, key, want):
    # catches: a wrong multiplier, Weyl constant, round count or word order
    got = oracle.philox4x32_10(ctr, key)
    assert [int(x) for x in got] == want


def test_uniform_is_uniform():
    # catches: a bit-assembly mistake that skews or truncates the 53-bit uniform
    u = np.array([oracle.uniform(7, i) for i in range(20000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # different seeds give different streams
    assert oracle.uniform(7, 0) != oracle.uniform(8, 0)


# --------------------------------------------------------------------------
# Assignment
# --------------------------------------------------------------------------
def _exact_assign(Xi, Ci):
    """Brute force in exact integer arithmetic (inputs are small integers)."""
    labels, best, second = [], [], []
    for x in Xi:
        ds = [sum((int(a) - int(b)) ** 2 for a, b in zip(x, c)) for c in Ci]
        m = min(ds)
        j = ds.index(m)  # first (lowest) index attaining the minimum
        labels.append(j)
        best.append(m)
        rest = ds[:j] + ds[j + 1:]
        second.append(min(rest) if rest else math.inf)
    return labels, best, second


def test_assign_exact_integers_with_ties():
    # catches: a dropped term, wrong sign, '<=' tie-break, wrong runner-up
    rng = np.random.default_rng(3)
    Xi = rng.integers(-3, 4, size=(40, 5))
    Ci = rng.integers(-3, 4, size=(9, 5))
    Ci[6] = Ci[2]  # duplicate centroid: exact ties must go to index 2
    labels, best, second, inertia = oracle.assign(Xi.astype(np.float32), Ci.astype(np.float32))
    want_l, want_b, want_s = _exact_assign(Xi, Ci)
    assert labels.tolist() == want_l
    assert best.tolist() == [float(v) for v in want_b]
    assert second.tolist() == [float(v) for v in want_s]
    assert inertia == float(sum(want_b))
    assert 6 not in set(labels.tolist())


def test_assign_matches_scipy_cdist_on_the_probe_check_shape():
    # n=512, k=17, d=64: the separate float32 problem the fusion-probe page
    # uses to check its running-loop labels.  scipy's cdist is an independent
    # implementation of the squared Euclidean distance.
    X = synth.gaussian((512, 64), seed=11)
    C = synth.gaussian((17, 64), seed=12)
    labels, best, second, _ = oracle.assign(X, C)
    D = cdist(X.astype(np.float64), C.astype(np.float64), metric="sqeuclidean")
    np.testing.assert_allclose(best, D.min(axis=1), rtol=1e-12)
    srt = np.sort(D, axis=1)
    np.testing.assert_allclose(second, srt[:, 1], rtol=1e-12)
    gap = srt[:, 1] - srt[:, 0]
    clear = gap > 1e-9 * srt[:, 0]
    assert clear.all()
    np.testing.assert_array_equal(labels, D.argmin(axis=1))


def test_assign_gram_identity():
    # ||x - c||^2 = ||x||^2 + ||c||^2 - 2 x.c (the Gram form of the
    # "Gram assignment" section), evaluated by a matmul in float64.
    X = synth.gaussian((300, 96), seed=21, scale=2.0)
    C = synth.gaussian((23, 96), seed=22, scale=2.0)
    labels, best, _, _ = oracle.assign(X, C)
    X64, C64 = X.astype(np.float64), C.astype(np.float64)
    G = (X64 ** 2).sum(1)[:, None] + (C64 ** 2).sum(1)[None, :] - 2.0 * X64 @ C64.T
    np.testing.assert_allclose(best, G[np.arange(300), labels], rtol=1e-10, atol=1e-9)
    assert np.all(G.min(axis=1) >= best - 1e-9 * (1 + np.abs(best)))


def test_assign_recovers_planted_blobs():
    # with C = the planted centers the nearest center is the sample's own blob
    # (gap ~ 2d against noise sigma = 0.5); catches any transposed operand
    X, centers, blob = synth.planted_blobs(2048, 128, 64, seed=5)
    labels, best, second, _ = oracle.assign(X, centers)
    np.testing.assert_array_equal(labels, blob)
    assert np.all(second - best > 50.0)


def test_assign_single_centroid():
    X = synth.gaussian((100, 7), seed=31)
    C = synth.gaussian((1, 7), seed=32)
    labels, best, second, inertia = oracle.assign(X, C)
    assert (labels == 0).all()
    assert np.isinf(second).all()
    np.testing.assert_allclose(best, ((X.astype(np.float64) - C[0]) ** 2).sum(1), rtol=1e-13)
    assert inertia == pytest.approx(best.sum(), rel=1e-14)


def test_assign_one_feature_matches_sorted_search():
    # d = 1: nearest neighbour on a line by binary search over sorted centroids
    x = synth.gaussian((1000, 1), seed=41)[:, 0]
    c = synth.gaussian((37, 1), seed=42)[:, 0]
    labels, _, _, _ = oracle.assign(x[:, None], c[:, None])
    order = np.argsort(c, kind="stable")
    cs = c[order].astype(np.float64)
    pos = np.searchsorted(cs, x.astype(np.float64))
    want = []
    for xi, p in zip(x.astype(np.float64), pos):
        cands = [q for q in (p - 1, p) if 0 <= q < len(cs)]
        dist = [(xi - cs[q]) ** 2 for q in cands]
        m = min(dist)
        want.append(min(order[q] for q, dq in zip(cands, dist) if dq == m))
    np.testing.assert_array_equal(labels, want)


def test_assign_permutation_and_translation():
    # relabelling centroids relabels the answer; a common shift changes nothing
    X = synth.gaussian((400, 33), seed=51)
    C = synth.gaussian((29, 33), seed=52)
    labels, best, _, _ = oracle.assign(X, C)
    perm = np.random.default_rng(1).permutation(29)
    l2, b2, _, _ = oracle.assign(X, C[perm])
    np.testing.assert_array_equal(perm[l2], labels)
    np.testing.assert_array_equal(b2, best)
    shift = np.float32(0.25)  # exact in binary32 for these magnitudes: small
    l3, b3, _, _ = oracle.assign(X + shift, C + shift)
    np.testing.assert_array_equal(l3, labels)
    np.testing.assert_allclose(b3, best, rtol=1e-5)


# --------------------------------------------------------------------------
# Update
# --------------------------------------------------------------------------
def test_update_single_cluster_is_global_mean():
    X = synth.gaussian((5000, 20), seed=61, scale=3.0)
    C_old = np.zeros((1, 20), np.float32)
    C_new, counts = oracle.update(X, np.zeros(5000, np.int64), C_old)
    assert counts.tolist() == [5000]
    want = X.astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(C_new[0], want, rtol=2e-7, atol=1e-9)


def test_update_matches_unbuffered_scatter_add():
    # np.add.at accumulates each member into its cluster in sample order
    X = synth.gaussian((3000, 17), seed=71)
    labels = np.random.default_rng(2).integers(0, 40, size=3000)
    C_old = synth.gaussian((41, 17), seed=72)  # cluster 40 stays empty
    C_new, counts = oracle.update(X, labels, C_old)
    sums = np.zeros((41, 17), np.float64)
    np.add.at(sums, labels, X.astype(np.float64))
    cnt = np.bincount(labels, minlength=41)
    np.testing.assert_array_equal(counts, cnt)
    nz = cnt > 0
    np.testing.assert_array_equal(C_new[nz], (sums[nz] / cnt[nz, None]).astype(np.float32))
    assert cnt[40] == 0
    np.testing.assert_array_equal(C_new[40], C_old[40])  # bit-for-bit kept


def test_update_far_centroid_stays_empty_and_unchanged():
    X, centers, _ = synth.planted_blobs(1024, 16, 8, seed=81)
    C = centers.copy()
    C[3] += np.float32(1e3)
    labels, _, _, _ = oracle.assign(X, C)
    C_new, counts = oracle.update(X, labels, C)
    assert counts[3] == 0
    assert C_new[3].tobytes() == C[3].tobytes()
    # centroid * count = member sum for the others
    for j in range(8):
        if counts[j]:
            s = X[labels == j].astype(np.float64).sum(0)
            np.testing.assert_allclose(C_new[j].astype(np.float64) * counts[j], s,
                                       rtol=1e-6, atol=1e-4)


def test_update_rejects_bad_labels():
    X = synth.gaussian((10, 3), seed=1)
    with pytest.raises(ValueError):
        oracle.update(X, np.full(10, 5, np.int64), np.zeros((5, 3), np.float32))


def test_random_rows_init_never_empties_first_iteration():
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 4096, 64, 32, 64, 1, 9, 19, ""))
    labels, best, _, _ = oracle.assign(X, C0)
    _, counts = oracle.update(X, labels, C0)
    assert (counts > 0).all()


def test_lloyd_inertia_never_increases():
    X, C, _ = synth.workload_inputs(synth.Workload("t", 2048, 32, 24, 32, 1, 13, 23, ""))
    prev = math.inf
    for _ in range(10):
        C, labels, best, _, inertia, counts = oracle.lloyd_iter(X, C)
        assert inertia <= prev * (1 + 1e-12)
        prev = inertia


def test_fit_runs_to_a_fixed_point_with_zero_tolerance():
    # catches a stopping rule that fires early or a returned C that is not
    # the last update: at tol = 0 the fit ends where another iteration
    # changes nothing (same labels, same centroids bit for bit)
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 3000, 24, 16, 24, 1, 31, 32, ""))
    C, labels, best, hist, n_iter = oracle.fit(X, C0, max_iter=200, tol=0.0)
    assert n_iter < 200 and len(hist) == n_iter
    C_again, labels_again, _, _, inertia_again, _ = oracle.lloyd_iter(X, C)
    np.testing.assert_array_equal(labels_again, labels)
    assert C_again.tobytes() == C.tobytes()
    assert inertia_again == hist[-1]
    assert np.all(np.diff(hist) <= 1e-12 * hist[:-1])


def test_fit_stops_at_the_first_small_relative_improvement():
    # catches an off-by-one in the iteration count or a reversed comparison
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 3000, 24, 16, 24, 1, 33, 34, ""))
    full = oracle.fit(X, C0, max_iter=200, tol=0.0)[3]
    tol = 1e-3
    _, _, _, hist, n_iter = oracle.fit(X, C0, max_iter=200, tol=tol)
    np.testing.assert_array_equal(hist, full[:n_iter])
    rel = (full[:-1] - full[1:]) / full[:-1]  # rel[t - 1]: improvement of iteration t
    first = int(np.argmax(rel <= tol)) + 1    # the first iteration whose improvement is small
    assert n_iter == first + 1
    assert oracle.fit(X, C0, max_iter=3, tol=0.0)[4] == 3


def test_fit_from_planted_centers_stops_one_iteration_after_the_fixed_point():
    # planted, well separated blobs with C0 = the blob centers: iteration 1
    # moves each centroid to its blob's mean without changing any label;
    # iteration 2 (inertia against the means, lower) keeps them; iteration 3
    # sees the same inertia again and the fit stops
    X, centers, blob = synth.planted_blobs(2048, 32, 16, seed=41)
    C, labels, _, hist, n_iter = oracle.fit(X, centers, max_iter=50, tol=0.0)
    assert n_iter == 3
    assert hist[1] < hist[0] and hist[2] == hist[1]
    np.testing.assert_array_equal(labels, blob)
    means = np.stack([X[blob == j].astype(np.float64).mean(0) for j in range(16)])
    assert np.abs(C - means).max() <= 1e-6 * np.abs(means).max()


# --------------------------------------------------------------------------
# empty-cluster relocation (the reading of "relocates empty clusters")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("labels,best,k,want", [
    # clusters 2 and 4 are empty; the two farthest samples (3 and 7) move,
    # in index order, to clusters 2 and 4
    ([0, 0, 1, 1, 1, 0, 3, 3], [1.0, 4.0, 2.0, 9.0, 0.5, 4.0, 3.0, 7.0], 5, [0, 0, 1, 2, 1, 0, 3, 4]),
    # three samples tie at the largest distance: the two lowest indices move
    ([0, 0, 0, 0, 1, 1], [5.0, 2.0, 5.0, 1.0, 5.0, 0.0], 4, [2, 0, 3, 0, 1, 1]),
    # the farthest sample is its cluster's only member: cluster 0 is left empty
    ([0, 1, 1, 1], [9.0, 1.0, 1.0, 1.0], 3, [2, 1, 1, 1]),
    # no empty cluster: nothing moves
    ([2, 0, 1, 0], [3.0, 8.0, 1.0, 2.0], 3, [2, 0, 1, 0]),
    # every distance zero and one occupied cluster of four: samples 0..2 move
    ([1, 1, 1, 1, 1], [0.0, 0.0, 0.0, 0.0, 0.0], 4, [0, 2, 3, 1, 1]),
])
def test_relocate_hand_worked_cases(labels, best, k, want):
    # catches: the wrong end of the distance order, ties broken towards the
    # higher index, pairing by distance instead of by index, a moved sample
    # keeping its old label
    got, moved = oracle.relocate_empty(np.array(labels, np.int64), np.array(best, np.float32), k)
    assert got.tolist() == want
    assert moved.tolist() == [i for i in range(len(labels)) if labels[i] != want[i]]


def _relocate_by_repeated_argmax(labels, best, k):
    # the rule taken literally: m times, remove the farthest remaining
    # sample (first among equals); then hand them out in index order
    labels = [int(v) for v in labels]
    present = set(labels)
    empty = [j for j in range(k) if j not in present]
    left = list(range(len(labels)))
    taken = []
    for _ in empty:
        far = max(best[i] for i in left)
        i = min(i for i in left if best[i] == far)
        left.remove(i)
        taken.append(i)
    for j, i in zip(empty, sorted(taken)):
        labels[i] = j
    return labels


def test_relocate_matches_repeated_argmax_on_small_inputs():
    # catches a mistake in the sort keys on inputs with many ties and many
    # empty clusters (distances from a handful of values, -0.0 among them)
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, n + 1))
        used = rng.choice(k, size=int(rng.integers(1, k + 1)), replace=False)
        labels = rng.choice(used, size=n).astype(np.int64)
        best = rng.choice(np.array([0.0, -0.0, 1.0, 2.5, 2.5, 7.0], np.float32), size=n)
        got, _ = oracle.relocate_empty(labels, best, k)
        assert got.tolist() == _relocate_by_repeated_argmax(labels, best.astype(np.float64), k), trial


def test_fit_relocation_revives_a_far_centroid():
    # planted, well separated blobs with C0 = the blob centers except one
    # moved far away.  Keeping empty clusters leaves that centroid unused
    # for good and one blob merged into another; relocating hands it the
    # farthest sample (one of the orphaned blob's), and the fit recovers
    # every blob with a lower inertia
    X, centers, blob = synth.planted_blobs(2048, 32, 16, seed=43)
    C0 = centers.copy()
    C0[3] += np.float32(1e3)
    C_keep, labels_keep, _, hist_keep, _ = oracle.fit(X, C0, max_iter=50, tol=0.0)
    assert np.bincount(labels_keep, minlength=16)[3] == 0
    assert C_keep[3].tobytes() == C0[3].tobytes()
    C_rel, labels_rel, _, hist_rel, _ = oracle.fit(X, C0, max_iter=50, tol=0.0, relocate=True)
    np.testing.assert_array_equal(labels_rel, blob)
    assert hist_rel[-1] < hist_keep[-1]
    means = np.stack([X[blob == j].astype(np.float64).mean(0) for j in range(16)])
    assert np.abs(C_rel - means).max() <= 1e-6 * np.abs(means).max()
    assert np.all(np.diff(hist_rel) <= 1e-12 * hist_rel[:-1])


def test_fit_relocation_never_raises_the_inertia():
    # moving a sample onto its own new centroid lowers its cost, and the
    # mean update lowers it further: the inertia still never rises, even
    # from an initialisation with most clusters empty
    X = synth.gaussian((600, 8), seed=95)
    C0 = synth.gaussian((60, 8), seed=96) * np.float32(30.0)
    _, labels, _, hist, n_iter = oracle.fit(X, C0, max_iter=100, tol=0.0, relocate=True)
    assert np.all(np.diff(hist) <= 1e-12 * hist[:-1])
    assert (np.bincount(labels, minlength=60) > 0).all()


def test_oracle_thread_count_does_not_change_bits():
    X = synth.gaussian((777, 45), seed=91)
    C = synth.gaussian((31, 45), seed=92)
    a = oracle.lloyd_iter(X, C, nthreads=1)
    b = oracle.lloyd_iter(X, C, nthreads=4)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(np.asarray(u), np.asarray(v))


# --------------------------------------------------------------------------
# k-means++
# --------------------------------------------------------------------------
def test_kmeanspp_trial_count():
    # "2 + log(n_clusters)", natural log, floored
    assert oracle.n_trials_for(1) == 2
    assert oracle.n_trials_for(1024) == 8
    assert oracle.n_trials_for(2) == 2
    assert oracle.n_trials_for(3) == 3


def test_kmeanspp_first_center_is_uniform_draw():
    X = synth.gaussian((1000, 4), seed=3)
    for seed in (0, 1, 99):
        idx, _, _ = oracle.kmeanspp(X, 1, seed)
        assert idx[0] == int(math.floor(oracle.uniform(seed, 0) * 1000))


def test_kmeanspp_second_draw_follows_d2_law():
    # with one trial, center 1 is sampled with probability D^2_i / sum D^2
    pts = np.array([[0.0], [1.0], [2.0], [4.0], [7.0], [11.0]], np.float32)
    n = len(pts)
    expected = np.zeros(n)
    observed = np.zeros(n)
    for seed in range(3000):
        idx, _, _ = oracle.kmeanspp(pts, 2, seed, n_trials=1)
        d2 = (pts[:, 0].astype(np.float64) - pts[idx[0], 0]) ** 2
        expected += d2 / d2.sum()
        observed[idx[1]] += 1
    assert observed[expected == 0].sum() == 0
    keep = expected > 0
    chi = stats.chisquare(observed[keep], expected[keep] * observed.sum() / expected[keep].sum())
    assert chi.pvalue > 1e-3


def test_kmeanspp_distinct_points_never_repeat():
    # a chosen point has D^2 = 0, so with the strict '>' search it is never
    # drawn again: k = n gives a permutation
    X = synth.gaussian((40, 3), seed=5)
    idx, margins, pots = oracle.kmeanspp(X, 40, 7, n_trials=3)
    assert sorted(idx.tolist()) == list(range(40))
    assert pots[-1] == 0.0
    assert np.all(np.diff(pots) <= 1e-12)  # potential never increases


def test_kmeanspp_identical_points_take_last_index():
    # sum D^2 = 0: no running sum exceeds the target, the draw clips to n - 1
    X = np.ones((10, 4), np.float32)
    idx, _, _ = oracle.kmeanspp(X, 3, 1, n_trials=2)
    assert idx[1] == 9 and idx[2] == 9


def test_kmeanspp_hits_every_separated_blob():
    # 16 blobs, centers 100 apart: greedy D^2 seeding with 4 trials puts one
    # center in each blob
    centers = np.arange(16, dtype=np.float32)[:, None] * 100.0 * np.ones((1, 8), np.float32)
    X = np.repeat(centers, 30, axis=0) + synth.gaussian((480, 8), seed=8, scale=0.5)
    idx, _, _ = oracle.kmeanspp(X, 16, 2024, n_trials=4)
    assert sorted((idx // 30).tolist()) == list(range(16))


def test_kmeanspp_margins_are_fractions():
    X = synth.gaussian((500, 6), seed=9)
    idx, margins, _ = oracle.kmeanspp(X, 20, 3)
    assert len(margins) == 1 + 19 * oracle.n_trials_for(20)
    assert np.all(margins >= 0) and np.all(margins <= 0.5)


# --------------------------------------------------------------------------
# Input generator
# --------------------------------------------------------------------------
def test_blob_generator_statistics_and_determinism():
    X, centers, blob = synth.planted_blobs(4096, 64, 16, seed=3, threads=3)
    X2, _, _ = synth.planted_blobs(4096, 64, 16, seed=3, threads=1)
    assert X.tobytes() == X2.tobytes()  # thread count does not change bytes
    noise = X - centers[blob]
    assert abs(noise.std() - 0.5) < 0.01
    assert abs(centers.std() - 1.0) < 0.05
    assert (blob == np.arange(4096) % 16).all()


# --------------------------------------------------------------------------
# k-means++: the greedy choice among trials and the draw numbering
# ("004 — tile sizes, a Cython Lloyd step, and k-means++", section
# "k-means++": each new center is the best of 2 + log(n_clusters) D^2-drawn
# candidates, the best being the one that leaves the smallest potential)
# --------------------------------------------------------------------------
def _d2_pick(D2, u):
    """Plain loop: the first sample whose running sum of D^2 exceeds
    u * sum(D^2); the last sample when none does."""
    total = 0.0
    for v in D2:
        total += v
    target = u * total
    run = 0.0
    for i, v in enumerate(D2):
        run += v
        if run > target:
            return i
    return len(D2) - 1


def _kmeanspp_loops(X, k, seed, T, rule="lowest", numbering="paper"):
    """Greedy k-means++ restated with plain Python loops, for tiny inputs of
    small integers (every distance, sum and potential is then exact in
    binary64).  ``rule`` and ``numbering`` select deliberately wrong variants,
    so a test can show that the oracle's answers tell them apart."""
    n = len(X)

    def sq(a, b):
        return float(sum((float(p) - float(q)) ** 2 for p, q in zip(a, b)))

    idx = [min(int(math.floor(oracle.uniform(seed, 0) * n)), n - 1)]
    D2 = [sq(X[i], X[idx[0]]) for i in range(n)]
    for c in range(1, k):
        cands = []
        for t in range(T):
            draw = 1 + (c - 1) * T + t if numbering == "paper" else c * T + t
            cands.append(_d2_pick(D2, oracle.uniform(seed, draw)))
        pots = [sum(min(D2[i], sq(X[i], X[j])) for i in range(n)) for j in cands]
        if rule == "lowest":          # smallest potential, lowest trial on ties
            bt = min(range(T), key=lambda t: (pots[t], t))
        elif rule == "highest":
            bt = max(range(T), key=lambda t: (pots[t], -t))
        elif rule == "first":
            bt = 0
        elif rule == "last":
            bt = T - 1
        else:                         # smallest potential, lowest index on ties
            bt = min(range(T), key=lambda t: (pots[t], cands[t]))
        best = cands[bt]
        idx.append(best)
        D2 = [min(D2[i], sq(X[i], X[best])) for i in range(n)]
    return idx


def test_kmeanspp_hand_worked_best_trial_is_the_middle_one():
    # 1-D points 0, 2, 5, 9, 14; k = 2 with T = 3 trials.  With seed 103:
    #   u0 = 0.0252 -> first center floor(0.0252 * 5) = sample 0 (x = 0);
    #   D^2 = 0, 4, 25, 81, 196 (total 306), running sums 0, 4, 29, 110, 306;
    #   trial 0: u = 0.0592, target 18.1 -> sample 2 (x = 5);
    #   trial 1: u = 0.2165, target 66.3 -> sample 3 (x = 9);
    #   trial 2: u = 0.8702, target 266.3 -> sample 4 (x = 14).
    # Potentials sum_i min(D^2_i, (x_i - x_cand)^2):
    #   x = 5:  0 + 4 + 0 + 16 + 81 = 101
    #   x = 9:  0 + 4 + 16 + 0 + 25 = 45   <- smallest: the middle trial
    #   x = 14: 0 + 4 + 25 + 25 + 0 = 54
    # A first-trial rule gives sample 2, a last-trial rule sample 4 and a
    # largest-potential rule sample 2.  Seed 594 draws the same three
    # candidates in the reverse order (4, 3, 2) and must give sample 3 too.
    X = np.array([[0.0], [2.0], [5.0], [9.0], [14.0]], np.float32)
    for seed, us in ((103, (0.0252, 0.0592, 0.2165, 0.8702)), (594, (0.0328, 0.8765, 0.2855, 0.0236))):
        for draw, want in enumerate(us):
            assert abs(oracle.uniform(seed, draw) - want) < 5e-5
        idx, _, pots = oracle.kmeanspp(X, 2, seed, n_trials=3)
        assert idx.tolist() == [0, 3]
        assert pots.tolist() == [306.0, 45.0]


@pytest.mark.parametrize("seed,want", [(0, 2), (2, 0)])
def test_kmeanspp_equal_potentials_go_to_the_lowest_trial(seed, want):
    # 1-D points -1, 0, 1; the first center is sample 1 (u0 in [1/3, 2/3) for
    # both seeds), so D^2 = 1, 0, 1 and a draw picks sample 0 when u < 1/2,
    # sample 2 otherwise.  Either candidate leaves potential 1: an exact tie.
    # Seed 0 draws (sample 2, sample 0), seed 2 draws (sample 0, sample 2); the
    # lowest trial wins, so a lowest-index or last-trial rule fails one of them.
    X = np.array([[-1.0], [0.0], [1.0]], np.float32)
    u = [oracle.uniform(seed, i) for i in range(3)]
    assert 1 / 3 <= u[0] < 2 / 3
    assert (u[1] >= 0.5) == (want == 2) and (u[2] >= 0.5) == (want == 0)
    idx, _, pots = oracle.kmeanspp(X, 2, seed, n_trials=2)
    assert idx.tolist() == [1, want]
    assert pots.tolist() == [2.0, 1.0]


def test_kmeanspp_draw_numbering_with_several_trials():
    # Scaled one-hot rows: every pair of distinct samples is 2 s^2 apart, so
    # every unchosen sample carries the same D^2 and every candidate leaves
    # the same potential.  The lowest trial then always wins, and center c is
    # the candidate of draw 1 + (c - 1) T (trial 0): the floor(u m)-th of the
    # m samples not yet chosen, in index order.  A numbering that used draw
    # c T + t, or (c - 1) T + t, gives another sequence for this seed.
    n, k, T, s = 9, 6, 3, 2.0
    X = (s * np.eye(n)).astype(np.float32)

    def closed_form(draw_of):
        chosen = [min(int(math.floor(oracle.uniform(5, 0) * n)), n - 1)]
        for c in range(1, k):
            free = [i for i in range(n) if i not in chosen]
            chosen.append(free[int(math.floor(oracle.uniform(5, draw_of(c)) * len(free)))])
        return chosen

    want = closed_form(lambda c: 1 + (c - 1) * T)
    idx, _, pots = oracle.kmeanspp(X, k, 5, n_trials=T)
    assert idx.tolist() == want
    assert pots.tolist() == [2 * s * s * (n - 1 - c) for c in range(k)]
    assert closed_form(lambda c: c * T) != want
    assert closed_form(lambda c: (c - 1) * T) != want


def test_kmeanspp_matches_plain_loops_and_not_the_wrong_rules():
    # Tiny integer point sets over many seeds: the oracle picks exactly what
    # the loop restatement picks, index by index, and each wrong rule (largest
    # potential, first trial, last trial, lowest index on equal potentials,
    # draws numbered c T + t) disagrees with the oracle somewhere.
    rng = np.random.default_rng(2024)
    wrong = {"highest": 0, "first": 0, "last": 0, "lowest_index": 0, "numbering": 0}
    middle_wins = 0
    for case in range(120):
        n = int(rng.integers(3, 13))
        d = int(rng.integers(1, 4))
        X = rng.integers(-6, 7, size=(n, d)).astype(np.float32)
        k = int(rng.integers(2, n + 1))
        T = int(rng.integers(2, 5))
        seed = int(rng.integers(0, 2**63))
        o_idx, _, _ = oracle.kmeanspp(X, k, seed, n_trials=T)
        got = o_idx.tolist()
        assert got == _kmeanspp_loops(X, k, seed, T), f"case {case}"
        for rule in ("highest", "first", "last", "lowest_index"):
            wrong[rule] += got != _kmeanspp_loops(X, k, seed, T, rule=rule)
        wrong["numbering"] += got != _kmeanspp_loops(X, k, seed, T, numbering="shifted")
        if T >= 3:
            # does the strictly best trial sit strictly inside the trial list?
            idx0 = got[0]
            D2 = [float(((X[i].astype(np.float64) - X[idx0]) ** 2).sum()) for i in range(n)]
            cands = [_d2_pick(D2, oracle.uniform(seed, 1 + t)) for t in range(T)]
            pots = [sum(min(D2[i], float(((X[i].astype(np.float64) - X[j]) ** 2).sum())) for i in range(n))
                    for j in cands]
            bt = min(range(T), key=lambda t: (pots[t], t))
            middle_wins += 0 < bt < T - 1 and pots[bt] < min(pots[0], pots[-1])
    assert all(v > 0 for v in wrong.values()), wrong
    assert middle_wins > 0
