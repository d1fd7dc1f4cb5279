"""Pins for bucketing: stable (expert, token, slot) order, and the distinct-experts closed
form checked against the figures printed on the expert-parallelism page."""
import numpy as np
import pytest

from oracle import moe
from conftest import read_fixture


def test_bucket_is_stable_counting_sort():
    rng = np.random.default_rng(0)
    n, k, e = 40, 3, 7
    idx = np.stack([rng.choice(e, k, replace=False) for _ in range(n)])
    counts, offsets, perm, rowof = moe.bucket(idx, e)
    assert counts.tolist() == [int((idx == i).sum()) for i in range(e)]
    assert offsets[0] == 0 and offsets[-1] == n * k
    flat = idx.reshape(-1)
    for ex in range(e):
        seg = perm[offsets[ex]:offsets[ex + 1]]
        assert np.all(flat[seg] == ex)
        assert np.all(np.diff(seg) > 0)  # ascending (token, slot)
    assert np.all(perm[rowof] == np.arange(n * k))


def test_imbalance_bound_matches_printed_figures():
    fx = read_fixture("imbalance_arc_pr89.txt")
    for row in fx["_rows"]:
        e, k, b, pct, dec = int(row[0]), int(row[1]), int(row[2]), float(row[3]), int(row[4])
        assert round(100 * moe.imbalance_bound(e, k, b), dec) == pytest.approx(pct, abs=1e-9)


def test_expected_distinct_matches_monte_carlo():
    rng = np.random.default_rng(1)
    e, k, b, trials = 256, 6, 128, 400
    got = []
    for _ in range(trials):
        idx = np.argsort(rng.random((b, e)), axis=1)[:, :k]  # uniform random k-subsets
        counts, *_ = moe.bucket(idx, e)
        got.append(int((counts > 0).sum()))
    mean, sem = np.mean(got), np.std(got) / np.sqrt(trials)
    assert abs(mean - moe.expected_distinct(e, k, b)) < 4 * sem + 1e-9


def test_hash_prefix_touches_nearly_all_experts():
    # 1024 table-routed tokens with 8 of 256 experts each: E(1 - (1 - 8/256)^1024) is 256 to 1e-11
    assert 256 - moe.expected_distinct(256, 8, 1024) < 1e-10
