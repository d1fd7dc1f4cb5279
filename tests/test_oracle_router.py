"""Pins for the oracle's router: closed-form sigmoid scores, the tie rule, bias-only
routing, renormalisation and table routing."""
import struct

import numpy as np

from oracle import moe
from conftest import read_fixture


def test_router_closed_form_fixture():
    fx = read_fixture("router_small.txt")
    col0 = [struct.unpack("<f", bytes.fromhex(h))[0] for h in fx["wr_col0"].split()]
    wr = np.zeros((4, 2), np.float32)
    wr[:, 0] = col0
    x = np.array([[1.0, 0.0]])
    s = moe.router_scores(x, wr, None)
    np.testing.assert_allclose(s[0], [float(v) for v in fx["scores"].split()], atol=1e-7)
    idx, w, margin = moe.select_topk(s, 2)
    assert list(idx[0]) == [int(v) for v in fx["top2"].split()]
    np.testing.assert_allclose(w[0], [float(v) for v in fx["w"].split()], atol=1e-7)
    np.testing.assert_allclose(margin[0], 0.75 - 0.5, atol=1e-7)


def test_zero_router_ties_go_to_lower_index():
    # W_r = 0, no bias: every score is exactly 1/2, so the top-k is experts 0..k-1, weights 1/k
    x = np.random.default_rng(0).standard_normal((3, 16))
    s = moe.router_scores(x, np.zeros((8, 16), np.float32), None)
    assert np.all(s == 0.5)
    idx, w, margin = moe.select_topk(s, 3)
    assert (idx == np.arange(3)).all()
    np.testing.assert_array_equal(w, np.full((3, 3), 1 / 3))
    assert np.all(margin == 0)


def test_bias_only_router_is_argsort_of_bias():
    rng = np.random.default_rng(1)
    b = rng.standard_normal(32).astype(np.float32)
    x = rng.standard_normal((2, 8))
    s = moe.router_scores(x, np.zeros((32, 8), np.float32), b)
    idx, w, _ = moe.select_topk(s, 5)
    want = np.argsort(-b.astype(np.float64), kind="stable")[:5]
    assert (idx == want).all()
    sel = 1 / (1 + np.exp(-b[want].astype(np.float64)))
    np.testing.assert_allclose(w[0], sel / sel.sum(), rtol=1e-15)


def test_weights_sum_to_one_and_scores_descend():
    rng = np.random.default_rng(2)
    s = moe.router_scores(rng.standard_normal((50, 64)), (rng.standard_normal((16, 64)) * 0.1).astype(np.float32),
                          rng.standard_normal(16).astype(np.float32))
    idx, w, margin = moe.select_topk(s, 4)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    sel = np.take_along_axis(s, idx, 1)
    assert np.all(np.diff(sel, axis=1) <= 0)
    assert np.all(margin >= 0)
    for t in range(50):  # every unselected score is at most the k-th
        rest = np.setdiff1d(np.arange(16), idx[t])
        assert s[t, rest].max() <= sel[t, -1]


def test_hash_route_reads_table_rows():
    table = np.array([[3, 1, 2, 0], [0, 2, 1, 3], [1, 0, 3, 2]], np.int32)
    idx, w = moe.hash_route(np.array([2, 0, 2, 1]), table, 2)
    assert idx.tolist() == [[1, 0], [3, 1], [1, 0], [0, 2]]
    assert np.all(w == 0.5)


def test_sigmoid_and_silu_closed_forms():
    assert moe.sigmoid(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(moe.sigmoid(np.log([3.0, 9.0, 1 / 3])), [0.75, 0.9, 0.25], rtol=1e-15)
    np.testing.assert_allclose(moe.silu(np.log([3.0])), [0.75 * np.log(3.0)], rtol=1e-15)
    assert moe.silu(np.array([0.0]))[0] == 0.0
