"""Host logic of the pooled full-size oracle runs used by the GPU parity tests: the expert
partitions cover every touched expert exactly once, and the pooled sum of partials equals the
plain oracle forward (sampled rows and a route override included)."""
import numpy as np

import synthetic
from oracle import moe
import oracle_pool

SPEC = synthetic.Spec("pool-small", d=512, n_experts=12, top_k=3, f=256, f_shared=256, n_shared=1,
                      fmt_gate_up="q2_k", fmt_down="q8_0", fmt_shared="q8_0", n_tokens=20, seed=41,
                      bias="normal", n_hash=4, hash_vocab=50)


def test_partitions_cover_touched_experts_once_and_balance():
    idx = np.random.default_rng(3).integers(0, 40, size=(300, 4))
    groups = oracle_pool.partition_experts(idx, 6)
    flat = sorted(e for g in groups for e in g)
    assert flat == sorted(set(idx.ravel().tolist()))
    counts = np.bincount(idx.ravel())
    loads = [int(counts[g].sum()) for g in groups]
    assert max(loads) - min(loads) <= counts.max()  # LPT: within one expert of each other


def test_pooled_forward_equals_plain_forward():
    p = synthetic.make_problem(SPEC)
    ref = moe.forward(p)
    got = oracle_pool.forward(p, workers=3)
    assert np.array_equal(got["idx"], ref["idx"])
    np.testing.assert_allclose(got["out"], ref["out"], rtol=0, atol=1e-12 * np.max(np.abs(ref["out"])))
    rows = [0, 3, 4, 19]  # table/learned boundary and the last row
    ov = ref["idx"].copy()
    ov[7] = ov[7][::-1]  # a permuted route for one learned token
    ov[9, 0] = (set(range(SPEC.n_experts)) - set(ov[9].tolist())).pop()
    ref2 = moe.forward(p, tokens=rows + [9], route_override=ov)
    got2 = oracle_pool.forward(p, tokens=rows + [9], route_override=ov, workers=2)
    np.testing.assert_allclose(got2["out"], ref2["out"], rtol=0, atol=1e-12 * np.max(np.abs(ref2["out"])))
