"""Pins for the oracle's layer forward: brute force on tiny problems, closed-form
one-hot experts, the partition (expert parallel) invariant, masking of unowned slots,
placement invariance and table routing."""
import dataclasses

import numpy as np
import pytest

import synthetic
from oracle import brute, moe

TINY_Q2K = synthetic.Spec("tiny-q2k", d=256, n_experts=6, top_k=2, f=256, f_shared=256, n_shared=1,
                          fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0", n_tokens=3, seed=11,
                          bias="normal")
TINY_HASH = synthetic.Spec("tiny-hash", d=256, n_experts=8, top_k=3, f=128, f_shared=128, n_shared=1,
                           fmt_gate_up="q8_0", fmt_down="q8_0", fmt_shared="q8_0", n_tokens=5, seed=12,
                           n_hash=2, hash_vocab=40)
SMALL = synthetic.Spec("small-q2k", d=512, n_experts=8, top_k=3, f=256, f_shared=256, n_shared=1,
                       fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0", n_tokens=12, seed=13,
                       bias="normal")


def _rel_err(a, b):
    return np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("spec", [synthetic.CONFIGS[0], TINY_Q2K, TINY_HASH], ids=lambda s: s.name)
def test_numpy_oracle_matches_brute_force(spec):
    p = synthetic.make_problem(spec)
    ref = moe.forward(p)
    out, idx, w = brute.forward(p)
    assert ref["idx"].tolist() == idx
    np.testing.assert_allclose(ref["w"], np.array(w), rtol=1e-13)
    assert _rel_err(ref["out"], np.array(out)) < 1e-12


def _q8_rows(rows, k, entries):
    """Q8_0 [rows x k] with scale 1 in every block and the given {(r, c): q} entries."""
    t = np.zeros((rows, k // 32, 34), np.uint8)
    t[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    for (r, c), q in entries.items():
        t[r, c // 32, 2 + c % 32] = np.uint8(q & 0xFF)
    return t.reshape(rows, -1)


def test_one_hot_expert_closed_form():
    d, f, a, b, c = 32, 32, 5, 17, 9
    spec = synthetic.Spec("one-hot", d=d, n_experts=1, top_k=1, f=f, f_shared=f, n_shared=0,
                          fmt_gate_up="q8_0", fmt_down="q8_0", fmt_shared="q8_0", n_tokens=4, seed=3)
    p = synthetic.make_problem(spec)
    p = dataclasses.replace(p, gate=_q8_rows(f, d, {(0, a): 1})[None], up=_q8_rows(f, d, {(0, b): 1})[None],
                            down=_q8_rows(d, f, {(c, 0): 1})[None])
    x = moe.bf16_bits_to_f64(p.x_bits)
    out = moe.forward(p)["out"]
    want = np.zeros_like(out)
    want[:, c] = x[:, a] / (1 + np.exp(-x[:, a])) * x[:, b]
    np.testing.assert_allclose(out, want, rtol=1e-15, atol=0)


def test_zero_gate_leaves_only_shared_expert():
    p = synthetic.make_problem(TINY_Q2K)
    zero = np.zeros((TINY_Q2K.n_experts,) + p.gate[0].shape, np.uint8)
    pz = dataclasses.replace(p, gate=zero)
    x = moe.bf16_bits_to_f64(p.x_bits)
    np.testing.assert_allclose(moe.forward(pz)["out"], moe.shared_expert(p, x), rtol=1e-15)


def _partitions(counts, n_parts, rng):
    e = len(counts)
    contiguous = [list(range(r * e // n_parts, (r + 1) * e // n_parts)) for r in range(n_parts)]
    assign = rng.integers(0, n_parts, size=e)
    random = [list(np.nonzero(assign == r)[0]) for r in range(n_parts)]
    load = [0] * n_parts
    lpt = [[] for _ in range(n_parts)]
    for ex in sorted(range(e), key=lambda i: (-counts[i], i)):  # longest processing time first
        r = int(np.argmin(load))
        lpt[r].append(ex)
        load[r] += counts[ex]
    return {"contiguous": contiguous, "random": random, "lpt": lpt}


@pytest.mark.parametrize("n_parts", [1, 2, 4])
def test_partials_over_any_partition_sum_to_output(n_parts):
    p = synthetic.make_problem(SMALL)
    ref = moe.forward(p)
    x = moe.bf16_bits_to_f64(p.x_bits)
    counts = np.bincount(ref["idx"].ravel(), minlength=SMALL.n_experts)
    shared = moe.shared_expert(p, x)
    for name, parts in _partitions(counts, n_parts, np.random.default_rng(n_parts)).items():
        assert sorted(sum(parts, [])) == list(range(SMALL.n_experts))
        total = shared.copy()
        for part in parts:
            total += moe.routed_sum(p, x, ref["idx"], ref["w"], owned=part)
        assert _rel_err(total, ref["out"]) < 1e-12, name


def test_masking_unowned_slots_equals_owned_partial():
    p = synthetic.make_problem(SMALL)
    ref = moe.forward(p)
    x = moe.bf16_bits_to_f64(p.x_bits)
    owned = [0, 3, 5, 6]
    wm = np.where(np.isin(ref["idx"], owned), ref["w"], 0.0)
    masked = moe.routed_sum(p, x, ref["idx"], wm)
    part = moe.routed_sum(p, x, ref["idx"], ref["w"], owned=owned)
    assert _rel_err(masked, part) < 1e-13
    # and zeroing the unowned experts' weights instead gives the same partial
    zero_g = np.stack([p.gate[e] if e in owned else np.zeros_like(p.gate[e]) for e in range(SMALL.n_experts)])
    pz = dataclasses.replace(p, gate=zero_g)
    assert _rel_err(moe.routed_sum(pz, x, ref["idx"], ref["w"]), part) < 1e-13


def _permuted(p, perm):
    """Store expert e at position perm[e]; ids in the hash table follow."""
    inv = np.argsort(perm)
    st = lambda s: np.stack([s[int(inv[i])] for i in range(len(perm))])
    kw = dict(router_w=p.router_w[inv], gate=st(p.gate), up=st(p.up), down=st(p.down))
    if p.router_b is not None:
        kw["router_b"] = p.router_b[inv]
    if p.hash_table is not None:
        kw["hash_table"] = perm[p.hash_table].astype(np.int32)
    return dataclasses.replace(p, **kw)


@pytest.mark.parametrize("spec", [SMALL, TINY_HASH], ids=lambda s: s.name)
def test_expert_placement_does_not_change_output(spec):
    p = synthetic.make_problem(spec)
    ref = moe.forward(p)
    perm = np.random.default_rng(5).permutation(spec.n_experts)
    got = moe.forward(_permuted(p, perm))
    assert (got["idx"] == perm[ref["idx"]]).all()
    assert _rel_err(got["out"], ref["out"]) < 1e-12


def test_sampled_rows_equal_full_rows():
    p = synthetic.make_problem(SMALL)
    full = moe.forward(p)["out"]
    part = moe.forward(p, tokens=[7, 2, 11])["out"]
    assert _rel_err(part, full[[7, 2, 11]]) < 1e-13  # BLAS blocking may reorder sums


def test_route_override_with_own_route_is_identity():
    p = synthetic.make_problem(SMALL)
    ref = moe.forward(p)
    again = moe.forward(p, route_override=ref["idx"])
    np.testing.assert_array_equal(again["out"], ref["out"])
    # a different expert set for one token changes only that token's row
    ov = ref["idx"].copy()
    ov[4] = [e for e in range(SMALL.n_experts) if e not in ref["idx"][4]][:SMALL.top_k]
    other = moe.forward(p, route_override=ov)
    rows = [t for t in range(SMALL.n_tokens) if t != 4]
    assert _rel_err(other["out"][rows], ref["out"][rows]) < 1e-13  # rows batched differently
    assert not np.allclose(other["out"][4], ref["out"][4])
    np.testing.assert_allclose(other["w"][4].sum(), 1.0, rtol=1e-15)


def test_hash_tokens_use_table_and_equal_weights():
    p = synthetic.make_problem(TINY_HASH)
    r = moe.forward(p)
    for t in range(TINY_HASH.n_hash):
        assert r["idx"][t].tolist() == p.hash_table[p.token_ids[t]][:TINY_HASH.top_k].tolist()
        assert np.all(r["w"][t] == 1 / TINY_HASH.top_k)
        assert np.isinf(r["margin"][t])
    tab = p.hash_table
    assert all(len(set(row)) == TINY_HASH.top_k for row in tab.tolist())
