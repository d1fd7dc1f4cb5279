"""GPU: expert-subset handles (the expert-parallel partial of arc PR #89, "Stage 1 -- EP=2", on
one GPU). For contiguous, random and load-balanced (LPT) partitions of the experts into 2 and 4
parts, on the decode and the batched path: every handle routes exactly as the full handle does;
each partial matches the fp64 oracle's sum over its owned slots (plus the shared expert for the
one part that includes it); the partials add up to the full forward."""
import numpy as np
import pytest

import synthetic
from oracle import moe
import moe_gpu
from quantized_moe_gb300 import ds4moe as api
from test_gpu_parity import SMALL_MIX

pytestmark = pytest.mark.gpu

MARGIN = 1e-6


def partitions(counts: np.ndarray, n_parts: int, seed: int):
    """Contiguous blocks, a random split, and LPT on the observed per-expert slot counts."""
    E = counts.size
    out = {"contiguous": [list(range(i * E // n_parts, (i + 1) * E // n_parts)) for i in range(n_parts)]}
    perm = np.random.default_rng(seed).permutation(E)
    out["random"] = [sorted(perm[i::n_parts].tolist()) for i in range(n_parts)]
    load, lpt = [0] * n_parts, [[] for _ in range(n_parts)]
    for e in sorted(range(E), key=lambda e: (-counts[e], e)):
        g = min(range(n_parts), key=lambda i: (load[i], i))
        lpt[g].append(e)
        load[g] += int(counts[e])
    out["lpt"] = [sorted(g) for g in lpt]
    return out


@pytest.mark.parametrize("n_tokens", [6, 37], ids=["decode", "batched"])
@pytest.mark.parametrize("n_parts", [2, 4])
def test_partials_over_expert_partitions(n_tokens, n_parts):
    spec = SMALL_MIX.with_(n_tokens=n_tokens, n_hash=min(5, n_tokens))
    p = synthetic.make_problem(spec)
    h_full = moe_gpu.create(p)
    try:
        full, idx_full, w_full = moe_gpu.forward(h_full, p)
    finally:
        api.ds4moe_destroy(h_full)
    x = moe.bf16_bits_to_f64(p.x_bits)
    ref_idx, ref_w, margin, _ = moe.route(p, x)
    clear = margin > MARGIN  # tokens whose route is unique (table-routed ones have margin inf)
    assert np.array_equal(np.sort(idx_full[clear], 1), np.sort(ref_idx[clear], 1))
    shared = moe.shared_expert(p, x)
    counts = np.bincount(idx_full.ravel(), minlength=spec.n_experts)
    for name, parts in partitions(counts, n_parts, seed=n_parts).items():
        total = np.zeros_like(full, dtype=np.float64)
        for i, owned in enumerate(parts):
            h = moe_gpu.create(p, owned=owned, include_shared=(i == 0))
            try:
                got, idx, w = moe_gpu.forward(h, p)
                st = api.ds4moe_get_stats(h)
            finally:
                api.ds4moe_destroy(h)
            # the same routing as the full handle (same kernels, same inputs)
            assert np.array_equal(idx, idx_full) and np.array_equal(w.view(np.uint32), w_full.view(np.uint32))
            held = np.zeros(spec.n_experts, bool)
            held[owned] = True
            assert np.array_equal(st["counts"][:spec.n_experts], np.where(held, counts, 0)), (name, i)
            assert st["distinct_experts"] == int((counts[held] > 0).sum())
            want = moe.routed_sum(p, x, ref_idx, ref_w, owned=owned) + (shared if i == 0 else 0.0)
            err = np.max(np.abs(got[clear] - want[clear]))
            tol = 2e-3 * float(np.max(np.abs(want[clear]))) + 1e-5
            print(f"{name} part {i} ({len(owned)} experts): max err {err:.3e}, tol {tol:.3e}")
            assert err <= tol, (name, i, err, tol)
            total += got
        # the partials add up to the full forward
        assert np.max(np.abs(total - full)) <= moe_gpu.tolerance(full), name
