"""Full-size oracle runs in a process pool -- TEST INFRASTRUCTURE.

The layer output is the plain sum over experts of the routed partials sum_{owned j} w_j E_j(x),
plus the shared expert (the expert-parallel combine of arc PR #89, "Stage 1 -- EP=2"; the
oracle's own partition invariant is pinned in test_oracle_layer.py). A full-size workload is
therefore split into expert partitions balanced by slot count, each partial is computed by
``oracle.moe.routed_sum(owned=...)`` in its own process, and the partials are added in partition
order. The routing itself is computed once, here, by ``oracle.moe.route``. Nothing in this module
does any of the layer's arithmetic beyond that final sum.

Workers are started with ``spawn`` (safe after the CUDA context exists) and rebuild the problem
from its Spec (the expert stacks are drawn lazily per expert from their own seeded streams), so
only problems made by ``synthetic.make_problem(spec)`` can be evaluated this way.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from typing import Optional, Sequence

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _partial(args):
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import synthetic
    from oracle import moe

    spec, rows, x_bits, idx, w, owned, with_shared = args
    p = synthetic.make_problem(spec)
    x = moe.bf16_bits_to_f64(x_bits[rows])
    out = moe.routed_sum(p, x, idx[rows], w[rows], owned=owned)
    if with_shared:
        out = out + moe.shared_expert(p, x)
    return out


def partition_experts(idx: np.ndarray, parts: int) -> list[list[int]]:
    """Touched experts split into `parts` groups, largest slot counts first onto the lightest
    group (LPT); empty groups are dropped."""
    counts = np.bincount(np.asarray(idx).ravel(), minlength=int(np.max(idx)) + 1)
    order = sorted((e for e in range(counts.size) if counts[e] > 0), key=lambda e: (-counts[e], e))
    groups: list[list[int]] = [[] for _ in range(parts)]
    load = [0] * parts
    for e in order:
        g = min(range(parts), key=lambda i: (load[i], i))
        groups[g].append(e)
        load[g] += int(counts[e])
    return [sorted(g) for g in groups if g]


def forward(p, tokens: Optional[Sequence[int]] = None, route_override: Optional[np.ndarray] = None,
            workers: Optional[int] = None) -> dict:
    """As oracle.moe.forward(p, tokens=..., route_override=...) for a problem built from its Spec,
    with the expert partials evaluated in `workers` processes. Returns the same keys."""
    from oracle import moe

    s = p.spec
    x = moe.bf16_bits_to_f64(p.x_bits)
    idx, w, margin, scores = moe.route(p, x)
    if route_override is not None:
        ov = np.asarray(route_override, dtype=np.int64)
        for t in np.nonzero(~np.isnan(scores[:, 0]))[0]:
            idx[t] = ov[t]
            sel = scores[t, ov[t]]
            w[t] = sel / sel.sum()
    rows = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    n = workers or max(1, min(16, os.cpu_count() or 1))
    groups = partition_experts(idx[rows], n)
    tasks = [(s, rows, p.x_bits, idx, w, g, i == 0 and bool(s.n_shared)) for i, g in enumerate(groups)]
    if not tasks:  # nothing routed: the shared expert alone
        tasks = [(s, rows, p.x_bits, idx, w, [], bool(s.n_shared))]
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:  # one BLAS thread per worker process (the children inherit this environment)
        os.environ[v] = "1"
    try:
        with mp.get_context("spawn").Pool(min(n, len(tasks))) as pool:
            parts = pool.map(_partial, tasks)
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val
    out = parts[0].copy()
    for part in parts[1:]:
        out += part
    return dict(out=out, idx=idx, w=w, margin=margin, scores=scores, tokens=rows)
