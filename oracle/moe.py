"""fp64 CPU oracle of the quantized MoE layer forward -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module. It is a plain, slow, single-threaded restatement of what the layer computes, in
float64, with its own decoders. It shares no code with the CUDA library.

What it follows (sources are the three pages on the quantized MoE layer):

* Tensor mix -- routed experts in 2-bit super-block quants (Q2_K) and the shared expert in
  Q8_0 (ds4 PR #754 "CUDA: add DGX Spark network expert/tensor parallelism", section
  "Supported paths and safety"; TrevorS/ds4 PR #13 "DGX Spark / GB10 backend support",
  the model line under "Tested").
* Combine -- the layer output is the plain sum over the selected experts of the routing
  weight times the expert output, which is why any partition of the experts into rank
  partials sums back to it (arc PR #89 "expert parallelism stage 0 + stage 1 (EP=2) for
  V4's MoE", section "Stage 1 -- EP=2").
* Hash routing -- early layers route by a fixed token-id -> expert table (arc PR #89,
  section "Stage 0", third item).
* The benchmark workload definition fixes the rest: fp32 router with sigmoid scores,
  top-k, weights renormalised to sum 1; SwiGLU experts h = silu(W_g x) * (W_u x),
  y = W_d h; one always-on shared expert added unscaled; block formats
  Q8_0 (w = scale * q) and Q2_K (w = d * s * q - dmin * m).

Readings where the sources are silent (each also listed in the design notes):

* a router bias is added to the logits before the sigmoid, so it moves both the choice and
  the weights;
* top-k orders experts by (score descending, expert index ascending): ties go to the lower
  index;
* no routed scaling factor, no group-limited routing, no SwiGLU clamp;
* the routing weight multiplies the expert output after the down projection;
* hash-routed tokens skip the router and weigh each of their k experts 1/k.

Parity unpinned: the Zipf and hash-table input recipes (data, not arithmetic) and the
absolute output values of the full-size workloads (the pages print no worked example).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

Q8_0_BLOCK, Q8_0_BYTES = 32, 34
Q2_K_BLOCK, Q2_K_BYTES = 256, 84


# --------------------------------------------------------------------------- decoders

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact: bf16 is the top half of fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _f16(b: np.ndarray) -> np.ndarray:
    """Little-endian byte pairs [..., 2] -> float64 through IEEE binary16."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    return b.view("<f2")[..., 0].astype(np.float64)


def dequant_q8_0(row_bytes: np.ndarray, k: int) -> np.ndarray:
    """Q8_0 rows -> float64 [rows, k]; block of 32: fp16 scale then 32 int8, w = scale * q."""
    rb = np.asarray(row_bytes, dtype=np.uint8)
    rows = rb.reshape(-1, rb.shape[-1]).shape[0]
    blk = rb.reshape(rows, k // Q8_0_BLOCK, Q8_0_BYTES)
    scale = _f16(blk[:, :, 0:2])                                    # [rows, nb]
    q = blk[:, :, 2:].view(np.int8).astype(np.float64)              # [rows, nb, 32]
    return (scale[:, :, None] * q).reshape(rows, k)


def dequant_q2_k(row_bytes: np.ndarray, k: int) -> np.ndarray:
    """Q2_K rows -> float64 [rows, k].

    Super-block of 256 weights = 16 sub-blocks of 16. Bytes 0..15 hold the sub-block
    scale s_j (low nibble) and min m_j (high nibble); bytes 16..79 hold the 2-bit quants
    (weight i at byte i >> 2, bit offset 2 * (i & 3)); bytes 80..83 hold fp16 d, dmin.
    w_i = d * s_j * q_i - dmin * m_j with j = i // 16.
    """
    rb = np.asarray(row_bytes, dtype=np.uint8)
    rows = rb.reshape(-1, rb.shape[-1]).shape[0]
    nb = k // Q2_K_BLOCK
    blk = rb.reshape(rows, nb, Q2_K_BYTES)
    s = (blk[:, :, 0:16] & 0x0F).astype(np.float64)                 # [rows, nb, 16]
    m = (blk[:, :, 0:16] >> 4).astype(np.float64)
    qb = blk[:, :, 16:80]                                           # [rows, nb, 64]
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    q = ((qb[:, :, :, None] >> shifts) & 3).reshape(rows, nb, 16, 16)  # [.., sub-block j, i % 16]
    d = _f16(blk[:, :, 80:82])[:, :, None]                          # [rows, nb, 1]
    dmin = _f16(blk[:, :, 82:84])[:, :, None]
    w = q * (d * s)[..., None] - (dmin * m)[..., None]
    return w.reshape(rows, k)


def dequant(fmt: str, row_bytes: np.ndarray, k: int) -> np.ndarray:
    if fmt == "q8_0":
        return dequant_q8_0(row_bytes, k)
    if fmt == "q2_k":
        return dequant_q2_k(row_bytes, k)
    raise ValueError(f"unsupported format {fmt!r}")


# --------------------------------------------------------------------------- routing

def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def router_scores(x: np.ndarray, router_w: np.ndarray, router_b: Optional[np.ndarray]) -> np.ndarray:
    """s = sigmoid(W_r x + b) for each token row of x (float64 throughout)."""
    z = x @ np.asarray(router_w, dtype=np.float64).T
    if router_b is not None:
        z = z + np.asarray(router_b, dtype=np.float64)[None, :]
    return sigmoid(z)


def select_topk(scores: np.ndarray, k: int):
    """Top-k per row ordered by (score desc, index asc); returns idx, renormalised w, margin.

    margin = k-th largest score minus (k+1)-th largest (inf when k equals the expert count).
    """
    n, e = scores.shape
    idx = np.empty((n, k), dtype=np.int64)
    margin = np.full(n, np.inf)
    for t in range(n):
        order = np.lexsort((np.arange(e), -scores[t]))   # primary: -score, secondary: index
        idx[t] = order[:k]
        if k < e:
            margin[t] = scores[t, order[k - 1]] - scores[t, order[k]]
    sel = np.take_along_axis(scores, idx, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return idx, w, margin


def hash_route(token_ids: np.ndarray, table: np.ndarray, k: int):
    """Table routing: expert set = table[token id], equal weights 1/k."""
    idx = np.asarray(table, dtype=np.int64)[np.asarray(token_ids, dtype=np.int64)][:, :k]
    w = np.full(idx.shape, 1.0 / k)
    return idx, w


# --------------------------------------------------------------------------- experts

def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_ffn(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """y = W_d (silu(W_g x) * (W_u x)) for each row of x (float64)."""
    g = x @ wg.T
    u = x @ wu.T
    return (silu(g) * u) @ wd.T


def _expert_weights(p, e: int):
    s = p.spec
    wg = dequant(s.fmt_gate_up, p.gate[e], s.d)
    wu = dequant(s.fmt_gate_up, p.up[e], s.d)
    wd = dequant(s.fmt_down, p.down[e], s.f)
    return wg, wu, wd


def shared_expert(p, x: np.ndarray) -> np.ndarray:
    s = p.spec
    if not s.n_shared:
        return np.zeros_like(x)
    wg = dequant(s.fmt_shared, p.shared_gate, s.d)
    wu = dequant(s.fmt_shared, p.shared_up, s.d)
    wd = dequant(s.fmt_shared, p.shared_down, s.f_shared)
    return swiglu_ffn(x, wg, wu, wd)


def route(p, x: np.ndarray, token_ids: Optional[np.ndarray] = None, n_hash: Optional[int] = None):
    """Routing of every token: hash table for the first n_hash tokens, learned router after.

    Returns idx [N, k] (int64), w [N, k] (float64), margin [N] (inf for hash tokens) and the
    learned scores [N, E] (NaN rows for hash tokens).
    """
    s = p.spec
    n = x.shape[0]
    k = s.top_k
    if n_hash is None:
        n_hash = s.n_hash
    if token_ids is None:
        token_ids = p.token_ids
    n_hash = min(n_hash, n)
    idx = np.zeros((n, k), dtype=np.int64)
    w = np.zeros((n, k))
    margin = np.full(n, np.inf)
    scores = np.full((n, s.n_experts), np.nan)
    if n_hash:
        idx[:n_hash], w[:n_hash] = hash_route(token_ids[:n_hash], p.hash_table, k)
    if n > n_hash:
        sc = router_scores(x[n_hash:], p.router_w, p.router_b)
        scores[n_hash:] = sc
        idx[n_hash:], w[n_hash:], margin[n_hash:] = select_topk(sc, k)
    return idx, w, margin, scores


def routed_sum(p, x: np.ndarray, idx: np.ndarray, w: np.ndarray,
               owned: Optional[Sequence[int]] = None) -> np.ndarray:
    """sum_j w_j * E_{idx_j}(x) over the slots whose expert is in `owned` (all if None)."""
    n = x.shape[0]
    out = np.zeros((n, p.spec.d))
    owned_set = None if owned is None else set(int(e) for e in owned)
    for e in np.unique(idx):
        if owned_set is not None and int(e) not in owned_set:
            continue
        tok, slot = np.nonzero(idx == e)
        wg, wu, wd = _expert_weights(p, int(e))
        y = swiglu_ffn(x[tok], wg, wu, wd)
        np.add.at(out, tok, w[tok, slot][:, None] * y)
    return out


def forward(p, x_bits: Optional[np.ndarray] = None, tokens: Optional[Sequence[int]] = None,
            route_override: Optional[np.ndarray] = None, token_ids: Optional[np.ndarray] = None,
            n_hash: Optional[int] = None):
    """Layer forward: out = S(x) + sum_j w_j E_{idx_j}(x).

    tokens          compute the output only for these token rows (routing is always
                    computed for all rows, so sampled rows equal the full run's rows)
    route_override  int [N, k] expert ids to use instead of the oracle's own top-k for the
                    learned tokens; weights are then renormalised from the oracle's scores
    Returns dict(out [len(tokens), d] float64, idx, w, margin, scores, tokens).
    """
    if x_bits is None:
        x_bits = p.x_bits
    x = bf16_bits_to_f64(x_bits)
    n = x.shape[0]
    idx, w, margin, scores = route(p, x, token_ids, n_hash)
    if route_override is not None:
        ov = np.asarray(route_override, dtype=np.int64)
        learned = ~np.isnan(scores[:, 0])
        for t in np.nonzero(learned)[0]:
            idx[t] = ov[t]
            sel = scores[t, ov[t]]
            w[t] = sel / sel.sum()
    rows = np.arange(n) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xs = x[rows]
    out = routed_sum(p, xs, idx[rows], w[rows]) + shared_expert(p, xs)
    return dict(out=out, idx=idx, w=w, margin=margin, scores=scores, tokens=rows)


# --------------------------------------------------------------------------- bucketing

def bucket(idx: np.ndarray, n_experts: int):
    """Group (token, slot) pairs by expert, stably by (expert, token, slot).

    Returns counts [E], offsets [E+1] (exclusive scan), perm [N*k] (flat slot id t*k+j at
    each bucketed position) and rowof [N*k] (bucketed position of each flat slot id).
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=n_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm = np.argsort(flat, kind="stable")
    rowof = np.empty_like(perm)
    rowof[perm] = np.arange(perm.size)
    return counts, offsets, perm, rowof


def expected_distinct(n_experts: int, k: int, batch: int) -> float:
    """Expected number of distinct experts touched by `batch` tokens that each pick a
    uniformly random k-subset: E * (1 - (1 - k/E)^B)."""
    return n_experts * (1.0 - (1.0 - k / n_experts) ** batch)


def imbalance_bound(n_experts: int, k: int, batch: int) -> float:
    """Per-rank byte imbalance bound E / distinct - 1 (arc PR #89, "A correction to
    wave44-BV section 3.2": above E/N coverage the rank count cancels)."""
    return n_experts / expected_distinct(n_experts, k, batch) - 1.0
