"""Pure-Python brute force of the MoE layer forward on tiny inputs -- TEST INFRASTRUCTURE.

A second, independent restatement of the same definitions as the numpy oracle: it
decodes every weight from its bytes one at a time with integer operations and
``struct``, and runs every dot product as a Python loop over floats. It is used only
to pin the numpy oracle on small problems (a few hundred thousand multiply-adds).
"""
from __future__ import annotations

import math
import struct


def _half(lo: int, hi: int) -> float:
    return struct.unpack("<e", bytes((lo, hi)))[0]


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def decode_row(fmt: str, row: bytes, k: int) -> list:
    """One quantised row -> list of k Python floats."""
    out = []
    if fmt == "q8_0":
        for b in range(k // 32):
            blk = row[b * 34:(b + 1) * 34]
            scale = _half(blk[0], blk[1])
            for i in range(32):
                q = blk[2 + i]
                if q >= 128:
                    q -= 256
                out.append(scale * q)
    elif fmt == "q2_k":
        for b in range(k // 256):
            blk = row[b * 84:(b + 1) * 84]
            d = _half(blk[80], blk[81])
            dmin = _half(blk[82], blk[83])
            for i in range(256):
                j = i // 16
                s = blk[j] & 15
                m = blk[j] >> 4
                q = (blk[16 + i // 4] >> (2 * (i % 4))) & 3
                out.append(d * s * q - dmin * m)
    else:
        raise ValueError(fmt)
    return out


def decode_matrix(fmt: str, rows, k: int) -> list:
    return [decode_row(fmt, bytes(bytearray(r)), k) for r in rows]


def _dot(a, b) -> float:
    acc = 0.0
    for u, v in zip(a, b):
        acc += u * v
    return acc


def _ffn(x, wg, wu, wd):
    h = []
    for rg, ru in zip(wg, wu):
        g = _dot(rg, x)
        u = _dot(ru, x)
        h.append(g / (1.0 + math.exp(-g)) * u)
    return [_dot(rd, h) for rd in wd]


def forward(p, x_bits=None):
    """Full forward of a tiny synthetic problem; returns (out rows, idx rows, w rows)."""
    s = p.spec
    if x_bits is None:
        x_bits = p.x_bits
    xs = [[_bf16(b) for b in row] for row in x_bits]
    wr = [[float(v) for v in row] for row in p.router_w]
    bias = None if p.router_b is None else [float(v) for v in p.router_b]
    experts = {}
    out_rows, idx_rows, w_rows = [], [], []
    for t, x in enumerate(xs):
        if t < s.n_hash:
            chosen = [int(e) for e in p.hash_table[int(p.token_ids[t])][: s.top_k]]
            weights = [1.0 / s.top_k] * s.top_k
        else:
            scores = []
            for e in range(s.n_experts):
                z = _dot(wr[e], x) + (bias[e] if bias is not None else 0.0)
                scores.append(1.0 / (1.0 + math.exp(-z)))
            # repeated selection of the maximum; the first (lowest) index wins ties
            remaining = list(range(s.n_experts))
            chosen = []
            for _ in range(s.top_k):
                best = remaining[0]
                for e in remaining[1:]:
                    if scores[e] > scores[best]:
                        best = e
                chosen.append(best)
                remaining.remove(best)
            tot = sum(scores[e] for e in chosen)
            weights = [scores[e] / tot for e in chosen]
        y = [0.0] * s.d
        for e, wt in zip(chosen, weights):
            if e not in experts:
                experts[e] = (decode_matrix(s.fmt_gate_up, p.gate[e], s.d),
                              decode_matrix(s.fmt_gate_up, p.up[e], s.d),
                              decode_matrix(s.fmt_down, p.down[e], s.f))
            ye = _ffn(x, *experts[e])
            for i in range(s.d):
                y[i] += wt * ye[i]
        if s.n_shared:
            if "shared" not in experts:
                experts["shared"] = (decode_matrix(s.fmt_shared, p.shared_gate, s.d),
                                     decode_matrix(s.fmt_shared, p.shared_up, s.d),
                                     decode_matrix(s.fmt_shared, p.shared_down, s.f_shared))
            ys = _ffn(x, *experts["shared"])
            for i in range(s.d):
                y[i] += ys[i]
        out_rows.append(y)
        idx_rows.append(chosen)
        w_rows.append(weights)
    return out_rows, idx_rows, w_rows
