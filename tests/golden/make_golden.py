"""Writes the hand-packed block and router fixtures in this folder.

Every expected value here comes from the closed form of the format or of the sigmoid,
evaluated on the integer fields the fixture packs; nothing is computed by the oracle's
decoders or by the CUDA library. Run: python tests/golden/make_golden.py
"""
from __future__ import annotations

import math
import os
import struct

HERE = os.path.dirname(os.path.abspath(__file__))


def f16_bytes(v: float) -> bytes:
    return struct.pack("<e", v)


def q8_0_fixture() -> str:
    scale = 0.5  # exact in fp16
    q = [-127, -100, -64, -33, -8, -2, -1, 0, 1, 2, 3, 5, 8, 13, 21, 34,
         55, 89, 127, 126, 64, 32, 16, 4, -4, -16, -32, -126, 100, 77, -77, 0]
    blk = f16_bytes(scale) + bytes((v & 0xFF) for v in q)
    w = [scale * v for v in q]
    return ("# Q8_0 block (34 bytes): fp16 scale 0.5 then 32 int8; expected w = 0.5 * q\n"
            "# Format named in ds4 PR #754 'CUDA: add DGX Spark network expert/tensor\n"
            "# parallelism', section 'Supported paths and safety' (Q8_0 shared/attention).\n"
            f"bytes {blk.hex()}\n"
            "w " + " ".join(repr(v) for v in w) + "\n")


def q2_k_fixture(d: float, dmin: float, qpat) -> tuple[bytes, list]:
    s = list(range(16))           # s_j = j
    m = [15 - j for j in range(16)]  # m_j = 15 - j
    scales = bytes((s[j] | (m[j] << 4)) for j in range(16))
    q = [qpat(i) for i in range(256)]
    qs = bytearray(64)
    for i, v in enumerate(q):
        qs[i >> 2] |= (v & 3) << (2 * (i & 3))
    blk = scales + bytes(qs) + f16_bytes(d) + f16_bytes(dmin)
    w = [d * s[i // 16] * q[i] - dmin * m[i // 16] for i in range(256)]
    return blk, w


def q2_k_text() -> str:
    lines = ["# Q2_K super-blocks (84 bytes): 16 scale bytes (low nibble s_j = j, high nibble",
             "# m_j = 15 - j), 64 quant bytes (weight i at byte i>>2, bits 2*(i&3)), fp16 d, fp16 dmin.",
             "# Expected w_i = d*s_j*q_i - dmin*m_j with j = i // 16, evaluated on the packed integers.",
             "# Format named in ds4 PR #754, section 'Supported paths and safety' (Q2_K routed down).",
             "# Block A enumerates every (s, q) pair: q_i = (i + i // 16) % 4 with d = dmin = 1.",
             "# Block B uses d = 0.5, dmin = 0.25 and q_i = (7 * i) % 4."]
    for name, d, dmin, pat in (("A", 1.0, 1.0, lambda i: (i + i // 16) % 4),
                               ("B", 0.5, 0.25, lambda i: (7 * i) % 4)):
        blk, w = q2_k_fixture(d, dmin, pat)
        lines.append(f"bytes{name} {blk.hex()}")
        lines.append(f"w{name} " + " ".join(repr(v) for v in w))
    return "\n".join(lines) + "\n"


def router_text() -> str:
    # one token x = (1, 0); logits are W_r[:, 0]; sigmoid(ln a) = a / (1 + a)
    ln = [0.0, math.log(3.0), -math.log(3.0), math.log(9.0)]
    w32 = [struct.unpack("<f", struct.pack("<f", v))[0] for v in ln]  # fp32 weights
    scores = [1.0 / (1.0 + math.exp(-v)) for v in w32]
    # exact targets: 1/2, 3/4, 1/4, 9/10 (to ~1e-8 after fp32 rounding of the logs)
    top = [3, 1]
    tot = scores[3] + scores[1]
    return ("# Router: 4 experts, d = 2, one token x = (1, 0) (bf16 exact), no bias.\n"
            "# W_r[:, 0] = (0, ln 3, -ln 3, ln 9) rounded to fp32, W_r[:, 1] = 0.\n"
            "# sigmoid(ln a) = a / (1 + a): scores 1/2, 3/4, 1/4, 9/10; top-2 = experts 3, 1;\n"
            "# weights 0.9 / 1.65 and 0.75 / 1.65 (tolerance 1e-7 for the fp32 logs).\n"
            "wr_col0 " + " ".join(struct.pack("<f", v).hex() for v in ln) + "\n"
            "scores 0.5 0.75 0.25 0.9\n"
            f"top2 {top[0]} {top[1]}\n"
            f"w {0.9 / 1.65!r} {0.75 / 1.65!r}\n")


def main() -> None:
    with open(os.path.join(HERE, "q8_0_block.txt"), "w") as fh:
        fh.write(q8_0_fixture())
    with open(os.path.join(HERE, "q2_k_blocks.txt"), "w") as fh:
        fh.write(q2_k_text())
    with open(os.path.join(HERE, "router_small.txt"), "w") as fh:
        fh.write(router_text())


if __name__ == "__main__":
    main()
