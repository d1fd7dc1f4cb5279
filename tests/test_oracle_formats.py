"""Pins for the oracle's block decoders: hand-packed blocks with closed-form values,
the nibble order, and agreement with the independent pure-Python decoder."""
import numpy as np
import pytest

import synthetic
from oracle import brute, moe
from conftest import read_fixture


def test_q8_0_hand_packed_block():
    fx = read_fixture("q8_0_block.txt")
    blk = np.frombuffer(bytes.fromhex(fx["bytes"]), dtype=np.uint8)
    want = np.array([float(v) for v in fx["w"].split()])
    got = moe.dequant_q8_0(blk[None, :], 32)[0]
    np.testing.assert_array_equal(got, want)


def test_q8_0_unit_scale_is_identity():
    # scale 1.0 (fp16 0x3C00): w = q for every int8 value in [-127, 127]
    q = np.arange(-127, 128, dtype=np.int8)
    q = np.concatenate([q, np.zeros(256 - q.size, np.int8)])  # 8 blocks of 32
    rows = []
    for b in range(8):
        rows.append(np.concatenate([np.array([0x00, 0x3C], np.uint8), q[b * 32:(b + 1) * 32].view(np.uint8)]))
    row = np.concatenate(rows)
    np.testing.assert_array_equal(moe.dequant_q8_0(row[None, :], 256)[0], q.astype(np.float64))


@pytest.mark.parametrize("name", ["A", "B"])
def test_q2_k_hand_packed_blocks(name):
    fx = read_fixture("q2_k_blocks.txt")
    blk = np.frombuffer(bytes.fromhex(fx["bytes" + name]), dtype=np.uint8)
    want = np.array([float(v) for v in fx["w" + name].split()])
    got = moe.dequant_q2_k(blk[None, :], 256)[0]
    np.testing.assert_array_equal(got, want)


def test_q2_k_block_a_covers_every_scale_quant_pair():
    # block A: d = dmin = 1, s_j = j, m_j = 15 - j, so w = j*q - (15 - j); all 64 (j, q) pairs occur
    fx = read_fixture("q2_k_blocks.txt")
    blk = np.frombuffer(bytes.fromhex(fx["bytesA"]), dtype=np.uint8)
    w = moe.dequant_q2_k(blk[None, :], 256)[0]
    seen = set()
    for i in range(256):
        j = i // 16
        q = (w[i] + (15 - j)) / j if j else None
        if j:
            assert q == int(q) and 0 <= q <= 3
            seen.add((j, int(q)))
        else:
            assert w[i] == -15.0
    assert len(seen) == 15 * 4


def test_q2_k_nibble_order_matters():
    fx = read_fixture("q2_k_blocks.txt")
    blk = np.frombuffer(bytes.fromhex(fx["bytesA"]), dtype=np.uint8).copy()
    base = moe.dequant_q2_k(blk[None, :], 256)[0]
    sw = blk.copy()
    sw[:16] = ((blk[:16] & 0x0F) << 4) | (blk[:16] >> 4)
    assert not np.array_equal(moe.dequant_q2_k(sw[None, :], 256)[0], base)


@pytest.mark.parametrize("fmt,k", [("q8_0", 128), ("q2_k", 512)])
def test_decoders_match_pure_python(fmt, k):
    t = synthetic.quant_tensor(fmt, 5, k, 123, 99, 0)
    got = moe.dequant(fmt, t, k)
    want = np.array(brute.decode_matrix(fmt, t, k))
    np.testing.assert_array_equal(got, want)


def test_generator_value_ranges():
    t = synthetic.quant_tensor("q2_k", 64, 1024, 7, 3, 0).reshape(64, 4, 84)
    d = t[:, :, 80:82].copy().view("<f2").astype(np.float64)
    assert d.min() >= 1e-3 - 1e-6 and d.max() <= 4e-3 + 1e-6
    t8 = synthetic.quant_tensor("q8_0", 64, 256, 7, 3, 0).reshape(64, 8, 34)
    q = t8[:, :, 2:].view(np.int8)
    assert q.min() >= -127 and q.max() <= 127
    sc = t8[:, :, 0:2].copy().view("<f2").astype(np.float64)
    assert sc.min() >= 0.5e-3 - 1e-6 and sc.max() <= 2e-3 + 1e-6
