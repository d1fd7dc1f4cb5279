"""Plants plausible mistakes in the oracle (on the CPU, via monkeypatch) and checks that
the pins catch each one: a dropped term, swapped nibbles, a wrong bit order, a wrong
sign, a wrong tie rule, a dropped weight, a transposed operand."""
import numpy as np
import pytest

import synthetic
from oracle import moe
import test_oracle_formats as tf
import test_oracle_layer as tl
import test_oracle_router as tr

_orig_q2k = moe.dequant_q2_k
_orig_q8 = moe.dequant_q8_0
_orig_topk = moe.select_topk


def _q2k_variant(drop_min=False, swap_nibbles=False, reverse_bits=False):
    def dq(row_bytes, k):
        rb = np.asarray(row_bytes, dtype=np.uint8)
        rows = rb.reshape(-1, rb.shape[-1]).shape[0]
        nb = k // 256
        blk = rb.reshape(rows, nb, 84).copy()
        if swap_nibbles:
            blk[:, :, :16] = ((blk[:, :, :16] & 0x0F) << 4) | (blk[:, :, :16] >> 4)
        if reverse_bits:
            q = blk[:, :, 16:80]
            r = np.zeros_like(q)
            for i in range(4):
                r |= ((q >> (2 * i)) & 3) << (6 - 2 * i)
            blk[:, :, 16:80] = r
        w = _orig_q2k(blk.reshape(rows, -1), k)
        if drop_min:
            m = (blk[:, :, 0:16] >> 4).astype(np.float64)
            dmin = blk[:, :, 82:84].copy().view("<f2")[..., 0].astype(np.float64)
            w = w + (dmin[:, :, None] * m[:, :, np.arange(256) // 16]).reshape(rows, k)
        return w
    return dq


def _q8_unsigned(row_bytes, k):
    rb = np.asarray(row_bytes, dtype=np.uint8)
    rows = rb.reshape(-1, rb.shape[-1]).shape[0]
    blk = rb.reshape(rows, k // 32, 34)
    scale = blk[:, :, 0:2].copy().view("<f2")[..., 0].astype(np.float64)
    return (scale[:, :, None] * blk[:, :, 2:].astype(np.float64)).reshape(rows, k)


def _topk_high_index_wins(scores, k):
    n, e = scores.shape
    rev = scores[:, ::-1]
    idx, w, margin = _orig_topk(rev, k)
    return e - 1 - idx, w, margin


def _topk_no_renorm(scores, k):
    idx, w, margin = _orig_topk(scores, k)
    return idx, np.take_along_axis(scores, idx, 1), margin


def _ffn_gate_for_up(x, wg, wu, wd):
    g = x @ wg.T
    return (moe.silu(g) * g) @ wd.T


def _silu_wrong_sign(g):
    return g / (1.0 + np.exp(g))


_orig_routed_sum = moe.routed_sum


def _routed_sum_unweighted(p, x, idx, w, owned=None):
    return _orig_routed_sum(p, x, idx, np.ones_like(w), owned)


_orig_scores = moe.router_scores


def _scores_no_bias(x, router_w, router_b):
    return _orig_scores(x, router_w, None)


MUTATIONS = {
    "q2k_drop_min": ("dequant_q2_k", _q2k_variant(drop_min=True)),
    "q2k_swap_nibbles": ("dequant_q2_k", _q2k_variant(swap_nibbles=True)),
    "q2k_reverse_bits": ("dequant_q2_k", _q2k_variant(reverse_bits=True)),
    "q8_unsigned": ("dequant_q8_0", _q8_unsigned),
    "tie_high_index": ("select_topk", _topk_high_index_wins),
    "no_renorm": ("select_topk", _topk_no_renorm),
    "gate_for_up": ("swiglu_ffn", _ffn_gate_for_up),
    "silu_sign": ("silu", _silu_wrong_sign),
    "unweighted_combine": ("routed_sum", _routed_sum_unweighted),
    "bias_ignored": ("router_scores", _scores_no_bias),
}

PINS = [
    tf.test_q8_0_hand_packed_block,
    lambda: tf.test_q2_k_hand_packed_blocks("A"),
    lambda: tf.test_q2_k_hand_packed_blocks("B"),
    tr.test_router_closed_form_fixture,
    tr.test_zero_router_ties_go_to_lower_index,
    tr.test_bias_only_router_is_argsort_of_bias,
    tl.test_one_hot_expert_closed_form,
    lambda: tl.test_numpy_oracle_matches_brute_force(synthetic.CONFIGS[0]),
    lambda: tl.test_numpy_oracle_matches_brute_force(tl.TINY_Q2K),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(moe, attr, fn)
    caught = []
    for i, pin in enumerate(PINS):
        try:
            pin()
        except AssertionError:
            caught.append(i)
    assert caught, f"no pin caught mutation {name}"
