"""The routing entry point for callers that cannot allocate device memory (an engine with a
fixed, pre-carved memory pool, a plugin whose host owns the budget, a latency-critical path
where cudaMalloc may synchronise the device). Its scratch lives in a static device array. On
two calls in a row it must give the fp64 oracle's routes (bit-exact expert sets except where the
oracle's k-th and (k+1)-th scores are within 1e-6) and the routes of the handle-based forward
under the same rule. Kept in its own file so that pytest collects it last."""
import numpy as np
import pytest

import synthetic
import moe_gpu
from oracle import moe
from quantized_moe_gb300 import ds4moe as api

pytestmark = pytest.mark.gpu

MARGIN = 1e-6

SPECS = [
    # the handle routes these 48 tokens on its batched path (tensor-core router)
    synthetic.Spec("noalloc-route", d=1024, n_experts=64, top_k=6, f=256, f_shared=256, n_shared=1,
                   fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0", n_tokens=48, seed=31, bias="normal"),
    # the full router shape (d=4096, 256 experts, top-8; 64 KB of staged activations per CTA, above
    # the default shared-memory limit) with 16 tokens: the handle routes them on its batched path
    # (fp32 FMA router below 33 tokens)
    synthetic.Spec("noalloc-ds-shape", d=4096, n_experts=256, top_k=8, f=256, f_shared=256, n_shared=1,
                   fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0", n_tokens=16, seed=32, bias="normal"),
]


def _same_sets_except_near_ties(idx, want, margin):
    for t in range(idx.shape[0]):
        if margin[t] > MARGIN:
            assert sorted(idx[t].tolist()) == sorted(want[t].tolist()), (t, idx[t], want[t])


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_route_noalloc_matches_oracle_and_handle_forward_twice(spec):
    import torch

    p = synthetic.make_problem(spec)
    h = moe_gpu.create(p)
    wr = torch.from_numpy(p.router_w).cuda()
    wb = torch.from_numpy(p.router_b).cuda()
    idx = torch.empty((spec.n_tokens, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((spec.n_tokens, spec.top_k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    try:
        for call in range(2):  # two calls in a row, on different tokens
            xb = synthetic.activations(spec.with_(seed=spec.seed + call))
            _, idx_fwd, w_fwd = moe_gpu.forward(h, p, x_bits=xb)
            ref_idx, _, margin, scores = moe.route(p, moe.bf16_bits_to_f64(xb))
            x = torch.from_numpy(xb.view(np.int16)).cuda()
            idx.fill_(-1)
            w.fill_(-1.0)
            api.ds4moe_route_noalloc(wr.data_ptr(), wb.data_ptr(), x.data_ptr(), spec.n_tokens, spec.d,
                                     spec.n_experts, spec.top_k, idx.data_ptr(), w.data_ptr(), stream)
            torch.cuda.synchronize()
            got_idx, got_w = idx.cpu().numpy(), w.cpu().numpy()
            # against the oracle: sets, score-descending order, weights renormalised from its scores
            _same_sets_except_near_ties(got_idx, ref_idx, margin)
            for t in range(spec.n_tokens):
                sc = scores[t, got_idx[t]]
                assert len(set(got_idx[t].tolist())) == spec.top_k
                assert np.all(np.diff(sc) <= MARGIN)
                np.testing.assert_allclose(got_w[t], sc / sc.sum(), rtol=2e-6, atol=1e-7)
            # against the handle's forward: the same rule, and equal weights wherever the sets agree
            _same_sets_except_near_ties(got_idx, idx_fwd, margin)
            for t in range(spec.n_tokens):
                if sorted(got_idx[t].tolist()) == sorted(idx_fwd[t].tolist()):
                    o1, o2 = np.argsort(got_idx[t]), np.argsort(idx_fwd[t])
                    np.testing.assert_allclose(got_w[t][o1], w_fwd[t][o2], rtol=2e-6, atol=1e-7)
    finally:
        api.ds4moe_destroy(h)


def test_route_noalloc_rejects_sizes_beyond_its_static_scratch():
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_route_noalloc(16, None, 16, api.DS4MOE_NOALLOC_MAX_LOGITS // 64 + 1, 1024, 64, 6, 16, 16)
    assert ei.value.code == api.DS4MOE_ERR_CAPACITY
    assert "static scratch" in api.ds4moe_last_error()
