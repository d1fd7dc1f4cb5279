"""The routing entry point for callers that cannot allocate device memory (an engine with a
fixed, pre-carved memory pool, a plugin whose host owns the budget, a latency-critical path
where cudaMalloc may synchronise the device). It must give the same routes and weights as the
routing inside the handle-based forward, call after call, while its scratch lives in a static
device array. Kept in its own file so that pytest collects it last."""
import numpy as np
import pytest

import synthetic
import moe_gpu
from quantized_moe_gb300 import ds4moe as api

pytestmark = pytest.mark.gpu

SPEC = synthetic.Spec("noalloc-route", d=1024, n_experts=64, top_k=6, f=256, f_shared=256, n_shared=1,
                      fmt_gate_up="q2_k", fmt_down="q2_k", fmt_shared="q8_0", n_tokens=48, seed=31,
                      bias="normal")


def test_route_noalloc_matches_handle_forward_twice():
    import torch

    p = synthetic.make_problem(SPEC)
    h = moe_gpu.create(p)
    wr = torch.from_numpy(p.router_w).cuda()
    wb = torch.from_numpy(p.router_b).cuda()
    idx = torch.empty((SPEC.n_tokens, SPEC.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((SPEC.n_tokens, SPEC.top_k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    try:
        for call in range(2):  # two calls in a row, on different tokens
            xb = synthetic.activations(SPEC.with_(seed=SPEC.seed + call))
            _, idx_ref, w_ref = moe_gpu.forward(h, p, x_bits=xb)
            x = torch.from_numpy(xb.view(np.int16)).cuda()
            idx.fill_(-1)
            w.fill_(-1.0)
            api.ds4moe_route_noalloc(wr.data_ptr(), wb.data_ptr(), x.data_ptr(), SPEC.n_tokens, SPEC.d,
                                     SPEC.n_experts, SPEC.top_k, idx.data_ptr(), w.data_ptr(), stream)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
            np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=0)
    finally:
        api.ds4moe_destroy(h)


def test_route_noalloc_rejects_sizes_beyond_its_static_scratch():
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_route_noalloc(16, None, 16, api.DS4MOE_NOALLOC_MAX_LOGITS // 64 + 1, 1024, 64, 6, 16, 16)
    assert ei.value.code == api.DS4MOE_ERR_CAPACITY
    assert "static scratch" in api.ds4moe_last_error()
