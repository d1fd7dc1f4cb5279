"""Test-side helpers: create a library handle from a synthetic problem and run forwards
through the C ABI with torch-owned device buffers."""
from __future__ import annotations

import numpy as np

import synthetic
from quantized_moe_gb300 import ds4moe as api


def create(p: synthetic.Problem, max_tokens: int | None = None, device: int = 0, workspace_limit: int = 0,
           owned=None, include_shared: bool = True):
    """A handle for the problem; with `owned`, one holding only those routed experts."""
    s = p.spec
    shapes = api.make_shapes(s.d, s.f, s.f_shared, s.n_experts, s.top_k, s.n_shared, s.fmt_gate_up, s.fmt_down,
                             s.fmt_shared, p.router_b is not None, s.hash_vocab,
                             max_tokens or s.n_tokens, device, workspace_limit)
    keep = [p.router_w, p.router_b, p.gate.full() if hasattr(p.gate, "full") else p.gate,
            p.up.full() if hasattr(p.up, "full") else p.up, p.down.full() if hasattr(p.down, "full") else p.down,
            p.shared_gate, p.shared_up, p.shared_down, p.hash_table]
    keep = [None if a is None else np.ascontiguousarray(a) for a in keep]
    weights = api.make_weights(*keep)
    if owned is not None:
        return api.ds4moe_create_subset(weights, shapes, owned, include_shared)
    return api.ds4moe_create(weights, shapes)


def forward(h: int, p: synthetic.Problem, x_bits: np.ndarray | None = None, n_hash: int | None = None,
            token_ids: np.ndarray | None = None):
    """Runs one forward on the current torch stream; returns (out fp32 [N, d], idx, w)."""
    import torch

    s = p.spec
    xb = p.x_bits if x_bits is None else x_bits
    n = xb.shape[0]
    nh = min(s.n_hash if n_hash is None else n_hash, n)
    tid = p.token_ids if token_ids is None else token_ids
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda()
    out = torch.empty((n, s.d), dtype=torch.float32, device="cuda")
    tids = torch.from_numpy(np.ascontiguousarray(tid[:nh], dtype=np.int32)).cuda() if nh else None
    stream = torch.cuda.current_stream().cuda_stream
    api.ds4moe_forward_ex(h, x.data_ptr(), n, None if tids is None else tids.data_ptr(), nh, out.data_ptr(), stream)
    torch.cuda.synchronize()
    idx, w = api.ds4moe_get_route(h, n, s.top_k)
    return out.cpu().numpy(), idx, w


def tolerance(ref_out: np.ndarray) -> float:
    """max |gpu - oracle| allowed: 2e-3 of the largest oracle magnitude plus 1e-5."""
    return 2e-3 * float(np.max(np.abs(ref_out))) + 1e-5
