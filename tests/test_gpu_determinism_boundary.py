"""GPU: bitwise run-to-run determinism, placement invariance on the device, and the C-ABI
error paths that need a device (capacity, pointer checks, workspace cap, bad token ids)."""
import dataclasses

import numpy as np
import pytest

import synthetic
from oracle import moe
import moe_gpu
from quantized_moe_gb300 import ds4moe as api
from test_gpu_parity import SMALL_MIX

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("spec", [synthetic.CONFIGS[0], synthetic.CONFIGS[1], synthetic.CONFIGS[2],
                                  synthetic.CONFIGS[3], synthetic.CONFIGS[4], SMALL_MIX],
                         ids=lambda v: v.name)
def test_repeated_forwards_are_bitwise_identical(spec):
    """20 forwards of the same inputs give the same output, routes and weights bit for bit (the
    combine has a fixed order and no float atomics; prefill-4096 is the size at which an atomic
    down projection drifts)."""
    import torch

    reps = 20
    p = synthetic.make_problem(spec)
    h = moe_gpu.create(p)
    try:
        x = torch.from_numpy(np.ascontiguousarray(p.x_bits).view(np.int16)).cuda()
        tids = torch.from_numpy(p.token_ids).cuda() if spec.n_hash else None
        out = torch.empty((spec.n_tokens, spec.d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        first = idx0 = w0 = None
        for _ in range(reps):
            out.fill_(float("nan"))
            api.ds4moe_forward_ex(h, x.data_ptr(), spec.n_tokens, None if tids is None else tids.data_ptr(),
                                  spec.n_hash, out.data_ptr(), stream)
            torch.cuda.synchronize()
            idx, w = api.ds4moe_get_route(h, spec.n_tokens, spec.top_k)
            if first is None:
                first, idx0, w0 = out.view(torch.int32).clone(), idx, w
                assert bool(torch.isfinite(out).all())
            else:
                assert torch.equal(out.view(torch.int32), first)
                assert np.array_equal(idx, idx0) and np.array_equal(w.view(np.uint32), w0.view(np.uint32))
    finally:
        api.ds4moe_destroy(h)


def test_expert_placement_invariance_on_device():
    p = synthetic.make_problem(SMALL_MIX)
    perm = np.random.default_rng(9).permutation(SMALL_MIX.n_experts)
    inv = np.argsort(perm)
    st = lambda s: np.stack([s[int(inv[i])] for i in range(len(perm))])
    q = dataclasses.replace(p, router_w=p.router_w[inv], router_b=p.router_b[inv], gate=st(p.gate), up=st(p.up),
                            down=st(p.down), hash_table=perm[p.hash_table].astype(np.int32))
    ha, hb = moe_gpu.create(p), moe_gpu.create(q)
    try:
        a, ia, _ = moe_gpu.forward(ha, p)
        b, ib, _ = moe_gpu.forward(hb, q)
    finally:
        api.ds4moe_destroy(ha)
        api.ds4moe_destroy(hb)
    assert np.array_equal(np.sort(perm[ia], 1), np.sort(ib, 1))
    assert np.max(np.abs(a - b)) <= moe_gpu.tolerance(a)


def test_token_count_edges():
    p = synthetic.make_problem(SMALL_MIX)
    h = moe_gpu.create(p, max_tokens=64)
    try:
        import torch
        x = torch.zeros((1, SMALL_MIX.d), dtype=torch.int16, device="cuda")
        out = torch.zeros((1, SMALL_MIX.d), dtype=torch.float32, device="cuda")
        api.ds4moe_forward(h, x.data_ptr(), 0, out.data_ptr(), 0)  # n = 0 is a no-op
        with pytest.raises(api.Ds4MoeError) as ei:
            api.ds4moe_forward(h, x.data_ptr(), 65, out.data_ptr(), 0)
        assert ei.value.code == api.DS4MOE_ERR_CAPACITY
        host = np.zeros((1, SMALL_MIX.d), np.uint16)
        with pytest.raises(api.Ds4MoeError) as ei:
            api.ds4moe_forward(h, host, 1, out.data_ptr(), 0)
        assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG
        # all-zero activations: every learned score is 1/2, ties go to experts 0..k-1
        got, idx, w = moe_gpu.forward(h, p, x_bits=np.zeros((3, SMALL_MIX.d), np.uint16), n_hash=0)
        b = p.router_b.astype(np.float64)
        want = np.argsort(-b, kind="stable")[:SMALL_MIX.top_k]
        assert all(sorted(r) == sorted(want.tolist()) for r in idx.tolist())
        assert np.all(got == 0.0)  # zero input -> zero expert outputs
        # a single token and a token count that is not a multiple of the pass size
        for n in (1, 6, 8, 16, 17, 63):  # decode path below 8 tokens, the batched path from 8
            xb = synthetic.activations(SMALL_MIX, n)
            got, idx, _ = moe_gpu.forward(h, p, x_bits=xb, n_hash=min(n, 5))
            ref = moe.forward(p, x_bits=xb, n_hash=min(n, 5))
            assert np.max(np.abs(got - ref["out"])) <= moe_gpu.tolerance(ref["out"])
    finally:
        api.ds4moe_destroy(h)


def test_out_of_range_token_id_sets_error_flag():
    p = synthetic.make_problem(SMALL_MIX)
    h = moe_gpu.create(p)
    try:
        bad = p.token_ids.copy()
        bad[2] = SMALL_MIX.hash_vocab + 7
        got, idx, w = moe_gpu.forward(h, p, token_ids=bad)
        st = api.ds4moe_get_stats(h)
        assert st["error_flags"] & 1
        assert np.all(w[2] == 0)
        assert np.all(np.isfinite(got))
    finally:
        api.ds4moe_destroy(h)


def test_workspace_limit_reports_oom():
    p = synthetic.make_problem(SMALL_MIX)
    with pytest.raises(api.Ds4MoeError) as ei:
        moe_gpu.create(p, workspace_limit=1 << 20)
    assert ei.value.code == api.DS4MOE_ERR_OOM


def test_host_entry_point_matches_device_entry_point():
    p = synthetic.make_problem(SMALL_MIX)
    h = moe_gpu.create(p)
    try:
        dev, _, _ = moe_gpu.forward(h, p)
        out = np.zeros((SMALL_MIX.n_tokens, SMALL_MIX.d), np.float32)
        api.ds4moe_forward_host(h, np.ascontiguousarray(p.x_bits), SMALL_MIX.n_tokens,
                                np.ascontiguousarray(p.token_ids), SMALL_MIX.n_hash, out, 0)
        assert np.array_equal(out.view(np.uint32), dev.view(np.uint32))
    finally:
        api.ds4moe_destroy(h)


def test_host_entry_point_pinned_decode_graph_matches_device_entry_point():
    """Decode-sized forwards from page-locked host buffers run as one graph with the copies; the
    result equals the device entry point bitwise, on repeat and with other buffers."""
    import torch
    p = synthetic.make_problem(SMALL_MIX)
    h = moe_gpu.create(p)
    try:
        n, nh = 6, 2
        xb = np.ascontiguousarray(p.x_bits[:n])
        dev, _, _ = moe_gpu.forward(h, p, x_bits=xb, n_hash=nh)
        for _ in range(2):  # two sets of buffers, each used twice (capture, then replay)
            x_h = torch.from_numpy(xb.view(np.int16)).pin_memory()
            t_h = torch.from_numpy(np.ascontiguousarray(p.token_ids[:nh], dtype=np.int32)).pin_memory()
            o_h = torch.empty((n, SMALL_MIX.d), dtype=torch.float32).pin_memory()
            for _ in range(2):
                o_h.zero_()
                api.ds4moe_forward_host(h, x_h.data_ptr(), n, t_h.data_ptr(), nh, o_h.data_ptr(), 0)
                assert np.array_equal(o_h.numpy().view(np.uint32), dev.view(np.uint32))
    finally:
        api.ds4moe_destroy(h)


def test_table_entries_outside_the_expert_range_are_refused():
    p = synthetic.make_problem(SMALL_MIX)
    bad = p.hash_table.copy()
    bad[7, 1] = SMALL_MIX.n_experts
    with pytest.raises(api.Ds4MoeError) as ei:
        moe_gpu.create(dataclasses.replace(p, hash_table=bad))
    assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG


def test_graph_replay_matches_direct_launches(monkeypatch):
    """Decode forwards replay cached CUDA graphs; results must equal direct launches bitwise,
    also after the graph cache has been cycled through more distinct buffers than it keeps."""
    import torch

    spec = synthetic.CONFIGS[0]
    p = synthetic.make_problem(spec)
    monkeypatch.setenv("DS4MOE_NO_GRAPHS", "1")
    h_direct = moe_gpu.create(p)
    monkeypatch.delenv("DS4MOE_NO_GRAPHS")
    h_graph = moe_gpu.create(p)
    try:
        for rep in range(20):  # 20 distinct input buffers: more than the 16 cached graphs
            xb = synthetic.activations(spec.with_(seed=100 + rep))
            a, ia, _ = moe_gpu.forward(h_direct, p, x_bits=xb)
            b, ib, _ = moe_gpu.forward(h_graph, p, x_bits=xb)
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)) and np.array_equal(ia, ib)
        x = torch.from_numpy(p.x_bits.view(np.int16)).cuda()
        out = torch.empty((spec.n_tokens, spec.d), device="cuda")
        for _ in range(3):  # the same buffers: one cached graph replayed
            api.ds4moe_forward(h_graph, x.data_ptr(), spec.n_tokens, out.data_ptr(), 0)
        torch.cuda.synchronize()
        a, _, _ = moe_gpu.forward(h_direct, p)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), a.view(np.uint32))
    finally:
        api.ds4moe_destroy(h_direct)
        api.ds4moe_destroy(h_graph)


def test_q2k_scale_beyond_fp16_dequant_range_is_refused():
    """The batched path dequantizes Q2_K in fp16 (q * 2^-16 times 2^16 d s): a super-block
    scale d >= 1/15 would overflow, so create refuses it by name (decode-only handles accept it)."""
    p = synthetic.make_problem(SMALL_MIX)
    gate = np.stack([p.gate[e] for e in range(SMALL_MIX.n_experts)]).copy()
    blk = gate.reshape(SMALL_MIX.n_experts, SMALL_MIX.f, -1, 84)
    blk[3, 5, 1, 80:82] = np.frombuffer(np.float16(0.1).tobytes(), np.uint8)
    q = dataclasses.replace(p, gate=gate)
    with pytest.raises(api.Ds4MoeError) as ei:
        moe_gpu.create(q, max_tokens=64)
    assert ei.value.code == api.DS4MOE_ERR_UNSUPPORTED_FORMAT
    h = moe_gpu.create(q, max_tokens=4)  # decode path only: no fp16 dequant, accepted
    api.ds4moe_destroy(h)
    # up to 16 tokens the decode kernels can serve every forward: such a handle accepts the
    # weights too and keeps its 16-token forwards on the decode path
    h = moe_gpu.create(q, max_tokens=16)
    try:
        assert api.ds4moe_launches_per_forward(h, 16) == 3
    finally:
        api.ds4moe_destroy(h)


@pytest.mark.parametrize("batched_from", [None, "17"], ids=["default", "decode-up-to-16"])
def test_path_selection_and_the_decode_kernels_up_to_16_tokens(monkeypatch, batched_from):
    """Below 8 tokens a forward takes the decode path (3 launches), from 8 tokens the batched
    path (12); with DS4MOE_BATCHED_FROM=17 at create the decode kernels serve up to 16 tokens.
    Every token count matches the oracle either way."""
    if batched_from:
        monkeypatch.setenv("DS4MOE_BATCHED_FROM", batched_from)
    spec = synthetic.CONFIGS[2]  # decode-16: d=4096, 256 experts top-8
    p = synthetic.make_problem(spec)
    h = moe_gpu.create(p, max_tokens=16)
    ref = moe.forward(p)["out"]  # tokens are independent: a forward of the first n rows gives ref[:n]
    try:
        for n in (1, 7, 8, 16):
            want = 3 if (batched_from or n < 8) else 12
            assert api.ds4moe_launches_per_forward(h, n) == want, n
            xb = np.ascontiguousarray(p.x_bits[:n])
            got, _, _ = moe_gpu.forward(h, p, x_bits=xb, n_hash=min(n, spec.n_hash))
            assert np.max(np.abs(got - ref[:n])) <= moe_gpu.tolerance(ref[:n]), n
    finally:
        api.ds4moe_destroy(h)


def test_batched_forward_with_every_token_table_routed():
    """Whole-layer table routing (every token hash-routed, as in a model's first layers): the
    batched path runs without the router, and matches the oracle."""
    p = synthetic.make_problem(SMALL_MIX)
    n = 40  # above the decode limit: the batched path
    tids = np.random.default_rng(31).integers(0, SMALL_MIX.hash_vocab, n).astype(np.int32)
    xb = synthetic.activations(SMALL_MIX, n)
    h = moe_gpu.create(p, max_tokens=n)
    try:
        got, idx, w = moe_gpu.forward(h, p, x_bits=xb, n_hash=n, token_ids=tids)
        st = api.ds4moe_get_stats(h)
    finally:
        api.ds4moe_destroy(h)
    ref = moe.forward(p, x_bits=xb, token_ids=tids, n_hash=n)
    assert np.array_equal(idx, ref["idx"])
    assert np.all(w == np.float32(1.0 / SMALL_MIX.top_k))
    assert int(st["counts"].sum()) == n * SMALL_MIX.top_k and st["error_flags"] == 0
    assert np.max(np.abs(got - ref["out"])) <= moe_gpu.tolerance(ref["out"])


@pytest.mark.parametrize("n", [6, 40], ids=["decode", "batched"])
def test_forward_captured_in_the_callers_graph(n):
    """A forward is stream-ordered with no host synchronisation, so a caller can capture it in its
    own CUDA graph: replays on new inputs (written into the captured buffer) equal direct forwards
    bitwise, on the decode path and on the batched path."""
    import torch

    spec = SMALL_MIX.with_(n_tokens=n, n_hash=min(5, n))
    p = synthetic.make_problem(spec)
    h = moe_gpu.create(p, max_tokens=64)
    try:
        cap = torch.cuda.Stream()
        x = torch.empty((n, spec.d), dtype=torch.int16, device="cuda")
        tids = torch.from_numpy(np.ascontiguousarray(p.token_ids[:spec.n_hash])).cuda()
        out = torch.empty((n, spec.d), dtype=torch.float32, device="cuda")

        def run():
            api.ds4moe_forward_ex(h, x.data_ptr(), n, tids.data_ptr(), spec.n_hash, out.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)

        x.copy_(torch.from_numpy(synthetic.activations(spec.with_(seed=100)).view(np.int16)))
        with torch.cuda.stream(cap):
            run()  # warm-up outside the capture (first-use checks of the buffers)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            run()
        for seed in (101, 102):
            xb = synthetic.activations(spec.with_(seed=seed))
            x.copy_(torch.from_numpy(xb.view(np.int16)))
            out.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            want, _, _ = moe_gpu.forward(h, p, x_bits=xb)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), seed
    finally:
        api.ds4moe_destroy(h)
