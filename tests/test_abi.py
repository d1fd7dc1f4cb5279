"""CPU: the C-ABI library builds, loads, exports every function the header declares, and
rejects bad arguments on the host before touching a device."""
import os
import re

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def api():
    from quantized_moe_gb300 import build as b
    b.build()
    from quantized_moe_gb300 import ds4moe
    return ds4moe


def _declared():
    src = open(os.path.join(ROOT, "include", "ds4moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4moe_\w+)\s*\(", src)))


def test_every_declared_function_is_exported(api):
    lib = api.lib()
    names = _declared()
    assert "ds4moe_create" in names and "ds4moe_forward" in names and "ds4moe_destroy" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(api.EXPORTED)


def test_last_error_and_null_arguments(api):
    lib = api.lib()
    assert lib.ds4moe_create(None, None, None) == api.DS4MOE_ERR_INVALID_ARG
    assert "NULL" in api.ds4moe_last_error()
    assert lib.ds4moe_forward(None, None, 1, None, None) == api.DS4MOE_ERR_INVALID_ARG
    api.ds4moe_destroy(None)  # NULL-safe


def _shapes(api, **kw):
    base = dict(d=512, f_routed=256, f_shared=256, n_experts=8, top_k=2, n_shared=1, fmt_gate_up="q2_k",
                fmt_down="q2_k", fmt_shared="q8_0", has_bias=False, hash_vocab=0, max_tokens=16)
    base.update(kw)
    return api.make_shapes(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(d=100), -1), (dict(d=12800), -1), (dict(f_routed=0), -1), (dict(n_experts=300), -1), (dict(top_k=9, n_experts=8), -1),
    (dict(max_tokens=0), -1), (dict(n_shared=2), -1), (dict(fmt_gate_up=7), -2), (dict(fmt_down=-1), -2),
    (dict(d=384), -2),  # Q2_K needs K a multiple of 256
])
def test_create_rejects_bad_shapes_on_host(api, kw, code):
    w = np.zeros(16, np.float32)
    weights = api.make_weights(w, None, w, w, w, w, w, w)
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_create(weights, _shapes(api, **kw))
    assert ei.value.code == code
    assert api.ds4moe_last_error()


def test_create_requires_shared_tensors_and_bias(api):
    w = np.zeros(16, np.float32)
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_create(api.make_weights(w, None, w, w, w), _shapes(api))
    assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_create(api.make_weights(w, None, w, w, w, w, w, w), _shapes(api, has_bias=True))
    assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("owned,msg", [([], "n_owned"), (list(range(9)), "n_owned"), ([0, 8], "outside"),
                                       ([-1], "outside"), ([3, 1, 3], "twice")])
def test_create_subset_rejects_bad_expert_lists_on_host(api, owned, msg):
    """An expert subset names 1..n_experts distinct ids in range; refused before any device work."""
    w = np.zeros(16, np.float32)
    weights = api.make_weights(w, None, w, w, w, w, w, w)
    with pytest.raises(api.Ds4MoeError) as ei:
        api.ds4moe_create_subset(weights, _shapes(api), owned, True)
    assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG
    assert msg in api.ds4moe_last_error()


def test_create_subset_null_list(api):
    lib = api.lib()
    w = np.zeros(16, np.float32)
    weights = api.make_weights(w, None, w, w, w, w, w, w)
    import ctypes
    h = ctypes.c_void_p()
    assert lib.ds4moe_create_subset(ctypes.byref(weights), ctypes.byref(_shapes(api)), None, 2, 1,
                                    ctypes.byref(h)) == api.DS4MOE_ERR_INVALID_ARG
    assert "owned is NULL" in api.ds4moe_last_error()
