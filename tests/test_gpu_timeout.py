"""GPU: the bounded waits of the batched expert GEMM end with an error status, not a hang. A test
hook withholds one dequant arrival in the first CTA of the routed gate/up GEMM and limits every
wait of that launch to about 1 ms: the waits that depend on that stage run out, the CTA unwinds
(its copies and issued MMAs finish, its tensor memory is freed) and error bit 2 plus the bits of
the waits that gave up appear in the stats. The context stays usable: the next forward is correct and clean."""
import numpy as np
import pytest

import synthetic
from oracle import moe
import moe_gpu
from quantized_moe_gb300 import ds4moe as api
from test_gpu_parity import SMALL_MIX

pytestmark = pytest.mark.gpu

WAIT_SITES = {17: "weight producer", 18: "activation producer", 19: "dequant (raw)", 20: "dequant (stage free)",
              21: "epilogue", 22: "MMA (accumulator free)", 23: "MMA (stage full)"}


@pytest.mark.parametrize("stage", [0, 2, 7])
def test_withheld_arrival_times_out_and_the_next_forward_is_clean(stage):
    p = synthetic.make_problem(SMALL_MIX)  # 37 tokens: the batched path; d = 512 gives 8 K stages per item
    h = moe_gpu.create(p)
    try:
        api.ds4moe_set_test_stall(h, stage)
        moe_gpu.forward(h, p)
        flags = api.ds4moe_get_stats(h)["error_flags"]
        sites = [name for bit, name in WAIT_SITES.items() if flags & (1 << bit)]
        print(f"stage {stage}: error flags {flags:#x}, waits that gave up: {sites}")
        assert flags & 4, f"no timeout recorded (flags {flags:#x})"
        # Every wait downstream of the withheld stage may run out (whichever started first gives up
        # first; the rest see the abort): the MMA's wait for the stage, the epilogue's wait for the
        # accumulator, and the waits for the stage slot to come free. Producer and dequant waits on
        # weights that did arrive must not be among them.
        downstream = (1 << 18) | (1 << 20) | (1 << 21) | (1 << 23)
        site_bits = flags & (0x7F << 17)
        assert site_bits and not (site_bits & ~downstream), f"unexpected waits gave up: {sites}"
        # the hook cleared itself; the context and the handle still work
        got, idx, w = moe_gpu.forward(h, p)
        assert api.ds4moe_get_stats(h)["error_flags"] == 0
        ref = moe.forward(p)
        assert np.max(np.abs(got - ref["out"])) <= moe_gpu.tolerance(ref["out"])
    finally:
        api.ds4moe_destroy(h)


def test_stall_hook_refuses_negative_stage():
    p = synthetic.make_problem(SMALL_MIX)
    h = moe_gpu.create(p)
    try:
        with pytest.raises(api.Ds4MoeError) as ei:
            api.ds4moe_set_test_stall(h, -1)
        assert ei.value.code == api.DS4MOE_ERR_INVALID_ARG
    finally:
        api.ds4moe_destroy(h)
