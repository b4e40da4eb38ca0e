"""The profiling hook moe_set_profile_events on the GPU (needs a B300).

The hook records caller-owned events around the expert up- and down-projection GEMMs of
the layer calls. The brackets must be in stream order, lie inside the call, and leave the
results unchanged; turning the hook off stops the recording.
"""
import ctypes

import numpy as np
import pytest

import moe_synth
from helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


def _events(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()   # creates the CUDA event behind the handle
    return evs


@pytest.mark.parametrize("T", [64, 2048])
def test_hook_brackets_the_expert_gemms(moe, T):
    w = moe_synth.Workload("hook", T=T, H=512, E=16, k=2, F=256, seed=T)
    d = {key: to_dev(v) for key, v in moe_synth.layer_inputs(w).items()}
    L = moe.lib()
    y0 = moe.moe_forward(d["x"], d["w_router"], d["bias"], d["w_up"], d["w_down"], w.k)
    start, end = _events(2)
    hook = _events(4)
    handles = (ctypes.c_void_p * 4)(*[e.cuda_event for e in hook])
    torch.cuda.synchronize()
    assert L.moe_set_profile_events(handles, 4) == 0
    start.record()
    y1 = moe.moe_forward(d["x"], d["w_router"], d["bias"], d["w_up"], d["w_down"], w.k)
    end.record()
    assert L.moe_set_profile_events(None, 0) == 0
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    t = [start.elapsed_time(e) for e in hook] + [start.elapsed_time(end)]
    assert all(t[i] <= t[i + 1] for i in range(4)), t
    assert t[0] > 0 and t[1] > t[0] and t[3] > t[2]
    # off: a further call does not record the events again
    stamp = start.elapsed_time(hook[3])
    moe.moe_forward(d["x"], d["w_router"], d["bias"], d["w_up"], d["w_down"], w.k)
    torch.cuda.synchronize()
    assert start.elapsed_time(hook[3]) == stamp


def test_hook_rejects_bad_arguments(moe):
    L = moe.lib()
    assert L.moe_set_profile_events(None, 4) == 1
    assert L.moe_set_profile_events((ctypes.c_void_p * 4)(0, 0, 0, 0), 4) == 1
    assert L.moe_set_profile_events(None, 3) == 1
    assert L.moe_set_profile_events(None, 0) == 0
