"""The MOE_DEBUG build, libmoe_debug.so, on the GPU (needs a B300).

That build adds a 256-byte guard region after every workspace slice, filled before each call's
first kernel and checked after its last one, and device-side range checks of indices the
library produced itself; all of them report on the device status word. A child process loads
it (MOE_DEBUG=1) and runs small calls through every workspace-taking entry point: every call
must leave the status word clear (no guard damaged, no index out of range), and every output
must equal the release library's bit for bit, since the checks must not change results. The
detector itself is checked by damaging one guard byte from the host (cudaMemsetAsync, not a
kernel), which must be reported as MOE_ERR_WORKSPACE.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))
MOE_ERR_WORKSPACE = 3


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


def test_debug_build_matches_release(moe, tmp_path):
    out = tmp_path / "debug_outputs.npz"
    env = dict(os.environ, MOE_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_calls.py"), str(out)],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    dbg = np.load(out)
    assert int(dbg["debug_build"][0]) == 1, "the child did not load libmoe_debug.so"
    assert moe.lib().moe_debug_build() == 0
    import debug_build_calls
    rel = debug_build_calls.run_calls(moe)
    assert set(rel) == set(dbg.files) - {"debug_build"}
    for name, a in rel.items():
        assert np.array_equal(a, dbg[name]), f"{name}: the debug build gives other results"


def test_debug_guard_detector(moe, tmp_path):
    """In the debug build, a damaged guard is reported (checked in a child process)."""
    code = (
        "import torch, ctypes, sparse_mixture_experts_57_b300 as m\n"
        "L = m.lib(); assert L.moe_debug_build() == 1\n"
        "ws = torch.zeros(16384, dtype=torch.uint8, device='cuda')\n"
        "assert m.get_device_status() == 0\n"
        "assert L.moe_debug_guard_selftest(ws.data_ptr(), ws.numel(),"
        " torch.cuda.current_stream().cuda_stream) == 0\n"
        "torch.cuda.synchronize()\n"
        f"assert m.get_device_status() == {MOE_ERR_WORKSPACE}\n"
        "assert m.get_device_status() == 0\n"
        "print('ok')\n")
    env = dict(os.environ, MOE_DEBUG="1", PYTHONPATH=os.path.dirname(HERE))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
    # the release build has no guards
    ws = torch.zeros(16384, dtype=torch.uint8, device="cuda")
    assert moe.lib().moe_debug_guard_selftest(ws.data_ptr(), ws.numel(),
                                              torch.cuda.current_stream().cuda_stream) == 2
