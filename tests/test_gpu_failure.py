"""Failure detection on the GPU without a fault (needs a B300).

Every pipeline wait in the library's tensor-core kernels is bounded. When one gives up, the
kernel records MOE_ERR_TIMEOUT on the device status word, stops the CTA's other roles through
an abort flag, waits for its copies in flight and releases its tensor memory. The self-test
entry point builds that situation on purpose: a wait on a barrier that nothing arrives on,
with a 1 ms limit. No trap, no unbounded wait, no bad address: the kernel returns, and the
GPU stays usable, which the grouped GEMM run afterwards on every SM checks (it allocates
tensor memory on each SM, which would wait forever if the self-test had kept its own).
"""
import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle as O
from helpers import assert_close, bf16_out, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


def _grouped_ffn_check(moe):
    counts, H, F = [300, 0, 1, 129, 57, 200], 256, 128
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off[-1])
    xp = moe_synth.normal_bf16(11, 50, (rows, H), 1.0)
    wu = moe_synth.expert_stack(11, moe_synth.TAG_UP, E, F, H)
    wd = moe_synth.expert_stack(11, moe_synth.TAG_DOWN, E, H, F)
    y = moe.moe_grouped_ffn(to_dev(xp), to_dev(off), to_dev(wu), to_dev(wd))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    assert_close(bf16_out(y), O.grouped_ffn(xp, off, wu, wd), "grouped ffn after the self-test")


@pytest.mark.parametrize("limit_us", [1000, 200])
def test_bounded_wait_gives_up_and_releases(moe, limit_us):
    L = moe.lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = 2 * sms
    src = torch.arange(4096, dtype=torch.int32, device="cuda").to(torch.uint8)
    report = torch.full((blocks * 8,), -1, dtype=torch.int32, device="cuda")
    assert moe.get_device_status() == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert L.moe_selftest_wait_timeout(src.data_ptr(), limit_us, blocks, report.data_ptr(),
                                       stream) == 0
    torch.cuda.synchronize()
    # the timeout is reported on the status word, and reading it clears it
    assert moe.get_device_status() == MOE_ERR_TIMEOUT
    assert moe.get_device_status() == 0
    rep = report.view(blocks, 8).cpu().numpy()
    assert (rep[:, 0] == 1).all(), "every producer wait gave up"
    assert (rep[:, 1] == 1).all(), "every MMA role left through the abort flag"
    assert (rep[:, 2] == 1).all(), "every epilogue role left through the abort flag"
    assert (rep[:, 3] == 1).all(), "every copy in flight landed before its CTA exited"
    # the hand-off cut the other roles' 2 s limit short: each CTA ended soon after its limit
    assert rep[:, 4].min() >= limit_us * 0.9
    assert rep[:, 4].max() < limit_us + 50_000, rep[:, 4].max()
    # tensor memory was released and the context is intact: a GEMM on every SM still works
    _grouped_ffn_check(moe)


def test_selftest_rejects_bad_arguments(moe):
    L = moe.lib()
    src = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    rep = torch.zeros(64, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.moe_selftest_wait_timeout(None, 1000, 8, rep.data_ptr(), s) == 1
    assert L.moe_selftest_wait_timeout(src.data_ptr(), 0, 8, rep.data_ptr(), s) == 1
    assert L.moe_selftest_wait_timeout(src.data_ptr(), 1000, 0, rep.data_ptr(), s) == 1
    assert L.moe_selftest_wait_timeout(src.data_ptr() + 4, 1000, 8, rep.data_ptr(), s) == 2
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
