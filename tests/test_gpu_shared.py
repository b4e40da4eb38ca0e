"""Shared expert beside the routed experts: GPU path vs the fp64 oracle (needs a B300).

Standard layer (moe_forward_shared) and LatentMoE (latent_moe_shared, shared expert in H),
compared in full on seeded inputs, with the bf16 output bars: relative Frobenius error
<= 1e-2 and max |err| <= 3e-2 * rms(oracle).
"""
import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle as O
from helpers import assert_close, bf16_out, check_selection, to_dev

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


@pytest.mark.parametrize("T,H,E,k,F,Fs", [(256, 256, 16, 2, 128, 256), (513, 512, 32, 4, 192, 128),
                                          (40, 320, 8, 2, 64, 192),
                                          (64, 2688, 128, 6, 1856, 1856)])
def test_layer_shared(moe, T, H, E, k, F, Fs):
    w = moe_synth.Workload("shared", T=T, H=H, E=E, k=k, F=F, seed=T + H + 7)
    inp = moe_synth.layer_inputs(w)
    inp.update(moe_synth.shared_expert_inputs(w, Fs))
    d = {key: to_dev(v) for key, v in inp.items()}
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    y = moe.moe_forward_shared(d["x"], d["w_router"], d["bias"], d["w_up"], d["w_down"],
                               d["w_up_shared"], d["w_down_shared"], k, topk_idx_out=idx)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = O.moe_layer_shared(inp["x"], inp["w_router"], inp["bias"], inp["w_up"], inp["w_down"],
                             inp["w_up_shared"], inp["w_down_shared"], k)
    same = check_selection(idx.cpu().numpy(), ref, inp["bias"], k)
    assert_close(bf16_out(y)[same], ref["y"][same], f"shared layer T={T}")


@pytest.mark.parametrize("router_on_latent", [True, False])
@pytest.mark.parametrize("T", [300, 40])       # rows-as-M and weights-as-M output projections
def test_latent_shared(moe, router_on_latent, T):
    w = moe_synth.Workload("latent_shared", T=T, H=512, E=32, k=8, F=128, seed=11 + T,
                           latent=128, router_on_latent=router_on_latent)
    Fs = 256
    inp = moe_synth.layer_inputs(w)
    inp.update(moe_synth.shared_expert_inputs(w, Fs))
    d = {key: to_dev(v) for key, v in inp.items()}
    idx = torch.empty((T, w.k), dtype=torch.int32, device="cuda")
    y = moe.latent_moe_shared(d["x"], d["w_in"], d["w_out"], d["w_router"], d["bias"],
                              d["w_up"], d["w_down"], d["w_up_shared"], d["w_down_shared"], w.k,
                              router_on_latent=router_on_latent, topk_idx_out=idx)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = O.latent_moe_shared(inp["x"], inp["w_in"], inp["w_out"], inp["w_router"], inp["bias"],
                              inp["w_up"], inp["w_down"], inp["w_up_shared"],
                              inp["w_down_shared"], w.k, router_on_latent)
    same = check_selection(idx.cpu().numpy(), ref, inp["bias"], w.k)
    assert_close(bf16_out(y)[same], ref["y"][same], f"latent shared T={T}")
