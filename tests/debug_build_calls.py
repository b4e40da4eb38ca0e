"""Small calls through every workspace-taking entry point, shared by the debug-build test.

run_calls() runs them with whichever library the package loaded (the release libmoe.so, or
libmoe_debug.so when MOE_DEBUG=1 was set before the first load), checks the device status
word after each call, and returns every output as numpy arrays. Run as a script it writes
them to the .npz file named on the command line.
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402

# (T, H, E, k, F): fused small-batch routing with weights-as-M FFNs; multi-kernel routing;
# CTA-pair FFN tiles with one-CTA tails
SHAPES = [(64, 256, 16, 2, 128), (300, 320, 24, 3, 192), (2048, 256, 8, 2, 128)]


def run_calls(moe) -> dict:
    import torch

    out = {}

    def done(name, *tensors):
        torch.cuda.synchronize()
        st = moe.get_device_status()
        assert st == 0, f"{name}: device status {st}"
        for i, t in enumerate(tensors):
            a = t.detach().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            out[f"{name}.{i}"] = a.cpu().numpy()

    for T, H, E, k, F in SHAPES:
        w = moe_synth.Workload("dbg", T=T, H=H, E=E, k=k, F=F, seed=T + 9)
        d = {n: moe_synth.to_torch(v, "cuda") for n, v in moe_synth.layer_inputs(w).items()}
        tag = f"T{T}"
        done(f"forward.{tag}", moe.moe_forward(d["x"], d["w_router"], d["bias"], d["w_up"],
                                               d["w_down"], k))
        done(f"gathered.{tag}", moe.moe_forward(d["x"], d["w_router"], d["bias"], d["w_up"],
                                                d["w_down"], k, gathered=True))
        done(f"fused_combine.{tag}", moe.moe_forward(d["x"], d["w_router"], d["bias"],
                                                     d["w_up"], d["w_down"], k,
                                                     fused_combine=True))
        s = {n: moe_synth.to_torch(v, "cuda")
             for n, v in moe_synth.shared_expert_inputs(w, 128).items()}
        done(f"shared.{tag}", moe.moe_forward_shared(d["x"], d["w_router"], d["bias"],
                                                     d["w_up"], d["w_down"], s["w_up_shared"],
                                                     s["w_down_shared"], k))
        idx, gates, tie = moe.moe_route(d["x"], d["w_router"], d["bias"], k)
        done(f"route.{tag}", idx, gates, tie)
        ridx, rg, rt, p = moe.moe_route_dispatch(d["x"], d["w_router"], d["bias"], k)
        done(f"dispatch.{tag}", ridx, rg, *p.values())
        p = moe.moe_permute(idx, d["x"], E)
        done(f"permute.{tag}", *p.values())
        yp = moe.moe_grouped_ffn(p["x_perm"], p["offsets"], d["w_up"], d["w_down"])
        done(f"ffn.{tag}", yp)
        done(f"combine.{tag}", moe.moe_combine(yp, p["slot_row"], gates, T, k))
        nu = moe.moe_quantize_nvfp4_weights(d["w_up"])
        nd = moe.moe_quantize_nvfp4_weights(d["w_down"])
        done(f"nvfp4.{tag}", moe.moe_forward_nvfp4(d["x"], d["w_router"], d["bias"], nu, nd, k),
             moe.moe_grouped_ffn_nvfp4(p["x_perm"], p["offsets"], nu, nd))
        fu = moe.moe_quantize_fp8_weights(d["w_up"])
        fd = moe.moe_quantize_fp8_weights(d["w_down"])
        done(f"fp8.{tag}", moe.moe_forward_fp8(d["x"], d["w_router"], d["bias"], fu, fd, k),
             moe.moe_grouped_ffn_fp8(p["x_perm"], p["offsets"], fu, fd))
    for T in (200, 1100):
        for rol in (True, False):
            w = moe_synth.Workload("dbgl", T=T, H=512, E=32, k=8, F=128, seed=T + 3, latent=128,
                                   router_on_latent=rol)
            d = {n: moe_synth.to_torch(v, "cuda") for n, v in moe_synth.layer_inputs(w).items()}
            s = {n: moe_synth.to_torch(v, "cuda")
                 for n, v in moe_synth.shared_expert_inputs(w, 128).items()}
            tag = f"T{T}.{int(rol)}"
            done(f"latent.{tag}", moe.latent_moe(d["x"], d["w_in"], d["w_out"], d["w_router"],
                                                 d["bias"], d["w_up"], d["w_down"], w.k,
                                                 router_on_latent=rol))
            done(f"latent_shared.{tag}",
                 moe.latent_moe_shared(d["x"], d["w_in"], d["w_out"], d["w_router"], d["bias"],
                                       d["w_up"], d["w_down"], s["w_up_shared"],
                                       s["w_down_shared"], w.k, router_on_latent=rol))
    return out


if __name__ == "__main__":
    import sparse_mixture_experts_57_b300 as moe
    moe.lib()
    moe.get_device_status()
    res = run_calls(moe)
    res["debug_build"] = np.array([moe.lib().moe_debug_build()])
    np.savez(sys.argv[1], **res)
