"""Backward of the causal prefill on the GPU vs the fp64 oracle.

The oracle's gradients are pinned by finite differences of the plain-C
forward oracle.  Both sides see the same rounded inputs; the GPU computes in
fp32, so each gradient is held to 1e-3 of its largest magnitude (plus 1e-6
absolute, for gradients that are exactly zero).
"""
import numpy as np
import pytest
import torch

from gpu_util import dev

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, T, d, dtype, floor_order)
    (1, 1, 1, 64, "f32", 1), (1, 2, 64, 64, "f32", 1), (1, 1, 130, 128, "f32", 1),
    (2, 2, 200, 64, "bf16", 1), (1, 2, 300, 128, "bf16", 2), (1, 1, 2100, 64, "bf16", 1),
]


def _close(got, ref, what):
    got = got.detach().float().cpu().numpy() if isinstance(got, torch.Tensor) else got
    scale = max(float(np.abs(ref).max()), 1e-6)
    err = float(np.abs(got - ref).max())
    # absolute floor: at n = 1 the count term is tanh(0) = 0, so dq is exactly 0
    assert err <= 1e-3 * scale + 1e-6, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


@pytest.mark.parametrize("B,H,T,d,dtype,floor_order", CASES)
def test_backward_vs_oracle(B, H, T, d, dtype, floor_order):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype=dtype, seed=7000 + T + d,
                       needles=1 if T >= 8 else 0)
    x = inputs.make_prefill(wl, "cpu")
    g = torch.Generator().manual_seed(7001 + T)
    dout = torch.randn(x["q"].shape, generator=g).to(x["q"].dtype)
    ref = oracle_bwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], dout,
                     consts={"floor_order": floor_order})
    t = {kk: x[kk].to(dev()) for kk in ("q", "k", "v", "w_count")}
    dq, dk, dv, dw = pa.bwd(t["q"], t["k"], t["v"], t["w_count"], dout.to(dev()),
                            consts=pa.default_consts(floor_order=floor_order))
    torch.cuda.synchronize()
    _close(dq, ref["dq"], "dq")
    _close(dk, ref["dk"], "dk")
    _close(dv, ref["dv"], "dv")
    _close(dw, ref["dw"], "dw")
    assert pa.device_status() == 0
