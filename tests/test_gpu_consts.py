"""Every call with constants other than the defaults, against the oracle.

polar_consts_t carries the neutral length of the temperature law (log_t0),
the scale of the count's tanh-log map (kappa), the key noise scale of the
null floor (sigma_k), the unit-sphere guard (eps) and the floor order.  The
other parity tests run the defaults (T0 = 2048, kappa = ln 2048, sigma_k =
1, eps = 1e-6) and vary only the floor order; here T0 = 256 (so the
temperature sharpens from row 256 on), kappa = 2.5, sigma_k = 0.625 and
eps = 2^-9, all exact in fp32 so both sides use the same numbers, with one
head's values scaled by 1e-4 so that the guard is active on its rows.
Calls: the bf16 prefill (one-wave and multi-wave orders, d = 128 and 64),
the fp32 prefill, the split decode (bf16, fp32), the paged decode (tensor
cores for bf16, CUDA cores for fp32), both backward paths and the memory
step (its own eps).
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import assert_within, dev, errors

pytestmark = pytest.mark.gpu

LOG_T0 = float(np.float32(math.log(256.0)))
C = {"log_t0": LOG_T0, "kappa": 2.5, "sigma_k": 0.625, "eps": 2.0 ** -9}


def _pc(floor_order=1):
    import long_context_attention_causal_gb300 as pa
    return pa.Consts(C["log_t0"], C["kappa"], C["sigma_k"], C["eps"], floor_order)


def _oc(floor_order=1):
    return dict(C, floor_order=floor_order)


def _small_values(x, key, h, scale=1e-4):
    """Head h of x[key] scaled down (in the tensor's own dtype) so that the
    attention average of the values falls below eps."""
    t = x[key].float()
    t[:, h] *= scale
    x[key] = t.to(x[key].dtype)
    return x


PREFILL = [
    # (B, H, T, d, dtype, floor_order): one wave, one wave d = 64, several
    # waves, fp32
    (1, 2, 1000, 128, "bf16", 1),
    (1, 3, 700, 64, "bf16", 2),
    (1, 40, 1024, 128, "bf16", 1),
    (1, 2, 300, 64, "f32", 2),
]


@pytest.mark.parametrize("B,H,T,d,dtype,fo", PREFILL)
def test_prefill_custom_consts(B, H, T, d, dtype, fo):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd
    x = inputs.make_prefill(inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype=dtype,
                                          seed=8100 + T + H, needles=2), "cpu")
    x = _small_values(x, "v", H - 1)
    g = {k: x[k].to(dev()) for k in ("q", "k", "v", "mem", "w_count")}
    out, neff, conf = pa.fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"], consts=_pc(fo),
                             want_conf=True)
    torch.cuda.synchronize()
    ref = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], consts=_oc(fo))
    assert_within(errors(out, neff, conf, *ref), dtype, f"prefill {B}x{H}x{T}x{d} {dtype}")
    # the constants matter: the defaults give a different result
    ref_def = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"],
                         consts={"floor_order": fo})
    assert np.abs(ref_def[2] - ref[2]).max() > 0.02


@pytest.mark.parametrize("Tkv,dtype,splits", [(3000, "bf16", 0), (1000, "f32", 3)])
def test_decode_custom_consts(Tkv, dtype, splits):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    x = inputs.make_decode(inputs.custom("decode", B=2, H=3, T=Tkv, d=128, dtype=dtype,
                                         seed=8200 + Tkv), "cpu")
    x = _small_values(x, "v_cache", 2)
    g = {k: x[k].to(dev()) for k in ("q", "k_cache", "v_cache", "mem", "w_count")}
    out, neff, conf = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                                num_splits=splits, consts=_pc(2), want_conf=True)
    torch.cuda.synchronize()
    ref = oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"],
                        consts=_oc(2))
    assert_within(errors(out, neff, conf, *ref), dtype, f"decode {Tkv} {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_paged_decode_custom_consts(dtype):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=3, Hq=8, Hkv=2, T=900, d=128, page=64, dtype=dtype, seed=8300)
    x = inputs.make_paged_decode(wl, "cpu")
    keys = ("q", "k_pages", "v_pages", "block_table", "seq_lens", "mem", "w_count")
    g = {k: x[k].to(dev()) for k in keys}
    pa.device_status(reset=True)
    out, neff, conf = pa.decode_paged(*(g[k] for k in keys), max_seq_len=wl.T,
                                      consts=_pc(1), want_conf=True)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    ref = oracle_decode_paged(*(x[k] for k in keys), consts=_oc(1))
    assert_within(errors(out, neff, conf, *ref), dtype, f"paged {dtype}")


def _close(got, ref, what, tol):
    got = got.detach().float().cpu().numpy()
    scale = max(float(np.abs(ref).max()), 1e-6)
    err = float(np.abs(got - ref).max())
    assert err <= tol * scale + 1e-6, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


@pytest.mark.parametrize("dtype,fo", [("bf16", 1), ("bf16", 2), ("f32", 1)])
def test_backward_custom_consts(dtype, fo):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd
    x = inputs.make_prefill(inputs.custom("prefill", B=1, H=2, T=600, d=128, dtype=dtype,
                                          seed=8400 + fo, needles=1), "cpu")
    dout = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(8401)).to(
        x["q"].dtype)
    ref = oracle_bwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], dout, consts=_oc(fo))
    t = {k: x[k].to(dev()) for k in ("q", "k", "v", "mem", "w_count")}
    tol = 2e-2 if dtype == "bf16" else 1e-3
    paths = [pa.bwd(t["q"], t["k"], t["v"], t["w_count"], dout.to(dev()), consts=_pc(fo))]
    if dtype == "bf16":
        o, ne, cf, st = pa.fwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"],
                                     consts=_pc(fo))
        paths.append(pa.bwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"], o, ne, cf,
                                  st, dout.to(dev()), consts=_pc(fo)))
    torch.cuda.synchronize()
    for grads in paths:
        for name, got in zip(("dq", "dk", "dv", "dw"), grads):
            _close(got, ref[name], f"{name} ({dtype}, floor {fo})", tol)
    assert pa.device_status() == 0


def test_memory_step_custom_eps():
    """The memory step's own guard: keys and queries of norm ~1e-4 in one
    head, eps = 2^-9, so k^ = k / eps and q^ = q / eps there."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_memory_step
    x = inputs.make_memory(inputs.MemoryWorkload("consts_mem", 2, 3, 4, 128, "f32", 8500),
                           "cpu")
    x["k"][:, 2] *= 1e-5
    x["q"][:, 2] *= 1e-5
    S_ref, mem_ref = oracle_memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"],
                                        x["beta"], eps=C["eps"])
    g = {k: t.to(dev()) for k, t in x.items()}
    mem = pa.memory_step(g["state"], g["q"], g["k"], g["v"], g["alpha"], g["beta"],
                         eps=C["eps"])
    torch.cuda.synchronize()
    assert np.abs(g["state"].cpu().double().numpy() - S_ref).max() <= 1e-4
    assert np.abs(mem.cpu().double().numpy() - mem_ref).max() <= 1e-4
