"""The decode entry point that allocates nothing.

polar_attn_decode_static_scratch serves callers that cannot allocate device
memory when they decode (a host framework or plugin that owns all device
memory, a serving loop that forbids cudaMalloc after start-up): its split
partials live in a fixed device array inside the library.  This test calls
it through the C ABI twice in a row, on different problems, and checks each
result against polar_attn_decode with a caller-provided workspace and
against the fp64 oracle, within the tolerances of the other parity tests
(bf16 and fp32 inputs).  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

KEYS = ("q", "k_cache", "v_cache", "mem", "w_count")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _static_decode(L, g, num_splits=0):
    import long_context_attention_causal_gb300 as pa
    B, H, Tkv, d = g["k_cache"].shape
    dtype = 1 if g["q"].dtype == torch.bfloat16 else 0
    out = torch.full_like(g["q"], float("nan"))
    n_eff = torch.full((B, H), float("nan"), device=g["q"].device)
    conf = torch.full((B, H), float("nan"), device=g["q"].device)
    c = pa.default_consts()
    st = L.polar_attn_decode_static_scratch(
        _ptr(g["q"]), _ptr(g["k_cache"]), _ptr(g["v_cache"]), _ptr(g["mem"]),
        _ptr(g["w_count"]), _ptr(out), _ptr(n_eff), _ptr(conf), B, H, Tkv, d, dtype,
        ctypes.byref(c), num_splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, n_eff, conf


TOL = {"bf16": (2e-2, 1e-2, 2e-2), "f32": (1e-4, 1e-4, 1e-4)}  # out, n_eff (rel), conf


def _check(out, n_eff, conf, ro, rn, rc, tol):
    ro, rn, rc = (torch.as_tensor(a, dtype=torch.float64) for a in (ro, rn, rc))
    assert (out.double().cpu() - ro).abs().max().item() <= tol[0]
    assert (n_eff.double().cpu() / rn - 1).abs().max().item() <= tol[1]
    assert (conf.double().cpu() - rc).abs().max().item() <= tol[2]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_static_scratch_decode_matches_workspace_decode(dtype):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    L = pa.lib()
    dev = torch.device("cuda:0")
    cases = [
        # a problem with many splits, then a smaller one that reuses the array
        inputs.custom("decode", B=4, H=8, T=8192, d=128, dtype=dtype, seed=501),
        inputs.custom("decode", B=2, H=3, T=777, d=64, dtype=dtype, seed=502),
    ]
    tol = TOL[dtype]
    for wl in cases:
        x = inputs.make_decode(wl, "cpu")
        g = {k: x[k].to(dev) for k in KEYS}
        st, out, n_eff, conf = _static_decode(L, g)
        assert st == 0, pa.strerror(st) + " " + L.polar_attn_last_error().decode()
        ref_out, ref_n, ref_c = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"],
                                          g["w_count"], want_conf=True)
        torch.cuda.synchronize()
        # against the workspace decode ...
        _check(out, n_eff, conf, ref_out.cpu(), ref_n.cpu(), ref_c.cpu(), tol)
        # ... and against the fp64 oracle
        _check(out, n_eff, conf,
               *oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"]), tol)
    assert pa.device_status() == 0


def test_static_scratch_rejects_oversized_request():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    L = pa.lib()
    wl = inputs.custom("decode", B=32, H=16, T=64, d=128, dtype="bf16", seed=503)
    x = inputs.make_decode(wl, "cpu")
    g = {k: x[k].to(torch.device("cuda:0")) for k in KEYS}
    # 32*16 heads * 40 splits * 132 floats * 4 bytes > 8 MiB
    st, out, _, _ = _static_decode(L, g, num_splits=40)
    torch.cuda.synchronize()
    assert st == 4
    assert b"static scratch" in L.polar_attn_last_error()
    assert torch.isnan(out.float()).all()  # nothing was launched
