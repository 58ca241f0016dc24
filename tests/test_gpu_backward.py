"""Backward of the causal prefill on the GPU vs the fp64 oracle.

The oracle's gradients are pinned by finite differences of the plain-C
forward oracle.  Both sides see the same rounded inputs.

* fp32 inputs run on the FP32 pipes in fp32: each gradient is held to 1e-3
  of its largest magnitude.
* bf16 inputs run on the tensor cores, whose operands P, dS' and dA are
  rounded to bf16 (relative 2^-9 each) with fp32 accumulation: each gradient
  is held to 2e-2 of its largest magnitude, the bound of the bf16 forward.
An absolute floor of 1e-6 covers gradients that are exactly zero (at n = 1
the count term is tanh(0) = 0, so dq vanishes).
"""
import numpy as np
import pytest
import torch

from gpu_util import dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "bf16": 2e-2}

CASES = [
    # (B, H, T, d, dtype, floor_order)
    (1, 1, 1, 64, "f32", 1), (1, 2, 64, 64, "f32", 1), (1, 1, 130, 128, "f32", 1),
    (1, 1, 300, 64, "f32", 2),
    (1, 1, 1, 128, "bf16", 1), (1, 2, 2, 64, "bf16", 1), (1, 2, 130, 128, "bf16", 1),
    (2, 2, 200, 64, "bf16", 1), (1, 2, 300, 128, "bf16", 2), (1, 1, 640, 128, "bf16", 2),
    (1, 1, 2100, 64, "bf16", 1), (1, 1, 4096, 128, "bf16", 1),
]


def _close(got, ref, what, tol):
    got = got.detach().float().cpu().numpy()
    scale = max(float(np.abs(ref).max()), 1e-6)
    err = float(np.abs(got - ref).max())
    print(f"{what}: max err / scale = {err / scale:.2e}")
    assert err <= tol * scale + 1e-6, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


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
    tol = TOL[dtype]
    _close(dq, ref["dq"], "dq", tol)
    _close(dk, ref["dk"], "dk", tol)
    _close(dv, ref["dv"], "dv", tol)
    _close(dw, ref["dw"], "dw", tol)
    assert pa.device_status() == 0


def test_backward_workspace_is_reusable():
    """Two calls through one caller-owned workspace give identical results."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=2, T=333, d=128, dtype="bf16", seed=71, needles=1)
    x = inputs.make_prefill(wl, dev())
    dout = torch.randn_like(x["q"])
    ws = torch.empty(pa.bwd_workspace_bytes(1, 2, 333, 128), dtype=torch.uint8, device=dev())
    a = pa.bwd(x["q"], x["k"], x["v"], x["w_count"], dout, workspace=ws)
    ws.fill_(0xFF)  # poison: every byte the next call reads must be rewritten
    b = pa.bwd(x["q"], x["k"], x["v"], x["w_count"], dout, workspace=ws)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u, w)
    assert pa.device_status() == 0


def _saved_run(B, H, T, d, floor_order):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd, oracle_row_stats
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16", seed=7100 + T + d,
                       needles=1 if T >= 8 else 0)
    x = inputs.make_prefill(wl, "cpu")
    g = torch.Generator().manual_seed(7101 + T)
    dout = torch.randn(x["q"].shape, generator=g).to(x["q"].dtype)
    c = {"floor_order": floor_order}
    ref = oracle_bwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], dout, consts=c)
    t = {kk: x[kk].to(dev()) for kk in ("q", "k", "v", "mem", "w_count")}
    pc = pa.default_consts(floor_order=floor_order)
    out, n_eff, conf, stats = pa.fwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"], consts=pc)
    # the statistics themselves: logsumexp and |a| of every row
    fo = oracle_row_stats(x["q"], x["k"], x["v"], consts=c)
    st = stats.cpu().numpy()
    assert np.abs(st[..., 0] - fo["lse"]).max() <= 2e-3 * max(1.0, np.abs(fo["lse"]).max())
    assert np.abs(st[..., 1] - fo["anorm"]).max() <= 2e-2 * np.abs(fo["anorm"]).max() + 1e-6
    dq, dk, dv, dw = pa.bwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"], out, n_eff,
                                  conf, stats, dout.to(dev()), consts=pc)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    return {"dq": dq, "dk": dk, "dv": dv, "dw": dw}, ref


@pytest.mark.parametrize("B,H,T,d,floor_order", [
    (1, 2, 130, 128, 1), (2, 2, 200, 64, 1), (1, 2, 300, 128, 2),
    (1, 1, 2100, 64, 1), (1, 1, 4096, 128, 1)])
def test_backward_from_saved_stats_vs_oracle(B, H, T, d, floor_order):
    """fwd_stats + bwd_stats (no forward recomputation) against the oracle.
    The direction is recovered from the bf16 output, one more bf16 rounding
    of the same size as the others: the bf16 bound of 2e-2 holds."""
    got, ref = _saved_run(B, H, T, d, floor_order)
    for name in ("dq", "dk", "dv", "dw"):
        _close(got[name], ref[name], name, TOL["bf16"])


def test_backward_from_saved_stats_single_key():
    """n = 1: dq and dk are exactly 0 in the definition (dS = dP - D
    cancels).  From saved statistics D uses the direction recovered from the
    bf16 output, so the cancellation leaves a residual of the size of that
    rounding (2^-9 relative): dq and dk stay within 5e-3 of dv's scale, the
    row's nonzero gradient."""
    got, ref = _saved_run(1, 1, 1, 128, 1)
    for name in ("dv", "dw"):
        _close(got[name], ref[name], name, TOL["bf16"])
    scale = float(np.abs(ref["dv"]).max())
    assert float(got["dq"].abs().max()) <= 5e-3 * scale
    assert float(got["dk"].abs().max()) <= 5e-3 * scale


def test_backward_from_saved_stats_into_given_buffers():
    """Caller-owned gradient buffers (NaN-poisoned beforehand) receive the
    same gradients, bit for bit, as freshly allocated ones; buffers of the
    wrong shape are rejected before the library is called."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    x = inputs.make_prefill(inputs.custom("prefill", B=1, H=2, T=700, d=128, dtype="bf16",
                                          seed=7300, needles=1), dev())
    dout = torch.randn(x["q"].shape, generator=torch.Generator(device=dev()).manual_seed(7301),
                       device=dev()).to(torch.bfloat16)
    fo = pa.fwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    ref = pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], *fo, dout)
    bufs = [torch.full(x["q"].shape, float("nan"), device=dev()) for _ in range(3)]
    dw = torch.full((2, 128), float("nan"), device=dev())
    got = pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], *fo, dout,
                       dq=bufs[0], dk=bufs[1], dv=bufs[2], dw=dw)
    torch.cuda.synchronize()
    assert got[0] is bufs[0] and got[3] is dw
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    with pytest.raises(ValueError):
        pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], *fo, dout,
                     dw=torch.empty((2, 64), device=dev()))


def test_stats_calls_reject_fp32():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=1, T=64, d=64, dtype="f32", seed=3, needles=0)
    x = inputs.make_prefill(wl, dev())
    with pytest.raises(Exception):
        pa.fwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"])


@pytest.mark.parametrize("from_stats", [False, True])
def test_backward_full_size_keyscale_16k_sampled(from_stats):
    """The bench's prefill workload (B2 H16 T16384 d128 bf16) in the launch
    configuration bench.py times: dq at sampled rows and dk, dv at sampled
    keys of one head against the sampled oracle (exact per output, fp64),
    and dw of that head over both batch entries."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd_sampled
    wl = inputs.WORKLOADS["keyscale_16k"]
    x = inputs.make_prefill(wl, "cpu")
    g = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(77)).to(x["q"].dtype)
    t = {kk: x[kk].to(dev()) for kk in ("q", "k", "v", "mem", "w_count")}
    gd = g.to(dev())
    if from_stats:
        out, ne, cf, st = pa.fwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"])
        dq, dk, dv, dw = pa.bwd_stats(t["q"], t["k"], t["v"], t["mem"], t["w_count"], out, ne,
                                      cf, st, gd)
    else:
        dq, dk, dv, dw = pa.bwd(t["q"], t["k"], t["v"], t["w_count"], gd)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    T, h = wl.T, 5
    rng = np.random.default_rng(78)
    rows = sorted(set([0, 1, 127, 128, 2047, 2048, 4095, 8191, T - 1] +
                      rng.integers(0, T, 16).tolist()))
    keys = sorted(set([0, 1, 127, 128, 2048, 8000, T - 2, T - 1] +
                      rng.integers(0, T, 8).tolist()))
    dw_ref = 0.0
    for b in range(wl.B):
        ref = oracle_bwd_sampled(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["w_count"][h],
                                 g[b, h], rows, keys)
        dw_ref = dw_ref + (ref["count"][:, None] * g[b, h].double().numpy()).sum(axis=0)
        if b == 1:
            _close(dq[b, h, rows], ref["dq"], "dq", TOL["bf16"])
            _close(dk[b, h, keys], ref["dk"], "dk", TOL["bf16"])
            _close(dv[b, h, keys], ref["dv"], "dv", TOL["bf16"])
    _close(dw[h], dw_ref, "dw", TOL["bf16"])
    # invariant at every output: finite
    for name, tt in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(tt).all(), name
