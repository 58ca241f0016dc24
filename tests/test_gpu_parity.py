"""GPU vs oracle, element by element, on small seeded inputs.

Sizes here finish in seconds on the oracle and still span several 128-row
tiles, ragged tails, both head dimensions, both dtypes and the degenerate
cases (one row, one key, empty problems, all-zero queries, planted
needles).  Every call goes through the C ABI (libpolarattn.so) via the thin
binding; the oracle is the fp64 plain-C implementation.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, assert_within, dev, errors, invariants_prefill, to_dev

pytestmark = pytest.mark.gpu

PKEYS = ("q", "k", "v", "mem", "w_count")
DKEYS = ("q", "k_cache", "v_cache", "mem", "w_count")


def _pa():
    import long_context_attention_causal_gb300 as pa
    return pa


def run_prefill(x, want_conf=True):
    g = to_dev(x, PKEYS)
    out = torch.full_like(g["q"], float("nan"))  # poisoned: every row must be written
    out, neff, conf = _pa().fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"],
                                out=out, want_conf=want_conf)
    torch.cuda.synchronize()
    return out, neff, conf


def oracle_prefill(x):
    from oracle import oracle_fwd
    return oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"])


def test_tiny_f32_workload():
    """B=1, H=2, T=256, d=64, fp32 from seed 0, memory zeros."""
    from long_context_attention_causal_gb300 import inputs
    x = inputs.make_prefill(inputs.WORKLOADS["tiny_f32"], "cpu")
    out, neff, conf = run_prefill(x)
    e = errors(out, neff, conf, *oracle_prefill(x))
    assert_within(e, "f32", "tiny_f32")
    invariants_prefill(out, neff, conf)


PREFILL_SHAPES = [
    # (B, H, T, d)
    (1, 1, 1, 64), (1, 2, 2, 128), (1, 2, 127, 64), (1, 1, 128, 128),
    (1, 1, 129, 64), (2, 3, 300, 64), (1, 2, 256, 128), (1, 1, 385, 128),
    (1, 2, 640, 64), (1, 1, 1000, 128),
]


@pytest.mark.parametrize("B,H,T,d", PREFILL_SHAPES)
def test_prefill_bf16_shapes(B, H, T, d):
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16",
                       seed=1000 + T + d, needles=1 if T >= 8 else 0)
    x = inputs.make_prefill(wl, "cpu")
    out, neff, conf = run_prefill(x)
    e = errors(out, neff, conf, *oracle_prefill(x))
    assert_within(e, "bf16", f"bf16 {B}x{H}x{T}x{d}")
    invariants_prefill(out, neff, conf)


@pytest.mark.parametrize("B,H,T,d", [(1, 1, 1, 64), (1, 2, 129, 128), (2, 1, 300, 64)])
def test_prefill_f32_shapes(B, H, T, d):
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="f32", seed=2000 + T)
    x = inputs.make_prefill(wl, "cpu")
    out, neff, conf = run_prefill(x)
    e = errors(out, neff, conf, *oracle_prefill(x))
    assert_within(e, "f32", f"f32 {B}x{H}x{T}x{d}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 128)])
def test_prefill_zero_queries_closed_form(dtype, d):
    """q = 0: uniform attention, n_eff = i + 1 and conf = n/(n+1) exactly
    in the mathematics; the kernel must reproduce them to tolerance."""
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=1, T=300, d=d, dtype=dtype, seed=31)
    x = inputs.make_prefill(wl, "cpu")
    x["q"].zero_()
    out, neff, conf = run_prefill(x)
    n = np.arange(1, 301, dtype=np.float64)
    tol = TOL[dtype]
    assert np.abs(neff.cpu().numpy()[0, 0] / n - 1).max() <= tol["neff"]
    assert np.abs(conf.cpu().numpy()[0, 0] - n / (n + 1)).max() <= tol["conf"]
    e = errors(out, neff, conf, *oracle_prefill(x))
    assert_within(e, dtype, "zero queries")


def test_prefill_memory_is_additive():
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=2, T=200, d=64, dtype="bf16", seed=41)
    x = inputs.make_prefill(wl, "cpu")
    o1, n1, _ = run_prefill(x, want_conf=False)
    x0 = dict(x, mem=torch.zeros_like(x["mem"]))
    o0, n0, _ = run_prefill(x0, want_conf=False)
    torch.testing.assert_close(n1, n0, rtol=0, atol=0)
    d = (o1.float() - o0.float() - x["mem"].float().to(dev())).abs().max().item()
    assert d <= 2e-2


def test_prefill_empty_is_noop():
    pa = _pa()
    z = torch.empty((1, 2, 0, 64), device=dev(), dtype=torch.bfloat16)
    w = torch.zeros((2, 64), device=dev())
    out, neff, _ = pa.fwd(z, z, z, z, w)
    assert out.numel() == 0 and neff.numel() == 0


def test_prefill_deterministic():
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=2, T=500, d=128, dtype="bf16", seed=51)
    x = inputs.make_prefill(wl, "cpu")
    a = run_prefill(x)
    b = run_prefill(x)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


# ----------------------------------------------------------------- decode

DECODE_CASES = [
    # (B, H, Tkv, d, dtype, splits)
    (1, 1, 1, 64, "bf16", 0), (2, 2, 2, 128, "bf16", 1), (1, 3, 100, 64, "bf16", 3),
    (2, 2, 1000, 128, "bf16", 0), (1, 2, 4097, 128, "bf16", 7), (1, 1, 5, 128, "bf16", 7),
    (2, 1, 777, 64, "f32", 0), (1, 2, 3000, 128, "f32", 5),
    # more splits than the combine's threads (chunks of d splits, a ragged
    # last chunk) and, at 700 keys in 300 splits, trailing empty splits
    (1, 2, 5000, 64, "bf16", 200), (1, 1, 700, 128, "f32", 300),
]


def run_decode(x, splits, want_conf=True):
    g = to_dev(x, DKEYS)
    out = torch.full_like(g["q"], float("nan"))
    out, neff, conf = _pa().decode(g["q"], g["k_cache"], g["v_cache"], g["mem"],
                                   g["w_count"], num_splits=splits, out=out,
                                   want_conf=want_conf)
    torch.cuda.synchronize()
    return out, neff, conf


@pytest.mark.parametrize("B,H,Tkv,d,dtype,splits", DECODE_CASES)
def test_decode_vs_oracle(B, H, Tkv, d, dtype, splits):
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    wl = inputs.custom("decode", B=B, H=H, T=Tkv, d=d, dtype=dtype, seed=3000 + Tkv)
    x = inputs.make_decode(wl, "cpu")
    out, neff, conf = run_decode(x, splits)
    ref = oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"])
    assert_within(errors(out, neff, conf, *ref), dtype, f"decode {B}x{H}x{Tkv}x{d}")


def test_decode_split_count_invariance():
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("decode", B=2, H=2, T=5000, d=128, dtype="bf16", seed=61)
    x = inputs.make_decode(wl, "cpu")
    o1, n1, c1 = run_decode(x, 1)
    for s in (0, 2, 16, 40):
        o, n, c = run_decode(x, s)
        assert (o.float() - o1.float()).abs().max().item() <= 1e-2
        assert (n / n1 - 1).abs().max().item() <= 1e-4
        assert (c - c1).abs().max().item() <= 1e-4


def test_decode_equals_last_prefill_row():
    """The decode query at position T-1 against the first T keys sees the
    same keys as prefill row T-1."""
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=2, T=700, d=128, dtype="bf16", seed=71)
    x = inputs.make_prefill(wl, "cpu")
    po, pn, pc = run_prefill(x)
    xd = {"q": x["q"][:, :, -1].contiguous(), "k_cache": x["k"], "v_cache": x["v"],
          "mem": x["mem"][:, :, -1].contiguous(), "w_count": x["w_count"]}
    do, dn, dc = run_decode(xd, 0)
    assert (do.float() - po[:, :, -1].float()).abs().max().item() <= 2e-2
    assert (dn / pn[:, :, -1] - 1).abs().max().item() <= 1e-2
    assert (dc - pc[:, :, -1]).abs().max().item() <= 2e-2


def test_combine_entry_point_matches_decode():
    """Partials left in the workspace by decode, merged again by the public
    combine call, give the same result."""
    from long_context_attention_causal_gb300 import inputs
    pa = _pa()
    wl = inputs.custom("decode", B=2, H=3, T=2000, d=64, dtype="bf16", seed=81)
    x = inputs.make_decode(wl, "cpu")
    g = to_dev(x, DKEYS)
    S = 4
    nbytes = pa.decode_workspace_bytes(2, 3, 2000, 64, S)
    ws = torch.empty(nbytes, device=dev(), dtype=torch.uint8)
    o1, n1, c1 = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                           num_splits=S, workspace=ws, want_conf=True)
    parts = ws.view(torch.float32).view(2, 3, S, 64 + 4)
    o2, n2, c2 = pa.combine(parts, g["q"], g["mem"], g["w_count"], 2000, want_conf=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(n1, n2) and torch.equal(c1, c2)
    # partial records: reserved slot is zero, l >= 1 (the max key counts 1)
    assert (parts[..., 3] == 0).all() and (parts[..., 1] >= 1 - 1e-6).all()


def test_decode_workspace_too_small_is_rejected():
    import ctypes
    pa = _pa()
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("decode", B=1, H=1, T=64, d=64, dtype="bf16", seed=91)
    g = to_dev(inputs.make_decode(wl, "cpu"), DKEYS)
    ws = torch.empty(16, device=dev(), dtype=torch.uint8)
    with pytest.raises(pa.PolarError) as ei:
        pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                  num_splits=2, workspace=ws)
    assert ei.value.status == 4


def test_bounded_wait_selftest_reports_and_recovers():
    """A wait that nothing completes ends with status 2, and the device
    stays usable for the next call."""
    pa = _pa()
    pa.device_status(reset=True)
    pa.selftest_wait_timeout(2000)
    assert pa.device_status(reset=True) == 2
    assert pa.device_status() == 0
    test_prefill_bf16_shapes(1, 1, 129, 64)
    assert pa.device_status() == 0


# ------------------------------------------- second-order null floor (NEXT)

@pytest.mark.parametrize("dtype,d,T", [("bf16", 128, 300), ("bf16", 64, 1000), ("f32", 64, 200)])
def test_prefill_second_order_floor(dtype, d, T):
    """floor_order = 2: the null floor is the second-order expected maximum
    of n noise logits; conf (and through it count and out) follow it."""
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd
    pa = _pa()
    wl = inputs.custom("prefill", B=1, H=2, T=T, d=d, dtype=dtype, seed=4000 + T, needles=2)
    x = inputs.make_prefill(wl, "cpu")
    g = to_dev(x, PKEYS)
    out, neff, conf = pa.fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"],
                             consts=pa.default_consts(floor_order=2), want_conf=True)
    torch.cuda.synchronize()
    ref = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"],
                     consts={"floor_order": 2})
    assert_within(errors(out, neff, conf, *ref), dtype, f"floor2 {T}x{d}")
    # the floor moved: the gate differs from the leading-order one
    lead = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    assert np.abs(lead[2] - ref[2]).max() > 1e-3


def test_decode_second_order_floor():
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    pa = _pa()
    wl = inputs.custom("decode", B=2, H=2, T=3000, d=128, dtype="bf16", seed=4100)
    x = inputs.make_decode(wl, "cpu")
    g = to_dev(x, DKEYS)
    c = pa.default_consts(floor_order=2)
    out, neff, conf = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                                consts=c, want_conf=True)
    torch.cuda.synchronize()
    ref = oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"],
                        consts={"floor_order": 2})
    assert_within(errors(out, neff, conf, *ref), "bf16", "decode floor2")


@pytest.mark.parametrize("T,d", [(1100, 64), (1500, 128)])
def test_prefill_tile_pairings_agree(T, d):
    """Grids of at most one wave of CTAs pair query tile p with tile
    n_qt - 1 - p; larger grids pair adjacent tiles.  The same two heads run
    alone (one wave, balanced pairs; n_qt odd at T = 1100, so one CTA owns
    the middle tile alone) and inside a batch of 40 heads (several waves,
    adjacent pairs): every row is computed by the same products in the same
    order, so the two results are bit-identical, and within the bar of the
    oracle."""
    from long_context_attention_causal_gb300 import inputs
    H_big = 40
    x = inputs.make_prefill(inputs.custom("prefill", B=1, H=H_big, T=T, d=d, dtype="bf16",
                                          seed=777 + T), "cpu")
    small = {k: (x[k][:, :2].contiguous() if k != "w_count" else x[k][:2].contiguous())
             for k in PKEYS}
    o_big, n_big, c_big = run_prefill(x)
    o_sm, n_sm, c_sm = run_prefill(small)
    assert torch.equal(o_big[:, :2], o_sm) and torch.equal(n_big[:, :2], n_sm)
    assert torch.equal(c_big[:, :2], c_sm)
    e = errors(o_sm, n_sm, c_sm, *oracle_prefill(small))
    assert_within(e, "bf16", f"pairings T{T} d{d}")


# ------------------------------------------ unit-sphere guard (eps = 1e-6)

def _guard_values(x):
    """Three heads whose |a| sits around the guard eps = 1e-6 with q = 0
    (uniform weights, a_i = running mean of the values): head 0 values of
    scale 5e-7 (|a_i| falls through eps along the rows), head 1 every value
    1e-7 e_0 (u = 0.1 e_0), head 2 every value 1e-5 e_0 (u = e_0)."""
    x["q"].zero_()
    v = x["v"] if "v" in x else x["v_cache"]
    dt = v.dtype
    vf = v.float()
    vf[:, 0] *= 5e-7
    vf[:, 1] = 0
    vf[:, 1, ..., 0] = 1e-7
    vf[:, 2] = 0
    vf[:, 2, ..., 0] = 1e-5
    v.copy_(vf.to(dt))


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("f32", 128), ("bf16", 64), ("bf16", 128)])
def test_prefill_direction_guard_straddles_eps(dtype, d):
    """Rows on both sides of the unit-sphere guard (u = a/|a| above eps,
    a/eps below) against the oracle, element by element."""
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom("prefill", B=1, H=3, T=300, d=d, dtype=dtype, seed=5100 + d)
    x = inputs.make_prefill(wl, "cpu")
    _guard_values(x)
    x["w_count"][1:].zero_()  # heads 1, 2: out - mem is u alone
    an = (x["v"][0, 0].double().cumsum(0) / torch.arange(1, 301)[:, None]).norm(dim=1)
    assert (an > 2e-6).any() and (an < 0.5e-6).any()
    out, neff, conf = run_prefill(x)
    e = errors(out, neff, conf, *oracle_prefill(x))
    assert_within(e, dtype, f"guard prefill {dtype} d{d}")
    # head 1: u = 0.1 e_0, head 2: u = e_0 at every row
    u = out.float().cpu() - x["mem"].float()
    tol = 5e-3 if dtype == "bf16" else 1e-5
    assert (u[0, 1, :, 0] - 0.1).abs().max().item() < tol
    assert (u[0, 2, :, 0] - 1.0).abs().max().item() < tol
    assert u[0, 1:, :, 1:].abs().max().item() < tol


@pytest.mark.parametrize("dtype,Tkv", [("f32", 100), ("f32", 3000), ("bf16", 100), ("bf16", 3000)])
def test_decode_direction_guard_straddles_eps(dtype, Tkv):
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    wl = inputs.custom("decode", B=2, H=3, T=Tkv, d=128, dtype=dtype, seed=5200 + Tkv)
    x = inputs.make_decode(wl, "cpu")
    _guard_values(x)
    for splits in (0, 5):
        out, neff, conf = run_decode(x, splits)
        ref = oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"])
        assert_within(errors(out, neff, conf, *ref), dtype, f"guard decode {dtype} {Tkv}")
