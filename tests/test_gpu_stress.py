"""Stress and randomised shapes, GPU vs the oracle.

* Growing logits: key norms rise along the sequence and one key carries a
  logit spike far above the rest, so every row's running maximum keeps
  increasing from tile to tile and jumps by far more than the 2^8 factor at
  which the kernels rescale their running sums (and, in the tensor-core
  prefill, the accumulator in TMEM).
* Seeded random shapes, dtypes and floor orders for the prefill, the decode
  (random split counts) and the backward.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, assert_within, dev, errors, invariants_prefill, to_dev

pytestmark = pytest.mark.gpu

PKEYS = ("q", "k", "v", "mem", "w_count")


def _growing(x, T, spike_at=None):
    """Scale key j by 1 + 12 j / T; optionally plant a key aligned with the
    last query row at ~90 logit units (about 130 in log2)."""
    k = x["k"].float()
    ramp = 1.0 + 12.0 * torch.arange(T, dtype=torch.float32) / max(T, 1)
    k = k * ramp[None, None, :, None]
    if spike_at is not None:
        q = x["q"].float()
        qn = q[:, :, -1].norm(dim=-1, keepdim=True).clamp_min(1e-3)
        d = q.shape[-1]
        k[:, :, spike_at] = 90.0 * (d ** 0.5) * q[:, :, -1] / qn / qn
    x = dict(x)
    x["k"] = k.to(x["q"].dtype)
    return x


@pytest.mark.parametrize("dtype,d,T", [("bf16", 128, 1000), ("bf16", 64, 700), ("f32", 64, 300),
                                       ("f32", 128, 260)])
def test_prefill_growing_logits(dtype, d, T):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd
    wl = inputs.custom("prefill", B=1, H=2, T=T, d=d, dtype=dtype, seed=9000 + T, needles=0)
    x = _growing(inputs.make_prefill(wl, "cpu"), T, spike_at=T // 3)
    g = to_dev(x, PKEYS)
    out = torch.full_like(g["q"], float("nan"))
    out, neff, conf = pa.fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"], out=out,
                             want_conf=True)
    torch.cuda.synchronize()
    e = errors(out, neff, conf, *oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"]))
    assert_within(e, dtype, f"growing logits {dtype} d{d} T{T}")
    invariants_prefill(out, neff, conf)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_growing_logits(dtype):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    T = 3000
    wl = inputs.custom("decode", B=2, H=2, T=T, d=128, dtype=dtype, seed=9100)
    x = inputs.make_decode(wl, "cpu")
    ramp = 1.0 + 12.0 * torch.arange(T, dtype=torch.float32) / T
    x["k_cache"] = (x["k_cache"].float() * ramp[None, None, :, None]).to(x["q"].dtype)
    g = to_dev(x, ("q", "k_cache", "v_cache", "mem", "w_count"))
    out, neff, conf = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                                num_splits=5, want_conf=True)
    torch.cuda.synchronize()
    e = errors(out, neff, conf, *oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"],
                                               x["w_count"]))
    assert_within(e, dtype, f"decode growing logits {dtype}")


def _close_rel(got, ref, what, tol):
    got = got.detach().float().cpu().numpy()
    scale = max(float(np.abs(ref).max()), 1e-6)
    err = float(np.abs(got - ref).max())
    assert err <= tol * scale + 1e-6, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


def test_backward_growing_logits():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd
    T, d = 600, 128
    wl = inputs.custom("prefill", B=1, H=2, T=T, d=d, dtype="bf16", seed=9200, needles=0)
    x = _growing(inputs.make_prefill(wl, "cpu"), T)
    dout = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(9201)).to(x["q"].dtype)
    ref = oracle_bwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], dout)
    g = to_dev(x, PKEYS)
    got = pa.bwd(g["q"], g["k"], g["v"], g["w_count"], dout.to(dev()))
    torch.cuda.synchronize()
    for name, t in zip(("dq", "dk", "dv", "dw"), got):
        _close_rel(t, ref[name], name, 2e-2)
    assert pa.device_status() == 0


def _fuzz_cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        yield (int(rng.integers(1, 4)), int(rng.integers(1, 5)), int(rng.integers(1, 701)),
               int(rng.choice([64, 128])), str(rng.choice(["bf16", "f32"])),
               int(rng.choice([1, 2])), int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("B,H,T,d,dtype,fo,seed", list(_fuzz_cases(8, 31)))
def test_prefill_fuzz(B, H, T, d, dtype, fo, seed):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype=dtype, seed=seed % 100000,
                       needles=1 if T >= 8 else 0)
    x = inputs.make_prefill(wl, "cpu")
    g = to_dev(x, PKEYS)
    out = torch.full_like(g["q"], float("nan"))
    c = pa.default_consts(floor_order=fo)
    out, neff, conf = pa.fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"], out=out,
                             want_conf=True, consts=c)
    torch.cuda.synchronize()
    e = errors(out, neff, conf, *oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"],
                                            consts={"floor_order": fo}))
    assert_within(e, dtype, f"fuzz prefill {B}x{H}x{T}x{d} {dtype} floor{fo}")


@pytest.mark.parametrize("B,H,T,d,dtype,fo,seed", list(_fuzz_cases(6, 32)))
def test_decode_fuzz(B, H, T, d, dtype, fo, seed):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    Tkv = T * 7 + 1
    wl = inputs.custom("decode", B=B, H=H, T=Tkv, d=d, dtype=dtype, seed=seed % 100000)
    x = inputs.make_decode(wl, "cpu")
    g = to_dev(x, ("q", "k_cache", "v_cache", "mem", "w_count"))
    splits = int(np.random.default_rng(seed).integers(0, 20))
    c = pa.default_consts(floor_order=fo)
    out, neff, conf = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                                num_splits=splits, want_conf=True, consts=c)
    torch.cuda.synchronize()
    e = errors(out, neff, conf, *oracle_decode(x["q"], x["k_cache"], x["v_cache"], x["mem"],
                                               x["w_count"], consts={"floor_order": fo}))
    assert_within(e, dtype, f"fuzz decode {B}x{H}x{Tkv}x{d} {dtype} S{splits}")


@pytest.mark.parametrize("B,H,T,d,dtype,fo,seed", list(_fuzz_cases(4, 33)))
def test_backward_fuzz(B, H, T, d, dtype, fo, seed):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd
    T = min(T, 400)
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype=dtype, seed=seed % 100000,
                       needles=1 if T >= 8 else 0)
    x = inputs.make_prefill(wl, "cpu")
    dout = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(seed % 1000)).to(
        x["q"].dtype)
    ref = oracle_bwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], dout,
                     consts={"floor_order": fo})
    g = to_dev(x, PKEYS)
    got = pa.bwd(g["q"], g["k"], g["v"], g["w_count"], dout.to(dev()),
                 consts=pa.default_consts(floor_order=fo))
    torch.cuda.synchronize()
    tol = 2e-2 if dtype == "bf16" else 1e-3
    for name, t in zip(("dq", "dk", "dv", "dw"), got):
        _close_rel(t, ref[name], f"{name} {B}x{H}x{T}x{d} {dtype}", tol)
    assert pa.device_status() == 0


def _paged_fuzz_cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = int(rng.integers(1, 4))
        yield (int(rng.integers(1, 5)), G * Hkv, Hkv, int(rng.integers(1, 1500)),
               int(rng.choice([64, 128])), int(rng.choice([8, 16, 32, 64, 128, 256])),
               str(rng.choice(["bf16", "bf16", "f32"])), int(rng.integers(0, 12)),
               int(rng.choice([1, 2])), int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("B,Hq,Hkv,T,d,page,dtype,splits,fo,seed",
                         list(_paged_fuzz_cases(10, 34)))
def test_paged_decode_fuzz(B, Hq, Hkv, T, d, page, dtype, splits, fo, seed):
    """Seeded random paged decodes: group sizes 1-8, both head sizes, pages
    of 8-256 tokens, ragged lengths, split counts 0 (automatic) to 11, both
    floor orders; bf16 runs the tensor-core kernel, fp32 the CUDA-core one."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, page=page, dtype=dtype,
                             seed=seed % 100000)
    x = inputs.make_paged_decode(wl, "cpu")
    keys = ("q", "k_pages", "v_pages", "block_table", "seq_lens", "mem", "w_count")
    g = {k: x[k].to(dev()) for k in keys}
    pa.device_status(reset=True)
    out, neff, conf = pa.decode_paged(g["q"], g["k_pages"], g["v_pages"], g["block_table"],
                                      g["seq_lens"], g["mem"], g["w_count"], num_splits=splits,
                                      want_conf=True, consts=pa.default_consts(floor_order=fo))
    torch.cuda.synchronize()
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"], consts={"floor_order": fo})
    assert_within(errors(out, neff, conf, *ref), dtype,
                  f"fuzz paged {B}x{Hq}/{Hkv}x{T}x{d} p{page} {dtype} S{splits}")
    assert pa.device_status() == 0


# ------------------------------------------- repeated calls, same result

@pytest.mark.parametrize("B,H,T,d", [(1, 8, 4096, 64),    # one wave: balanced tile pairs
                                     (1, 2, 1500, 128),   # one wave, ragged tail
                                     (2, 16, 2048, 128),  # several waves: adjacent pairs
                                     (1, 24, 3000, 64)])
def test_prefill_repeated_calls_identical(B, H, T, d):
    """The prefill's schedule depends on warp timing (barrier hand-offs
    between the TMA, MMA and softmax warps); its arithmetic must not.  Fifty
    calls on the same inputs give bit-identical outputs and leave the device
    status word at 0 (no wait ran out)."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    x = to_dev(inputs.make_prefill(inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16",
                                                 seed=4242 + T), "cpu"), PKEYS)
    pa.device_status(reset=True)
    o0, n0, c0 = pa.fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], want_conf=True)
    for _ in range(50):
        o, n, c = pa.fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], want_conf=True)
        assert torch.equal(o, o0) and torch.equal(n, n0) and torch.equal(c, c0)
    torch.cuda.synchronize()
    assert pa.device_status(reset=True) == 0


def test_backward_repeated_calls_identical():
    """The backward's dQ kernel runs beside the dK/dV kernel on a second
    stream; twenty calls give bit-identical gradients and status 0."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    x = to_dev(inputs.make_prefill(inputs.custom("prefill", B=1, H=4, T=1300, d=128,
                                                 dtype="bf16", seed=4343), "cpu"), PKEYS)
    g = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(7)).to(
        x["q"].dtype).to(dev())
    pa.device_status(reset=True)
    ref = pa.bwd(x["q"], x["k"], x["v"], x["w_count"], g)
    for _ in range(20):
        got = pa.bwd(x["q"], x["k"], x["v"], x["w_count"], g)
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
    torch.cuda.synchronize()
    assert pa.device_status(reset=True) == 0
