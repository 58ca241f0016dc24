"""The host-buffer prefill (polar_attn_fwd_host) runs the prefill kernels on
pieces of the (b, h) range while the copies of other pieces are in flight;
each piece is a narrowed polar_attn_fwd launch, so every output element must
equal polar_attn_fwd's bit for bit, whatever the cut, and the pair must stay
within the parity bar of the oracle."""
import pytest
import torch

from gpu_util import assert_within, dev, errors

pytestmark = pytest.mark.gpu


def _inputs(B, H, T, d, dtype, seed):
    from long_context_attention_causal_gb300 import inputs
    return inputs.make_prefill(inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype=dtype,
                                             seed=seed), "cpu")


def _device_reference(x, want_conf):
    import long_context_attention_causal_gb300 as pa
    d = {k: x[k].to(dev()) for k in ("q", "k", "v", "mem", "w_count")}
    out, ne, cf = pa.fwd(d["q"], d["k"], d["v"], d["mem"], d["w_count"], want_conf=want_conf)
    torch.cuda.synchronize()
    return out.cpu(), ne.cpu(), (cf.cpu() if cf is not None else None)


@pytest.mark.parametrize("B,H,T,d,dtype", [(2, 3, 1000, 128, "bf16"), (3, 5, 777, 64, "bf16"),
                                           (2, 2, 300, 64, "f32"), (1, 1, 3000, 128, "bf16")])
@pytest.mark.parametrize("pieces", [0, 1, 2, 4, 7, 64])
def test_host_pipeline_equals_device_call(B, H, T, d, dtype, pieces):
    import long_context_attention_causal_gb300 as pa
    x = _inputs(B, H, T, d, dtype, seed=70 + pieces)
    ro, rn, rc = _device_reference(x, want_conf=True)
    h = {k: x[k].contiguous().pin_memory() for k in ("q", "k", "v", "mem", "w_count")}
    out, ne, cf = pa.fwd_host(h["q"], h["k"], h["v"], h["mem"], h["w_count"], want_conf=True,
                              num_pieces=pieces)
    assert torch.equal(out, ro) and torch.equal(ne, rn) and torch.equal(cf, rc)


def test_host_pipeline_pageable_buffers_and_reuse():
    """Pageable (not pinned) host tensors, caller-owned outputs and one
    workspace reused across calls with different inputs."""
    import long_context_attention_causal_gb300 as pa
    B, H, T, d = 2, 4, 2048, 128
    ws = torch.empty(pa.fwd_host_workspace_bytes(B, H, T, d), device=dev(), dtype=torch.uint8)
    out = torch.empty((B, H, T, d), dtype=torch.bfloat16)
    ne = torch.empty((B, H, T), dtype=torch.float32)
    for seed in (81, 82):
        x = _inputs(B, H, T, d, "bf16", seed)
        ro, rn, _ = _device_reference(x, want_conf=False)
        pa.fwd_host(x["q"], x["k"], x["v"], x["mem"], x["w_count"], out=out, n_eff=ne,
                    workspace=ws, num_pieces=3)
        assert torch.equal(out, ro) and torch.equal(ne, rn)


def test_host_pipeline_against_oracle():
    """Through the host path, the small bf16 case meets the parity bar
    against the oracle."""
    import long_context_attention_causal_gb300 as pa
    from oracle import oracle_fwd
    x = _inputs(1, 2, 300, 64, "bf16", seed=90)
    h = {k: x[k].contiguous().pin_memory() for k in ("q", "k", "v", "mem", "w_count")}
    out, ne, cf = pa.fwd_host(h["q"], h["k"], h["v"], h["mem"], h["w_count"], want_conf=True,
                              num_pieces=2)
    ro, rn, rc = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    assert_within(errors(out, ne, cf, ro, rn, rc), "bf16", "fwd_host")


def test_host_pipeline_orders_after_prior_stream_work():
    """The copies start only after what the caller's stream already holds:
    the workspace is overwritten by a kernel queued behind a long chain of
    products on the caller's stream, so copies that did not wait for it
    would be clobbered and the outputs would differ."""
    import long_context_attention_causal_gb300 as pa
    B, H, T, d = 1, 8, 4096, 128
    x = _inputs(B, H, T, d, "bf16", seed=91)
    ro, rn, _ = _device_reference(x, want_conf=False)
    h = {k: x[k].contiguous().pin_memory() for k in ("q", "k", "v", "mem", "w_count")}
    ws = torch.empty(pa.fwd_host_workspace_bytes(B, H, T, d), device=dev(), dtype=torch.uint8)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        big = torch.randn(8192, 8192, device=dev())
        for _ in range(8):
            big = big @ big / 8192.0  # keep the stream busy
        ws.fill_(255)  # NaN patterns everywhere, queued behind the products
        out, ne, _ = pa.fwd_host(h["q"], h["k"], h["v"], h["mem"], h["w_count"], stream=s,
                                 workspace=ws, synchronize=False, num_pieces=4)
    s.synchronize()
    assert torch.equal(out, ro) and torch.equal(ne, rn)


def test_host_pipeline_overlapping_steps_two_streams():
    """Consecutive steps pipelined the way a training or serving loop runs
    them: steps alternate between two caller streams and two workspaces, so
    step i + 1's inputs are copied in while step i's last pieces compute and
    its outputs are copied out.  Six steps on different inputs, each with its
    own pinned outputs, all enqueued before any synchronisation: each equals
    polar_attn_fwd on its inputs bit for bit."""
    import long_context_attention_causal_gb300 as pa
    B, H, T, d = 2, 4, 2048, 128
    nbytes = pa.fwd_host_workspace_bytes(B, H, T, d)
    ws = [torch.empty(nbytes, device=dev(), dtype=torch.uint8) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    steps = []
    for i in range(6):
        x = _inputs(B, H, T, d, "bf16", 90 + i)
        h = {k: x[k].contiguous().pin_memory() for k in ("q", "k", "v", "mem", "w_count")}
        out = torch.empty((B, H, T, d), dtype=torch.bfloat16).pin_memory()
        ne = torch.empty((B, H, T), dtype=torch.float32).pin_memory()
        steps.append((x, h, out, ne))
    for i, (_x, h, out, ne) in enumerate(steps):
        pa.fwd_host(h["q"], h["k"], h["v"], h["mem"], h["w_count"], out=out, n_eff=ne,
                    workspace=ws[i % 2], stream=streams[i % 2], synchronize=False)
    torch.cuda.synchronize()
    for x, _h, out, ne in steps:
        ro, rn, _ = _device_reference(x, want_conf=False)
        assert torch.equal(out, ro) and torch.equal(ne, rn)
