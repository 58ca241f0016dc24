"""The entry points are capturable into CUDA graphs (serving loops replay a
captured decode step instead of relaunching): with caller-owned workspaces
and outputs they allocate nothing and never synchronise the host, so a
captured call replayed on new inputs (copied into the captured buffers)
gives what an eager call gives."""
import pytest
import torch

from gpu_util import dev

pytestmark = pytest.mark.gpu


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the graph (function attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_graph_replay():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    B, H, T, d = 4, 8, 3000, 128
    x = inputs.make_decode(inputs.custom("decode", B=B, H=H, T=T, d=d, dtype="bf16", seed=61), dev())
    ws = torch.empty(pa.decode_workspace_bytes(B, H, T, d), device=dev(), dtype=torch.uint8)
    out = torch.empty_like(x["q"])
    ne = torch.empty((B, H), device=dev())
    g = _capture(lambda: pa.decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"],
                                   workspace=ws, out=out, n_eff=ne))
    for seed in (62, 63):
        y = inputs.make_decode(inputs.custom("decode", B=B, H=H, T=T, d=d, dtype="bf16",
                                             seed=seed), dev())
        for k in ("q", "k_cache", "v_cache", "mem", "w_count"):
            x[k].copy_(y[k])
        g.replay()
        torch.cuda.synchronize()
        eo, en, _ = pa.decode(y["q"], y["k_cache"], y["v_cache"], y["mem"], y["w_count"])
        torch.cuda.synchronize()
        assert torch.equal(out, eo) and torch.equal(ne, en)


def test_paged_decode_and_memory_step_graph_replay():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom_paged(B=4, Hq=8, Hkv=2, T=2000, d=128, page=64, dtype="bf16", seed=64)
    x = inputs.make_paged_decode(wl, dev())
    ws = torch.empty(max(16, pa.decode_paged_workspace_bytes(4, 8, 2, 2000, 128)), device=dev(),
                     dtype=torch.uint8)
    out = torch.empty_like(x["q"])
    ne = torch.empty((4, 8), device=dev())
    m = inputs.make_memory(inputs.MemoryWorkload("graph", 4, 8, 1, 128, "bf16", 65), dev())
    state0 = m["state"].clone()
    mem_out = torch.empty_like(m["q"])

    def step():
        pa.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                        x["mem"], x["w_count"], workspace=ws, out=out, n_eff=ne)
        pa.memory_step(m["state"], m["q"], m["k"], m["v"], m["alpha"], m["beta"], mem=mem_out)

    g = _capture(step)
    m["state"].copy_(state0)
    g.replay()
    torch.cuda.synchronize()
    eo, en, _ = pa.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                                x["seq_lens"], x["mem"], x["w_count"])
    st = state0.clone()
    em = pa.memory_step(st, m["q"], m["k"], m["v"], m["alpha"], m["beta"])
    torch.cuda.synchronize()
    assert torch.equal(out, eo) and torch.equal(ne, en)
    assert torch.equal(m["state"], st)
    assert torch.equal(mem_out, em)


def test_prefill_graph_replay():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    x = inputs.make_prefill(inputs.custom("prefill", B=1, H=4, T=1500, d=128, dtype="bf16",
                                          seed=66, needles=2), dev())
    out = torch.empty_like(x["q"])
    ne = torch.empty(x["q"].shape[:3], device=dev())
    g = _capture(lambda: pa.fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], out=out,
                                n_eff=ne))
    y = inputs.make_prefill(inputs.custom("prefill", B=1, H=4, T=1500, d=128, dtype="bf16",
                                          seed=67, needles=2), dev())
    for k in ("q", "k", "v", "mem", "w_count"):
        x[k].copy_(y[k])
    g.replay()
    torch.cuda.synchronize()
    eo, en, _ = pa.fwd(y["q"], y["k"], y["v"], y["mem"], y["w_count"])
    torch.cuda.synchronize()
    assert torch.equal(out, eo) and torch.equal(ne, en)


def test_backward_graph_replay():
    """The bf16 backward runs its dQ kernel on a library side stream, forked
    from and joined back into the caller's stream with events; captured into
    a graph that fork and join become graph edges, and replays on new inputs
    (copied into the captured buffers) give bit-identical gradients to eager
    calls."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    B, H, T, d = 1, 4, 1000, 128

    def make(seed):
        x = inputs.make_prefill(inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16",
                                              seed=seed, needles=1), dev())
        g = torch.Generator(device=dev())
        g.manual_seed(seed)
        x["dout"] = torch.randn(x["q"].shape, generator=g, device=dev()).to(torch.bfloat16)
        return x

    x = make(66)
    ws = torch.empty(pa.bwd_workspace_bytes(B, H, T, d), device=dev(), dtype=torch.uint8)
    held = {}

    def call():
        held["grads"] = pa.bwd(x["q"], x["k"], x["v"], x["w_count"], x["dout"], workspace=ws)

    g = _capture(call)
    for seed in (67, 68):
        y = make(seed)
        for k in ("q", "k", "v", "w_count", "dout"):
            x[k].copy_(y[k])
        g.replay()
        torch.cuda.synchronize()
        eager = pa.bwd(y["q"], y["k"], y["v"], y["w_count"], y["dout"])
        torch.cuda.synchronize()
        for a, b in zip(held["grads"], eager):
            assert torch.equal(a, b)
