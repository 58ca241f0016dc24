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
