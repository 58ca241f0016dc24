"""Calls from several host threads at once, each on its own CUDA stream.

The library keeps no per-call host state (tensor maps are built per call;
the host-buffer prefill and the backward's side stream are guarded by
mutexes), so concurrent calls must give exactly the results of the same
calls made one after another.  Four threads each run a mix of the public
calls -- the bf16 prefill at d = 128 and 64, the training pair (forward
with statistics, backward from them), the split decode, the paged decode,
the memory step and the host-buffer prefill -- several times on their own
stream and output buffers; every result is compared bit for bit with a
serial reference run, and the device status word must stay 0.
"""
import threading

import pytest
import torch

from gpu_util import dev

pytestmark = pytest.mark.gpu


def _inputs():
    from long_context_attention_causal_gb300 import inputs
    d = dev()
    x = {}
    x["p128"] = inputs.make_prefill(inputs.custom("prefill", B=1, H=4, T=1000, d=128,
                                                  dtype="bf16", seed=301, needles=2), d)
    x["p64"] = inputs.make_prefill(inputs.custom("prefill", B=2, H=2, T=700, d=64,
                                                 dtype="bf16", seed=302), d)
    g = torch.Generator(device=d)
    g.manual_seed(303)
    x["dout"] = torch.randn(x["p128"]["q"].shape, generator=g, device=d).to(torch.bfloat16)
    x["dec"] = inputs.make_decode(inputs.custom("decode", B=2, H=4, T=3000, d=128,
                                                dtype="bf16", seed=304), d)
    wl = inputs.PagedWorkload("threads_paged", 3, 8, 2, 1500, 128, 64, "bf16", 305,
                              ragged=True)
    x["paged"] = inputs.make_paged_decode(wl, d)
    x["paged_T"] = wl.T
    x["mem"] = inputs.make_memory(inputs.MemoryWorkload("threads_mem", 4, 4, 3, 128, "bf16",
                                                        306), d)
    hp = inputs.make_prefill(inputs.custom("prefill", B=1, H=3, T=900, d=128, dtype="bf16",
                                           seed=307), "cpu")
    x["host"] = {k: (t.pin_memory() if k != "needles" and torch.is_tensor(t) else t)
                 for k, t in hp.items()}
    return x


def _work(pa, x, stream):
    """One round of every call on `stream`; returns the results (device
    tensors and pinned host tensors), complete once the stream is."""
    r = {}
    with torch.cuda.stream(stream):
        p = x["p128"]
        r["fwd128"] = pa.fwd(p["q"], p["k"], p["v"], p["mem"], p["w_count"], want_conf=True)
        p = x["p64"]
        r["fwd64"] = pa.fwd(p["q"], p["k"], p["v"], p["mem"], p["w_count"], want_conf=True)
        p = x["p128"]
        out, ne, cf, st = pa.fwd_stats(p["q"], p["k"], p["v"], p["mem"], p["w_count"])
        r["stats"] = (out, ne, cf, st)
        r["bwd"] = pa.bwd_stats(p["q"], p["k"], p["v"], p["mem"], p["w_count"], out, ne, cf,
                                st, x["dout"])
        c = x["dec"]
        r["dec"] = pa.decode(c["q"], c["k_cache"], c["v_cache"], c["mem"], c["w_count"],
                             want_conf=True)
        c = x["paged"]
        r["paged"] = pa.decode_paged(c["q"], c["k_pages"], c["v_pages"], c["block_table"],
                                     c["seq_lens"], c["mem"], c["w_count"],
                                     max_seq_len=x["paged_T"], want_conf=True)
        m = x["mem"]
        state = m["state"].clone()
        r["mem"] = (pa.memory_step(state, m["q"], m["k"], m["v"], m["alpha"], m["beta"]), state)
        h = x["host"]
        out_h = torch.empty(h["q"].shape, dtype=h["q"].dtype).pin_memory()
        ne_h = torch.empty(h["q"].shape[:3], dtype=torch.float32).pin_memory()
        r["host"] = pa.fwd_host(h["q"], h["k"], h["v"], h["mem"], h["w_count"], out=out_h,
                                n_eff=ne_h, synchronize=False)
    return r


def _flat(r):
    out = []
    for key in sorted(r):
        for t in r[key]:
            if t is not None:
                out.append((key, t))
    return out


def test_concurrent_calls_from_four_threads():
    import long_context_attention_causal_gb300 as pa
    x = _inputs()
    pa.device_status(reset=True)
    s0 = torch.cuda.Stream()
    ref = _flat(_work(pa, x, s0))
    s0.synchronize()
    ref = [(k, t.clone()) for k, t in ref]

    n_threads, n_rounds = 4, 3
    results = [None] * n_threads
    errors = []

    def run(i):
        try:
            s = torch.cuda.Stream()
            got = [_flat(_work(pa, x, s)) for _ in range(n_rounds)]
            s.synchronize()
            results[i] = got
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert pa.device_status() == 0
    for i in range(n_threads):
        for rnd in results[i]:
            assert len(rnd) == len(ref)
            for (k, a), (_, b) in zip(ref, rnd):
                assert torch.equal(a, b), f"thread {i}: {k} differs from the serial run"
