"""Edges of the accepted sizes, against the oracle.

* A decode over 131,072 (b, h) problems of a few keys each (one split per
  problem, the combine grid at its widest).
* The paged decode with the largest page the call accepts (1,024 tokens:
  several TMA boxes per page slice) and with the smallest (8 tokens: many
  pages per stage), ragged sequence lengths, bf16 and fp32.
* The memory step over 1,000 tokens per head (the state stays in registers
  for the whole sequence).
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, assert_within, dev, errors

pytestmark = pytest.mark.gpu


def _pa():
    import long_context_attention_causal_gb300 as pa
    return pa


def test_decode_many_problems_few_keys():
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    B, H, Tkv, d = 1024, 128, 5, 128
    x = inputs.make_decode(inputs.custom("decode", B=B, H=H, T=Tkv, d=d, dtype="bf16",
                                         seed=9100), dev())
    assert _pa().decode_num_splits(B, H, Tkv, d) == 1
    out, neff, conf = _pa().decode(x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"],
                                   want_conf=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert ((neff >= 1 - 1e-3) & (neff <= Tkv * 1.001)).all()
    for b in (0, 511, 1023):
        sl = lambda t: t[b:b + 1].cpu()  # noqa: E731
        ref = oracle_decode(sl(x["q"]), sl(x["k_cache"]), sl(x["v_cache"]), sl(x["mem"]),
                            x["w_count"].cpu())
        assert_within(errors(out[b:b + 1], neff[b:b + 1], conf[b:b + 1], *ref), "bf16",
                      f"decode b={b}")


@pytest.mark.parametrize("page,dtype", [(1024, "bf16"), (1024, "f32"), (8, "bf16")])
def test_paged_decode_page_size_extremes(page, dtype):
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=3, Hq=8, Hkv=2, T=5000, d=128, page=page, dtype=dtype,
                             seed=9200 + page)
    x = inputs.make_paged_decode(wl, "cpu")
    keys = ("q", "k_pages", "v_pages", "block_table", "seq_lens", "mem", "w_count")
    g = {k: x[k].to(dev()) for k in keys}
    _pa().device_status(reset=True)
    out, neff, conf = _pa().decode_paged(*(g[k] for k in keys), max_seq_len=wl.T,
                                         want_conf=True)
    torch.cuda.synchronize()
    assert _pa().device_status() == 0
    ref = oracle_decode_paged(*(x[k] for k in keys))
    assert_within(errors(out, neff, conf, *ref), dtype, f"paged page={page} {dtype}")


def test_memory_step_long_sequence():
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_memory_step
    x = inputs.make_memory(inputs.MemoryWorkload("mem_long", 1, 2, 1000, 128, "f32", 9300),
                           "cpu")
    S_ref, mem_ref = oracle_memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"],
                                        x["beta"])
    g = {k: t.to(dev()) for k, t in x.items()}
    mem = _pa().memory_step(g["state"], g["q"], g["k"], g["v"], g["alpha"], g["beta"])
    torch.cuda.synchronize()
    # fp32 state on both sides; 1,000 updates accumulate rounding of order
    # 1e-6 relative on entries of order 1
    es = float(np.abs(g["state"].cpu().double().numpy() - S_ref).max())
    em = float(np.abs(mem.cpu().double().numpy() - mem_ref).max())
    print(f"[parity] memory step B1 H2 T1000 d128 fp32: max |state err| {es:.2e}, "
          f"max |mem err| {em:.2e}")
    assert es <= 1e-4 and em <= TOL["f32"]["out"]
