"""Paged, grouped-query split decode on the GPU vs the oracle.

The cache is paged ([num_pages, Hkv, page, d], scattered physical pages,
block table, ragged per-sequence lengths including one-token sequences) and
query heads are grouped (G = Hq / Hkv in {1, 2, 4, 8}).  Every call goes
through the C ABI via the binding.
"""
import pytest
import torch

from gpu_util import assert_within, dev, errors

pytestmark = pytest.mark.gpu

KEYS = ("q", "k_pages", "v_pages", "block_table", "seq_lens", "mem", "w_count")


def _run(x, num_splits=0, max_seq_len=None, consts=None):
    import long_context_attention_causal_gb300 as pa
    g = {k: x[k].to(dev()) for k in KEYS}
    out = torch.full_like(g["q"], float("nan"))
    out, neff, conf = pa.decode_paged(g["q"], g["k_pages"], g["v_pages"], g["block_table"],
                                      g["seq_lens"], g["mem"], g["w_count"],
                                      max_seq_len=max_seq_len, num_splits=num_splits,
                                      out=out, consts=consts, want_conf=True)
    torch.cuda.synchronize()
    return out, neff, conf


CASES = [
    # (B, Hq, Hkv, T, d, page, dtype, splits)
    (3, 8, 2, 300, 128, 64, "bf16", 0),
    (2, 4, 4, 100, 64, 16, "f32", 3),
    (2, 16, 2, 1000, 128, 32, "bf16", 0),
    (4, 8, 1, 777, 128, 128, "bf16", 5),
    (3, 4, 2, 513, 64, 8, "bf16", 0),
    (2, 8, 4, 2048, 128, 64, "f32", 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,T,d,page,dtype,splits", CASES)
def test_paged_decode_vs_oracle(B, Hq, Hkv, T, d, page, dtype, splits):
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    pa.device_status(reset=True)
    wl = inputs.custom_paged(B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, page=page, dtype=dtype,
                             seed=5000 + T + Hq)
    x = inputs.make_paged_decode(wl, "cpu")
    out, neff, conf = _run(x, splits)
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"])
    assert_within(errors(out, neff, conf, *ref), dtype, f"paged {B}x{Hq}/{Hkv}x{T}x{d} p{page}")
    assert pa.device_status() == 0


def test_paged_identity_layout_matches_contiguous_decode():
    """Pages in order with one query head per KV head: the paged kernel and
    the contiguous decode kernel agree (both GPU)."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    B, H, T, d, P = 2, 4, 1000, 128, 64
    wl = inputs.custom("decode", B=B, H=H, T=T, d=d, dtype="bf16", seed=5100)
    x = inputs.make_decode(wl, "cpu")
    npg = (T + P - 1) // P
    pad = npg * P - T
    k = torch.nn.functional.pad(x["k_cache"], (0, 0, 0, pad))
    v = torch.nn.functional.pad(x["v_cache"], (0, 0, 0, pad))
    kp = k.view(B, H, npg, P, d).permute(0, 2, 1, 3, 4).reshape(B * npg, H, P, d).contiguous()
    vp = v.view(B, H, npg, P, d).permute(0, 2, 1, 3, 4).reshape(B * npg, H, P, d).contiguous()
    xp = {"q": x["q"], "k_pages": kp, "v_pages": vp,
          "block_table": torch.arange(B * npg, dtype=torch.int32).view(B, npg),
          "seq_lens": torch.full((B,), T, dtype=torch.int32), "mem": x["mem"],
          "w_count": x["w_count"]}
    po, pn, pc = _run(xp)
    g = {kk: x[kk].to(dev()) for kk in ("q", "k_cache", "v_cache", "mem", "w_count")}
    do, dn, dc = pa.decode(g["q"], g["k_cache"], g["v_cache"], g["mem"], g["w_count"],
                           want_conf=True)
    torch.cuda.synchronize()
    assert (po.float() - do.float()).abs().max().item() <= 1e-2
    assert (pn / dn - 1).abs().max().item() <= 1e-4
    assert (pc - dc).abs().max().item() <= 1e-4


def test_paged_second_order_floor():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=3, Hq=8, Hkv=2, T=600, d=128, page=32, dtype="bf16", seed=5200)
    x = inputs.make_paged_decode(wl, "cpu")
    out, neff, conf = _run(x, consts=pa.default_consts(floor_order=2))
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"], consts={"floor_order": 2})
    assert_within(errors(out, neff, conf, *ref), "bf16", "paged floor2")


def test_paged_bad_page_index_is_reported_not_read():
    """A page index past the pool is skipped on the device and reported as
    status 3; the other sequences are unaffected."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=3, Hq=4, Hkv=2, T=200, d=128, page=16, dtype="bf16",
                             seed=5300, ragged=False)
    x = inputs.make_paged_decode(wl, "cpu")
    bad = x["block_table"].clone()
    bad[1, 3] = x["k_pages"].shape[0] + 1000
    xb = dict(x, block_table=bad)
    pa.device_status(reset=True)
    out, neff, conf = _run(xb)
    assert pa.device_status(reset=True) == 3
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"])
    keep = [0, 2]
    e = errors(out[keep], neff[keep], conf[keep], ref[0][keep], ref[1][keep], ref[2][keep])
    assert_within(e, "bf16", "untouched sequences")
    assert torch.isfinite(out.float()).all()


def test_paged_length_beyond_bound_is_clamped_and_reported():
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom_paged(B=2, Hq=4, Hkv=2, T=256, d=64, page=32, dtype="bf16",
                             seed=5400, ragged=False)
    x = inputs.make_paged_decode(wl, "cpu")
    lens = x["seq_lens"].clone()
    lens[0] = 0  # no visible key
    pa.device_status(reset=True)
    out, neff, conf = _run(dict(x, seq_lens=lens), max_seq_len=256)
    assert pa.device_status(reset=True) == 3
    # a row with no visible key: direction and count vanish, memory passes
    torch.testing.assert_close(out[0].float().cpu(), x["mem"][0].float(), rtol=0, atol=1e-6)
    assert (neff[0] == 0).all() and (conf[0] == 0).all()


def test_paged_gqa_32k_sampled():
    """The full paged workload (B=32, Hq=16, Hkv=4, 32K tokens, 64-token
    pages) in the bench's launch configuration, sampled sequences against
    the oracle."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.PAGED_WORKLOADS["paged_gqa_32k"]
    x = inputs.make_paged_decode(wl, dev())
    pa.device_status(reset=True)
    out, neff, conf = pa.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                                      x["seq_lens"], x["mem"], x["w_count"],
                                      max_seq_len=wl.T, want_conf=True)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    assert torch.isfinite(out.float()).all()
    for b in (0, 13, 31):
        pages = x["block_table"][b].long()
        ref = oracle_decode_paged(x["q"][b:b + 1].cpu(), x["k_pages"][pages].cpu(),
                                  x["v_pages"][pages].cpu(),
                                  torch.arange(len(pages), dtype=torch.int32)[None],
                                  x["seq_lens"][b:b + 1].cpu(), x["mem"][b:b + 1].cpu(),
                                  x["w_count"].cpu())
        e = errors(out[b:b + 1], neff[b:b + 1], conf[b:b + 1], *ref)
        assert_within(e, "bf16", f"paged_gqa_32k b={b}")


def _poison_tail_rows(x, value=float("nan")):
    """Rows of each sequence's last page past its length set to `value` in
    both K and V (cache memory that the sequence does not own)."""
    kp, vp = x["k_pages"].clone(), x["v_pages"].clone()
    P = kp.shape[2]
    for b in range(x["seq_lens"].shape[0]):
        n = int(x["seq_lens"][b])
        if n % P:
            pg = int(x["block_table"][b, (n - 1) // P])
            kp[pg, :, n % P:] = value
            vp[pg, :, n % P:] = value
    return dict(x, k_pages=kp, v_pages=vp)


@pytest.mark.parametrize("d,page,G", [(128, 64, 4), (64, 16, 2), (128, 256, 8)])
def test_paged_rows_past_the_end_are_never_used(d, page, G):
    """NaN in the cache rows past each sequence's end (inside its last page)
    must not reach the output: the keys are masked and their V rows are read
    as zeros."""
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=4, Hq=2 * G, Hkv=2, T=700, d=d, page=page, dtype="bf16",
                             seed=5500 + page)
    x = inputs.make_paged_decode(wl, "cpu")
    out, neff, conf = _run(_poison_tail_rows(x))
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"])
    assert torch.isfinite(out.float()).all()
    assert_within(errors(out, neff, conf, *ref), "bf16", f"poisoned tails d{d} p{page}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_paged_growing_logits(dtype):
    """Key norms rising 12x along each sequence, plus one spike late in the
    sequence, so every head's running maximum keeps moving and jumps far
    beyond any rescale threshold between stages."""
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.custom_paged(B=3, Hq=8, Hkv=2, T=1500, d=128, page=32, dtype=dtype,
                             seed=5600)
    x = inputs.make_paged_decode(wl, "cpu")
    kp = x["k_pages"].float().clone()
    P = kp.shape[2]
    for b in range(x["seq_lens"].shape[0]):
        n = int(x["seq_lens"][b])
        for lp in range((n + P - 1) // P):
            pg = int(x["block_table"][b, lp])
            j = torch.arange(lp * P, lp * P + P, dtype=torch.float32)
            kp[pg] *= (1.0 + 11.0 * j / n).view(1, P, 1)
        if n > 40:
            spike = n - 17
            pg = int(x["block_table"][b, spike // P])
            kp[pg, :, spike % P] = x["q"][b, 0].float() * 9.0
    x = dict(x, k_pages=kp.to(x["k_pages"].dtype))
    out, neff, conf = _run(x)
    ref = oracle_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], x["mem"], x["w_count"])
    assert_within(errors(out, neff, conf, *ref), dtype, "paged growing logits")
