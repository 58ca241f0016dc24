"""GPU vs oracle at the largest sizes the prefill and the decode are run at.

* A prefill whose tensors hold more than 2^31 elements (B1 H260 T65536
  d128 bf16: 2.18e9 elements, 4.4 GB per tensor): every byte and element
  offset past 2^31 goes through the TMA maps, the epilogue's stores and the
  per-row outputs.  Compared with the oracle on the heads on both sides of
  the 2^31-element boundary (head 256 starts exactly on it) and the last.
* A one-million-token causal row (B1 H1 T2^20 d128 bf16, 16 planted
  needles): the temperature law and the null floor at n = 2^20, 8,192
  query tiles of one head.
* A decode against a cache of 2^20 keys per head.
* The backward (forward with row statistics, then the gradients) on
  tensors of more than 2^31 elements.
* The gated-delta memory step on a state of more than 2^31 elements.
* The paged, grouped decode against a page pool of more than 2^31
  elements.

Inputs are drawn on the device by the seeded generator of the workloads
(the same recipe as the named workloads: q, k, v ~ N(0, 1), mem ~ N(0, 0.1),
w_count ~ N(0, 0.02), needles as in needles_4k); the oracle reads the same
rounded tensors.  Rows compared: the first 64, rows around every
power-of-two context length from the 2K temperature knee on, the last 64,
needle rows and seeded random rows; the properties that hold at any size
are checked at every row.  Each test prints the largest errors it saw.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_within, dev, errors, invariants_prefill

pytestmark = pytest.mark.gpu


def _pa():
    import long_context_attention_causal_gb300 as pa
    return pa


def _rows(T, extra, seed, n_random):
    g = np.random.default_rng(seed)
    rows = set(range(min(T, 64)))
    c = 2048
    while c <= T:
        rows.update(r for r in (c - 2, c - 1, c, c + 1) if 0 <= r < T)
        c *= 2
    rows.update(range(max(0, T - 64), T))
    rows.update(extra)
    rows.update(g.integers(0, T, n_random).tolist())
    return sorted(rows)


def _compare_head(x, out, neff, conf, b, h, rows, what):
    from oracle import oracle_rows
    sl = lambda t: t[b, h].cpu()  # noqa: E731
    ro, rn, rc = oracle_rows(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["mem"]),
                             x["w_count"][h].cpu(), rows)
    ridx = torch.tensor(rows)
    e = errors(out[b, h].cpu()[ridx], neff[b, h].cpu()[ridx], conf[b, h].cpu()[ridx],
               ro, rn, rc)
    assert_within(e, "bf16", f"{what} head ({b},{h})")
    return e


def _report(name, worst, n):
    print(f"[parity] {name}: {n} rows compared, max |out err| {worst['out']:.3e}, "
          f"max n_eff rel err {worst['neff']:.3e}, max |conf err| {worst['conf']:.3e}")


def _run_prefill(wl):
    from long_context_attention_causal_gb300 import inputs
    x = inputs.make_prefill(wl, dev())
    out, neff, conf = _pa().fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"],
                                want_conf=True)
    torch.cuda.synchronize()
    return x, out, neff, conf


def test_prefill_past_2g_elements():
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.Workload("heads260_64k", "prefill", 1, 260, 65536, 128, "bf16", 11)
    x, out, neff, conf = _run_prefill(wl)
    B, H, T, d = x["q"].shape
    assert B * H * T * d > 2 ** 31
    assert 256 * T * d == 2 ** 31  # head 256 starts on the boundary
    invariants_prefill(out, neff, conf)
    worst, n = {}, 0
    for h in (0, 255, 256, 259):
        rows = _rows(T, [], 101 + h, 256)
        e = _compare_head(x, out, neff, conf, 0, h, rows, "heads260_64k")
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
        n += len(rows)
    _report("B1 H260 T65536 d128 (2.18e9 elements per tensor), heads 0/255/256/259",
            worst, n)
    del x, out, neff, conf
    torch.cuda.empty_cache()


def test_prefill_million_token_row():
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.Workload("million_1h", "prefill", 1, 1, 1 << 20, 128, "bf16", 12,
                         needles=16)
    x, out, neff, conf = _run_prefill(wl)
    T = x["q"].shape[2]
    invariants_prefill(out, neff, conf)
    needle_rows = [i for (_b, _h, i, _j) in x["needles"]]
    assert len(needle_rows) == 16
    rows = _rows(T, needle_rows, 113, 64)
    e = _compare_head(x, out, neff, conf, 0, 0, rows, "million_1h")
    _report("B1 H1 T1048576 d128, 16 needles", e, len(rows))
    del x, out, neff, conf
    torch.cuda.empty_cache()


def test_decode_million_keys():
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode
    wl = inputs.Workload("decode_1m", "decode", 1, 2, 1 << 20, 128, "bf16", 13)
    x = inputs.make_decode(wl, dev())
    out, neff, conf = _pa().decode(x["q"], x["k_cache"], x["v_cache"], x["mem"],
                                   x["w_count"], want_conf=True)
    torch.cuda.synchronize()
    ro, rn, rc = oracle_decode(x["q"].cpu(), x["k_cache"].cpu(), x["v_cache"].cpu(),
                               x["mem"].cpu(), x["w_count"].cpu())
    e = errors(out, neff, conf, ro, rn, rc)
    assert_within(e, "bf16", "decode_1m")
    print(f"[parity] decode B1 H2 Tkv1048576 d128: max |out err| {e['out']:.3e}, "
          f"max n_eff rel err {e['neff']:.3e}, max |conf err| {e['conf']:.3e}")


def _close_scaled(got, ref, what, tol=2e-2):
    """Held to tol of the gradient's largest magnitude (the bf16 backward's
    bar), with an absolute floor of 1e-6 for gradients that vanish."""
    got = got.detach().float().cpu().numpy()
    scale = max(float(np.abs(ref).max()), 1e-6)
    err = float(np.abs(got - ref).max())
    assert err <= tol * scale + 1e-6, f"{what}: max err {err:.3e} vs scale {scale:.3e}"
    return err / scale


def test_backward_past_2g_elements():
    """The training pair (forward keeping its row statistics, backward from
    them) on B1 H1040 T16384 d128: 2.18e9 elements per tensor, head 1024
    starting on the 2^31-element boundary.  dq at sampled rows, dk and dv at
    sampled keys, dw of the head, against the sampled oracle (exact per
    output, fp64) on heads 1023, 1024 and 1039."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_bwd_sampled
    wl = inputs.Workload("heads1040_16k", "prefill", 1, 1040, 16384, 128, "bf16", 14)
    x = inputs.make_prefill(wl, dev())
    B, H, T, d = x["q"].shape
    assert 1024 * T * d == 2 ** 31
    gen = torch.Generator(device=dev())
    gen.manual_seed(15)
    g = torch.randn(x["q"].shape, generator=gen, device=dev()).to(x["q"].dtype)
    out, ne, cf, st = pa.fwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    dq, dk, dv, dw = pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], out, ne, cf,
                                  st, g)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    del out, ne, cf, st
    rng = np.random.default_rng(16)
    rows = sorted(set([0, 1, 127, 128, 2047, 2048, 8191, T - 1] +
                      rng.integers(0, T, 12).tolist()))
    keys = sorted(set([0, 1, 128, 2048, T - 2, T - 1] + rng.integers(0, T, 6).tolist()))
    worst = {}
    for h in (1023, 1024, 1039):
        cpu = lambda t: t[0, h].cpu()  # noqa: E731
        gh = cpu(g)
        ref = oracle_bwd_sampled(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), x["w_count"][h].cpu(),
                                 gh, rows, keys)
        dw_ref = (ref["count"][:, None] * gh.double().numpy()).sum(axis=0)
        for name, got, r in (("dq", dq[0, h, rows], ref["dq"]), ("dk", dk[0, h, keys], ref["dk"]),
                             ("dv", dv[0, h, keys], ref["dv"]), ("dw", dw[h], dw_ref)):
            worst[name] = max(worst.get(name, 0.0), _close_scaled(got, r, f"{name} head {h}"))
    for name, tt in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(tt).all(), name
    print("[parity] backward B1 H1040 T16384 d128 (2.18e9 elements per tensor), heads "
          "1023/1024/1039: max err / scale " +
          ", ".join(f"{k} {v:.2e}" for k, v in worst.items()))
    del x, g, dq, dk, dv, dw
    torch.cuda.empty_cache()


def test_memory_step_past_2g_state_elements():
    """The in-place gated-delta step on 139,264 heads of d = 128 (a state of
    2.28e9 fp32 elements; head 131,072 starts on the 2^31-element boundary),
    two tokens per head: the heads around the boundary and the last one
    against the oracle, state and memory stream."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_memory_step
    wl = inputs.MemoryWorkload("mem_139k", 1088, 128, 2, 128, "bf16", 17)
    x = inputs.make_memory(wl, dev())
    B, H, d = wl.B, wl.H, wl.d
    assert B * H * d * d > 2 ** 31 and 131072 * d * d == 2 ** 31
    picks = [divmod(bh, H) for bh in (0, 131071, 131072, B * H - 1)]
    S0 = {bh: x["state"][bh[0], bh[1]].clone() for bh in picks}
    mem = pa.memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    torch.cuda.synchronize()
    worst_s, worst_m = 0.0, 0.0
    for (b, h) in picks:
        sl = lambda t: t[b:b + 1, h:h + 1].cpu()  # noqa: E731
        S_ref, mem_ref = oracle_memory_step(S0[(b, h)][None, None].cpu(), sl(x["q"]),
                                            sl(x["k"]), sl(x["v"]), sl(x["alpha"]),
                                            sl(x["beta"]))
        es = float(np.abs(sl(x["state"]).double().numpy() - S_ref).max())
        em = float(np.abs(sl(mem).float().numpy() - mem_ref).max())
        assert es <= 1e-4 and em <= 2e-2, f"head ({b},{h}): state {es:.2e}, mem {em:.2e}"
        worst_s, worst_m = max(worst_s, es), max(worst_m, em)
    assert torch.isfinite(mem.float()).all()
    print(f"[parity] memory step B1088 H128 T2 d128 (2.28e9 state elements): max |state err| "
          f"{worst_s:.2e}, max |mem err| {worst_m:.2e}")
    del x, mem
    torch.cuda.empty_cache()


def test_paged_decode_past_2g_pool_elements():
    """The paged, grouped decode (tensor-core kernel) against a pool of
    33,792 pages of 8 KV heads x 64 tokens x d 128 (2.21e9 elements per
    pool; pages past index 32,768 lie beyond 2^31 elements), 66 sequences of
    32K tokens over a seeded permutation of the pool, 4 query heads per KV
    head: sampled sequences against the oracle."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_decode_paged
    wl = inputs.PagedWorkload("paged_66x32k", 66, 32, 8, 32768, 128, 64, "bf16", 18)
    x = inputs.make_paged_decode(wl, dev())
    assert x["k_pages"].numel() > 2 ** 31
    pa.device_status(reset=True)
    out, neff, conf = pa.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                                      x["seq_lens"], x["mem"], x["w_count"],
                                      max_seq_len=wl.T, want_conf=True)
    torch.cuda.synchronize()
    assert pa.device_status() == 0
    assert torch.isfinite(out.float()).all()
    beyond = 2 ** 31 // (wl.Hkv * wl.page * wl.d)
    worst = {}
    for b in (0, 33, 65):
        pages = x["block_table"][b].long()
        assert int(pages.max()) >= beyond  # the sequence reads past the boundary
        ref = oracle_decode_paged(x["q"][b:b + 1].cpu(), x["k_pages"][pages].cpu(),
                                  x["v_pages"][pages].cpu(),
                                  torch.arange(len(pages), dtype=torch.int32)[None],
                                  x["seq_lens"][b:b + 1].cpu(), x["mem"][b:b + 1].cpu(),
                                  x["w_count"].cpu())
        e = errors(out[b:b + 1], neff[b:b + 1], conf[b:b + 1], *ref)
        assert_within(e, "bf16", f"paged_66x32k b={b}")
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
    print(f"[parity] paged decode B66 Hq32 Hkv8 T32768 d128 page64 (2.21e9 pool elements), "
          f"sequences 0/33/65: max |out err| {worst['out']:.3e}, max n_eff rel err "
          f"{worst['neff']:.3e}, max |conf err| {worst['conf']:.3e}")
    del x, out, neff, conf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,H,T,d", [(16, 256, 100, 128), (8, 512, 300, 64)])
def test_prefill_many_short_heads(B, H, T, d):
    """Thousands of short heads (the multi-wave CTA order with its L2-sized
    head groups over 4,096 (b, h) slices of one or two query tiles, ragged
    tails): every row of heads spread over the grid against the oracle."""
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.Workload(f"short_{B}x{H}x{T}x{d}", "prefill", B, H, T, d, "bf16", 19,
                         needles=1)
    x, out, neff, conf = _run_prefill(wl)
    invariants_prefill(out, neff, conf)
    worst, n = {}, 0
    for (b, h) in [(0, 0), (0, H - 1), (B // 2, H // 3), (B - 1, 0), (B - 1, H - 1)]:
        rows = list(range(T))
        e = _compare_head(x, out, neff, conf, b, h, rows, wl.name)
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
        n += len(rows)
    _report(f"B{B} H{H} T{T} d{d} ({B * H} heads), five heads in full", worst, n)
