"""The bf16 prefill on grids of several waves of CTAs against the oracle.

Adjacent 128-row query tiles share a CTA there (heaviest pairs first); the
shapes below (many heads, d = 128 and 64) are chosen that way, with ragged
and odd tile counts: an odd number of tiles leaves a CTA with one tile
only, and a T that is not a multiple of 128 leaves rows past T in the last
tile.  fwd_stats (logsumexp and |a| per row) and the second-order floor go
through the same grids.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_within, errors, invariants_prefill, to_dev

pytestmark = pytest.mark.gpu

PKEYS = ("q", "k", "v", "mem", "w_count")


def _pa():
    import long_context_attention_causal_gb300 as pa
    return pa


def _run(x, **kw):
    g = to_dev(x, PKEYS)
    out = torch.full_like(g["q"], float("nan"))
    out, neff, conf = _pa().fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"], out=out,
                                want_conf=True, **kw)
    torch.cuda.synchronize()
    return out, neff, conf


@pytest.mark.parametrize("B,H,T,d", [(1, 160, 256, 128), (2, 80, 300, 128), (1, 96, 1000, 128),
                                     (3, 40, 1100, 128), (1, 48, 1300, 128), (1, 40, 2300, 128),
                                     (2, 12, 4224, 128), (2, 40, 1300, 64), (1, 24, 3000, 64)])
def test_multiwave_prefill_vs_oracle(B, H, T, d):
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16", seed=6000 + T + H,
                       needles=2, keyscale=True)
    x = inputs.make_prefill(wl, "cpu")
    out, neff, conf = _run(x)
    assert _pa().device_status() == 0
    invariants_prefill(out, neff, conf)
    ref = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    e = errors(out, neff, conf, *ref)
    print(f"[parity] multi-wave prefill B{B} H{H} T{T} d{d}: {e}")
    assert_within(e, "bf16", f"multi-wave {B}x{H}x{T}x{d}")


def test_multiwave_stats_and_second_order_floor():
    """fwd_stats (logsumexp and |a| per row) and floor_order = 2 on a grid of
    several waves."""
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_fwd, oracle_row_stats
    pa = _pa()
    wl = inputs.custom("prefill", B=1, H=80, T=640, d=128, dtype="bf16", seed=6200, needles=2)
    x = inputs.make_prefill(wl, "cpu")
    g = to_dev(x, PKEYS)
    out, neff, conf, st = pa.fwd_stats(g["q"], g["k"], g["v"], g["mem"], g["w_count"])
    torch.cuda.synchronize()
    hs = slice(0, 4)
    rs = oracle_row_stats(x["q"][:, hs], x["k"][:, hs], x["v"][:, hs])
    stc = st.cpu().numpy()[:, hs]
    assert np.abs(stc[..., 0] - rs["lse"]).max() <= 2e-3
    assert np.abs(stc[..., 1] - rs["anorm"]).max() <= 2e-2 * rs["anorm"].max()
    ref = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
    assert_within(errors(out, neff, conf, *ref), "bf16", "multi-wave fwd_stats")
    c2 = pa.default_consts(floor_order=2)
    out2, neff2, conf2 = pa.fwd(g["q"], g["k"], g["v"], g["mem"], g["w_count"], consts=c2,
                                want_conf=True)
    torch.cuda.synchronize()
    ref2 = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"], consts={"floor_order": 2})
    assert_within(errors(out2, neff2, conf2, *ref2), "bf16", "multi-wave floor_order 2")
