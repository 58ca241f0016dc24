"""The Python binding checks every tensor's shape against q's before it
reaches the C ABI: the library takes its sizes from the integers it is
given, so a mismatched operand would otherwise be read or written out of
bounds.  Each case here must raise ValueError and launch nothing."""
import pytest
import torch

from gpu_util import dev

pytestmark = pytest.mark.gpu

B, H, T, d = 1, 2, 64, 64


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, device=dev(), dtype=dtype)


def _prefill():
    return dict(q=_t(B, H, T, d), k=_t(B, H, T, d), v=_t(B, H, T, d), mem=_t(B, H, T, d),
                w_count=_t(H, d, dtype=torch.float32))


@pytest.mark.parametrize("name,bad", [("k", (B, H, T - 1, d)), ("v", (B, H, T, d + 8)),
                                      ("mem", (B, H + 1, T, d)), ("w_count", (H, d - 8))])
def test_fwd_and_fwd_stats_reject_mismatched_shapes(name, bad):
    import long_context_attention_causal_gb300 as pa
    for fn in (pa.fwd, pa.fwd_stats):
        x = _prefill()
        x[name] = _t(*bad, dtype=x[name].dtype)
        with pytest.raises(ValueError):
            fn(**x)


def test_fwd_rejects_wrong_output_buffers():
    import long_context_attention_causal_gb300 as pa
    x = _prefill()
    with pytest.raises(ValueError):
        pa.fwd(**x, out=_t(B, H, T - 1, d))
    with pytest.raises(ValueError):
        pa.fwd(**x, n_eff=_t(B, H, T - 1, dtype=torch.float32))
    with pytest.raises(ValueError):
        pa.fwd(**x, conf=_t(B, H, T + 1, dtype=torch.float32))


@pytest.mark.parametrize("name", ["k", "v", "dout", "w_count"])
def test_bwd_rejects_mismatched_shapes(name):
    import long_context_attention_causal_gb300 as pa
    x = _prefill()
    args = dict(q=x["q"], k=x["k"], v=x["v"], w_count=x["w_count"], dout=_t(B, H, T, d))
    args[name] = _t(*(args[name].shape[:-1] + (d * 2,)), dtype=args[name].dtype)
    with pytest.raises(ValueError):
        pa.bwd(**args)


@pytest.mark.parametrize("name", ["k", "mem", "out", "dout", "w_count", "n_eff", "conf",
                                  "stats"])
def test_bwd_stats_rejects_mismatched_shapes(name):
    import long_context_attention_causal_gb300 as pa
    x = _prefill()
    args = dict(x, out=_t(B, H, T, d), dout=_t(B, H, T, d),
                n_eff=_t(B, H, T, dtype=torch.float32), conf=_t(B, H, T, dtype=torch.float32),
                stats=_t(B, H, T, 2, dtype=torch.float32))
    shape = list(args[name].shape)
    shape[-1] += 1
    args[name] = _t(*shape, dtype=args[name].dtype)
    with pytest.raises(ValueError):
        pa.bwd_stats(**args)


def test_decode_variants_reject_mismatched_shapes():
    import long_context_attention_causal_gb300 as pa
    Tkv = 256
    base = dict(q=_t(B, H, d), k_cache=_t(B, H, Tkv, d), v_cache=_t(B, H, Tkv, d),
                mem=_t(B, H, d), w_count=_t(H, d, dtype=torch.float32))
    for fn in (pa.decode, pa.decode_static_scratch):
        for name, bad in (("v_cache", _t(B, H, Tkv - 1, d)),
                          ("w_count", _t(H + 1, d, dtype=torch.float32))):
            with pytest.raises(ValueError):
                fn(**dict(base, **{name: bad}))
        with pytest.raises(ValueError):
            fn(**base, out=_t(B, H, d + 8))
        with pytest.raises(ValueError):
            fn(**base, n_eff=_t(B, H + 1, dtype=torch.float32))


def test_decode_paged_rejects_mismatched_tables():
    import long_context_attention_causal_gb300 as pa
    page, pages = 16, 8
    base = dict(q=_t(B, H, d), k_pages=_t(pages, H, page, d), v_pages=_t(pages, H, page, d),
                block_table=_t(B, 4, dtype=torch.int32), seq_lens=_t(B, dtype=torch.int32),
                mem=_t(B, H, d), w_count=_t(H, d, dtype=torch.float32))
    for name, bad in (("block_table", _t(B + 1, 4, dtype=torch.int32)),
                      ("seq_lens", _t(B + 1, dtype=torch.int32)),
                      ("w_count", _t(H, d + 8, dtype=torch.float32))):
        with pytest.raises(ValueError):
            pa.decode_paged(**dict(base, **{name: bad}))


def test_combine_rejects_mismatched_shapes():
    import long_context_attention_causal_gb300 as pa
    S = 4
    partials = _t(B, H, S, d + 4, dtype=torch.float32)
    w = _t(H, d, dtype=torch.float32)
    with pytest.raises(ValueError):
        pa.combine(partials, _t(B, H, d + 8), _t(B, H, d), w, 256)
    with pytest.raises(ValueError):
        pa.combine(partials, _t(B, H, d), _t(B, H, d), _t(H + 1, d, dtype=torch.float32), 256)
