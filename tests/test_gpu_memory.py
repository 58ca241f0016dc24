"""Gated-delta memory step on the GPU vs the oracle.

The state is updated in place; the memory stream it returns is what the
prefill and decode calls add.  Every call goes through the C ABI.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, dev

pytestmark = pytest.mark.gpu


def _case(B, H, T, d, dtype, seed):
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.MemoryWorkload(f"m{seed}", B, H, T, d, dtype, seed)
    return inputs.make_memory(wl, "cpu")


def _gpu(x):
    import long_context_attention_causal_gb300 as pa
    g = {k: t.to(dev()) for k, t in x.items()}
    mem = pa.memory_step(g["state"], g["q"], g["k"], g["v"], g["alpha"], g["beta"])
    torch.cuda.synchronize()
    return g["state"].cpu().double().numpy(), mem.float().cpu().numpy()


@pytest.mark.parametrize("B,H,T,d,dtype", [(2, 3, 1, 128, "f32"), (1, 2, 17, 64, "f32"),
                                           (2, 2, 5, 128, "bf16"), (1, 1, 64, 128, "f32"),
                                           (3, 1, 1, 64, "bf16")])
def test_memory_step_vs_oracle(B, H, T, d, dtype):
    from oracle import oracle_memory_step
    x = _case(B, H, T, d, dtype, 6000 + T + d)
    S_ref, mem_ref = oracle_memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"],
                                        x["beta"])
    S, mem = _gpu(x)
    assert np.abs(S - S_ref).max() <= 1e-4          # fp32 state on both sides
    assert np.abs(mem - mem_ref).max() <= TOL[dtype]["out"]


def test_memory_step_delta_write_on_gpu():
    """alpha = beta = 1: after the step the state returns v at k^."""
    x = _case(2, 2, 1, 128, "f32", 6100)
    x["alpha"].fill_(1.0)
    x["beta"].fill_(1.0)
    S, _ = _gpu(x)
    k = x["k"].double().numpy()[:, :, 0]
    kh = k / np.linalg.norm(k, axis=-1, keepdims=True)
    got = np.einsum("bhij,bhj->bhi", S, kh)
    np.testing.assert_allclose(got, x["v"].double().numpy()[:, :, 0], atol=1e-4)


def test_memory_step_empty_is_noop():
    import long_context_attention_causal_gb300 as pa
    st = torch.zeros((1, 1, 64, 64), device=dev())
    z = torch.empty((1, 1, 0, 64), device=dev())
    a = torch.empty((1, 1, 0), device=dev())
    mem = pa.memory_step(st, z, z, z, a, a)
    assert mem.numel() == 0


def test_memstep_256_sampled():
    """The bench's memory workload (256 x 16 heads, d = 128, bf16, one
    step), sampled heads against the oracle."""
    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_memory_step
    wl = inputs.MEMORY_WORKLOADS["memstep_256"]
    x = inputs.make_memory(wl, dev())
    S0 = x["state"].clone()
    mem = pa.memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    torch.cuda.synchronize()
    for (b, h) in [(0, 0), (255, 15), (100, 7)]:
        sl = lambda t: t[b:b + 1, h:h + 1].cpu()  # noqa: E731
        S_ref, mem_ref = oracle_memory_step(sl(S0), sl(x["q"]), sl(x["k"]), sl(x["v"]),
                                            sl(x["alpha"]), sl(x["beta"]))
        assert np.abs(sl(x["state"]).double().numpy() - S_ref).max() <= 1e-4
        assert np.abs(sl(mem).float().numpy() - mem_ref).max() <= TOL["bf16"]["out"]
