"""Shared helpers of the GPU parity tests (imported by test files only)."""
import numpy as np
import torch

# Tolerances of the parity bar: bf16 inputs -> out max-abs <= 2e-2 and n_eff
# relative <= 1e-2; fp32 inputs -> 1e-4 on both.  The gate (conf) is held to
# the same absolute bound as out.
TOL = {
    "bf16": {"out": 2e-2, "neff": 1e-2, "conf": 2e-2},
    "f32": {"out": 1e-4, "neff": 1e-4, "conf": 1e-4},
}


def dev():
    return torch.device("cuda:0")


def to_dev(x, keys):
    return {k: x[k].to(dev()) for k in keys}


def errors(out, neff, conf, ro, rn, rc):
    out = out.float().cpu().numpy() if isinstance(out, torch.Tensor) else out
    neff = neff.cpu().numpy() if isinstance(neff, torch.Tensor) else neff
    e = {
        "out": float(np.abs(out - ro).max()) if ro.size else 0.0,
        "neff": float(np.abs(neff / rn - 1).max()) if rn.size else 0.0,
    }
    if conf is not None:
        conf = conf.cpu().numpy() if isinstance(conf, torch.Tensor) else conf
        e["conf"] = float(np.abs(conf - rc).max()) if rc.size else 0.0
    return e


def assert_within(e, dtype, what=""):
    tol = TOL[dtype]
    bad = {k: v for k, v in e.items() if not (v <= tol[k])}
    assert not bad, f"{what}: errors {e} exceed {tol}"


def invariants_prefill(out, neff, conf):
    """Properties that hold at any size: finite outputs, 1 <= n_eff <= i+1
    (with fp32 slack), 0 <= conf <= 1."""
    T = neff.shape[-1]
    n = torch.arange(1, T + 1, device=neff.device, dtype=torch.float32)
    assert torch.isfinite(out.float()).all(), "non-finite out"
    assert torch.isfinite(neff).all(), "non-finite n_eff"
    assert (neff >= 1 - 1e-3).all(), "n_eff below 1"
    assert (neff <= n * (1 + 1e-3) + 1e-3).all(), "n_eff above visible keys"
    if conf is not None:
        assert ((conf >= 0) & (conf <= 1)).all(), "conf outside [0, 1]"
