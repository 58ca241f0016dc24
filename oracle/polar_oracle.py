"""ctypes wrapper of the plain-C fp64 oracle (``polar_oracle.c``).

Test infrastructure only: the tests, the smoke check and the bench's
CPU-baseline leg use it; the product path never imports it.  It shares no
code with the CUDA library.  The arithmetic lives in ``polar_oracle.c``;
this file only compiles it with gcc, marshals numpy arrays and upcasts
inputs exactly to fp64.

Constants (the pinned reading of "ATMA: Length-Invariant Language Modeling
via Polar Attention and Gated-Delta Compression Memory", §2.1 and §3):
  log_t0  = ln 2048   (training length 2K sets the temperature neutral point)
  kappa   = ln 2048   (tanh-of-log saturation scale)
  sigma_k = 1         (null model: key components iid N(0, 1))
  eps     = 1e-6      (unit-sphere projection guard)
  floor_order = 1     (leading-order null floor; 2 = second order)
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "polar_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpolar_oracle.so")

DEFAULT_CONSTS = {
    "log_t0": math.log(2048.0),
    "kappa": math.log(2048.0),
    "sigma_k": 1.0,
    "eps": 1e-6,
    "floor_order": 1,   # 2: second-order (Gumbel) expected-maximum floor
}

_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with gcc (host C only; no CUDA)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
             "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # POLAR_ORACLE_LIB points at a separately built copy (the mutation
            # test builds deliberately broken copies to show the pins bite)
            path = os.environ.get("POLAR_ORACLE_LIB") or build_oracle()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            c_int, c_long, c_double = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.oracle_polar_rows.argtypes = [
                dp, dp, dp, dp, dp, c_int, c_int, c_double, c_double, c_double,
                c_double, c_int, lp, c_long, c_int, c_long, dp, dp, dp, c_int]
            lib.oracle_polar_rows.restype = c_int
            lib.oracle_polar_fwd.argtypes = [
                dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_double,
                c_double, c_double, c_double, c_int, c_int, c_long, dp, dp, dp,
                c_int]
            lib.oracle_polar_fwd.restype = c_int
            lib.oracle_polar_decode.argtypes = [
                dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_double,
                c_double, c_double, c_double, c_int, c_int, c_long, dp, dp, dp,
                c_int]
            lib.oracle_polar_decode.restype = c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast to a C-contiguous fp64 numpy array (torch or numpy in)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _consts(consts):
    c = dict(DEFAULT_CONSTS)
    if consts:
        c.update(consts)
    return c["log_t0"], c["kappa"], c["sigma_k"], c["eps"], int(c["floor_order"])


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def oracle_fwd(q, k, v, mem, w, consts=None, mode="definition", tile=64,
               nthreads=None):
    """Causal prefill over all rows.

    q, k, v, mem: [B, H, T, d]; w: [H, d].  Returns (out [B,H,T,d],
    n_eff [B,H,T], conf [B,H,T]) as fp64 numpy arrays.
    mode: "definition" (two passes, full logit row) or "streamed" (tiles of
    `tile` keys with squared correction factors).
    """
    q, k, v, mem, w = map(_f64, (q, k, v, mem, w))
    B, H, T, d = q.shape
    out = np.empty((B, H, T, d))
    neff = np.empty((B, H, T))
    conf = np.empty((B, H, T))
    lib = _load()
    st = lib.oracle_polar_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w), B, H, T, d,
        *_consts(consts), 0 if mode == "definition" else 1, int(tile),
        _ptr(out), _ptr(neff), _ptr(conf), _threads(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_polar_fwd failed ({st})")
    return out, neff, conf


def oracle_rows(q, k, v, mem, w, rows, consts=None, mode="definition", tile=64,
                nthreads=None):
    """Selected causal rows of ONE head: q, k, v, mem [T, d]; w [d].

    rows: query indices i (row i sees keys 0..i).  Returns (out [R, d],
    n_eff [R], conf [R]).
    """
    q, k, v, mem, w = map(_f64, (q, k, v, mem, w))
    T, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = rows.shape[0]
    out = np.empty((R, d))
    neff = np.empty(R)
    conf = np.empty(R)
    lib = _load()
    st = lib.oracle_polar_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w), T, d, *_consts(consts),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), R,
        0 if mode == "definition" else 1, int(tile), _ptr(out), _ptr(neff),
        _ptr(conf), _threads(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_polar_rows failed ({st})")
    return out, neff, conf


def oracle_decode(q, k, v, mem, w, consts=None, nsplit=0, tile=64, nthreads=None):
    """Decode: q, mem [B, H, d]; k, v [B, H, Tkv, d]; w [H, d].

    nsplit = 0: definition form; nsplit >= 1: split-KV partials merged.
    Returns (out [B,H,d], n_eff [B,H], conf [B,H]).
    """
    q, k, v, mem, w = map(_f64, (q, k, v, mem, w))
    B, H, Tkv, d = k.shape
    out = np.empty((B, H, d))
    neff = np.empty((B, H))
    conf = np.empty((B, H))
    lib = _load()
    st = lib.oracle_polar_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w), B, H, Tkv, d,
        *_consts(consts), int(nsplit), int(tile), _ptr(out), _ptr(neff),
        _ptr(conf), _threads(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_polar_decode failed ({st})")
    return out, neff, conf


def oracle_decode_paged(q, k_pages, v_pages, block_table, seq_lens, mem, w,
                        consts=None, nsplit=0):
    """Decode against a paged cache with grouped-query heads.

    q, mem [B, Hq, d]; k_pages, v_pages [num_pages, Hkv, page, d];
    block_table [B, max_pages] (logical page -> physical page);
    seq_lens [B] (keys visible to sequence b, n = seq_lens[b]); w [Hq, d].
    Key j of sequence b is row j % page of physical page
    block_table[b, j // page]; query head h reads key/value head
    h // (Hq / Hkv).  The cache of each sequence is gathered into rows
    (data movement only) and the decode definition applied per sequence.
    Returns (out [B,Hq,d], n_eff [B,Hq], conf [B,Hq]).
    """
    q, mem, w = map(_f64, (q, mem, w))
    kp, vp = _f64(k_pages), _f64(v_pages)
    table = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table)
    lens = np.asarray(seq_lens.cpu() if hasattr(seq_lens, "cpu") else seq_lens)
    B, Hq, d = q.shape
    _, Hkv, P, _ = kp.shape
    G = Hq // Hkv
    out = np.empty((B, Hq, d))
    neff = np.empty((B, Hq))
    conf = np.empty((B, Hq))
    for b in range(B):
        n = int(lens[b])
        pages = table[b, : (n + P - 1) // P]
        # [pages, Hkv, P, d] -> [Hkv, pages * P, d], first n keys
        kb = kp[pages].transpose(1, 0, 2, 3).reshape(Hkv, -1, d)[:, :n]
        vb = vp[pages].transpose(1, 0, 2, 3).reshape(Hkv, -1, d)[:, :n]
        kh = np.repeat(kb, G, axis=0)[None]  # query head h -> kv head h // G
        vh = np.repeat(vb, G, axis=0)[None]
        o, ne, cf = oracle_decode(q[b:b + 1], kh, vh, mem[b:b + 1], w, consts=consts,
                                  nsplit=nsplit)
        out[b], neff[b], conf[b] = o[0], ne[0], cf[0]
    return out, neff, conf


def oracle_memory_step(state, q, k, v, alpha, beta, eps=1e-6):
    """Gated-delta memory over T tokens ("ATMA", §2.1 item 3: the memory
    channel's gated delta rule with L2-normalised keys and queries; §2.2:
    the in-place step kernel).  Reading of the words, per token t and head:
        k^ = k / max(|k|, eps),  q^ = q / max(|q|, eps)
        S  <- alpha_t * S (I - beta_t k^ k^T) + beta_t v_t k^T
        mem_t = S q^
    state [B, H, d, d] (S maps keys to values: mem = S q^), q, k, v
    [B, H, T, d], alpha, beta [B, H, T].  Returns (new state, mem [B,H,T,d])
    in fp64; the input state is not modified.
    """
    S = _f64(state).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    alpha, beta = _f64(alpha), _f64(beta)
    B, H, T, d = q.shape
    mem = np.empty((B, H, T, d))
    eye = np.eye(d)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                kh = k[b, h, t] / max(np.linalg.norm(k[b, h, t]), eps)
                qh = q[b, h, t] / max(np.linalg.norm(q[b, h, t]), eps)
                a, bt = alpha[b, h, t], beta[b, h, t]
                S[b, h] = a * S[b, h] @ (eye - bt * np.outer(kh, kh)) + bt * np.outer(v[b, h, t], kh)
                mem[b, h, t] = S[b, h] @ qh
    return S, mem


def oracle_bwd(q, k, v, mem, w, dout, consts=None):
    """Gradients of the causal prefill output (out only; n_eff and conf are
    diagnostics).  The definition of the forward is restated with dense fp64
    torch operations (whole T x T logit matrix per head) and differentiated
    by torch autograd.  q, k, v, mem, dout [B, H, T, d]; w [H, d].
    Returns dict(dq, dk, dv, dmem, dw) as fp64 numpy arrays.
    """
    import torch
    c = dict(DEFAULT_CONSTS)
    if consts:
        c.update(consts)
    t = lambda x: torch.as_tensor(_f64(x))  # noqa: E731
    q, k, v, mem, w, g = (t(x).requires_grad_(i < 5) for i, x in
                          enumerate((q, k, v, mem, w, dout)))
    B, H, T, d = q.shape
    n = torch.arange(1, T + 1, dtype=torch.float64)
    tau = torch.clamp(torch.log(n) / c["log_t0"], min=1.0)           # [T]
    s = tau[:, None] * (q @ k.transpose(-1, -2)) / math.sqrt(d)      # [B,H,T,T]
    mask = torch.ones(T, T, dtype=torch.bool).triu(1)
    s = s.masked_fill(mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                                  # [B,H,T]
    p = torch.exp(s - lse[..., None])
    a = p @ v
    an = a.norm(dim=-1)
    u = a / torch.clamp(an, min=c["eps"])[..., None]
    q2 = (p * p).sum(-1)
    qn = q.norm(dim=-1)
    sigma = tau * c["sigma_k"] * qn / math.sqrt(d)
    r = torch.sqrt(2.0 * torch.log(n))
    if int(c["floor_order"]) == 2:
        rr = torch.where(n >= 2, r, torch.ones_like(r))
        f = torch.where(n >= 2, rr - (torch.log(torch.log(torch.clamp(n, min=2.0)))
                                      + math.log(4 * math.pi)) / (2 * rr) + 0.5772156649015329 / rr,
                        torch.zeros_like(r))
    else:
        f = r
    conf = torch.sigmoid(lse - sigma * f)
    count = conf * torch.tanh(-torch.log(q2) / c["kappa"])
    out = u + count[..., None] * w[None, :, None, :] + mem
    (out * g).sum().backward()
    return {"dq": q.grad.numpy(), "dk": k.grad.numpy(), "dv": v.grad.numpy(),
            "dmem": mem.grad.numpy(), "dw": w.grad.numpy()}


def oracle_row_stats(q, k, v, consts=None):
    """Per-row statistics of the causal prefill's streaming state (ATMA
    §2.2: the running max and sum give the logsumexp of the scaled logits;
    §2.1: a = sum_j p_j v_j is the value the unit-sphere projection
    normalises).  Dense fp64 numpy, whole logit row per query:
    lse_i = log sum_{j<=i} exp(s_ij), s_ij = tau_i q_i.k_j / sqrt(d), and
    |a_i|.  q, k, v [B, H, T, d].  Returns dict(lse [B,H,T], anorm [B,H,T]).
    """
    c = dict(DEFAULT_CONSTS)
    if consts:
        c.update(consts)
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d = q.shape
    n = np.arange(1, T + 1, dtype=np.float64)
    tau = np.maximum(1.0, np.log(n) / c["log_t0"])
    s = tau[:, None] * np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(d)
    s = np.where(np.triu(np.ones((T, T), dtype=bool), 1), -np.inf, s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    lse = (m + np.log(l))[..., 0]
    a = np.einsum("bhij,bhjd->bhid", e / l, v)
    return {"lse": lse, "anorm": np.linalg.norm(a, axis=-1)}


def _floor_factor(n, order):
    """Expected-maximum factor of the null floor (leading or second order)."""
    r = np.sqrt(2.0 * np.log(n))
    if int(order) != 2:
        return r
    rr = np.where(n >= 2, r, 1.0)
    return np.where(n >= 2, rr - (np.log(np.log(np.maximum(n, 2.0))) + math.log(4 * math.pi))
                    / (2 * rr) + 0.5772156649015329 / rr, 0.0)


def oracle_bwd_sampled(q, k, v, w_h, dout, rows, keys, consts=None, block=512):
    """Gradients of ONE head of the causal prefill at selected outputs, for
    lengths where the dense oracle_bwd does not fit (ATMA §2.1 forward; its
    exact gradient as in oracle_bwd).  Plain fp64 numpy in two passes:
    (1) per row i, by blocks of rows: the logits against keys 0..i, the
    softmax p, a = sum p v, the direction u and its gradient
    da = (g - u (u.g)) / max(|a|, eps) (g / eps below eps), and the count's
    gradients: conf = sigmoid(lse - b), T = tanh(-ln Q2 / kappa),
    dQ2 = -(g.w) conf (1 - T^2) / (kappa Q2), dlse = (g.w) T conf (1 - conf);
    ds_ij = p_ij (v_j.da_i - a_i.da_i + dlse - 2 dQ2 Q2 + 2 dQ2 p_ij);
    (2) dq_i = (tau_i / sqrt d) sum_j ds_ij k_j - dlse (sigma_i / |q_i|)
    f(n) q_i / |q_i| at the selected rows, and dk_j = sum_i (tau_i / sqrt d)
    ds_ij q_i, dv_j = sum_i p_ij da_i at the selected keys.
    q, k, v, dout [T, d]; w_h [d].  Returns dict(dq [R, d], dk [K, d],
    dv [K, d], count [T]) as fp64 numpy arrays.
    """
    c = dict(DEFAULT_CONSTS)
    if consts:
        c.update(consts)
    q, k, v, g, w_h = (_f64(x) for x in (q, k, v, dout, w_h))
    T, d = q.shape
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    n = np.arange(1, T + 1, dtype=np.float64)
    tau = np.maximum(1.0, np.log(n) / c["log_t0"])
    coef = tau / math.sqrt(d)
    lse = np.empty(T)
    da = np.empty((T, d))
    cmd = np.empty(T)   # dlse - 2 dQ2 Q2 - a.da
    e2 = np.empty(T)    # 2 dQ2
    dlse = np.empty(T)
    count = np.empty(T)
    for r0 in range(0, T, block):
        r1 = min(T, r0 + block)
        s = coef[r0:r1, None] * (q[r0:r1] @ k[:r1].T)                 # [R, r1]
        s = np.where(np.arange(r1)[None, :] > np.arange(r0, r1)[:, None], -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        p = e / l
        lse[r0:r1] = (m + np.log(l))[:, 0]
        a = p @ v[:r1]
        an = np.linalg.norm(a, axis=1)
        big = an > c["eps"]
        den = np.where(big, an, c["eps"])
        u = a / den[:, None]
        gg = g[r0:r1]
        ug = (u * gg).sum(axis=1)
        dab = np.where(big[:, None], (gg - u * ug[:, None]) / den[:, None], gg / c["eps"])
        da[r0:r1] = dab
        q2 = (p * p).sum(axis=1)
        qn = np.linalg.norm(q[r0:r1], axis=1)
        b = coef[r0:r1] * c["sigma_k"] * qn * _floor_factor(n[r0:r1], c["floor_order"])
        conf = 1.0 / (1.0 + np.exp(b - lse[r0:r1]))
        tt = np.tanh(-np.log(q2) / c["kappa"])
        gw = gg @ w_h
        dq2 = -gw * conf * (1.0 - tt * tt) / (c["kappa"] * q2)
        dl = gw * tt * conf * (1.0 - conf)
        dlse[r0:r1] = dl
        e2[r0:r1] = 2.0 * dq2
        cmd[r0:r1] = dl - 2.0 * dq2 * q2 - (a * dab).sum(axis=1)
        count[r0:r1] = conf * tt
    out_dq = np.empty((len(rows), d))
    for t, i in enumerate(rows):
        s = coef[i] * (k[: i + 1] @ q[i])
        p = np.exp(s - lse[i])
        ds = p * (v[: i + 1] @ da[i] + cmd[i] + e2[i] * p)
        qn = np.linalg.norm(q[i])
        f = _floor_factor(np.array([n[i]]), c["floor_order"])[0]
        floor = -dlse[i] * coef[i] * c["sigma_k"] * f / qn if qn > 0 else 0.0
        out_dq[t] = coef[i] * (ds @ k[: i + 1]) + floor * q[i]
    out_dk = np.empty((len(keys), d))
    out_dv = np.empty((len(keys), d))
    for t, j in enumerate(keys):
        i = np.arange(j, T)
        s = coef[i] * (q[i] @ k[j])
        p = np.exp(s - lse[i])
        ds = p * (da[i] @ v[j] + cmd[i] + e2[i] * p)
        out_dk[t] = (coef[i] * ds) @ q[i]
        out_dv[t] = p @ da[i]
    return {"dq": out_dq, "dk": out_dk, "dv": out_dv, "count": count}
