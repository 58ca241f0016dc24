"""Thin Python binding of libpolarattn.so (the C ABI in include/polar_attn.h).

Argument marshalling only: torch tensors provide device memory and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or the
device is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpolarattn.so")

POLAR_F32 = 0
POLAR_BF16 = 1

_lib = None
_lock = threading.Lock()


class PolarError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == 5:
            try:
                detail = " - " + lib().polar_attn_last_error().decode()
            except Exception:
                pass
        super().__init__(f"{where}: status {status} ({strerror(status)}){detail}")


class Consts(ctypes.Structure):
    """polar_consts_t: log_t0, kappa, sigma_k, eps (fp32), floor_order."""
    _fields_ = [("log_t0", ctypes.c_float), ("kappa", ctypes.c_float),
                ("sigma_k", ctypes.c_float), ("eps", ctypes.c_float),
                ("floor_order", ctypes.c_int)]


def default_consts(floor_order: int = 1) -> Consts:
    return Consts(math.log(2048.0), math.log(2048.0), 1.0, 1e-6, floor_order)


def lib() -> ctypes.CDLL:
    """Load libpolarattn.so (build it first with __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            vp, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)
            ci, cs = ctypes.c_int, ctypes.c_size_t
            cp = ctypes.POINTER(Consts)
            L.polar_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci,
                                         ci, ci, ci, cp, vp]
            L.polar_attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci,
                                            ci, ci, ci, ci, cp, ci, vp, cs, vp]
            L.polar_attn_combine.argtypes = [vp, ci, vp, vp, vp, vp, vp, vp, ci,
                                             ci, ci, ci, ci, cp, vp]
            L.polar_attn_decode_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
            L.polar_attn_decode_workspace_bytes.restype = cs
            L.polar_attn_decode_num_splits.argtypes = [ci, ci, ci, ci]
            L.polar_attn_strerror.argtypes = [ci]
            L.polar_attn_strerror.restype = ctypes.c_char_p
            L.polar_attn_device_status.argtypes = [ci]
            L.polar_attn_selftest_wait_timeout.argtypes = [ci, vp]
            L.polar_attn_default_consts.argtypes = [cp]
            L.polar_attn_decode_static_scratch.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cp, ci, vp]
            L.polar_attn_decode_static_scratch.restype = ci
            L.polar_attn_decode_paged.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci,
                ci, cp, ci, vp, cs, vp]
            L.polar_attn_decode_paged.restype = ci
            L.polar_attn_decode_paged_num_splits.argtypes = [ci, ci, ci, ci]
            L.polar_attn_decode_paged_num_splits.restype = ci
            L.polar_attn_decode_paged_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
            L.polar_attn_decode_paged_workspace_bytes.restype = cs
            L.polar_memory_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                                            ci, ctypes.c_float, vp]
            L.polar_memory_step.restype = ci
            L.polar_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci,
                                         ci, ci, cp, vp, cs, vp]
            L.polar_attn_bwd.restype = ci
            L.polar_attn_fwd_stats.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci,
                                               ci, ci, ci, cp, vp]
            L.polar_attn_fwd_stats.restype = ci
            L.polar_attn_bwd_stats.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                               vp, vp, vp, ci, ci, ci, ci, ci, cp, vp, cs, vp]
            L.polar_attn_bwd_stats.restype = ci
            L.polar_attn_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
            L.polar_attn_bwd_workspace_bytes.restype = cs
            L.polar_attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci,
                                              ci, ci, cp, ci, vp, cs, vp]
            L.polar_attn_fwd_host.restype = ci
            L.polar_attn_fwd_host_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
            L.polar_attn_fwd_host_workspace_bytes.restype = cs
            L.polar_attn_last_error.argtypes = []
            L.polar_attn_last_error.restype = ctypes.c_char_p
            for f in ("polar_attn_fwd", "polar_attn_decode", "polar_attn_combine",
                      "polar_attn_decode_num_splits", "polar_attn_device_status",
                      "polar_attn_selftest_wait_timeout", "polar_attn_version",
                      "polar_attn_default_consts"):
                getattr(L, f).restype = ci
            _lib = L
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().polar_attn_strerror(int(status)).decode()
    except ImportError:
        return "library not loaded"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return POLAR_F32
    if t.dtype == torch.bfloat16:
        return POLAR_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _shape(t, name, shape):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have the shape {tuple(shape)}, got {tuple(t.shape)}")


def _dec_outputs(q, out, n_eff, conf, bh):
    _dev(out, "out", q.dtype)
    _dev(n_eff, "n_eff", torch.float32)
    _dev(conf, "conf", torch.float32)
    _shape(out, "out", q.shape)
    _shape(n_eff, "n_eff", bh)
    _shape(conf, "conf", bh)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st, where):
    if st != 0:
        raise PolarError(st, where)


def fwd(q, k, v, mem, w_count, out=None, n_eff=None, conf=None, consts=None,
        want_conf=False, stream=None):
    """Causal prefill: q, k, v, mem [B, H, T, d] (bf16 or fp32, same dtype),
    w_count [H, d] fp32.  Returns (out, n_eff, conf or None)."""
    _dev(q, "q")
    dt = q.dtype
    for name, t in (("k", k), ("v", v), ("mem", mem)):
        _dev(t, name, dt)
    _dev(w_count, "w_count", torch.float32)
    B, H, T, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or mem.shape != q.shape:
        raise ValueError("q, k, v, mem must share the shape [B, H, T, d]")
    if tuple(w_count.shape) != (H, d):
        raise ValueError("w_count must be [H, d]")
    if out is None:
        out = torch.empty_like(q)
    if n_eff is None:
        n_eff = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    if conf is None and want_conf:
        conf = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    _dev(out, "out", dt)
    _dev(n_eff, "n_eff", torch.float32)
    _dev(conf, "conf", torch.float32)
    _shape(out, "out", q.shape)
    _shape(n_eff, "n_eff", (B, H, T))
    _shape(conf, "conf", (B, H, T))
    c = consts or default_consts()
    st = lib().polar_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w_count),
                              _ptr(out), _ptr(n_eff), _ptr(conf), B, H, T, d,
                              _dtype_code(q), ctypes.byref(c), _stream(stream))
    _check(st, "polar_attn_fwd")
    return out, n_eff, conf


def fwd_stats(q, k, v, mem, w_count, consts=None, stream=None):
    """Causal prefill (bf16) that also keeps the backward's row statistics.
    Returns (out, n_eff, conf, stats [B, H, T, 2] = logsumexp, |a|)."""
    _dev(q, "q", torch.bfloat16)
    for name, t in (("k", k), ("v", v), ("mem", mem)):
        _dev(t, name, torch.bfloat16)
    _dev(w_count, "w_count", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, d]")
    B, H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("mem", mem)):
        _shape(t, name, q.shape)
    _shape(w_count, "w_count", (H, d))
    out = torch.empty_like(q)
    n_eff = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    conf = torch.empty_like(n_eff)
    stats = torch.empty((B, H, T, 2), device=q.device, dtype=torch.float32)
    c = consts or default_consts()
    st = lib().polar_attn_fwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w_count),
                                    _ptr(out), _ptr(n_eff), _ptr(conf), _ptr(stats), B, H, T,
                                    d, _dtype_code(q), ctypes.byref(c), _stream(stream))
    _check(st, "polar_attn_fwd_stats")
    return out, n_eff, conf, stats


def _host(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def fwd_host_workspace_bytes(B, H, T, d, dtype=torch.bfloat16) -> int:
    code = 1 if dtype == torch.bfloat16 else 0
    return int(lib().polar_attn_fwd_host_workspace_bytes(B, H, T, d, code))


def fwd_host(q, k, v, mem, w_count, out=None, n_eff=None, conf=None, want_conf=False,
             num_pieces=0, workspace=None, consts=None, stream=None, synchronize=True):
    """Causal prefill from host (CPU) tensors: copies in, kernels and copies
    out overlap piece by piece inside the library.  Pinned tensors
    (pin_memory()) let the copies run asynchronously.  workspace: a CUDA
    uint8 tensor of fwd_host_workspace_bytes(...) bytes (allocated here if
    None).  With synchronize=False the CPU outputs are valid only after the
    stream has been synchronised.  Returns (out, n_eff, conf or None) on the
    CPU."""
    _host(q, "q")
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32")
    for name, t in (("k", k), ("v", v), ("mem", mem)):
        _host(t, name, dt)
    _host(w_count, "w_count", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, d]")
    B, H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("mem", mem)):
        _shape(t, name, q.shape)
    _shape(w_count, "w_count", (H, d))
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=dt, pin_memory=pin)
    if n_eff is None:
        n_eff = torch.empty((B, H, T), dtype=torch.float32, pin_memory=pin)
    if conf is None and want_conf:
        conf = torch.empty((B, H, T), dtype=torch.float32, pin_memory=pin)
    _host(out, "out", dt)
    _host(n_eff, "n_eff", torch.float32)
    _shape(out, "out", q.shape)
    _shape(n_eff, "n_eff", (B, H, T))
    if conf is not None:
        _host(conf, "conf", torch.float32)
        _shape(conf, "conf", (B, H, T))
    need = fwd_host_workspace_bytes(B, H, T, d, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 256), device="cuda", dtype=torch.uint8)
    _dev(workspace, "workspace", torch.uint8)
    c = consts or default_consts()
    st = lib().polar_attn_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w_count), _ptr(out), _ptr(n_eff),
        _ptr(conf), B, H, T, d, _dtype_code(q), ctypes.byref(c), int(num_pieces),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "polar_attn_fwd_host")
    if synchronize:
        (stream or torch.cuda.current_stream()).synchronize()
    return out, n_eff, conf


def decode_num_splits(B, H, Tkv, d) -> int:
    return int(lib().polar_attn_decode_num_splits(B, H, Tkv, d))


def decode_workspace_bytes(B, H, Tkv, d, num_splits=0) -> int:
    return int(lib().polar_attn_decode_workspace_bytes(B, H, Tkv, d, num_splits))


def decode(q, k_cache, v_cache, mem, w_count, num_splits=0, workspace=None,
           out=None, n_eff=None, conf=None, consts=None, want_conf=False,
           stream=None):
    """Split-KV decode: q, mem [B, H, d]; k_cache, v_cache [B, H, Tkv, d];
    w_count [H, d] fp32.  workspace: a CUDA uint8 tensor (allocated here if
    None).  Returns (out, n_eff, conf or None)."""
    _dev(q, "q")
    dt = q.dtype
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("mem", mem)):
        _dev(t, name, dt)
    _dev(w_count, "w_count", torch.float32)
    B, H, Tkv, d = k_cache.shape
    if tuple(q.shape) != (B, H, d) or tuple(mem.shape) != (B, H, d):
        raise ValueError("q and mem must be [B, H, d]")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share a shape")
    _shape(w_count, "w_count", (H, d))
    need = decode_workspace_bytes(B, H, Tkv, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _dev(workspace, "workspace")
    if out is None:
        out = torch.empty_like(q)
    if n_eff is None:
        n_eff = torch.empty((B, H), device=q.device, dtype=torch.float32)
    if conf is None and want_conf:
        conf = torch.empty((B, H), device=q.device, dtype=torch.float32)
    _dec_outputs(q, out, n_eff, conf, (B, H))
    c = consts or default_consts()
    st = lib().polar_attn_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mem), _ptr(w_count), _ptr(out),
        _ptr(n_eff), _ptr(conf), B, H, Tkv, d, _dtype_code(q), ctypes.byref(c),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "polar_attn_decode")
    return out, n_eff, conf


def decode_static_scratch(q, k_cache, v_cache, mem, w_count, num_splits=0,
                          out=None, n_eff=None, conf=None, consts=None,
                          want_conf=False, stream=None):
    """Split-KV decode that allocates nothing: the split partials live in
    the library's fixed device array (see polar_attn_decode_static_scratch).
    For callers that cannot allocate device memory when they decode.  Calls
    that overlap on the GPU share that array and must be serialised."""
    _dev(q, "q")
    dt = q.dtype
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("mem", mem)):
        _dev(t, name, dt)
    _dev(w_count, "w_count", torch.float32)
    B, H, Tkv, d = k_cache.shape
    if tuple(q.shape) != (B, H, d) or tuple(mem.shape) != (B, H, d):
        raise ValueError("q and mem must be [B, H, d]")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share a shape")
    _shape(w_count, "w_count", (H, d))
    if out is None:
        out = torch.empty_like(q)
    if n_eff is None:
        n_eff = torch.empty((B, H), device=q.device, dtype=torch.float32)
    if conf is None and want_conf:
        conf = torch.empty((B, H), device=q.device, dtype=torch.float32)
    _dec_outputs(q, out, n_eff, conf, (B, H))
    c = consts or default_consts()
    st = lib().polar_attn_decode_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mem), _ptr(w_count), _ptr(out),
        _ptr(n_eff), _ptr(conf), B, H, Tkv, d, _dtype_code(q), ctypes.byref(c),
        int(num_splits), _stream(stream))
    if st == 4:
        raise PolarError(st, "polar_attn_decode_static_scratch: "
                         + lib().polar_attn_last_error().decode())
    _check(st, "polar_attn_decode_static_scratch")
    return out, n_eff, conf


def decode_paged_workspace_bytes(B, Hq, Hkv, max_seq_len, d, num_splits=0) -> int:
    return int(lib().polar_attn_decode_paged_workspace_bytes(B, Hq, Hkv, max_seq_len, d,
                                                             num_splits))


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, mem, w_count,
                 max_seq_len=None, num_splits=0, workspace=None, out=None, n_eff=None,
                 conf=None, consts=None, want_conf=False, stream=None):
    """Decode against a paged cache with grouped-query heads.

    q, mem [B, Hq, d]; k_pages, v_pages [num_pages, Hkv, page, d];
    block_table [B, max_pages] int32; seq_lens [B] int32 (device);
    w_count [Hq, d] fp32.  max_seq_len bounds seq_lens (default: the
    table's capacity max_pages * page).  Returns (out, n_eff, conf)."""
    _dev(q, "q")
    dt = q.dtype
    for name, t in (("k_pages", k_pages), ("v_pages", v_pages), ("mem", mem)):
        _dev(t, name, dt)
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(w_count, "w_count", torch.float32)
    B, Hq, d = q.shape
    num_pages, Hkv, page, d2 = k_pages.shape
    if d2 != d or v_pages.shape != k_pages.shape or tuple(mem.shape) != (B, Hq, d):
        raise ValueError("shape mismatch between q, mem and the pages")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    _shape(seq_lens, "seq_lens", (B,))
    _shape(w_count, "w_count", (Hq, d))
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * page
    need = decode_paged_workspace_bytes(B, Hq, Hkv, max_seq_len, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if n_eff is None:
        n_eff = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    if conf is None and want_conf:
        conf = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    _dec_outputs(q, out, n_eff, conf, (B, Hq))
    c = consts or default_consts()
    st = lib().polar_attn_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
        _ptr(mem), _ptr(w_count), _ptr(out), _ptr(n_eff), _ptr(conf), B, Hq, Hkv, d,
        page, num_pages, max_pages, int(max_seq_len), _dtype_code(q), ctypes.byref(c),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "polar_attn_decode_paged")
    return out, n_eff, conf


def memory_step(state, q, k, v, alpha, beta, mem=None, eps=1e-6, stream=None):
    """Gated-delta memory over T tokens, state updated in place.

    state [B, H, d, d] fp32 (modified); q, k, v [B, H, T, d] (bf16 or fp32);
    alpha, beta [B, H, T] fp32.  Returns mem [B, H, T, d] (the memory
    stream)."""
    _dev(state, "state", torch.float32)
    _dev(q, "q")
    for name, t in (("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    _dev(alpha, "alpha", torch.float32)
    _dev(beta, "beta", torch.float32)
    B, H, T, d = q.shape
    if tuple(state.shape) != (B, H, d, d) or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("state [B,H,d,d] and q, k, v [B,H,T,d] shapes disagree")
    if tuple(alpha.shape) != (B, H, T) or tuple(beta.shape) != (B, H, T):
        raise ValueError("alpha and beta must be [B, H, T]")
    if mem is None:
        mem = torch.empty_like(q)
    _dev(mem, "mem", q.dtype)
    st = lib().polar_memory_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                 _ptr(beta), _ptr(mem), B, H, T, d, _dtype_code(q),
                                 float(eps), _stream(stream))
    _check(st, "polar_memory_step")
    return mem


def bwd_workspace_bytes(B, H, T, d) -> int:
    return int(lib().polar_attn_bwd_workspace_bytes(B, H, T, d))


def bwd(q, k, v, w_count, dout, consts=None, workspace=None, stream=None):
    """Gradients of the causal prefill output: returns (dq, dk, dv, dw_count)
    in fp32; d out / d mem is dout itself."""
    _dev(q, "q")
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _dev(t, name, q.dtype)
    _dev(w_count, "w_count", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, d]")
    B, H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _shape(t, name, q.shape)
    _shape(w_count, "w_count", (H, d))
    dq = torch.empty(q.shape, device=q.device, dtype=torch.float32)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    dw = torch.empty((H, d), device=q.device, dtype=torch.float32)
    need = int(lib().polar_attn_bwd_workspace_bytes(B, H, T, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    c = consts or default_consts()
    st = lib().polar_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w_count), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), _ptr(dw), B, H, T, d, _dtype_code(q),
                              ctypes.byref(c), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "polar_attn_bwd")
    return dq, dk, dv, dw


def bwd_stats(q, k, v, mem, w_count, out, n_eff, conf, stats, dout, consts=None,
              workspace=None, stream=None, dq=None, dk=None, dv=None, dw=None):
    """Gradients (bf16) from the outputs of fwd_stats: returns (dq, dk, dv,
    dw_count) in fp32 (written into dq, dk, dv, dw when given); d out / d mem
    is dout itself."""
    _dev(q, "q", torch.bfloat16)
    for name, t in (("k", k), ("v", v), ("mem", mem), ("out", out), ("dout", dout)):
        _dev(t, name, torch.bfloat16)
    for name, t in (("w_count", w_count), ("n_eff", n_eff), ("conf", conf), ("stats", stats)):
        _dev(t, name, torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, d]")
    B, H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("mem", mem), ("out", out), ("dout", dout)):
        _shape(t, name, q.shape)
    _shape(w_count, "w_count", (H, d))
    _shape(n_eff, "n_eff", (B, H, T))
    _shape(conf, "conf", (B, H, T))
    _shape(stats, "stats", (B, H, T, 2))
    if dq is None:
        dq = torch.empty(q.shape, device=q.device, dtype=torch.float32)
    if dk is None:
        dk = torch.empty(q.shape, device=q.device, dtype=torch.float32)
    if dv is None:
        dv = torch.empty(q.shape, device=q.device, dtype=torch.float32)
    if dw is None:
        dw = torch.empty((H, d), device=q.device, dtype=torch.float32)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv), ("dw", dw)):
        _dev(t, name, torch.float32)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _shape(t, name, q.shape)
    _shape(dw, "dw", (H, d))
    need = int(lib().polar_attn_bwd_workspace_bytes(B, H, T, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    c = consts or default_consts()
    st = lib().polar_attn_bwd_stats(
        _ptr(q), _ptr(k), _ptr(v), _ptr(mem), _ptr(w_count), _ptr(out), _ptr(n_eff), _ptr(conf),
        _ptr(stats), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dw), B, H, T, d,
        _dtype_code(q), ctypes.byref(c), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "polar_attn_bwd_stats")
    return dq, dk, dv, dw


def combine(partials, q, mem, w_count, Tkv, out=None, n_eff=None, conf=None,
            consts=None, want_conf=False, stream=None):
    """Merge split partials [B, H, S, d + 4] fp32 and apply the epilogue."""
    _dev(partials, "partials", torch.float32)
    _dev(q, "q")
    _dev(mem, "mem", q.dtype)
    _dev(w_count, "w_count", torch.float32)
    if partials.dim() != 4:
        raise ValueError("partials must be [B, H, S, d + 4]")
    B, H, S, d4 = partials.shape
    d = d4 - 4
    _shape(q, "q", (B, H, d))
    _shape(mem, "mem", (B, H, d))
    _shape(w_count, "w_count", (H, d))
    if out is None:
        out = torch.empty_like(q)
    if n_eff is None:
        n_eff = torch.empty((B, H), device=q.device, dtype=torch.float32)
    if conf is None and want_conf:
        conf = torch.empty((B, H), device=q.device, dtype=torch.float32)
    _dec_outputs(q, out, n_eff, conf, (B, H))
    c = consts or default_consts()
    st = lib().polar_attn_combine(_ptr(partials), S, _ptr(q), _ptr(mem), _ptr(w_count),
                                  _ptr(out), _ptr(n_eff), _ptr(conf), B, H, int(Tkv), d,
                                  _dtype_code(q), ctypes.byref(c), _stream(stream))
    _check(st, "polar_attn_combine")
    return out, n_eff, conf


def device_status(reset: bool = False) -> int:
    """Kernel-side status word (0 = no wait ran out).  Synchronises."""
    return int(lib().polar_attn_device_status(1 if reset else 0))


def selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    _check(lib().polar_attn_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "polar_attn_selftest_wait_timeout")


def version() -> int:
    return int(lib().polar_attn_version())
