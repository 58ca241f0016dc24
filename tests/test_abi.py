"""Host-side checks of the C ABI (no GPU needed, nothing launched).

The library must load, export every entry point include/polar_attn.h
declares, and reject bad arguments with the documented status before any
device work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "polar_attn.h")


@pytest.fixture(scope="module")
def L():
    from long_context_attention_causal_gb300 import _build
    _build.build()
    import long_context_attention_causal_gb300 as pa
    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                       r"(polar_attn_[A-Za-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("polar_attn_fwd", "polar_attn_decode", "polar_attn_combine",
              "polar_attn_decode_workspace_bytes", "polar_attn_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"not exported: {missing}"


def test_strerror_static_strings(L):
    for s in range(0, 8):
        msg = L.polar_attn_strerror(s)
        assert isinstance(msg, bytes) and len(msg) > 0
    assert L.polar_attn_strerror(0) == b"ok"


def test_default_consts(L):
    import math
    import long_context_attention_causal_gb300 as pa
    c = pa.Consts()
    assert L.polar_attn_default_consts(ctypes.byref(c)) == 0
    assert c.log_t0 == pytest.approx(math.log(2048), rel=1e-6)
    assert c.kappa == pytest.approx(math.log(2048), rel=1e-6)
    assert c.sigma_k == 1.0 and c.eps == pytest.approx(1e-6)
    assert c.floor_order == 1
    assert L.polar_attn_default_consts(None) == 1


ALIGNED = ctypes.c_void_p(1 << 20)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)
NULL = ctypes.c_void_p(0)


def fwd(L, q=ALIGNED, out=ALIGNED, B=1, H=1, T=8, d=64, dtype=1, consts=None):
    return L.polar_attn_fwd(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED, out, ALIGNED, NULL,
                            B, H, T, d, dtype, consts, NULL)


def test_fwd_argument_validation(L):
    import long_context_attention_causal_gb300 as pa
    assert fwd(L, B=-1) == 1
    assert fwd(L, d=96) == 2
    assert fwd(L, d=32) == 2
    assert fwd(L, dtype=7) == 2
    assert fwd(L, q=NULL) == 1
    assert fwd(L, out=NULL) == 1
    assert fwd(L, q=MISALIGNED) == 3
    bad = pa.Consts(0.0, 1.0, 1.0, 1e-6)
    assert fwd(L, consts=ctypes.byref(bad)) == 1
    bad = pa.Consts(1.0, 1.0, 1.0, 0.0)
    assert fwd(L, consts=ctypes.byref(bad)) == 1
    bad = pa.Consts(1.0, 1.0, 1.0, 1e-6, 3)
    assert fwd(L, consts=ctypes.byref(bad)) == 1
    # empty problems are a no-op, even with null pointers
    assert fwd(L, q=NULL, T=0) == 0
    assert fwd(L, q=NULL, B=0) == 0


def test_decode_argument_validation(L):
    def dec(Tkv=16, ws=ALIGNED, wsb=1 << 20, S=0, d=128, q=ALIGNED, B=1):
        return L.polar_attn_decode(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                   ALIGNED, NULL, B, 2, Tkv, d, 1, None, S, ws,
                                   ctypes.c_size_t(wsb), NULL)
    assert dec(Tkv=0) == 1
    assert dec(S=-1) == 1
    assert dec(d=80) == 2
    assert dec(q=NULL) == 1
    assert dec(q=MISALIGNED) == 3
    assert dec(B=0, q=NULL) == 0


def test_workspace_size_formula(L):
    L.polar_attn_decode_workspace_bytes.restype = ctypes.c_size_t
    assert L.polar_attn_decode_workspace_bytes(32, 16, 32768, 128, 10) == \
        32 * 16 * 10 * (128 + 4) * 4
    assert L.polar_attn_decode_workspace_bytes(1, 1, 0, 128, 1) == 0
    assert L.polar_attn_decode_workspace_bytes(1, 1, 10, 96, 1) == 0
    s = L.polar_attn_decode_num_splits(32, 16, 32768, 128)
    assert 1 <= s <= 64
    assert L.polar_attn_decode_num_splits(1, 1, 100, 128) == 1


def _expected_splits(BH, Tkv, sms):
    """The decode's split rule restated: from the count giving about eight
    waves of split CTAs (three per SM) up to twice it, the count whose last
    wave is fullest, the smaller on a tie, at least 512 keys per split."""
    slots = 3 * sms
    cap = max(1, min(1024, (Tkv + 511) // 512))
    lo = max(1, min(cap, -(-8 * slots // BH)))
    best, fill_best = lo, -1.0
    for s in range(lo, min(2 * lo, cap) + 1):
        ctas = BH * s
        fill = ctas / (-(-ctas // slots) * slots)
        if fill > fill_best + 1e-12:
            best, fill_best = s, fill
    return best


@pytest.mark.parametrize("B,H,Tkv", [(32, 16, 32768), (4, 16, 32768), (1, 2, 1 << 20),
                                     (2, 4, 3000), (8, 8, 8192), (3, 5, 700)])
def test_decode_split_rule(L, B, H, Tkv):
    # no device here: the library counts 148 SMs, as the rule's default
    got = L.polar_attn_decode_num_splits(B, H, Tkv, 128)
    assert got == _expected_splits(B * H, Tkv, 148)
    # the chosen count's last wave is at least as full as that of the
    # smallest count in the range
    slots = 3 * 148

    def fill(s):
        return B * H * s / (-(-(B * H * s) // slots) * slots)
    cap = max(1, min(1024, (Tkv + 511) // 512))
    lo = max(1, min(cap, -(-8 * slots // (B * H))))
    assert fill(got) >= fill(lo)


def _c(n):
    return ctypes.c_size_t(n)


def test_bwd_argument_validation(L):
    L.polar_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    need = L.polar_attn_bwd_workspace_bytes(1, 2, 64, 128)
    assert need >= 1 * 2 * 64 * (128 + 8) * 4
    assert L.polar_attn_bwd_workspace_bytes(1, 1, 10, 96) == 0
    assert L.polar_attn_bwd_workspace_bytes(-1, 1, 10, 64) == 0

    def bwd(q=ALIGNED, dq=ALIGNED, ws=ALIGNED, wsb=None, B=1, H=2, T=64, d=128, dtype=1):
        wsb = need if wsb is None else wsb
        return L.polar_attn_bwd(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED, dq, ALIGNED, ALIGNED,
                                ALIGNED, B, H, T, d, dtype, None, ws, _c(wsb), NULL)
    assert bwd(B=-1) == 1
    assert bwd(d=80) == 2
    assert bwd(dtype=5) == 2
    assert bwd(q=NULL) == 1
    assert bwd(dq=NULL) == 1
    assert bwd(q=MISALIGNED) == 3
    assert bwd(wsb=16) == 4
    assert bwd(ws=NULL) == 4
    assert bwd(ws=MISALIGNED) == 3
    assert bwd(T=0, q=NULL) == 0


def test_stats_pair_argument_validation(L):
    def fs(q=ALIGNED, stats=ALIGNED, conf=ALIGNED, dtype=1, d=128, T=64):
        return L.polar_attn_fwd_stats(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                      conf, stats, 1, 2, T, d, dtype, None, NULL)
    assert fs(dtype=0) == 2       # fp32: polar_attn_fwd + polar_attn_bwd instead
    assert fs(d=96) == 2
    assert fs(stats=NULL) == 1
    assert fs(conf=NULL) == 1
    assert fs(stats=ctypes.c_void_p((1 << 20) + 4)) == 3
    assert fs(q=MISALIGNED) == 3
    assert fs(T=0, q=NULL) == 0
    L.polar_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    need = L.polar_attn_bwd_workspace_bytes(1, 2, 64, 128)

    def bs(out=ALIGNED, stats=ALIGNED, wsb=None, dtype=1):
        wsb = need if wsb is None else wsb
        return L.polar_attn_bwd_stats(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, out, ALIGNED,
                                      ALIGNED, stats, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                      1, 2, 64, 128, dtype, None, ALIGNED, _c(wsb), NULL)
    assert bs(dtype=0) == 2
    assert bs(out=NULL) == 1
    assert bs(stats=NULL) == 1
    assert bs(out=MISALIGNED) == 3
    assert bs(wsb=8) == 4


def test_memory_step_argument_validation(L):
    def ms(state=ALIGNED, alpha=ALIGNED, eps=1e-6, d=128, dtype=1, T=1):
        return L.polar_memory_step(state, ALIGNED, ALIGNED, ALIGNED, alpha, ALIGNED, ALIGNED,
                                   2, 4, T, d, dtype, ctypes.c_float(eps), NULL)
    assert ms(eps=0.0) == 1
    assert ms(eps=float("nan")) == 1
    assert ms(d=32) == 2
    assert ms(dtype=3) == 2
    assert ms(state=NULL) == 1
    assert ms(state=MISALIGNED) == 3
    assert ms(alpha=ctypes.c_void_p((1 << 20) + 2)) == 3
    assert ms(T=0, state=NULL) == 0


def test_fwd_host_argument_validation(L):
    L.polar_attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    B, H, T, d = 2, 3, 100, 64

    def r256(x):
        return (x + 255) // 256 * 256
    need = L.polar_attn_fwd_host_workspace_bytes(B, H, T, d, 1)
    # device copies of q, k, v, mem, out (bf16), n_eff and conf (fp32), w_count
    assert need == 5 * r256(B * H * T * d * 2) + 2 * r256(B * H * T * 4) + r256(H * d * 4)
    assert L.polar_attn_fwd_host_workspace_bytes(B, H, T, d, 0) == \
        5 * r256(B * H * T * d * 4) + 2 * r256(B * H * T * 4) + r256(H * d * 4)
    assert L.polar_attn_fwd_host_workspace_bytes(B, H, T, 96, 1) == 0
    assert L.polar_attn_fwd_host_workspace_bytes(B, H, T, d, 5) == 0

    def call(q=ALIGNED, ws=ALIGNED, wsb=need, pieces=0, d=d, dtype=1, B=B):
        return L.polar_attn_fwd_host(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                     NULL, B, H, T, d, dtype, None, pieces, ws, _c(wsb), NULL)
    assert call(pieces=-1) == 1
    assert call(d=80) == 2
    assert call(dtype=3) == 2
    assert call(q=NULL) == 1
    assert call(ws=NULL) == 4
    assert call(wsb=need - 1) == 4
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == 3
    assert call(B=0, q=NULL, ws=NULL) == 0


def test_paged_decode_argument_validation(L):
    # workspace: one fp32 record of d + 4 floats per (sequence, query head, split)
    assert L.polar_attn_decode_paged_workspace_bytes(4, 16, 4, 4096, 128, 7) == \
        4 * 16 * 7 * (128 + 4) * 4
    assert L.polar_attn_decode_paged_workspace_bytes(4, 12, 4, 4096, 128, 7) == 0  # G = 3
    assert L.polar_attn_decode_paged_workspace_bytes(4, 16, 4, 4096, 96, 7) == 0
    assert L.polar_attn_decode_paged_workspace_bytes(4, 16, 4, 0, 128, 7) == 0
    assert L.polar_attn_decode_paged_num_splits(4, 4, 4096, 96) == 0

    def pg(q=ALIGNED, table=ALIGNED, B=2, Hq=8, Hkv=2, d=128, page=64, num_pages=64,
           max_pages=32, max_len=2048, dtype=1, S=0):
        return L.polar_attn_decode_paged(q, ALIGNED, ALIGNED, table, ALIGNED, ALIGNED,
                                         ALIGNED, ALIGNED, ALIGNED, NULL, B, Hq, Hkv, d, page,
                                         num_pages, max_pages, max_len, dtype, None, S,
                                         ALIGNED, _c(1 << 20), NULL)
    assert pg(Hq=6, Hkv=4) == 2        # Hq not a multiple of Hkv
    assert pg(Hq=48, Hkv=2) == 2       # 24 query heads per KV head
    assert pg(page=48) == 2            # not a power of two
    assert pg(page=4) == 2
    assert pg(d=80) == 2
    assert pg(dtype=9) == 2
    assert pg(S=-1) == 1
    assert pg(num_pages=0) == 1
    assert pg(max_pages=16) == 1       # 16 pages x 64 tokens < 2048
    assert pg(q=NULL) == 1
    assert pg(table=NULL) == 1
    assert pg(q=MISALIGNED) == 3
    assert pg(table=ctypes.c_void_p((1 << 20) + 2)) == 3
    assert pg(B=0, q=NULL) == 0


def test_combine_argument_validation(L):
    def cb(part=ALIGNED, S=4, Tkv=100, d=128, dtype=1, B=1, out=ALIGNED):
        return L.polar_attn_combine(part, S, ALIGNED, ALIGNED, ALIGNED, out, ALIGNED, NULL,
                                    B, 2, Tkv, d, dtype, None, NULL)
    assert cb(S=0) == 1
    assert cb(Tkv=0) == 1
    assert cb(d=96) == 2
    assert cb(dtype=4) == 2
    assert cb(part=NULL) == 1
    assert cb(out=NULL) == 1
    assert cb(part=MISALIGNED) == 3
    assert cb(B=0, part=NULL) == 0


def test_static_scratch_decode_argument_validation(L):
    def ss(q=ALIGNED, Tkv=100, d=128, dtype=1, B=1, S=0):
        return L.polar_attn_decode_static_scratch(q, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                                  ALIGNED, ALIGNED, NULL, B, 2, Tkv, d, dtype,
                                                  None, S, NULL)
    assert ss(Tkv=0) == 1
    assert ss(S=-1) == 1
    assert ss(d=96) == 2
    assert ss(dtype=6) == 2
    assert ss(S=70000) == 2
    assert ss(q=NULL) == 1
    assert ss(q=MISALIGNED) == 3
    assert ss(B=0, q=NULL) == 0
