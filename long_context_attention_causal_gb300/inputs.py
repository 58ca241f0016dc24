"""Seeded synthetic inputs for causal Polar Attention.

This module only draws random tensors; it holds none of the method's
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.

The five workloads stand in for the evaluation of "ATMA: Length-Invariant
Language Modeling via Polar Attention and Gated-Delta Compression Memory"
(§3: 2K training length, evaluation up to 64K tokens, needle-in-a-haystack
retrieval).  No dataset is used: haystacks are iid Gaussian, needles are
planted keys aligned with a query.

Recipe (every N(mu, x) is read as standard deviation x):
  * q, k, v ~ N(0, 1) drawn in fp32, then rounded to the workload dtype;
  * needles (prefill_needles): per head, `needles` distinct query rows i
    uniform in [0, T); for each a key position j uniform in [0, i] (key
    positions distinct per head); k_j <- 4 * q_i / |q_i|;
  * per-head key scale (prefill_keyscale): k[:, h] *= s_h, s_h ~ U[0.5, 2],
    one s_h per head shared across the batch;
  * mem ~ N(0, 0.1) in the workload dtype (zeros where stated);
  * w_count ~ N(0, 0.02), fp32, shape [H, d].
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "prefill" or "decode"
    B: int
    H: int
    T: int  # query length for prefill, cache length Tkv for decode
    d: int
    dtype: str  # "f32" or "bf16"
    seed: int
    needles: int = 0  # planted needles per head (prefill)
    keyscale: bool = False  # per-head key scale U[0.5, 2]
    mem_std: float = 0.1  # 0 => memory stream of zeros

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "prefill", 1, 2, 256, 64, "f32", 0,
                         mem_std=0.0),
    "needles_4k": Workload("needles_4k", "prefill", 1, 8, 4096, 64, "bf16", 1,
                           needles=8),
    "keyscale_16k": Workload("keyscale_16k", "prefill", 2, 16, 16384, 128,
                             "bf16", 2, keyscale=True),
    "needles_64k": Workload("needles_64k", "prefill", 1, 16, 65536, 128,
                            "bf16", 3, needles=64),
    "decode_32k": Workload("decode_32k", "decode", 32, 16, 32768, 128, "bf16",
                           4),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_prefill(wl: Workload, device="cpu"):
    """Returns dict(q, k, v, mem [B,H,T,d] in wl dtype, w_count [H,d] fp32,
    needles: list of (b, h, i, j) planted pairs, key_scale [H] or None)."""
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    g = _gen(device, wl.seed)
    shape = (B, H, T, d)
    q = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    key_scale = None
    if wl.keyscale:
        key_scale = torch.rand(H, generator=g, device=device,
                               dtype=torch.float32) * 1.5 + 0.5
        k *= key_scale.view(1, H, 1, 1)
    needles = []
    if wl.needles:
        # positions are drawn on the host from their own seeded stream
        gh = torch.Generator(device="cpu")
        gh.manual_seed(wl.seed * 7919 + 17)
        for b in range(B):
            for h in range(H):
                rows = torch.randperm(T, generator=gh)[: wl.needles].tolist()
                used = set()
                for i in rows:
                    while True:
                        j = int(torch.randint(0, i + 1, (1,), generator=gh))
                        if j not in used:
                            break
                        if len(used) >= i + 1:  # no free slot (tiny T)
                            j = None
                            break
                    if j is None:
                        continue
                    used.add(j)
                    qi = q[b, h, i]
                    k[b, h, j] = 4.0 * qi / qi.norm()
                    needles.append((b, h, i, j))
    if wl.mem_std > 0:
        mem = torch.randn(shape, generator=g, device=device,
                          dtype=torch.float32) * wl.mem_std
    else:
        mem = torch.zeros(shape, device=device, dtype=torch.float32)
    w = torch.randn((H, d), generator=g, device=device,
                    dtype=torch.float32) * 0.02
    dt = wl.torch_dtype
    return {
        "q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "mem": mem.to(dt),
        "w_count": w.contiguous(), "needles": needles, "key_scale": key_scale,
    }


def make_decode(wl: Workload, device="cpu"):
    """Returns dict(q [B,H,d], k_cache/v_cache [B,H,Tkv,d], mem [B,H,d] in wl
    dtype, w_count [H,d] fp32)."""
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    g = _gen(device, wl.seed)
    dt = wl.torch_dtype
    q = torch.randn((B, H, d), generator=g, device=device).to(dt)
    # draw the cache per (b) slab to bound fp32 scratch at large sizes
    k = torch.empty((B, H, T, d), device=device, dtype=dt)
    v = torch.empty((B, H, T, d), device=device, dtype=dt)
    for b in range(B):
        k[b] = torch.randn((H, T, d), generator=g, device=device).to(dt)
        v[b] = torch.randn((H, T, d), generator=g, device=device).to(dt)
    if wl.mem_std > 0:
        mem = (torch.randn((B, H, d), generator=g, device=device)
               * wl.mem_std).to(dt)
    else:
        mem = torch.zeros((B, H, d), device=device, dtype=dt)
    w = torch.randn((H, d), generator=g, device=device) * 0.02
    return {"q": q, "k_cache": k, "v_cache": v, "mem": mem,
            "w_count": w.contiguous()}


@dataclasses.dataclass(frozen=True)
class PagedWorkload:
    """Decode against a paged KV cache with grouped-query heads."""
    name: str
    B: int
    Hq: int  # query heads
    Hkv: int  # key/value heads (Hq = G * Hkv)
    T: int  # longest sequence (cache tokens, the current one included)
    d: int
    page: int  # tokens per page
    dtype: str
    seed: int
    ragged: bool = False  # sequence lengths uniform in [1, T] (else all T)
    mem_std: float = 0.1

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


PAGED_WORKLOADS = {
    # decode_32k's batch and context with 4 query heads per KV head
    "paged_gqa_32k": PagedWorkload("paged_gqa_32k", 32, 16, 4, 32768, 128, 64,
                                   "bf16", 5),
    # the same with 2 and 8 query heads per KV head
    "paged_gqa2_32k": PagedWorkload("paged_gqa2_32k", 32, 16, 8, 32768, 128, 64,
                                    "bf16", 7),
    "paged_gqa8_32k": PagedWorkload("paged_gqa8_32k", 32, 16, 2, 32768, 128, 64,
                                    "bf16", 8),
}


def make_paged_decode(wl: PagedWorkload, device="cpu"):
    """Returns dict(q, mem [B,Hq,d], k_pages, v_pages [num_pages, Hkv, page,
    d] in wl dtype, block_table [B, max_pages] int32, seq_lens [B] int32,
    w_count [Hq, d] fp32).  Physical pages are a seeded random permutation,
    so logically consecutive pages are scattered over the pool; unused
    table entries point at page 0."""
    B, Hq, Hkv, T, d, P = wl.B, wl.Hq, wl.Hkv, wl.T, wl.d, wl.page
    gh = torch.Generator(device="cpu")
    gh.manual_seed(wl.seed * 7919 + 29)
    if wl.ragged:
        lens = torch.randint(1, T + 1, (B,), generator=gh)
        lens[0] = T
        if B > 1:
            lens[1] = 1
    else:
        lens = torch.full((B,), T, dtype=torch.int64)
    npg = (lens + P - 1) // P
    max_pages = (T + P - 1) // P
    total = int(npg.sum())
    perm = torch.randperm(total, generator=gh)
    table = torch.zeros((B, max_pages), dtype=torch.int32)
    o = 0
    for b in range(B):
        table[b, : int(npg[b])] = perm[o: o + int(npg[b])].to(torch.int32)
        o += int(npg[b])
    g = _gen(device, wl.seed)
    dt = wl.torch_dtype
    q = torch.randn((B, Hq, d), generator=g, device=device).to(dt)
    kp = torch.empty((total, Hkv, P, d), device=device, dtype=dt)
    vp = torch.empty((total, Hkv, P, d), device=device, dtype=dt)
    step = max(1, (1 << 26) // (Hkv * P * d))  # bound the fp32 scratch
    for i in range(0, total, step):
        j = min(total, i + step)
        kp[i:j] = torch.randn((j - i, Hkv, P, d), generator=g, device=device).to(dt)
        vp[i:j] = torch.randn((j - i, Hkv, P, d), generator=g, device=device).to(dt)
    mem = (torch.randn((B, Hq, d), generator=g, device=device) * wl.mem_std).to(dt)
    w = torch.randn((Hq, d), generator=g, device=device) * 0.02
    return {"q": q, "k_pages": kp, "v_pages": vp, "block_table": table.to(device),
            "seq_lens": lens.to(torch.int32).to(device), "mem": mem,
            "w_count": w.contiguous()}


def custom_paged(B=2, Hq=8, Hkv=2, T=300, d=128, page=64, dtype="bf16", seed=0,
                 ragged=True) -> PagedWorkload:
    return PagedWorkload(f"custom_paged_{B}x{Hq}x{Hkv}x{T}x{d}_{page}_{dtype}", B, Hq,
                         Hkv, T, d, page, dtype, seed, ragged)


@dataclasses.dataclass(frozen=True)
class MemoryWorkload:
    """Gated-delta memory steps: B x H heads, T tokens, d x d fp32 state."""
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str
    seed: int

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


MEMORY_WORKLOADS = {
    # one decode step of 256 sequences x 16 heads: a 268 MB state, above L2
    "memstep_256": MemoryWorkload("memstep_256", 256, 16, 1, 128, "bf16", 6),
}


def make_memory(wl: MemoryWorkload, device="cpu"):
    """Returns dict(state [B,H,d,d] fp32 ~ N(0, 0.05), q, k, v [B,H,T,d] ~
    N(0,1) in wl dtype, alpha ~ U[0.8, 1], beta ~ U[0, 1] [B,H,T] fp32)."""
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    g = _gen(device, wl.seed)
    dt = wl.torch_dtype
    state = torch.randn((B, H, d, d), generator=g, device=device) * 0.05
    q = torch.randn((B, H, T, d), generator=g, device=device).to(dt)
    k = torch.randn((B, H, T, d), generator=g, device=device).to(dt)
    v = torch.randn((B, H, T, d), generator=g, device=device).to(dt)
    alpha = torch.rand((B, H, T), generator=g, device=device) * 0.2 + 0.8
    beta = torch.rand((B, H, T), generator=g, device=device)
    return {"state": state, "q": q, "k": k, "v": v, "alpha": alpha, "beta": beta}


def custom(kind="prefill", B=1, H=1, T=128, d=64, dtype="bf16", seed=0,
           needles=0, keyscale=False, mem_std=0.1) -> Workload:
    """A workload of any shape with the same recipe (tests, edge cases)."""
    return Workload(f"custom_{kind}_{B}x{H}x{T}x{d}_{dtype}", kind, B, H, T, d,
                    dtype, seed, needles, keyscale, mem_std)
