"""Seeded synthetic workloads for block-sparse prefill attention.

This module only draws inputs: queries, a paged key/value pool, a page table
and sequence lengths, shaped like the FlashPrefill V2 paper's operator
benchmarks (Sec.4.1: Llama-3.1-8B- and Qwen3-30B-A3B-shaped attention layers at
32K-128K tokens, needle-in-a-haystack style inputs, continuous batching). It
holds none of the method's arithmetic (no pooling, scoring, selection or
attention), so both the CUDA path and the CPU oracle consume exactly the same
bytes.

Generator (per request b and KV head h, each with its own seed):
  * u is a random unit vector of R^d (the shared "sink / stripe" direction);
  * every 128-token block J has a centre mu_J ~ N(0, mu_scale^2 I);
  * keys    k_p   = mu_J(p) + 0.3 N(0, I), with tokens 0..3 replaced by 4u;
  * queries q_p,j = mu_J(p) + 0.3 N(0, I) + 1.0 u   for each of the g heads j;
  * values  v_p   ~ N(0, I);
  * optional vertical stripes: in every 4096-token window, 8 distinct random
    positions (never tokens 0..3) get +3 sigma u, sigma = std of {k_p . u}.
The pool holds sum_b ceil(L_b / 64) pages plus 5% unused pages, randomly
permuted (or the identity for a contiguous layout) and dealt to the requests
in order; unused slots hold small finite filler values.

Chunked prefill after a cached prefix: with kv_lengths[b] = L_b^kv > L_b^q the
generator draws the whole sequence of L_b^kv positions, puts all L_b^kv keys and
values in the paged pool and keeps the queries of the last L_b^q positions (the
new chunk), so a chunked run sees exactly the tensors of the unchunked one.

FP8 workloads quantise the bf16 tensors to OCP E4M3 with per-tensor scales
c = absmax / 448 (the scales are part of the input, as in the paper's FP8
execution, Sec.3.3 Eq.15).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

BASE_SEED = 20260824
HEAD_DIM = 128
BLOCK = 128
PAGE = 64

# Workloads named by what they are, with their sizes.
WORKLOADS = {
    # single 2K sequence, 4 query heads on 1 KV head, contiguous KV
    "tiny_2k": dict(lengths=[2048], hq=4, hkv=1, dtype="bf16", alpha=0.1, paging="identity", stripes=False),
    # Llama-3.1-8B-shaped layer at 32K: 32 query heads, 8 KV heads, paged KV
    "llama8b_32k": dict(lengths=[32768], hq=32, hkv=8, dtype="bf16", alpha=0.1, paging="random", stripes=False),
    # Qwen3-30B-A3B-shaped layer at 128K: 32 query heads, 4 KV heads, paged KV, stripes
    "qwen30b_128k": dict(lengths=[131072], hq=32, hkv=4, dtype="bf16", alpha=0.1, paging="random", stripes=True),
    # the same layer in FP8 E4M3
    "qwen30b_128k_fp8": dict(lengths=[131072], hq=32, hkv=4, dtype="e4m3", alpha=0.2, paging="random",
                             stripes=True, base="qwen30b_128k"),
    # continuous batching: 16 requests, log-uniform lengths in [4096, 131072]
    "varlen16": dict(lengths="loguniform16", hq=32, hkv=4, dtype="bf16", alpha=0.1, paging="random",
                     stripes=False),
    "varlen16_fp8": dict(lengths="loguniform16", hq=32, hkv=4, dtype="e4m3", alpha=0.2, paging="random",
                         stripes=False, base="varlen16"),
    # chunked prefill: the last 8K tokens of the 128K Qwen3-30B-A3B-shaped sequence after its 120K-token
    # cached prefix (the same keys, values and queries as qwen30b_128k)
    "qwen30b_128k_chunk8k": dict(lengths=[8192], kv_lengths=[131072], hq=32, hkv=4, dtype="bf16", alpha=0.1,
                                 paging="random", stripes=True, base="qwen30b_128k"),
}
# FP8 variants draw the same bf16 data as their base workload before quantising it
WORKLOAD_INDEX = {name: i for i, name in enumerate(WORKLOADS)}
WORKLOAD_INDEX.update({name: WORKLOAD_INDEX[spec["base"]] for name, spec in WORKLOADS.items() if "base" in spec})


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor            # [T, hq, d] bf16 or float8_e4m3fn
    k_pages: torch.Tensor      # [num_pages, 64, hkv, d]
    v_pages: torch.Tensor      # [num_pages, 64, hkv, d]
    page_table: torch.Tensor   # [batch, max_pages] int32, -1 past a request's pages
    cu_seqlens: torch.Tensor   # [batch+1] int32 (same device as q)
    lengths: List[int]         # new-token (query) lengths L_b^q
    hq: int
    hkv: int
    dtype: str                 # "bf16" or "e4m3"
    c_q: float
    c_k: float
    c_v: float
    alpha: float
    sink_blocks: int
    window_blocks: int
    kv_lengths: Optional[List[int]] = None    # L_b^kv (cached prefix + new tokens); None: = lengths
    seqlens_kv: Optional[torch.Tensor] = None  # [batch] int32 copy of kv_lengths on q's device

    @property
    def batch(self) -> int:
        return len(self.lengths)

    @property
    def host_seqlens_kv(self) -> Optional[np.ndarray]:
        return None if self.kv_lengths is None else np.asarray(self.kv_lengths, dtype=np.int32)

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def host_cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)


def _mix(*xs: int) -> int:
    """SplitMix64-style hash of a tuple of integers into a 63-bit seed."""
    h = 0x9E3779B97F4A7C15
    for x in xs:
        h = (h ^ (int(x) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        h = (h + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        h = z ^ (z >> 31)
    return h & 0x7FFFFFFFFFFFFFFF


def loguniform_lengths(n: int, lo: int, hi: int, seed: int) -> List[int]:
    """n lengths drawn log-uniform in [lo, hi], rounded to the nearest multiple of 128, clamped."""
    rng = np.random.Generator(np.random.Philox(seed))
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    out = np.clip(np.rint(x / BLOCK) * BLOCK, lo, hi).astype(np.int64)
    return [int(v) for v in out]


def _gen_head(L: int, g: int, d: int, gen: torch.Generator, device, mu_scale: float, stripes: bool):
    nb = (L + BLOCK - 1) // BLOCK
    u = torch.randn(d, generator=gen, device=device, dtype=torch.float32)
    u = u / u.norm()
    mu = torch.randn(nb, d, generator=gen, device=device, dtype=torch.float32) * mu_scale
    blk = torch.arange(L, device=device) // BLOCK
    centre = mu[blk]
    k = centre + 0.3 * torch.randn(L, d, generator=gen, device=device, dtype=torch.float32)
    k[: min(4, L)] = 4.0 * u
    q = centre[:, None, :] + 0.3 * torch.randn(L, g, d, generator=gen, device=device, dtype=torch.float32) + u
    v = torch.randn(L, d, generator=gen, device=device, dtype=torch.float32)
    if stripes and L > 4:
        sigma = float((k @ u).std())
        for w0 in range(0, L, 4096):
            lo, hi = max(4, w0), min(w0 + 4096, L)
            if hi - lo <= 0:
                continue
            n = min(8, hi - lo)
            pos = lo + torch.randperm(hi - lo, generator=gen, device=device)[:n]
            k[pos] += 3.0 * sigma * u
    return q, k, v


def _e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    return (x.float() / scale).to(torch.float8_e4m3fn)


def make_workload(name: str, device="cpu", seed: int = BASE_SEED, lengths: Optional[List[int]] = None,
                  hq: Optional[int] = None, hkv: Optional[int] = None, dtype: Optional[str] = None,
                  paging: Optional[str] = None, stripes: Optional[bool] = None, mu_scale: float = 1.0,
                  alpha: Optional[float] = None, sink_blocks: int = 1, window_blocks: int = 1,
                  extra_page_frac: float = 0.05, page_size: int = PAGE,
                  kv_lengths: Optional[List[int]] = None) -> Workload:
    """Builds a named workload; keyword arguments override its shape (for small test cases).

    mu_scale < 1 gives the "stress" variant with much denser block selection. kv_lengths (>= lengths,
    element-wise) makes each request the last lengths[b] tokens of a kv_lengths[b]-token sequence whose
    earlier tokens are a cached prefix.
    """
    spec = dict(WORKLOADS[name])
    cfg_id = WORKLOAD_INDEX[name]
    if lengths is None and kv_lengths is None:
        kv_lengths = spec.get("kv_lengths")
    if lengths is None:
        lengths = spec["lengths"]
        if lengths == "loguniform16":
            lengths = loguniform_lengths(16, 4096, 131072, _mix(seed, cfg_id, 999))
    lengths = [int(x) for x in lengths]
    if kv_lengths is not None:
        kv_lengths = [int(x) for x in kv_lengths]
        if len(kv_lengths) != len(lengths) or any(kv < L for kv, L in zip(kv_lengths, lengths)):
            raise ValueError("kv_lengths must give one length >= the query length per request")
    kvl = kv_lengths if kv_lengths is not None else lengths
    hq = hq or spec["hq"]
    hkv = hkv or spec["hkv"]
    dtype = dtype or spec["dtype"]
    paging = paging or spec["paging"]
    stripes = spec["stripes"] if stripes is None else stripes
    alpha = spec["alpha"] if alpha is None else alpha
    g = hq // hkv
    d = HEAD_DIM
    device = torch.device(device)
    batch = len(lengths)
    T = sum(lengths)

    # page table: pages dealt to requests in order from a (permuted) pool
    PAGE = page_size
    pages_per = [(L + PAGE - 1) // PAGE for L in kvl]
    used = sum(pages_per)
    num_pages = max(1, used + int(math.ceil(extra_page_frac * used)))
    pgen = torch.Generator(device="cpu")
    pgen.manual_seed(_mix(seed, cfg_id, 7))
    if paging == "identity":
        perm = torch.arange(num_pages, dtype=torch.int64)
    else:
        perm = torch.randperm(num_pages, generator=pgen)
    max_pages = max(1, max(pages_per) if pages_per else 1)
    pt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n

    fgen = torch.Generator(device=device)
    fgen.manual_seed(_mix(seed, cfg_id, 11))
    kpool = 0.1 * torch.randn(num_pages * PAGE, hkv, d, generator=fgen, device=device)
    vpool = 0.1 * torch.randn(num_pages * PAGE, hkv, d, generator=fgen, device=device)
    q = torch.empty(T, hq, d, device=device, dtype=torch.float32)
    pt_dev = pt.to(device)
    start = 0
    for b, (L, Lkv) in enumerate(zip(lengths, kvl)):
        if Lkv:
            j = torch.arange(Lkv, device=device)
            slot = pt_dev[b, j // PAGE].long() * PAGE + (j % PAGE)
        for h in range(hkv):
            gen = torch.Generator(device=device)
            gen.manual_seed(_mix(seed, cfg_id, b, h))
            if Lkv == 0:
                continue
            qh, kh, vh = _gen_head(Lkv, g, d, gen, device, mu_scale, stripes)
            q[start:start + L, h * g:(h + 1) * g] = qh[Lkv - L:]
            kpool[slot, h] = kh
            vpool[slot, h] = vh
        start += L

    qb = q.to(torch.bfloat16)
    kb = kpool.to(torch.bfloat16).view(num_pages, PAGE, hkv, d)
    vb = vpool.to(torch.bfloat16).view(num_pages, PAGE, hkv, d)
    c_q = c_k = c_v = 1.0
    if dtype == "e4m3":
        def absmax(x):
            return float(x.float().abs().max()) if x.numel() else 1.0
        # scales from the real tokens only (filler slots are far smaller); with a cached prefix the query
        # scale covers the new tokens only
        c_q = max(absmax(qb), 1e-12) / 448.0
        c_k = max(absmax(kb), 1e-12) / 448.0
        c_v = max(absmax(vb), 1e-12) / 448.0
        qb, kb, vb = _e4m3(qb, c_q), _e4m3(kb, c_k), _e4m3(vb, c_v)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)
    skv = None if kv_lengths is None else torch.tensor(np.asarray(kv_lengths, dtype=np.int32), device=device)
    return Workload(name=name, q=qb.contiguous(), k_pages=kb.contiguous(), v_pages=vb.contiguous(),
                    page_table=pt_dev.contiguous(), cu_seqlens=cu, lengths=lengths, hq=hq, hkv=hkv, dtype=dtype,
                    c_q=c_q, c_k=c_k, c_v=c_v, alpha=alpha, sink_blocks=sink_blocks, window_blocks=window_blocks,
                    kv_lengths=kv_lengths, seqlens_kv=skv)
