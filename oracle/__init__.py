"""fp64 CPU oracle for FlashPrefill V2 block-sparse prefill attention with mean correction.

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg are its only users. The product library never imports it.

The arithmetic lives in ``fp_oracle.c`` (plain C, fp64, POSIX threads). This
wrapper marshals numpy arrays to it, and does host-side bookkeeping only:
segment enumeration (request b, KV head h, tile t), CSR assembly from the
oracle's own selection, scattering tile rows back to [T, Hq, d] through
the PackGQA row map (pos(r) = floor(r/g), head(r) = h g + r mod g; FlashPrefill
V2 Sec.3.3 Eq.13), and the integer work of Stage 2 under a given CSR (each
tile's visit order, correction masks and page rows; the KV-split plan).
"""
from __future__ import annotations

import ctypes
import os
import dataclasses
from typing import Optional, Sequence

import numpy as np

from .build import build as _build_lib, LIB_PATH

ORC_CORRECTION = 1
ORC_DENSE = 2
ORC_EQ15 = 4


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("block", ctypes.c_int32), ("page_size", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("c_q", ctypes.c_double), ("c_k", ctypes.c_double), ("c_v", ctypes.c_double),
        ("cu_seqlens", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("pt_stride", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
        ("seqlens_kv", ctypes.c_void_p),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _build_lib()  # compiles only when the library is missing or older than its source
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(_Problem)
        vp = ctypes.c_void_p
        L.orc_decode_bf16.restype = ctypes.c_double
        L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        L.orc_decode_e4m3.restype = ctypes.c_double
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        L.orc_round_e4m3_n.argtypes = [vp, vp, ctypes.c_int64]
        L.orc_validate.argtypes = [P]
        L.orc_pool.argtypes = [P, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        L.orc_pool_all.argtypes = [P, vp, vp, vp, vp]
        L.orc_energies.argtypes = [P, vp, ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_select.argtypes = [vp, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_attend_tile.argtypes = [P, vp, vp, ctypes.c_long, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp,
                                      ctypes.c_int, vp, vp]
        L.orc_run_segments.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp,
                                       ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                       ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _raw(x) -> np.ndarray:
    """Element bytes of a bf16 / float8_e4m3fn torch tensor (or an already-raw numpy array)."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x)
    import torch
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    if x.dtype == torch.float8_e4m3fn:
        return x.view(torch.uint8).numpy()
    raise TypeError(f"unsupported element type {x.dtype}")


def round_e4m3(x) -> np.ndarray:
    """The E4M3 values nearest to x (ties to even, saturating at +-448), elementwise."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty_like(x)
    lib().orc_round_e4m3_n(_ptr(x), _ptr(y), x.size)
    return y


@dataclasses.dataclass
class Problem:
    """Host copy of one attention layer's inputs, as raw element bytes."""
    q: np.ndarray            # [T, hq, d] uint16 (bf16 bits) or uint8 (e4m3 bits)
    k_pages: np.ndarray      # [num_pages, page, hkv, d]
    v_pages: np.ndarray
    cu_seqlens: np.ndarray   # [batch+1] int32
    page_table: np.ndarray   # [batch, stride] int32
    hq: int
    hkv: int
    dtype: str = "bf16"
    c_q: float = 1.0
    c_k: float = 1.0
    c_v: float = 1.0
    block: int = 128
    tile_rows: int = 128
    seqlens_kv: Optional[np.ndarray] = None  # [batch] L_b^kv >= L_b^q (cached prefix + new tokens); None: = L_b^q

    @classmethod
    def from_workload(cls, w, tile_rows: int = 128) -> "Problem":
        kv = getattr(w, "host_seqlens_kv", None)
        return cls(q=_raw(w.q), k_pages=_raw(w.k_pages), v_pages=_raw(w.v_pages),
                   cu_seqlens=np.asarray(w.host_cu_seqlens, dtype=np.int32),
                   page_table=np.ascontiguousarray(w.page_table.to("cpu").numpy().astype(np.int32)),
                   hq=w.hq, hkv=w.hkv, dtype=w.dtype, c_q=w.c_q, c_k=w.c_k, c_v=w.c_v, tile_rows=tile_rows,
                   seqlens_kv=None if kv is None else np.asarray(kv, dtype=np.int32))

    def __post_init__(self):
        self.q = np.ascontiguousarray(self.q)
        self.k_pages = np.ascontiguousarray(self.k_pages)
        self.v_pages = np.ascontiguousarray(self.v_pages)
        self.cu_seqlens = np.ascontiguousarray(self.cu_seqlens, dtype=np.int32)
        self.page_table = np.ascontiguousarray(self.page_table, dtype=np.int32)
        if self.page_table.ndim == 1:
            self.page_table = self.page_table[None, :]
        if self.seqlens_kv is not None:
            self.seqlens_kv = np.ascontiguousarray(self.seqlens_kv, dtype=np.int32)

    @property
    def d(self) -> int:
        return int(self.q.shape[-1])

    @property
    def page_size(self) -> int:
        return int(self.k_pages.shape[1])

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def g(self) -> int:
        return self.hq // self.hkv

    def lengths(self):
        """New-token (query) lengths L_b^q."""
        return np.diff(self.cu_seqlens).astype(np.int64)

    def kv_lengths(self):
        """KV lengths L_b^kv (cached prefix plus the new tokens)."""
        return self.lengths() if self.seqlens_kv is None else self.seqlens_kv.astype(np.int64)

    def q_shifts(self):
        """Absolute position of each request's first new token, L_b^kv - L_b^q."""
        return self.kv_lengths() - self.lengths()

    def c_struct(self) -> _Problem:
        s = _Problem()
        s.batch, s.hq, s.hkv, s.d = self.batch, self.hq, self.hkv, self.d
        s.block, s.page_size, s.tile_rows = self.block, self.page_size, self.tile_rows
        s.dtype = 0 if self.dtype == "bf16" else 1
        s.c_q, s.c_k, s.c_v = self.c_q, self.c_k, self.c_v
        s.cu_seqlens = self.cu_seqlens.ctypes.data
        s.page_table = self.page_table.ctypes.data
        s.pt_stride = self.page_table.shape[1]
        s.num_pages = self.k_pages.shape[0]
        s.q = self.q.ctypes.data
        s.k_pages = self.k_pages.ctypes.data
        s.v_pages = self.v_pages.ctypes.data
        s.seqlens_kv = None if self.seqlens_kv is None else self.seqlens_kv.ctypes.data
        return s


@dataclasses.dataclass
class Segments:
    """Segment enumeration in (request, KV head, tile) order; t is the tile's index within its request,
    T its index on the grid of absolute packed rows (T = t unless the request has a cached prefix)."""
    b: np.ndarray
    h: np.ndarray
    t: np.ndarray
    T: np.ndarray
    D: np.ndarray            # diagonal block of each tile
    full_off: np.ndarray     # offset of each segment's D+1 per-block entries
    full_total: int
    blk_base: np.ndarray     # first pooled row of each request
    total_blocks: int

    def __len__(self):
        return len(self.b)


def first_tiles(p: Problem) -> np.ndarray:
    """Absolute tile of each request's first tile: packed rows are numbered by absolute position
    (r = g pos + head mod g) and tiled from r = 0, and the new queries start at row g (L^kv - L^q)."""
    return (p.g * p.q_shifts()) // p.tile_rows


def segments(p: Problem) -> Segments:
    Lq, Lkv = p.lengths(), p.kv_lengths()
    nb = (Lkv + p.block - 1) // p.block
    T0 = first_tiles(p)
    ntiles = np.where(Lq > 0, (p.g * Lkv + p.tile_rows - 1) // p.tile_rows - T0, 0)
    bs, hs, ts, Ts = [], [], [], []
    for b in range(p.batch):
        for h in range(p.hkv):
            bs.append(np.full(ntiles[b], b))
            hs.append(np.full(ntiles[b], h))
            ts.append(np.arange(ntiles[b]))
            Ts.append(T0[b] + np.arange(ntiles[b]))
    cat = lambda xs: np.concatenate(xs).astype(np.int32) if xs else np.zeros(0, np.int32)
    b, h, t, T = cat(bs), cat(hs), cat(ts), cat(Ts)
    D = ((T.astype(np.int64) * p.tile_rows) // p.g) // p.block
    full_off = np.concatenate([[0], np.cumsum(D + 1)]).astype(np.int64)
    blk_base = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
    return Segments(b=b, h=h, t=t, T=T, D=D.astype(np.int64), full_off=full_off[:-1].copy(),
                    full_total=int(full_off[-1]), blk_base=blk_base[:-1].copy(), total_blocks=int(blk_base[-1]))


@dataclasses.dataclass
class Pooled:
    kbar: np.ndarray   # [total_blocks, hkv, d] fp64
    vbar: np.ndarray
    cnt: np.ndarray    # [total_blocks] int32


def pool(p: Problem, seg: Optional[Segments] = None) -> Pooled:
    """Block means of every (request, KV head) (Eq.5)."""
    seg = seg or segments(p)
    nb = max(seg.total_blocks, 1)
    kbar = np.zeros((nb, p.hkv, p.d))
    vbar = np.zeros((nb, p.hkv, p.d))
    cnt = np.zeros(nb, dtype=np.int32)
    s = p.c_struct()
    rc = lib().orc_pool_all(ctypes.byref(s), _ptr(seg.blk_base), _ptr(kbar), _ptr(vbar), _ptr(cnt))
    if rc:
        raise RuntimeError(f"oracle pool failed: {rc}")
    return Pooled(kbar, vbar, cnt)


def _threads(n: Optional[int]) -> int:
    return int(n) if n else max(1, os.cpu_count() or 1)


@dataclasses.dataclass
class Selection:
    sel_full: np.ndarray     # uint8 per (segment, J<=D)
    near_full: np.ndarray
    energy_full: Optional[np.ndarray]

    def selected(self, seg: Segments, s: int) -> np.ndarray:
        o = seg.full_off[s]
        return np.nonzero(self.sel_full[o:o + seg.D[s] + 1])[0].astype(np.int32)

    def near(self, seg: Segments, s: int) -> np.ndarray:
        o = seg.full_off[s]
        return np.nonzero(self.near_full[o:o + seg.D[s] + 1])[0].astype(np.int32)


def select(p: Problem, alpha: float, sink: int, window: int, seg: Optional[Segments] = None,
           pooled: Optional[Pooled] = None, seg_ids: Optional[Sequence[int]] = None, energies: bool = False,
           nthreads: Optional[int] = None) -> Selection:
    """Scoring (Eq.19) + thresholding with forced blocks (Eq.20) for the listed segments (all by default)."""
    seg = seg or segments(p)
    pooled = pooled or pool(p, seg)
    ids = np.arange(len(seg), dtype=np.int64) if seg_ids is None else np.asarray(seg_ids, dtype=np.int64)
    sel = np.zeros(max(seg.full_total, 1), np.uint8)
    near = np.zeros(max(seg.full_total, 1), np.uint8)
    en = np.zeros(max(seg.full_total, 1)) if energies else None
    s = p.c_struct()
    rc = lib().orc_run_segments(ctypes.byref(s), _ptr(ids), len(ids), _ptr(seg.b), _ptr(seg.h), _ptr(seg.t),
                                _ptr(seg.blk_base), _ptr(pooled.kbar), _ptr(pooled.vbar), _ptr(pooled.cnt),
                                _ptr(seg.full_off), 1, float(alpha), int(sink), int(window), _ptr(sel), _ptr(near),
                                _ptr(en), 0, 0, None, None, None, _threads(nthreads))
    if rc:
        raise RuntimeError(f"oracle select failed: {rc}")
    return Selection(sel, near, en)


def csr_from_selection(seg: Segments, selection: Selection):
    """CSR (cu, idx) over all segments in order; idx ascending block ids (Sec.3.3 Eq.17)."""
    counts = np.zeros(len(seg), dtype=np.int64)
    parts = []
    for s in range(len(seg)):
        ids = selection.selected(seg, s)
        counts[s] = len(ids)
        parts.append(ids)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    return cu, idx


def selection_from_csr(seg: Segments, cu: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Per-(segment, J<=D) selection bytes from a CSR produced elsewhere."""
    full = np.zeros(max(seg.full_total, 1), np.uint8)
    for s in range(len(seg)):
        ids = idx[cu[s]:cu[s + 1]]
        if len(ids) and (ids.min() < 0 or ids.max() > seg.D[s]):
            raise ValueError(f"segment {s}: block id outside [0, D]")
        full[seg.full_off[s] + ids.astype(np.int64)] = 1
    return full


def tiles64_from_csr(p: Problem, seg: Segments, cu: np.ndarray, idx: np.ndarray):
    """The CSR over 64-token physical KV tiles that covers the same tokens as a block CSR (FlashPrefill V2
    Sec.3.4 "Serving Integration", Alg.1 step 5): per segment, the ascending ids u of the 64-token tiles
    [64u, 64u + 64) that hold a token of a selected block J, i.e. of [128J, min(128J + 128, L_b^kv))."""
    L = p.kv_lengths()
    counts = np.zeros(len(seg), dtype=np.int64)
    parts = []
    for s in range(len(seg)):
        Lb = int(L[seg.b[s]])
        tiles = []
        for J in idx[cu[s]:cu[s + 1]]:
            lo, hi = p.block * int(J), min(p.block * (int(J) + 1), Lb)
            tiles.extend(range(lo // 64, (hi - 1) // 64 + 1))
        t = np.array(sorted(set(tiles)), dtype=np.int32)
        counts[s] = len(t)
        parts.append(t)
    tcu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    tidx = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    return tcu, tidx


def attend(p: Problem, sel_full: np.ndarray, correction: bool = True, dense: bool = False,
           seg: Optional[Segments] = None, pooled: Optional[Pooled] = None, seg_ids: Optional[Sequence[int]] = None,
           nthreads: Optional[int] = None, eq15: bool = False):
    """Mean-corrected block-sparse attention (Eq.6; Eq.4 without correction) of the listed segments.

    eq15 (E4M3 problems only): the online softmax of [V2] Sec.3.3 "FP8 Execution", Eq.15, with its probabilities
    quantised to E4M3 against the running row maximum, over the iterations of Eq.17 (selected blocks descending,
    then chunks of 128 correction means descending), the means in E4M3 operand format.

    Returns (O [n, tile_rows, d], lse [n, tile_rows]) for the n listed segments."""
    seg = seg or segments(p)
    pooled = pooled or pool(p, seg)
    ids = np.arange(len(seg), dtype=np.int64) if seg_ids is None else np.asarray(seg_ids, dtype=np.int64)
    O = np.zeros((len(ids), p.tile_rows, p.d))
    lse = np.zeros((len(ids), p.tile_rows))
    flags = (ORC_CORRECTION if correction else 0) | (ORC_DENSE if dense else 0) | (ORC_EQ15 if eq15 else 0)
    s = p.c_struct()
    sel_full = np.ascontiguousarray(sel_full, dtype=np.uint8)
    rc = lib().orc_run_segments(ctypes.byref(s), _ptr(ids), len(ids), _ptr(seg.b), _ptr(seg.h), _ptr(seg.t),
                                _ptr(seg.blk_base), _ptr(pooled.kbar), _ptr(pooled.vbar), _ptr(pooled.cnt),
                                _ptr(seg.full_off), 0, 0.0, 0, 0, None, None, None, 1, flags, _ptr(sel_full),
                                _ptr(O), _ptr(lse), _threads(nthreads))
    if rc:
        raise RuntimeError(f"oracle attention failed: {rc}")
    return O, lse


def tile_schedule(p: Problem, seg: Segments, s: int, cu: np.ndarray, idx: np.ndarray, correction: bool = True,
                  dense: bool = False) -> np.ndarray:
    """The Stage 2 iteration sequence of segment s under a given CSR, as rows (J, m0, m1, m2, m3, r0, r1).

    FlashPrefill V2 Sec.3.3 "Index-Driven Sparse Traversal" (Eq.17) walks a tile's selected blocks in descending
    order; each is one exact iteration (J >= 0) that reads the block's K/V through the page table (Eq.22):
    r0 and r1 are the pool rows (page * page_size + slot) of the block's first and last page chunk of
    min(page_size, 128) tokens, or num_pages * page_size for a chunk past the request's KV. Sec.3.2
    "Implementation" then adds the pruned causal blocks in chunks of 128 means with the mask
    todo = valid & ~selected, valid = {J < D}: one iteration per chunk c that holds a todo block, chunks in
    descending order, J = -1 - c, m0..m3 = the chunk's todo bits (bit i of word k: block 128c + 32k + i),
    r0 = the chunk's first pooled-mean row. Dense mode (alpha = 0) walks every block J <= D, no chunks."""
    D = int(seg.D[s])
    b = int(seg.b[s])
    if dense:
        S = np.arange(D, -1, -1)
    else:
        S = np.sort(np.asarray(idx[cu[s]:cu[s + 1]], dtype=np.int64))[::-1]
    Lkv = int(p.kv_lengths()[b])
    ps = p.page_size
    pse = min(ps, p.block)
    npc = p.block // pse
    oob = p.k_pages.shape[0] * ps
    rows = []

    def pool_row(tok):
        if tok >= Lkv:
            return oob
        return int(p.page_table[b, tok // ps]) * ps + tok % ps

    for J in S:
        rows.append((int(J), 0, 0, 0, 0, pool_row(int(J) * p.block), pool_row(int(J) * p.block + (npc - 1) * pse)))
    if correction and not dense and D > 0:
        todo = np.ones(D, dtype=bool)
        todo[S[S < D]] = False
        for c in range((D + 127) // 128 - 1, -1, -1):
            bits = np.zeros(128, dtype=bool)
            part = todo[128 * c:min(128 * c + 128, D)]
            bits[:len(part)] = part
            if not bits.any():
                continue
            words = [int(np.sum(bits[32 * k:32 * k + 32].astype(np.uint64) << np.arange(32, dtype=np.uint64)))
                     for k in range(4)]
            rows.append((-1 - c, *words, int(seg.blk_base[b]) + 128 * c, 0))
    return np.array(rows, dtype=np.int64).reshape(-1, 7)


def split_plan(costs: np.ndarray, n_sms: int, min_iters: int = 8, max_ctas: int = 160, tiles_per_sm: int = 4):
    """Count-balanced KV splits (FlashPrefill V2 Sec.3.3 Eq.18) as this build applies them: while the tiles
    number fewer than tiles_per_sm x n_sms, a tile of n > C* iterations runs as U = ceil(n / C*) contiguous
    runs of ceil(n / U) iterations, C* = max(min_iters, ceil(sum n / min(n_sms, max_ctas))). Returns
    (C* or None when splits are off, list of per-tile run lists [(it_lo, it_hi), ...])."""
    costs = np.asarray(costs, dtype=np.int64)
    if len(costs) >= tiles_per_sm * n_sms:
        return None, [[(0, int(c))] for c in costs]
    target = max(min_iters, -(-int(costs.sum()) // min(n_sms, max_ctas)))
    runs = []
    for c in costs.tolist():
        u = -(-c // target) if c > target else 1
        per = -(-c // u) if c else 0
        runs.append([(k * per, min(c, (k + 1) * per)) for k in range(u)])
    return target, runs


def tile_rows_to_tokens(p: Problem, seg: Segments, seg_ids: Sequence[int], O_tiles: np.ndarray,
                        lse_tiles: np.ndarray):
    """Scatter tile rows to O [T, hq, d] and LSE [T, hq] (NaN where a row was not computed)."""
    T = int(p.cu_seqlens[-1])
    O = np.full((T, p.hq, p.d), np.nan)
    lse = np.full((T, p.hq), np.nan)
    Lkv, shift = p.kv_lengths(), p.q_shifts()
    for i, s in enumerate(seg_ids):
        b, h = int(seg.b[s]), int(seg.h[s])
        base = int(seg.T[s]) * p.tile_rows          # absolute packed row of tile row 0
        r0 = max(base, p.g * int(shift[b]))
        r1 = min(base + p.tile_rows, p.g * int(Lkv[b]))
        r = np.arange(r0, r1)
        tok = p.cu_seqlens[b] + r // p.g - int(shift[b])
        head = h * p.g + r % p.g
        O[tok, head] = O_tiles[i, r0 - base:r1 - base]
        lse[tok, head] = lse_tiles[i, r0 - base:r1 - base]
    return O, lse


def run(p: Problem, alpha: float, sink: int, window: int, correction: bool = True, dense: bool = False,
        nthreads: Optional[int] = None, eq15: bool = False):
    """The whole layer: returns dict(cu, idx, sel, O [T,hq,d], lse [T,hq], pooled, seg); eq15 as in attend."""
    seg = segments(p)
    pooled = pool(p, seg)
    selection = select(p, alpha, sink, window, seg=seg, pooled=pooled, nthreads=nthreads)
    cu, idx = csr_from_selection(seg, selection)
    ids = np.arange(len(seg))
    Ot, lt = attend(p, selection.sel_full, correction=correction, dense=dense, seg=seg, pooled=pooled,
                    nthreads=nthreads, eq15=eq15)
    O, lse = tile_rows_to_tokens(p, seg, ids, Ot, lt)
    return dict(cu=cu, idx=idx, selection=selection, O=O, lse=lse, pooled=pooled, seg=seg)
