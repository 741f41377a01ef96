"""Shared GPU-vs-oracle comparison for the parity tests (imported by tests only).

The CUDA path runs through the C ABI (binding -> libfp.so); the oracle runs on
the host copy of the same seeded inputs. Stage 2 is compared on the GPU's own
CSR so that a legitimately flipped near-threshold block cannot pollute the
output error; the flips themselves are counted.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from block_sparse_long_mean_gb300 import binding as B
from block_sparse_long_mean_gb300 import synth

# Tolerances (output vs fp64 oracle), as required for the two precisions.
BF16_REL_RMS, BF16_MAX_ABS = 1e-2, 3e-2
FP8_REL_RMS = 6e-2


@dataclasses.dataclass
class GpuRun:
    w: synth.Workload
    p: B.Problem
    bufs: B.Buffers
    flags: int
    alpha: float
    sink: int
    window: int


def run_gpu(w: synth.Workload, alpha: Optional[float] = None, flags: int = B.FP_MEAN_CORRECTION,
            capacity: Optional[int] = None) -> GpuRun:
    alpha = w.alpha if alpha is None else alpha
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p, capacity=capacity)
    B.run_layer(p, w.q, w.k_pages, w.v_pages, alpha, w.sink_blocks, w.window_blocks, bufs, flags=flags)
    torch.cuda.synchronize()
    return GpuRun(w, p, bufs, flags, alpha, w.sink_blocks, w.window_blocks)


@dataclasses.dataclass
class Report:
    segments_checked: int
    near_flips: int
    csr_mismatch: int
    rel_rms: float
    max_abs: float
    lse_max_abs: float
    mean_max_err: float
    density: float


def sample_segments(seg: oracle.Segments, n_random: int, seed: int = 0) -> np.ndarray:
    """Every segment for small problems; else each (request, KV head)'s last tiles, first tiles and
    a seeded random sample."""
    if len(seg) <= 4096:
        return np.arange(len(seg))
    rng = np.random.default_rng(seed)
    ids = set(rng.choice(len(seg), size=min(n_random, len(seg)), replace=False).tolist())
    keys = np.stack([seg.b, seg.h]).T
    for b, h in {tuple(k) for k in keys.tolist()}:
        mine = np.nonzero((seg.b == b) & (seg.h == h))[0]
        ids.update(mine[-2:].tolist())
        ids.update(mine[:1].tolist())
    return np.array(sorted(ids))


def compare(run: GpuRun, seg_ids: Optional[Sequence[int]] = None, n_random: int = 48,
            check_means: bool = True, eq15: bool = False) -> Report:
    w, bufs = run.w, run.bufs
    code = B.fp_device_status(bufs.workspace)
    assert code == B.FP_OK, B.STATUS.get(code, code)
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    pooled = oracle.pool(op, seg)
    ids = sample_segments(seg, n_random) if seg_ids is None else np.asarray(seg_ids)

    mean_err = 0.0
    if check_means and seg.total_blocks:
        kb = bufs.kbar.cpu().double().numpy()[:seg.total_blocks]
        vb = bufs.vbar.cpu().double().numpy()[:seg.total_blocks]
        mean_err = max(np.max(np.abs(kb - pooled.kbar)), np.max(np.abs(vb - pooled.vbar)))

    cu = bufs.csr_cu.cpu().numpy().astype(np.int64)
    nnz = int(cu[-1])
    idx = bufs.csr_idx[:nnz].cpu().numpy()
    dense = bool(run.flags & B.FP_DENSE)
    near_flips = mismatch = 0
    if not dense:
        sel = oracle.select(op, run.alpha, run.sink, run.window, seg=seg, pooled=pooled, seg_ids=ids)
        for s in ids:
            mine = idx[cu[s]:cu[s + 1]]
            want = sel.selected(seg, s)
            if not np.array_equal(mine, want):
                diff = np.setxor1d(mine, want)
                near = sel.near(seg, s)
                flips = np.intersect1d(diff, near)
                near_flips += len(flips)
                mismatch += len(diff) - len(flips)
        gpu_sel = oracle.selection_from_csr(seg, cu, idx)
    else:
        gpu_sel = np.ones(max(seg.full_total, 1), np.uint8)
    O_t, lse_t = oracle.attend(op, gpu_sel, correction=bool(run.flags & B.FP_MEAN_CORRECTION), dense=dense,
                               seg=seg, pooled=pooled, seg_ids=ids, eq15=eq15)
    O_ref, lse_ref = oracle.tile_rows_to_tokens(op, seg, ids, O_t, lse_t)
    have = ~np.isnan(lse_ref)
    out = bufs.out.float().cpu().double().numpy()
    lse = bufs.lse.cpu().double().numpy()
    diff = out[have] - O_ref[have]
    rel_rms = float(np.sqrt(np.sum(diff ** 2) / max(np.sum(O_ref[have] ** 2), 1e-300)))
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    lse_err = float(np.max(np.abs(lse[have] - lse_ref[have]))) if diff.size else 0.0
    causal = int((seg.D + 1).sum())
    return Report(len(ids), near_flips, mismatch, rel_rms, max_abs, lse_err, float(mean_err),
                  nnz / max(causal, 1))
