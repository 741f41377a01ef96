#!/usr/bin/env python3
"""Benchmark of one FlashPrefill V2 attention layer (Stage 1 + Stage 2) on GB300.

A step is one pass of the whole hot path over one layer: fp_select (pooling,
scoring, thresholding, CSR) followed by fp_attention (exact blocks + mean
correction + epilogue), both through the C ABI, inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is milliseconds per layer for the whole
job (N GPUs each run one layer per step, so value = step time / N); lower is
better. `--impl reference` times the fp64 CPU oracle on the host cores instead
(a bounded sample of the same workload, extrapolated to a layer).

Besides the timed steps the line reports this build's own dense (alpha = 0)
mode of the same kernels and the speedup over it, Stage 1 against its floor
max(HBM, MMA, MUFU), the output error of the corrected and uncorrected layer
against that dense output, and the fp64 oracle timed over the whole layer on
the host cores (the `cpu_baseline` leg).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_long_mean_gb300 import synth  # noqa: E402

METRIC = "sparse prefill-attn ms/layer & dense-equiv TFLOP/s at 128K; tensor-pipe %"
UNIT = "ms/layer"
DEFAULT_WORKLOAD = "qwen30b_128k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet dense tensor peaks (no 2:4 sparsity), for a second fraction beside the measured one
NOMINAL_TFLOPS = {"bf16": 2250.0, "e4m3": 4500.0}
# exp2 (MUFU) throughput of one SM per clock: 31.4 ex2.approx.ftz.f32 per clock per SM measured on GB300 with a
# throughput probe (independent chains, all SMs), i.e. 32 per clock
MUFU_EX2_PER_CLK_SM = 32.0
# fp_select: prep, pool, score, csr scan, csr expand; fp_attention: prep, meta, bucket, scatter, attention, and the
# split combine when the tiles number fewer than 4 x SMs (the library's rule for enabling KV splits)
KERNELS_PER_STEP = 10


def kernels_per_step(nseg: int) -> int:
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return KERNELS_PER_STEP + (1 if nseg < 4 * sms else 0)

# DRAM bytes (read + write) of one attention-kernel launch on this workload, from one stored ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid while the kernel's sources are those the capture ran.
ATTN_TRAFFIC = {"sources_sha256": "c97d351f211582b7795886202cf33508bbe913a601268ce00faf0d35b54ef214",
                "bytes": {"qwen30b_128k": 1365835776 + 1029804800, "qwen30b_128k_fp8": 692387584 + 1018726144}}


def attn_traffic(workload: str):
    import hashlib
    h = hashlib.sha256()
    for f in ("fp_stage2.cu", "fp_internal.cuh", "sm100_ptx.cuh"):
        with open(os.path.join(ROOT, "block_sparse_long_mean_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() == ATTN_TRAFFIC["sources_sha256"]:
        return ATTN_TRAFFIC["bytes"].get(workload)
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ work accounting

def accounting(w, cu: np.ndarray, idx: np.ndarray):
    """FLOP and byte counts of one layer from the workload and its CSR."""
    op_seg = segments_of(w)
    D = op_seg["D"]
    rows = op_seg["rows"]
    counts = np.diff(cu)
    nseg = len(D)
    # mean-correction chunks per tile: 128-block chunks of [0, D) holding a pruned block
    chunks = np.zeros(nseg, np.int64)
    sel_lo = 0
    for s in range(nseg):
        ids = idx[cu[s]:cu[s + 1]]
        d = int(D[s])
        if d == 0:
            continue
        nch = (d + 127) // 128
        full = np.bincount(ids[ids < d] // 128, minlength=nch)[:nch]
        cap = np.minimum(128, d - 128 * np.arange(nch))
        chunks[s] = int(np.sum(full < cap))
    tile = 4.0 * 128 * 128 * 128
    executed = tile * float(np.sum(counts) + np.sum(chunks))
    d = 128
    kvl = kv_lengths_of(w)
    # dense causal work: query i of a request sits at position L^kv - L^q + i and sees that many keys + 1
    dense_equiv = 4.0 * d * w.hq * sum(Lq * (Lkv - Lq) + Lq * (Lq + 1) / 2 for Lq, Lkv in zip(w.lengths, kvl))
    eb = 2 if w.dtype == "bf16" else 1
    T = w.total_tokens
    nblk = sum((L + 127) // 128 for L in kvl)
    stage1_bytes = (T * w.hq * d * eb + 2 * sum(kvl) * w.hkv * d * eb  # Q, K, V read once
                    + nblk * w.hkv * d * (4 + 4 + 2 * eb)            # means written (fp32 + operand copies)
                    + 4 * (nseg + 1) + 4 * int(cu[-1]))              # CSR written
    causal_blocks = int(np.sum(D + 1))
    # Stage 1's own arithmetic as the method states it (Eq.19): one dot product of d MACs and one exponential
    # per (query row, causal block J <= D) of every tile
    row_blocks = float(np.sum(rows * (D + 1)))
    return dict(executed_flop=executed, dense_equiv_flop=dense_equiv, stage1_bytes=stage1_bytes,
                dense_mode_executed_flop=tile * float(np.sum(D + 1)),
                stage1_mma_flop=2.0 * d * row_blocks, stage1_exps=row_blocks,
                nnz=int(cu[-1]), causal_blocks=causal_blocks, density=int(cu[-1]) / max(causal_blocks, 1),
                corr_chunks=int(np.sum(chunks)), segments=nseg, rows=rows)


def kv_lengths_of(w):
    return list(w.kv_lengths) if getattr(w, "kv_lengths", None) is not None else list(w.lengths)


def segments_of(w):
    """Diagonal block and query-row count of every segment: tiles of 128 packed rows on the absolute grid
    (row = g position + head mod g) that hold one of the request's query rows."""
    g = w.hq // w.hkv
    Ds, rows = [], []
    for Lq, Lkv in zip(w.lengths, kv_lengths_of(w)):
        if Lq == 0:
            continue
        t0 = g * (Lkv - Lq) // 128
        T = np.arange(t0, (g * Lkv + 127) // 128)
        for _ in range(w.hkv):
            Ds.append((T * 128 // g) // 128)
            rows.append(np.minimum(128, g * Lkv - 128 * T) - np.maximum(0, g * (Lkv - Lq) - 128 * T))
    cat = lambda x: np.concatenate(x) if x else np.zeros(0, np.int64)
    return dict(D=cat(Ds).astype(np.int64), rows=cat(rows).astype(np.int64))


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index
        self.path = os.path.join("/tmp", f"fp_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------- CPU oracle

def oracle_layer_time(w, threads: int | None = None):
    """Times the fp64 oracle on the whole layer: pooling, selection of every segment and mean-corrected
    attention of every tile, on all host cores."""
    import oracle
    threads = threads or max(1, os.cpu_count() or 1)
    op = oracle.Problem.from_workload(w)
    t0 = time.perf_counter()
    seg = oracle.segments(op)
    pooled = oracle.pool(op, seg)
    sel = oracle.select(op, w.alpha, w.sink_blocks, w.window_blocks, seg=seg, pooled=pooled, nthreads=threads)
    oracle.attend(op, sel.sel_full, seg=seg, pooled=pooled, nthreads=threads)
    elapsed = time.perf_counter() - t0
    return elapsed * 1e3, threads, f"the whole layer: {len(seg)} segments pooled, selected and attended"


def oracle_sample_time(w, cu: np.ndarray, idx: np.ndarray, target_s: float = 12.0, threads: int | None = None):
    """Times the fp64 oracle on a seeded sample of segments of the workload and extrapolates to one layer
    by the oracle's per-segment work (pooling is timed in full)."""
    import oracle
    threads = threads or max(1, os.cpu_count() or 1)
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    t0 = time.perf_counter()
    pooled = oracle.pool(op, seg)
    t_pool = time.perf_counter() - t0
    counts = np.diff(cu)
    # per-segment oracle work: scoring rows x (D+1) x d, attention rows x (exact keys + corrections) x 2d
    D = seg.D
    rows = segments_of(w)["rows"]
    work = rows * (D + 1) * 128 + rows * (counts * 128 + np.maximum(D - counts + 1, 0)) * 256
    rng = np.random.default_rng(1234)
    order = rng.permutation(len(seg))
    # calibrate on a handful of segments, then size the sample for ~target_s seconds
    n = min(len(seg), max(threads, 4))
    elapsed, done = 0.0, 0
    taken = []
    while done < len(seg):
        ids = order[done:done + n]
        t0 = time.perf_counter()
        sel = oracle.select(op, w.alpha, w.sink_blocks, w.window_blocks, seg=seg, pooled=pooled, seg_ids=ids,
                            nthreads=threads)
        oracle.attend(op, sel.sel_full, seg=seg, pooled=pooled, seg_ids=ids, nthreads=threads)
        elapsed += time.perf_counter() - t0
        done += len(ids)
        taken.extend(ids.tolist())
        if elapsed >= target_s:
            break
        per = elapsed / max(float(np.sum(work[np.array(taken)])), 1.0)
        n = int(min(len(seg) - done, max(threads, (target_s - elapsed) / max(per * np.mean(work), 1e-12))))
        if n <= 0:
            break
    frac = float(np.sum(work[np.array(taken)])) / max(float(np.sum(work)), 1.0)
    ms_layer = (t_pool + elapsed / max(frac, 1e-12)) * 1e3
    sample = (f"{len(taken)} of {len(seg)} segments ({100 * frac:.3f}% of the layer's oracle work) "
              f"selected + attended, pooling in full; extrapolated by per-segment work")
    return ms_layer, threads, sample, elapsed + t_pool


# ---------------------------------------------------------------------- our arm

def run_ours(args, rank: int, world: int, dist_on: bool):
    from block_sparse_long_mean_gb300 import binding as B
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = synth.make_workload(args.workload, device=dev, seed=synth.BASE_SEED + rank)
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p, device=dev)
    # every launch and copy goes to a stream of its own (made the current one): the legacy default stream would
    # order itself against the copy streams of the end-to-end pipeline
    torch.cuda.synchronize(dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    flags = B.FP_MEAN_CORRECTION
    # a chunk after a cached prefix: the prefix's block means were pooled by the previous chunk's selection
    # (here: one fp_select before the warm-up) and fp_select_chunk pools only the blocks holding new tokens
    chunked = w.kv_lengths is not None and args.prefix_means == "carried"
    select = B.fp_select_chunk if chunked else B.fp_select
    if chunked:
        B.fp_select(p, w.q, w.k_pages, w.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs.csr_cu,
                    bufs.csr_idx, bufs.kbar, bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace, stream)

    def step(s1=None, s2=None, s3=None):
        if s1 is not None:
            s1.record(stream)
        select(p, w.q, w.k_pages, w.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs.csr_cu,
               bufs.csr_idx, bufs.kbar, bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace, stream)
        if s2 is not None:
            s2.record(stream)
        B.fp_attention(p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op, flags,
                       bufs.out, None, bufs.workspace, stream)
        if s3 is not None:
            s3.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    code = B.fp_device_status(bufs.workspace, stream)
    if code != 0:
        raise RuntimeError(f"device status {B.STATUS.get(code, code)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    start.record(stream)
    for i in range(args.steps):
        step(*ev[i])
    stop.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if dist_on:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    s1 = [e[0].elapsed_time(e[1]) for e in ev]
    s2 = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = max_over_ranks(total_ms, dist_on, dev)
    ms_step = total_ms / args.steps

    # end to end through the public API from pinned host buffers: every step copies its inputs in and its
    # output out. Serial: copy in, compute, copy out, one after the other on one stream. Pipelined (the
    # reported value): two device input and output buffers, so that step i's inputs are copied in (one copy
    # stream) while step i - 1 computes and step i - 2's output is copied out (another copy stream), as a
    # server overlaps the next request's transfer with the current one's compute.
    h_q = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
    h_k = torch.empty(w.k_pages.shape, dtype=w.k_pages.dtype, pin_memory=True)
    h_v = torch.empty(w.v_pages.shape, dtype=w.v_pages.dtype, pin_memory=True)
    h_q.copy_(w.q)
    h_k.copy_(w.k_pages)
    h_v.copy_(w.v_pages)
    h_pt = w.page_table.cpu().pin_memory()
    h_cu = w.cu_seqlens.cpu().pin_memory()
    h_kv = w.seqlens_kv.cpu().pin_memory() if w.seqlens_kv is not None else None
    hosts = [t for t in (h_q, h_k, h_v, h_pt, h_cu, h_kv) if t is not None]
    h_out = [torch.empty(bufs.out.shape, dtype=bufs.out.dtype, pin_memory=True) for _ in range(2)]
    e2e_steps = max(2, min(args.steps, 10))
    # the second set of device inputs and outputs, and the layer through the C ABI on either set
    w2 = synth.Workload(**{**w.__dict__, "q": torch.empty_like(w.q), "k_pages": torch.empty_like(w.k_pages),
                           "v_pages": torch.empty_like(w.v_pages), "page_table": torch.empty_like(w.page_table),
                           "cu_seqlens": torch.empty_like(w.cu_seqlens),
                           "seqlens_kv": None if w.seqlens_kv is None else torch.empty_like(w.seqlens_kv)})
    sets = [(w, p, bufs.out), (w2, B.Problem.from_workload(w2), torch.empty_like(bufs.out))]

    def devs(x):
        return [t for t in (x.q, x.k_pages, x.v_pages, x.page_table, x.cu_seqlens, x.seqlens_kv) if t is not None]

    def layer(ws, pb, out, st):
        select(pb, ws.q, ws.k_pages, ws.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs.csr_cu, bufs.csr_idx,
               bufs.kbar, bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace, st)
        B.fp_attention(pb, ws.q, ws.k_pages, ws.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op, flags,
                       out, None, bufs.workspace, st)

    def e2e_serial():
        for d, h in zip(devs(w), hosts):
            d.copy_(h, non_blocking=True)
        layer(w, p, bufs.out, stream)
        h_out[0].copy_(bufs.out, non_blocking=True)

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipelined(n, start=None, stop=None):
        if start is not None:
            start.record(stream)
            s_in.wait_event(start)
        for i in range(n):
            b = i & 1
            ws, pb, out = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])  # step i - 2 has finished reading this input set
                for d, h in zip(devs(ws), hosts):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i - 2's output has been copied out of this buffer
            layer(ws, pb, out, stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                h_out[b].copy_(out, non_blocking=True)
                ev_out[b].record(s_out)
        if stop is not None:
            stop.record(s_out)
            s_in.wait_event(stop)
            stream.wait_event(stop)

    e2e_serial()
    e2e_pipelined(2)
    torch.cuda.synchronize(dev)
    # the host link is shared with the rest of the machine and has slow periods (both modes see them): each mode
    # is timed five times and the median reported, with every sample in the line
    serial_runs, piped_runs = [], []
    for _ in range(5):
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(stream)
        for _ in range(e2e_steps):
            e2e_serial()
        ee.record(stream)
        torch.cuda.synchronize(dev)
        serial_runs.append(es.elapsed_time(ee) / e2e_steps)
        ps, pe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_pipelined(e2e_steps, ps, pe)
        torch.cuda.synchronize(dev)
        piped_runs.append(ps.elapsed_time(pe) / e2e_steps)
    e2e_serial_ms = float(np.median(serial_runs))
    e2e_ms = float(np.median(piped_runs))
    code = B.fp_device_status(bufs.workspace, stream)
    if code != 0:
        raise RuntimeError(f"device status {B.STATUS.get(code, code)}")
    if not torch.equal(h_out[(e2e_steps - 1) & 1], bufs.out.cpu()):
        raise RuntimeError("the pipelined end-to-end output differs from the layer's")
    h2d = sum(t.numel() * t.element_size() for t in hosts)
    d2h = h_out[0].numel() * h_out[0].element_size()
    del w2, sets

    cu = bufs.csr_cu.cpu().numpy().astype(np.int64)
    idx = bufs.csr_idx[:int(cu[-1])].cpu().numpy()
    acc = accounting(w, cu, idx)
    pk, pk_src = peaks()
    s1_ms, s2_ms = float(np.median(s1)), float(np.median(s2))
    s2_mean = float(np.mean(s2))
    achieved_tflops = acc["executed_flop"] / (s2_mean * 1e-3) / 1e12
    peak_t = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if w.dtype == "e4m3":
        peak_t *= 2.0   # no FP8 GEMM is measured: the BF16 burst times the nominal FP8/BF16 ratio (4.5 / 2.25)
    nominal_t = NOMINAL_TFLOPS[w.dtype]
    s1_mean = float(np.mean(s1))
    stage1_gbs = acc["stage1_bytes"] / (s1_mean * 1e-3) / 1e9
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_ghz = (clk or {}).get("sm_mhz") or float(pk.get("sm_max_mhz", 2070.0))
    sm_ghz = sm_ghz / 1e3
    # Stage 1 floor: its bytes at the measured HBM rate, its pooled-key MACs at the tensor peak of its operand
    # type, its exponentials at the MUFU rate (one per query row and causal block, as Eq.19 states them)
    floor_hbm = acc["stage1_bytes"] / (hbm * 1e9) * 1e3
    floor_mma = acc["stage1_mma_flop"] / (peak_t * 1e12) * 1e3
    floor_mufu = acc["stage1_exps"] / (MUFU_EX2_PER_CLK_SM * sms * sm_ghz * 1e9) * 1e3
    floor_ms = max(floor_hbm, floor_mma, floor_mufu)
    res = dict(metric=METRIC, value=ms_step / world, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
               ms_per_step=ms_step, higher_is_better=False, scaling="weak", vs_baseline=None,
               dtype=w.dtype, data="synthetic",
               config=dict(workload_config(args.workload, w, world),
                           **({"prefix_block_means": "carried from the previous chunk (fp_select_chunk)" if chunked
                               else "pooled again (fp_select)"} if w.kv_lengths is not None else {})),
               stage1_ms=s1_ms, stage2_ms=s2_ms,
               executed_tflops=achieved_tflops,
               dense_equiv_tflops=acc["dense_equiv_flop"] / (ms_step * 1e-3) / 1e12,
               stage1_gbs=stage1_gbs, density=acc["density"], correction_chunks=acc["corr_chunks"],
               roofline=dict(bound="tensor", kernel="fp_attention (Stage 2: meta, bucket, scatter, attention kernels)",
                             achieved=achieved_tflops,
                             peak=peak_t, unit="TFLOP/s", frac=achieved_tflops / peak_t,
                             peak_source=(f"{pk_src} bf16 burst (cuBLAS GEMM)" if w.dtype == "bf16" else
                                          f"{pk_src} bf16 burst x2, the nominal e4m3/bf16 ratio (assumed: no "
                                          f"e4m3 GEMM measured)"),
                             nominal_peak=nominal_t, frac_of_nominal=achieved_tflops / nominal_t,
                             nominal_source="GB300 datasheet dense (no 2:4 sparsity) tensor peak",
                             traffic=attn_traffic(args.workload), traffic_unit="bytes per launch",
                             traffic_source="stored ncu capture of these kernel sources (null once they change)"),
               stage1_roofline=dict(bound="hbm", achieved=stage1_gbs, peak=hbm, unit="GB/s", frac=stage1_gbs / hbm,
                                    floor_ms=floor_ms, frac_of_floor=floor_ms / s1_mean,
                                    floor_parts_ms=dict(hbm=floor_hbm, mma=floor_mma, mufu=floor_mufu),
                                    floor_rule=("max of: Stage 1 bytes at the measured HBM rate; 2 d MACs per "
                                                "(query row, causal block) at the tensor peak; one exp per "
                                                f"(query row, causal block) at {MUFU_EX2_PER_CLK_SM:g} ex2 per "
                                                f"clock per SM x {sms} SMs x {sm_ghz * 1e3:.0f} MHz")),
               e2e=dict(value=e2e_ms, unit=UNIT, h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                        serial_ms=e2e_serial_ms, runs_ms=[round(x, 4) for x in piped_runs],
                        serial_runs_ms=[round(x, 4) for x in serial_runs],
                        how=("pipelined over two device input/output sets: step i's host-to-device copy overlaps "
                             "step i-1's compute and step i-2's device-to-host copy; every step's copies lie in "
                             "the timed region (serial_ms: copy in, compute, copy out, one after the other); "
                             "each the median of five timed runs of the same steps")),
               gpu_launches=kernels_per_step(acc["segments"]) * args.steps,
               clocks=clk)
    if args.dense_steps > 0:
        # this build's own dense mode (alpha = 0: every causal block exact, no correction) through the same
        # attention kernel; it needs no selection, so it is timed as the fp_attention call alone
        out_corr = bufs.out.clone()
        B.fp_attention(p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op, 0,
                       bufs.out, None, bufs.workspace, stream)
        out_nocorr = bufs.out.clone()
        dstart, dstop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        B.fp_attention(p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op,
                       B.FP_DENSE, bufs.out, None, bufs.workspace, stream)
        dstart.record(stream)
        for _ in range(args.dense_steps):
            B.fp_attention(p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op,
                           B.FP_DENSE, bufs.out, None, bufs.workspace, stream)
        dstop.record(stream)
        torch.cuda.synchronize(dev)
        code = B.fp_device_status(bufs.workspace, stream)
        if code != 0:
            raise RuntimeError(f"device status {B.STATUS.get(code, code)}")
        dense_ms = dstart.elapsed_time(dstop) / args.dense_steps
        res["dense_mode_ms"] = dense_ms
        res["dense_mode_executed_tflops"] = acc["dense_mode_executed_flop"] / (dense_ms * 1e-3) / 1e12
        res["speedup_vs_dense_mode"] = dense_ms / ms_step

        def rel_rms(a, b):
            a, b = a.float(), b.float()
            return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))

        # Sec.4.4 "Effect of Mean Correction": how far the sparse layer lies from dense attention, with and
        # without the correction (the dense mode is itself checked against the oracle by the parity tests)
        res["output_rel_rms_vs_dense_mode"] = dict(correction_on=rel_rms(out_corr, bufs.out),
                                                   correction_off=rel_rms(out_nocorr, bufs.out))
        del out_corr, out_nocorr
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if args.cpu_mode == "full":
            ms_cpu, cores, sample = oracle_layer_time(w)
        else:
            ms_cpu, cores, sample, _ = oracle_sample_time(w, cu, idx, target_s=args.cpu_seconds)
        res["cpu_baseline"] = dict(value=ms_cpu, unit=UNIT, cores=cores, kind="oracle", sample=sample)
    return res


def max_over_ranks(ms: float, dist_on: bool, device) -> float:
    """The job's time: the slowest rank's (every rank receives it)."""
    if not dist_on:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def workload_config(name: str, w, world: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    prefix = (f" new tokens after a {max(kv_lengths_of(w)) - max(w.lengths)}-token prefix"
              if w.kv_lengths is not None else "")
    return dict(workload=f"{name}: batch {w.batch}, L={max(w.lengths)}{prefix}, Hq={w.hq}, Hkv={w.hkv}, d=128, "
                         f"B=128, page 64, alpha={w.alpha}, sink {w.sink_blocks}, window {w.window_blocks}",
                tokens=w.total_tokens, inputs_larger_than_l2=True, l2_flush=False, parallelism=f"replicas x{world}")


def run_reference(args):
    """The fp64 CPU oracle as the reference arm: each step times a bounded sample of the layer."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_workload(args.workload, device=dev)
    # the oracle's own selection defines the CSR used for work accounting
    import oracle
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    pooled = oracle.pool(op, seg)
    sample_ids = np.random.default_rng(7).choice(len(seg), size=min(len(seg), 64), replace=False)
    sel = oracle.select(op, w.alpha, w.sink_blocks, w.window_blocks, seg=seg, pooled=pooled, seg_ids=sample_ids)
    # selected counts: forced set estimate for unsampled segments, the oracle's own for sampled ones
    counts = np.minimum(seg.D + 1, 3)
    for s in sample_ids:
        counts[s] = len(sel.selected(seg, s))
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    idx = np.zeros(int(cu[-1]), np.int64)
    per_step = max(2.0, min(args.cpu_seconds, 150.0 / max(args.steps + args.warmup, 1)))
    times = []
    for i in range(args.warmup + args.steps):
        ms, cores, sample, _ = oracle_sample_time(w, cu, idx, target_s=per_step)
        if i >= args.warmup:
            times.append(ms)
    v = float(np.mean(times))
    return dict(impl="reference", metric=METRIC, value=v, unit=UNIT, n_gpus=1, steps=args.steps,
                warmup=args.warmup, ms_per_step=v, higher_is_better=False, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic",
                config=workload_config(args.workload, w, int(os.environ.get("WORLD_SIZE", "1"))),
                cpu_baseline=dict(value=v, unit=UNIT, cores=cores, kind="oracle", sample=sample),
                e2e=dict(value=v, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--dense-steps", type=int, default=3, help="timed steps of the alpha = 0 dense mode (0: skip)")
    ap.add_argument("--cpu-mode", default="full", choices=["full", "sample"],
                    help="cpu_baseline: the oracle over the whole layer, or a timed sample extrapolated to it")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--prefix-means", default="carried", choices=["carried", "pooled"],
                    help="workloads with a cached prefix: keep the prefix's block means from the previous chunk "
                         "(fp_select_chunk) or pool them again (fp_select)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    dist_on = world > 1
    if dist_on:
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, dist_on)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
