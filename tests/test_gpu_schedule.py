"""GPU parity of the attention stage's integer work within a fixed CSR.

The oracle's own CSR (its selection over every segment) goes to
fp_attention_trace, which records what the attention kernel actually walked:
the scheduler's work list, each tile's visit sequence, the correction chunks
with their masks and the page-table rows of every block. The host recomputes
all of it from the same CSR with oracle.tile_schedule and oracle.split_plan
(FlashPrefill V2 Sec.3.3 Eq.17, "Sparsity-Aware Load Balancing", Eq.18; Sec.3.2
"Implementation" for todo = valid & ~selected) and the two must agree bit for
bit. Where several results are correct (the order of equal-cost tiles in the
work list) the test checks that the order is valid instead.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from block_sparse_long_mean_gb300 import binding as B  # noqa: E402
from block_sparse_long_mean_gb300 import synth  # noqa: E402


def parse_trace(tr: np.ndarray):
    used, overflow, nitems = int(tr[0]), int(tr[1]), int(tr[2])
    assert overflow == 0
    items = {}
    o, end = 8, 8 + used
    while o < end:
        w, b, h, T, D, lo, hi, ne = (int(x) for x in tr[o:o + 8])
        n = hi - lo
        ent = tr[o + 8:o + 8 + 8 * n].reshape(n, 8).astype(np.int64)
        assert w not in items
        items[w] = dict(b=b, h=h, T=T, D=D, lo=lo, hi=hi, n_exact=ne, ent=ent)
        o += 8 + 8 * n
    assert o == end
    return nitems, items


def check_integer_work(w, flags, alpha=None, sink=None, window=None):
    alpha = w.alpha if alpha is None else alpha
    sink = w.sink_blocks if sink is None else sink
    window = w.window_blocks if window is None else window
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p)
    # Stage 1 on the GPU: its CSR must be the oracle's (near-threshold blocks excepted, counted)
    B.fp_select(p, w.q, w.k_pages, w.v_pages, alpha, sink, window, bufs.csr_cu, bufs.csr_idx, bufs.kbar,
                bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace)
    assert B.fp_device_status(bufs.workspace) == B.FP_OK
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    sel = oracle.select(op, alpha, sink, window, seg=seg)
    cu, idx = oracle.csr_from_selection(seg, sel)
    gcu = bufs.csr_cu.cpu().numpy()
    gsel = oracle.selection_from_csr(seg, gcu, bufs.csr_idx[:int(gcu[-1])].cpu().numpy())
    flips = np.nonzero(gsel[:seg.full_total] != sel.sel_full[:seg.full_total])[0]
    assert np.all(sel.near_full[flips]), "CSR differs from the oracle's outside near-threshold blocks"

    # Stage 2 on the oracle's CSR, traced
    d_cu = torch.from_numpy(cu.astype(np.int32)).cuda()
    d_idx = torch.from_numpy(np.concatenate([idx, [0]]).astype(np.int32)).cuda()
    dense = bool(flags & B.FP_DENSE)
    corr = bool(flags & B.FP_MEAN_CORRECTION) and not dense
    seqs = [oracle.tile_schedule(op, seg, s, cu, idx, correction=corr, dense=dense) for s in range(len(seg))]
    costs = np.array([len(x) for x in seqs])
    # one 8-word header per work item (a split tile has one per run: at most 320 runs beyond the tiles) and
    # one 8-word entry per iteration
    words = 8 + 8 * (len(seg) + 320 + int(costs.sum()))
    trace = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    B.fp_attention_trace(p, w.q, w.k_pages, w.v_pages, d_cu, d_idx, bufs.kbar_op, bufs.vbar_op, flags, bufs.out,
                         bufs.lse, bufs.workspace, trace)
    assert B.fp_device_status(bufs.workspace) == B.FP_OK
    nitems, items = parse_trace(trace.cpu().numpy())

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    target, runs = oracle.split_plan(costs, sms)
    assert nitems == sum(len(r) for r in runs) == len(items)
    assert sorted(items) == list(range(nitems))
    key = {(int(seg.b[s]), int(seg.h[s]), int(seg.T[s])): s for s in range(len(seg))}
    by_seg = {}
    for wi in range(nitems):
        it = items[wi]
        s = key[(it["b"], it["h"], it["T"])]
        by_seg.setdefault(s, []).append(wi)
        assert it["D"] == int(seg.D[s])
        assert it["n_exact"] == (int(seg.D[s]) + 1 if dense else int(cu[s + 1] - cu[s]))
        # the visited iterations, in order, with masks and page rows
        want = seqs[s][it["lo"]:it["hi"]]
        ent = it["ent"]
        assert np.array_equal(ent[:, 0], want[:, 0]), (s, ent[:, 0], want[:, 0])
        assert np.array_equal(ent[:, 2:6] & 0xffffffff, want[:, 1:5]), s
        assert np.array_equal(ent[:, 6:8], want[:, 5:7]), s
        fl = np.zeros(len(ent), np.int64)
        if len(ent):
            fl[0] |= 1
            fl[-1] |= 2
        assert np.array_equal(ent[:, 1], fl), s
    # every tile once, its runs contiguous in the work list and in iteration order, as the split plan says
    assert sorted(by_seg) == list(range(len(seg)))
    for s, ws in by_seg.items():
        assert ws == list(range(ws[0], ws[0] + len(ws)))
        assert [(items[x]["lo"], items[x]["hi"]) for x in ws] == runs[s], (s, runs[s])
    # heaviest tiles first (equal costs in any order)
    order_costs = [costs[key[(items[x]["b"], items[x]["h"], items[x]["T"])]] for x in range(nitems)]
    assert all(a >= b for a, b in zip(order_costs, order_costs[1:]))
    n_chunks = int(sum(int(np.sum(x[:, 0] < 0)) for x in seqs))
    print(f"items {nitems}, tiles {len(seg)}, split target {target}, iterations {int(costs.sum())}, "
          f"correction chunks {n_chunks}, near-threshold flips {len(flips)}")
    return target


STRESS = dict(lengths=[1000, 333, 0, 2112, 129], hq=16, hkv=2, mu_scale=0.5, alpha=0.05, paging="random",
              page_size=32, seed=21)


def test_integer_work_tiny_2k_split():
    w = synth.make_workload("tiny_2k", device="cuda")
    assert check_integer_work(w, B.FP_MEAN_CORRECTION) is not None   # 64 tiles: split plan active


@pytest.mark.parametrize("flags", [B.FP_MEAN_CORRECTION, 0, B.FP_DENSE])
def test_integer_work_stress_varlen(flags):
    w = synth.make_workload("tiny_2k", device="cuda", **STRESS)
    check_integer_work(w, flags)


@pytest.mark.parametrize("flags", [B.FP_DENSE, B.FP_MEAN_CORRECTION])
def test_integer_work_split_runs(flags):
    # one 8K request on one head: 64 tiles, the heavy last ones cut into many count-balanced runs (Eq.18)
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[8192], hq=1, hkv=1, mu_scale=0.5,
                            alpha=0.02)
    assert check_integer_work(w, flags) is not None


def test_integer_work_chunked_prefill():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1000, 77, 1, 0, 130], kv_lengths=[2600, 300, 129, 64, 130],
                            hq=8, hkv=2, mu_scale=0.5, alpha=0.05, paging="random", page_size=16, seed=44)
    check_integer_work(w, B.FP_MEAN_CORRECTION)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_integer_work_without_splits(dtype):
    # 938 tiles (more than 4 x SMs): every tile is one work item
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[12000, 3000], hq=8, hkv=2, dtype=dtype,
                            alpha=0.2 if dtype == "e4m3" else 0.1, paging="random")
    assert check_integer_work(w, B.FP_MEAN_CORRECTION) is None


def test_integer_work_paper_forced_set():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[2048, 900], hq=8, hkv=2, mu_scale=0.6)
    check_integer_work(w, B.FP_MEAN_CORRECTION, sink=2, window=4)


def test_trace_reports_overflow_without_writing_past_its_end():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1024], hq=4, hkv=1)
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p)
    B.run_layer(p, w.q, w.k_pages, w.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs)
    ref = bufs.out.clone()
    buf = torch.full((64 + 16,), -7, dtype=torch.int32, device="cuda")
    trace = buf[:64]
    B.fp_attention_trace(p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op,
                         B.FP_MEAN_CORRECTION, bufs.out, None, bufs.workspace, trace)
    assert B.fp_device_status(bufs.workspace) == B.FP_OK
    t = trace.cpu().numpy()
    assert t[1] == 1                                     # ran out of room
    assert bool((buf[64:] == -7).all())                  # nothing written past the capacity
    assert torch.equal(bufs.out, ref)                    # the outputs are fp_attention's
