"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Criteria: CSR bit-exact except blocks whose oracle energy lies within 1e-3
relative of the threshold (counted); BF16 output rel-RMS <= 1e-2 and max-abs
<= 3e-2; FP8 rel-RMS <= 6e-2; integer work bit-exact and deterministic.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from block_sparse_long_mean_gb300 import binding as B  # noqa: E402
from block_sparse_long_mean_gb300 import synth  # noqa: E402

from parity import BF16_MAX_ABS, BF16_REL_RMS, FP8_REL_RMS, compare, run_gpu  # noqa: E402


def check_bf16(rep):
    print(rep)
    assert rep.csr_mismatch == 0
    assert rep.rel_rms <= BF16_REL_RMS and rep.max_abs <= BF16_MAX_ABS
    assert rep.lse_max_abs <= 2e-2
    assert rep.mean_max_err <= 1e-4


def check_fp8(rep):
    print(rep)
    assert rep.csr_mismatch == 0
    assert rep.rel_rms <= FP8_REL_RMS


# ------------------------------------------------------------------ small, full parity

def test_tiny_2k_full_parity():
    w = synth.make_workload("tiny_2k", device="cuda")
    check_bf16(compare(run_gpu(w)))


@pytest.mark.parametrize("g,hkv,page", [(8, 2, 64), (4, 1, 16), (1, 3, 128), (16, 1, 32), (2, 2, 8)])
def test_stress_varlen_parity(g, hkv, page):
    # denser selection (mu ~ N(0, 0.5^2 I)), ragged lengths, an empty request, several page sizes
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1000, 333, 0, 2112, 129], hq=g * hkv, hkv=hkv,
                            mu_scale=0.5, alpha=0.05, paging="random", page_size=page, seed=g * 10 + hkv)
    rep = compare(run_gpu(w))
    check_bf16(rep)
    assert rep.density > 0.3


def test_dense_mode_matches_oracle_dense():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1536, 700], hq=8, hkv=2)
    check_bf16(compare(run_gpu(w, flags=B.FP_DENSE)))


def test_alpha_zero_selects_every_causal_block():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1024, 300], hq=8, hkv=2)
    rep = compare(run_gpu(w, alpha=0.0))
    check_bf16(rep)
    assert rep.density == 1.0


def test_correction_off_matches_oracle_eq4():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[2048, 640], hq=8, hkv=2, mu_scale=0.7)
    check_bf16(compare(run_gpu(w, flags=0)))


def test_fp8_small_parity():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[2048, 517], hq=8, hkv=2, dtype="e4m3", alpha=0.2,
                            paging="random")
    check_fp8(compare(run_gpu(w)))


# ------------------------------------------------------------ integer work, determinism

def test_repeat_runs_and_page_placement_are_bit_identical():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1500, 900], hq=8, hkv=2, mu_scale=0.5,
                            alpha=0.05, paging="random")
    a = run_gpu(w)
    b = run_gpu(w)
    for name in ("csr_cu", "out", "lse", "kbar", "vbar"):
        assert torch.equal(getattr(a.bufs, name), getattr(b.bufs, name)), name
    nnz = int(a.bufs.csr_cu[-1])
    assert torch.equal(a.bufs.csr_idx[:nnz], b.bufs.csr_idx[:nnz])
    # move every page to another slot of the pool
    n = w.num_pages
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3)).to("cuda")
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n, device="cuda")
    w2 = synth.Workload(**{**w.__dict__})
    w2.k_pages = w.k_pages[perm].contiguous()
    w2.v_pages = w.v_pages[perm].contiguous()
    w2.page_table = torch.where(w.page_table >= 0, inv[w.page_table.clamp(min=0).long()].int(),
                                w.page_table).contiguous()
    c = run_gpu(w2)
    assert torch.equal(a.bufs.csr_cu, c.bufs.csr_cu)
    assert torch.equal(a.bufs.csr_idx[:nnz], c.bufs.csr_idx[:nnz])
    assert torch.equal(a.bufs.out, c.bufs.out)


def test_csr_counts_and_offsets_are_consistent():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[777, 2048], hq=8, hkv=2, mu_scale=0.5,
                            alpha=0.05)
    r = run_gpu(w)
    cu = r.bufs.csr_cu.cpu().numpy()
    idx = r.bufs.csr_idx[:cu[-1]].cpu().numpy()
    assert cu[0] == 0 and np.all(np.diff(cu) >= 1)        # the diagonal block is always kept
    for s in range(len(cu) - 1):
        seg = idx[cu[s]:cu[s + 1]]
        assert np.all(np.diff(seg) > 0)


# ------------------------------------------------------------------- device-side errors

def test_out_of_range_page_is_reported_not_faulted():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[512], hq=4, hkv=1, paging="random")
    w.page_table[0, 3] = w.num_pages + 7
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p)
    B.fp_select(p, w.q, w.k_pages, w.v_pages, 0.1, 1, 1, bufs.csr_cu, bufs.csr_idx, bufs.kbar, bufs.vbar,
                bufs.kbar_op, bufs.vbar_op, bufs.workspace)
    assert B.fp_device_status(bufs.workspace) == B.STATUS_CODE["FP_ERR_DEVICE_PAGE"]


def test_malformed_csr_is_reported():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1024], hq=4, hkv=1)
    r = run_gpu(w)
    bufs = r.bufs
    nnz = int(bufs.csr_cu[-1])
    bad = bufs.csr_idx.clone()
    bad[nnz - 1] = 10 ** 6     # outside [0, D]
    B.fp_attention(r.p, w.q, w.k_pages, w.v_pages, bufs.csr_cu, bad, bufs.kbar_op, bufs.vbar_op,
                   B.FP_MEAN_CORRECTION, bufs.out, None, bufs.workspace)
    assert B.fp_device_status(bufs.workspace) == B.STATUS_CODE["FP_ERR_DEVICE_CSR"]


def test_csr_capacity_overflow_is_reported():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1024], hq=4, hkv=1)
    p = B.Problem.from_workload(w)
    bufs = B.Buffers(p, capacity=5)
    B.fp_select(p, w.q, w.k_pages, w.v_pages, 0.1, 1, 1, bufs.csr_cu, bufs.csr_idx, bufs.kbar, bufs.vbar,
                bufs.kbar_op, bufs.vbar_op, bufs.workspace)
    assert B.fp_device_status(bufs.workspace) == B.STATUS_CODE["FP_ERR_DEVICE_OVERFLOW"]


# ----------------------------------------------------- full-size workloads, sampled parity

def test_llama8b_32k_sampled_parity():
    w = synth.make_workload("llama8b_32k", device="cuda")
    check_bf16(compare(run_gpu(w)))


def test_qwen30b_128k_sampled_parity():
    w = synth.make_workload("qwen30b_128k", device="cuda")
    check_bf16(compare(run_gpu(w), n_random=32))


def test_qwen30b_128k_fp8_sampled_parity_with_and_without_correction():
    w = synth.make_workload("qwen30b_128k_fp8", device="cuda")
    on = compare(run_gpu(w), n_random=24)
    check_fp8(on)
    off = compare(run_gpu(w, flags=0), n_random=24, check_means=False)
    print("fp8 correction on/off rel-RMS vs the oracle of each mode:", on.rel_rms, off.rel_rms)
    assert off.rel_rms <= FP8_REL_RMS


@pytest.mark.parametrize("name", ["varlen16", "varlen16_fp8"])
def test_varlen16_sampled_parity(name):
    w = synth.make_workload(name, device="cuda")
    rep = compare(run_gpu(w), n_random=32)
    (check_fp8 if w.dtype == "e4m3" else check_bf16)(rep)


# ------------------------------------------------- serving formats and the paper's forced set

@pytest.mark.parametrize("page", [64, 16])
def test_tiles64_expansion_matches_oracle(page):
    import oracle
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1000, 333, 0, 2112, 129, 64], hq=8, hkv=2,
                            mu_scale=0.5, alpha=0.05, paging="random", page_size=page)
    r = run_gpu(w)
    nseg = B.fp_num_segments(r.p)
    nnz = int(r.bufs.csr_cu[-1])
    tile_cu = torch.empty(nseg + 1, dtype=torch.int32, device="cuda")
    tile_idx = torch.full((2 * nnz + 16,), -7, dtype=torch.int32, device="cuda")
    B.fp_csr_expand64(r.p, r.bufs.csr_cu, r.bufs.csr_idx, tile_cu, tile_idx, r.bufs.workspace)
    assert B.fp_device_status(r.bufs.workspace) == B.FP_OK
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    cu = r.bufs.csr_cu.cpu().numpy()
    want_cu, want_idx = oracle.tiles64_from_csr(op, seg, cu, r.bufs.csr_idx[:nnz].cpu().numpy())
    got_cu = tile_cu.cpu().numpy()
    assert np.array_equal(got_cu, want_cu)
    assert np.array_equal(tile_idx[:got_cu[-1]].cpu().numpy(), want_idx)
    assert bool((tile_idx[got_cu[-1]:] == -7).all())   # nothing written past the result


def test_tiles64_expansion_reports_bad_ids_and_overflow():
    w = synth.make_workload("tiny_2k", device="cuda", lengths=[1024, 300], hq=4, hkv=1)
    r = run_gpu(w)
    nseg = B.fp_num_segments(r.p)
    nnz = int(r.bufs.csr_cu[-1])
    tile_cu = torch.empty(nseg + 1, dtype=torch.int32, device="cuda")
    full = torch.empty(2 * nnz, dtype=torch.int32, device="cuda")
    B.fp_csr_expand64(r.p, r.bufs.csr_cu, r.bufs.csr_idx, tile_cu, full, r.bufs.workspace)
    assert B.fp_device_status(r.bufs.workspace) == B.FP_OK
    # too small a capacity: reported, and the result is cut off at the capacity
    small = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    B.fp_csr_expand64(r.p, r.bufs.csr_cu, r.bufs.csr_idx, tile_cu, small, r.bufs.workspace)
    assert B.fp_device_status(r.bufs.workspace) == B.STATUS_CODE["FP_ERR_DEVICE_OVERFLOW"]
    assert torch.equal(small, full[:3])
    # a block id past the request: reported and skipped
    bad = r.bufs.csr_idx.clone()
    bad[nnz - 1] = 10 ** 6
    B.fp_csr_expand64(r.p, r.bufs.csr_cu, bad, tile_cu, full, r.bufs.workspace)
    assert B.fp_device_status(r.bufs.workspace) == B.STATUS_CODE["FP_ERR_DEVICE_CSR"]


@pytest.mark.parametrize("name", ["tiny_2k", "llama8b_32k"])
def test_paper_default_forced_set_parity(name):
    # 256 sink tokens and a 512-token local window = 2 sink blocks and 4 window blocks of 128 tokens
    kw = dict(lengths=[2048, 900], hq=8, hkv=2, mu_scale=0.6) if name == "tiny_2k" else {}
    w = synth.make_workload(name, device="cuda", **kw)
    w.sink_blocks, w.window_blocks = 2, 4
    rep = compare(run_gpu(w), n_random=32)
    check_bf16(rep)
