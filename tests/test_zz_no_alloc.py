"""fp_select_noalloc: Stage 1 for callers that cannot allocate device memory.

Such callers (an engine plugin handed only its tensors, or code where
cudaMalloc's implicit device synchronisation is not allowed) cannot provide a
workspace, so this entry point takes its scratch from a fixed 16 MiB array
inside the library. It must produce exactly what fp_select produces. This file
is named to be collected last, so a failure here never hides another test.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from block_sparse_long_mean_gb300 import binding as B  # noqa: E402
from block_sparse_long_mean_gb300 import synth  # noqa: E402


def _select_with_workspace(p, w):
    bufs = B.Buffers(p)
    B.fp_select(p, w.q, w.k_pages, w.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs.csr_cu, bufs.csr_idx,
                bufs.kbar, bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace)
    assert B.fp_device_status(bufs.workspace) == B.FP_OK
    return bufs


def _select_noalloc(p, w):
    bufs = B.Buffers(p)
    for t in (bufs.csr_cu, bufs.csr_idx):
        t.fill_(-7)                 # outputs must be fully written by the call
    bufs.kbar.fill_(float("nan"))
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    B.fp_select_noalloc(p, w.q, w.k_pages, w.v_pages, w.alpha, w.sink_blocks, w.window_blocks, bufs.csr_cu,
                        bufs.csr_idx, bufs.kbar, bufs.vbar, bufs.kbar_op, bufs.vbar_op, status)
    torch.cuda.synchronize()
    assert int(status.item()) == B.FP_OK
    return bufs


def _same(a, b):
    assert torch.equal(a.csr_cu, b.csr_cu)
    nnz = int(a.csr_cu[-1])
    assert torch.equal(a.csr_idx[:nnz], b.csr_idx[:nnz])
    for name in ("kbar", "vbar", "kbar_op", "vbar_op"):
        x, y = getattr(a, name).float(), getattr(b, name).float()
        assert torch.equal(x, y), name


def test_noalloc_select_matches_workspace_select_on_consecutive_calls():
    # two different problems, then the first again: the shared scratch keeps the previous call's
    # contents, which must not leak into the next result
    wa = synth.make_workload("tiny_2k", device="cuda", lengths=[1000, 333, 0, 2112], hq=16, hkv=2, mu_scale=0.5,
                             alpha=0.05, paging="random")
    wb = synth.make_workload("tiny_2k", device="cuda", lengths=[4096], hq=8, hkv=1, mu_scale=0.6, alpha=0.1,
                             paging="random", seed=5)
    for w in (wa, wb, wa):
        p = B.Problem.from_workload(w)
        _same(_select_noalloc(p, w), _select_with_workspace(p, w))


def test_noalloc_select_rejects_problems_beyond_its_scratch():
    # 4 x 1M-token requests need far more than 16 MiB of scratch: rejected on the host
    lengths = [1 << 20] * 4
    import numpy as np
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pt = torch.zeros(4, (1 << 20) // 64, dtype=torch.int32, device="cuda")
    p = B.Problem(torch.from_numpy(cu).cuda(), cu, pt, 32, 4, num_pages=1 << 16)
    assert B.fp_workspace_bytes(p) > 16 << 20
    code = B.fp_select_noalloc(p, None, None, None, 0.1, 1, 1, None, None, None, None, None, None, check=False)
    assert code == B.STATUS_CODE["FP_ERR_WORKSPACE"]
