"""CPU checks of the C-ABI library: it loads, exports every entry point the
header declares, sizes problems like the oracle's segment enumeration and
rejects invalid descriptions on the host (no device work is enqueued for them)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_mean_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "fp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_entry_point():
    names = header_functions()
    assert set(names) == set(B.EXPORTS), names
    for n in names:
        assert hasattr(B.lib, n), n
        assert callable(getattr(B, n)), n


def problem(lengths, hq=32, hkv=4, page=64, dtype="bf16", kv_lengths=None, **kw):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    kvl = lengths if kv_lengths is None else kv_lengths
    stride = max(1, max((L + page - 1) // page for L in kvl) if kvl else 1)
    pt = torch.zeros(len(lengths), stride, dtype=torch.int32)
    if kv_lengths is not None:
        kv = np.asarray(kv_lengths, dtype=np.int32)
        kw.update(seqlens_kv=torch.from_numpy(kv.copy()), host_seqlens_kv=kv)
    return B.Problem(torch.from_numpy(cu), cu, pt, hq, hkv, num_pages=1 << 20, page_size=page, dtype=dtype, **kw)


@pytest.mark.parametrize("lengths,hq,hkv,kv_lengths", [
    ([131072], 32, 4, None), ([32768], 32, 8, None), ([2048], 4, 1, None), ([300, 0, 129, 4096], 8, 2, None),
    ([1], 16, 1, None), ([], 8, 8, None),
    # chunked prefill after a cached prefix: on and off the tile grid, one query, an empty chunk
    ([8192], 32, 4, [131072]), ([77, 200, 1, 0, 130], 8, 2, [300, 456, 129, 64, 130]), ([5], 4, 4, [1000]),
])
def test_sizing_matches_oracle_segments(lengths, hq, hkv, kv_lengths):
    p = problem(lengths, hq, hkv, kv_lengths=kv_lengths)
    op = oracle.Problem(q=np.zeros((1, hq, 128), np.uint16), k_pages=np.zeros((1, 64, hkv, 128), np.uint16),
                        v_pages=np.zeros((1, 64, hkv, 128), np.uint16),
                        cu_seqlens=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32),
                        page_table=np.zeros((max(len(lengths), 1), 1), np.int32), hq=hq, hkv=hkv,
                        seqlens_kv=None if kv_lengths is None else np.asarray(kv_lengths, np.int32))
    seg = oracle.segments(op)
    assert B.fp_num_segments(p) == len(seg)
    assert B.fp_num_blocks(p) == seg.total_blocks
    assert B.fp_csr_capacity(p) == int((seg.D + 1).sum())
    assert B.fp_workspace_bytes(p) > 0


@pytest.mark.parametrize("kw,code", [
    (dict(lengths=[256], hq=12, hkv=4), -2),      # g = 3 is not a power of two
    (dict(lengths=[256], hq=64, hkv=2), -2),      # g = 32 > 16
    (dict(lengths=[256], hq=10, hkv=4), -2),      # Hq % Hkv != 0
    (dict(lengths=[256], page=48), -2),           # page size not a power of two
    (dict(lengths=[256], page=256), -2),          # page larger than a block
    (dict(lengths=[(1 << 20) + 128]), -2),        # longer than the supported maximum
])
def test_host_rejects_unsupported_descriptions(kw, code):
    assert B.lib.fp_num_segments(problem(**kw).ref) == code


def test_host_rejects_bad_arguments_before_any_device_work():
    p = problem([256], hq=8, hkv=2)
    p.c.head_dim = 64
    assert B.lib.fp_workspace_bytes(p.ref) == -2
    p = problem([256], hq=8, hkv=2)
    fake = ctypes.c_void_p(1 << 20)    # never dereferenced: validation fails first
    need = B.fp_workspace_bytes(p)
    # workspace too small
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need - 1, None) == -3
    # negative alpha / window, null CSR
    assert B.lib.fp_select(p.ref, fake, fake, fake, -0.5, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need, None) == -1
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, -1, fake, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need, None) == -1
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, None, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need, None) == -1
    # misaligned workspace
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake,
                           ctypes.c_void_p((1 << 20) + 8), need, None) == -1
    # unknown flags, missing means with correction on
    assert B.lib.fp_attention(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 8, fake, None, fake, need,
                              None) == -1
    assert B.lib.fp_attention(p.ref, fake, fake, fake, fake, fake, 10, None, None, 1, fake, None, fake, need,
                              None) == -1
    # misaligned tensors: TMA-read inputs and the output need 16 bytes, lse 4
    odd8, odd2 = ctypes.c_void_p((1 << 20) + 8), ctypes.c_void_p((1 << 20) + 2)
    assert B.lib.fp_select(p.ref, odd8, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need, None) == -1
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, odd8, fake, fake,
                           need, None) == -1
    assert B.lib.fp_attention(p.ref, fake, odd8, fake, fake, fake, 10, fake, fake, 1, fake, None, fake, need,
                              None) == -1
    assert B.lib.fp_attention(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 1, odd8, None, fake, need,
                              None) == -1
    assert B.lib.fp_attention(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 1, fake, odd2, fake, need,
                              None) == -1
    assert B.lib.fp_select_noalloc(p.ref, fake, fake, odd8, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake,
                                   None, None) == -1
    # int32 / fp32 arrays need 4 bytes
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, odd2, fake, 10 ** 6, fake, fake, fake, fake, fake,
                           need, None) == -1
    assert B.lib.fp_select(p.ref, fake, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, odd2, fake, fake, fake, fake,
                           need, None) == -1
    assert B.lib.fp_attention(p.ref, fake, fake, fake, fake, odd2, 10, fake, fake, 1, fake, None, fake, need,
                              None) == -1
    assert B.lib.fp_csr_expand64(p.ref, fake, fake, fake, odd2, 10, fake, need, None) == -1
    # the chunk variant validates like fp_select
    assert B.lib.fp_select_chunk(p.ref, fake, fake, fake, 0.1, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake,
                                 fake, need - 1, None) == -3
    assert B.lib.fp_select_chunk(p.ref, fake, fake, fake, -0.5, 1, 1, fake, fake, 10 ** 6, fake, fake, fake, fake,
                                 fake, need, None) == -1
    # the traced attention: a trace buffer that is null, misaligned or smaller than its 8-word header
    assert B.lib.fp_attention_trace(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 1, fake, None, fake, need,
                                    None, None, 64) == -1
    assert B.lib.fp_attention_trace(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 1, fake, None, fake, need,
                                    None, odd8, 64) == -1
    assert B.lib.fp_attention_trace(p.ref, fake, fake, fake, fake, fake, 10, fake, fake, 1, fake, None, fake, need,
                                    None, fake, 7) == -1
    # statistics read-back: null workspace or output
    stats = B.fp_select_stats()
    assert B.lib.fp_read_select_stats(None, ctypes.byref(stats), None) == -1
    assert B.lib.fp_read_select_stats(fake, None, None) == -1
    # FP8 without scales
    p8 = problem([256], hq=8, hkv=2, dtype="e4m3", c_q=0.0, c_k=1.0, c_v=1.0)
    assert B.lib.fp_workspace_bytes(p8.ref) == -1
    # a misaligned device int32 array in the description
    p = problem([256], hq=8, hkv=2)
    p.c.page_table = (1 << 20) + 2
    assert B.lib.fp_num_segments(p.ref) == -1
    # device cu_seqlens missing although tokens exist
    p = problem([256], hq=8, hkv=2)
    p.c.cu_seqlens = None
    assert B.lib.fp_num_segments(p.ref) == -1


def test_host_rejects_bad_kv_lengths():
    # L^kv < L^q, one of the two seqlens_kv pointers missing, L^kv past the maximum, a page table too short
    assert B.lib.fp_num_segments(problem([256], hq=8, hkv=2, kv_lengths=[255]).ref) == -1
    p = problem([256], hq=8, hkv=2, kv_lengths=[512])
    p.c.host_seqlens_kv = None
    assert B.lib.fp_num_segments(p.ref) == -1
    p = problem([256], hq=8, hkv=2, kv_lengths=[512])
    p.c.seqlens_kv = None
    assert B.lib.fp_num_segments(p.ref) == -1
    assert B.lib.fp_num_segments(problem([256], hq=8, hkv=2, kv_lengths=[(1 << 20) + 1]).ref) == -2
    p = problem([256], hq=8, hkv=2, kv_lengths=[512])
    p.c.page_table_stride = 7                    # 512 keys need 8 pages of 64
    assert B.lib.fp_num_segments(p.ref) == -1
    # KV blocks but no query: pooling still needs the K/V buffers
    p = problem([0], hq=8, hkv=2, kv_lengths=[300])
    assert B.fp_num_segments(p) == 0 and B.fp_num_blocks(p) == 3
    need = B.fp_workspace_bytes(p)
    fake = ctypes.c_void_p(1 << 20)
    assert B.lib.fp_select(p.ref, None, None, fake, 0.1, 1, 1, fake, None, 0, fake, fake, fake, fake, fake,
                           need, None) == -1


def test_status_strings():
    for code, name in B.STATUS.items():
        assert B.fp_status_string(code) and "unknown" not in B.fp_status_string(code), name
