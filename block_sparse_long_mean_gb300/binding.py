"""Thin ctypes binding of libfp.so (include/fp.h): argument marshalling only.

Every function has the name of the C entry point it calls and passes device
pointers of torch tensors and the current torch CUDA stream. No step of the
method runs in Python. If the library is missing or cannot be loaded the
import of this module fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp.so")

FP_OK = 0
FP_MEAN_CORRECTION = 1
FP_DENSE = 2
FP_DTYPE_BF16 = 0
FP_DTYPE_E4M3 = 1

STATUS = {
    0: "FP_OK", -1: "FP_ERR_INVALID_ARG", -2: "FP_ERR_UNSUPPORTED", -3: "FP_ERR_WORKSPACE", -4: "FP_ERR_CUDA",
    -5: "FP_ERR_CAPACITY", -16: "FP_ERR_DEVICE_PAGE", -17: "FP_ERR_DEVICE_CSR", -18: "FP_ERR_DEVICE_OVERFLOW",
    -19: "FP_ERR_DEVICE_TIMEOUT", -20: "FP_ERR_DEVICE_SEQLEN",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}
EXPORTS = ["fp_workspace_bytes", "fp_num_segments", "fp_num_blocks", "fp_csr_capacity", "fp_select",
           "fp_attention", "fp_device_status", "fp_status_string", "fp_select_noalloc", "fp_csr_expand64",
           "fp_read_select_stats", "fp_attention_trace", "fp_select_chunk"]


class FpError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class fp_problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("c_q", ctypes.c_float), ("c_k", ctypes.c_float), ("c_v", ctypes.c_float),
        ("cu_seqlens", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("page_table_stride", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("host_cu_seqlens", ctypes.c_void_p),
        ("seqlens_kv", ctypes.c_void_p), ("host_seqlens_kv", ctypes.c_void_p),
    ]


class fp_select_stats(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int32), ("exact_tiles", ctypes.c_int32), ("exact_blocks", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libfp.so not built at {_LIB_PATH}; run block_sparse_long_mean_gb300/build_lib.py")
    L = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER(fp_problem)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    for name in ("fp_workspace_bytes", "fp_num_segments", "fp_num_blocks", "fp_csr_capacity"):
        getattr(L, name).restype = i64
        getattr(L, name).argtypes = [P]
    L.fp_select.restype = ctypes.c_int
    L.fp_select.argtypes = [P, vp, vp, vp, f32, i32, i32, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]
    L.fp_select_chunk.restype = ctypes.c_int
    L.fp_select_chunk.argtypes = [P, vp, vp, vp, f32, i32, i32, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]
    L.fp_select_noalloc.restype = ctypes.c_int
    L.fp_select_noalloc.argtypes = [P, vp, vp, vp, f32, i32, i32, vp, vp, i64, vp, vp, vp, vp, vp, vp]
    L.fp_attention.restype = ctypes.c_int
    L.fp_attention.argtypes = [P, vp, vp, vp, vp, vp, i64, vp, vp, i32, vp, vp, vp, sz, vp]
    L.fp_csr_expand64.restype = ctypes.c_int
    L.fp_csr_expand64.argtypes = [P, vp, vp, vp, vp, i64, vp, sz, vp]
    L.fp_device_status.restype = ctypes.c_int
    L.fp_device_status.argtypes = [vp, vp]
    L.fp_read_select_stats.restype = ctypes.c_int
    L.fp_read_select_stats.argtypes = [vp, ctypes.POINTER(fp_select_stats), vp]
    L.fp_attention_trace.restype = ctypes.c_int
    L.fp_attention_trace.argtypes = [P, vp, vp, vp, vp, vp, i64, vp, vp, i32, vp, vp, vp, sz, vp, vp, i64]
    L.fp_status_string.restype = ctypes.c_char_p
    L.fp_status_string.argtypes = [ctypes.c_int]
    return L


lib = _load()


class Problem:
    """fp_problem plus the host copies of cu_seqlens and seqlens_kv it points to (kept alive here).

    seqlens_kv / host_seqlens_kv (optional, both or neither) give each request's KV length L^kv >= L^q:
    the request's new tokens are then the last L^q of L^kv positions (chunked prefill after a cached prefix).
    """

    def __init__(self, cu_seqlens: torch.Tensor, host_cu_seqlens, page_table: torch.Tensor, num_q_heads: int,
                 num_kv_heads: int, num_pages: int, page_size: int = 64, dtype: str = "bf16", c_q: float = 1.0,
                 c_k: float = 1.0, c_v: float = 1.0, head_dim: int = 128, block_size: int = 128,
                 seqlens_kv: Optional[torch.Tensor] = None, host_seqlens_kv=None):
        self.host_cu = np.ascontiguousarray(np.asarray(host_cu_seqlens, dtype=np.int32))
        self.host_kv = None if host_seqlens_kv is None else np.ascontiguousarray(
            np.asarray(host_seqlens_kv, dtype=np.int32))
        self.cu_seqlens = cu_seqlens
        self.seqlens_kv = seqlens_kv
        self.page_table = page_table
        s = fp_problem()
        s.batch = len(self.host_cu) - 1
        s.num_q_heads, s.num_kv_heads = num_q_heads, num_kv_heads
        s.head_dim, s.block_size, s.page_size = head_dim, block_size, page_size
        s.dtype = FP_DTYPE_BF16 if dtype == "bf16" else FP_DTYPE_E4M3
        s.c_q, s.c_k, s.c_v = c_q, c_k, c_v
        s.cu_seqlens = cu_seqlens.data_ptr() if cu_seqlens is not None and cu_seqlens.numel() else None
        s.page_table = page_table.data_ptr() if page_table is not None and page_table.numel() else None
        s.page_table_stride = int(page_table.shape[-1]) if page_table is not None and page_table.dim() == 2 else 0
        s.num_pages = num_pages
        s.host_cu_seqlens = self.host_cu.ctypes.data
        s.seqlens_kv = seqlens_kv.data_ptr() if seqlens_kv is not None and seqlens_kv.numel() else None
        s.host_seqlens_kv = self.host_kv.ctypes.data if self.host_kv is not None and self.host_kv.size else None
        self.c = s
        self.dtype = dtype

    @classmethod
    def from_workload(cls, w) -> "Problem":
        return cls(w.cu_seqlens, w.host_cu_seqlens, w.page_table, w.hq, w.hkv, w.num_pages,
                   page_size=int(w.k_pages.shape[1]), dtype=w.dtype, c_q=w.c_q, c_k=w.c_k, c_v=w.c_v,
                   seqlens_kv=getattr(w, "seqlens_kv", None), host_seqlens_kv=getattr(w, "host_seqlens_kv", None))

    @property
    def ref(self):
        return ctypes.byref(self.c)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, where: str):
    if code != FP_OK:
        raise FpError(code, where)


def fp_workspace_bytes(p: Problem) -> int:
    n = lib.fp_workspace_bytes(p.ref)
    _check(0 if n >= 0 else n, "fp_workspace_bytes")
    return n


def fp_num_segments(p: Problem) -> int:
    n = lib.fp_num_segments(p.ref)
    _check(0 if n >= 0 else n, "fp_num_segments")
    return n


def fp_num_blocks(p: Problem) -> int:
    n = lib.fp_num_blocks(p.ref)
    _check(0 if n >= 0 else n, "fp_num_blocks")
    return n


def fp_csr_capacity(p: Problem) -> int:
    n = lib.fp_csr_capacity(p.ref)
    _check(0 if n >= 0 else n, "fp_csr_capacity")
    return n


def fp_select(p: Problem, q, k_pages, v_pages, alpha: float, sink_blocks: int, window_blocks: int, csr_cu, csr_idx,
              kbar, vbar, kbar_op, vbar_op, workspace, stream=None, check: bool = True) -> int:
    code = lib.fp_select(p.ref, _p(q), _p(k_pages), _p(v_pages), float(alpha), int(sink_blocks), int(window_blocks),
                         _p(csr_cu), _p(csr_idx), int(csr_idx.numel()) if csr_idx is not None else 0, _p(kbar),
                         _p(vbar), _p(kbar_op), _p(vbar_op), _p(workspace),
                         int(workspace.numel() * workspace.element_size()), _stream(stream))
    if check:
        _check(code, "fp_select")
    return code


def fp_select_chunk(p: Problem, q, k_pages, v_pages, alpha: float, sink_blocks: int, window_blocks: int, csr_cu,
                    csr_idx, kbar, vbar, kbar_op, vbar_op, workspace, stream=None, check: bool = True) -> int:
    """fp_select for a chunk after a cached prefix whose block means are already in kbar/vbar/kbar_op/vbar_op."""
    code = lib.fp_select_chunk(p.ref, _p(q), _p(k_pages), _p(v_pages), float(alpha), int(sink_blocks),
                               int(window_blocks), _p(csr_cu), _p(csr_idx),
                               int(csr_idx.numel()) if csr_idx is not None else 0, _p(kbar), _p(vbar), _p(kbar_op),
                               _p(vbar_op), _p(workspace), int(workspace.numel() * workspace.element_size()),
                               _stream(stream))
    if check:
        _check(code, "fp_select_chunk")
    return code


def fp_attention(p: Problem, q, k_pages, v_pages, csr_cu, csr_idx, kbar_op, vbar_op, flags: int, out, lse,
                 workspace, stream=None, check: bool = True) -> int:
    code = lib.fp_attention(p.ref, _p(q), _p(k_pages), _p(v_pages), _p(csr_cu), _p(csr_idx),
                            int(csr_idx.numel()) if csr_idx is not None else 0, _p(kbar_op), _p(vbar_op),
                            int(flags), _p(out), _p(lse), _p(workspace),
                            int(workspace.numel() * workspace.element_size()), _stream(stream))
    if check:
        _check(code, "fp_attention")
    return code


def fp_attention_trace(p: Problem, q, k_pages, v_pages, csr_cu, csr_idx, kbar_op, vbar_op, flags: int, out, lse,
                       workspace, trace, stream=None, check: bool = True) -> int:
    """fp_attention that also records its integer work (work list, visit sequences, correction masks) in
    `trace`, a device int32 tensor (format in include/fp.h)."""
    code = lib.fp_attention_trace(p.ref, _p(q), _p(k_pages), _p(v_pages), _p(csr_cu), _p(csr_idx),
                                  int(csr_idx.numel()) if csr_idx is not None else 0, _p(kbar_op), _p(vbar_op),
                                  int(flags), _p(out), _p(lse), _p(workspace),
                                  int(workspace.numel() * workspace.element_size()), _stream(stream), _p(trace),
                                  int(trace.numel()) if trace is not None else 0)
    if check:
        _check(code, "fp_attention_trace")
    return code


def fp_select_noalloc(p: Problem, q, k_pages, v_pages, alpha: float, sink_blocks: int, window_blocks: int, csr_cu,
                      csr_idx, kbar, vbar, kbar_op, vbar_op, device_status=None, stream=None,
                      check: bool = True) -> int:
    """fp_select using the library's static scratch: for callers that cannot allocate a workspace."""
    code = lib.fp_select_noalloc(p.ref, _p(q), _p(k_pages), _p(v_pages), float(alpha), int(sink_blocks),
                                 int(window_blocks), _p(csr_cu), _p(csr_idx),
                                 int(csr_idx.numel()) if csr_idx is not None else 0, _p(kbar), _p(vbar),
                                 _p(kbar_op), _p(vbar_op), _p(device_status), _stream(stream))
    if check:
        _check(code, "fp_select_noalloc")
    return code


def fp_csr_expand64(p: Problem, csr_cu, csr_idx, tile_cu, tile_idx, workspace, stream=None,
                    check: bool = True) -> int:
    """fp_select's CSR over 128-token blocks -> the same CSR over 64-token KV tiles."""
    code = lib.fp_csr_expand64(p.ref, _p(csr_cu), _p(csr_idx), _p(tile_cu), _p(tile_idx),
                               int(tile_idx.numel()) if tile_idx is not None else 0, _p(workspace),
                               int(workspace.numel() * workspace.element_size()), _stream(stream))
    if check:
        _check(code, "fp_csr_expand64")
    return code


def fp_device_status(workspace, stream=None) -> int:
    return lib.fp_device_status(_p(workspace), _stream(stream))


def fp_read_select_stats(workspace, stream=None) -> dict:
    """Counters of the last fp_select on this workspace (status, tiles and blocks that took the fp32 path)."""
    st = fp_select_stats()
    _check(lib.fp_read_select_stats(_p(workspace), ctypes.byref(st), _stream(stream)), "fp_read_select_stats")
    return dict(status=st.status, exact_tiles=st.exact_tiles, exact_blocks=st.exact_blocks)


def fp_status_string(code: int) -> str:
    return lib.fp_status_string(int(code)).decode()


# ------------------------------------------------------------------ allocation helpers

class Buffers:
    """Caller-owned device buffers for one layer (the library allocates nothing)."""

    def __init__(self, p: Problem, device="cuda", capacity: Optional[int] = None):
        dev = torch.device(device)
        nseg, nblk = fp_num_segments(p), fp_num_blocks(p)
        hkv = p.c.num_kv_heads
        cap = fp_csr_capacity(p) if capacity is None else capacity
        T = int(p.host_cu[-1])
        op_dtype = torch.bfloat16 if p.dtype == "bf16" else torch.float8_e4m3fn
        self.workspace = torch.empty(max(fp_workspace_bytes(p), 256), dtype=torch.uint8, device=dev)
        self.csr_cu = torch.empty(nseg + 1, dtype=torch.int32, device=dev)
        self.csr_idx = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        self.kbar = torch.empty(max(nblk, 1), hkv, 128, dtype=torch.float32, device=dev)
        self.vbar = torch.empty_like(self.kbar)
        self.kbar_op = torch.empty(max(nblk, 1), hkv, 128, dtype=op_dtype, device=dev)
        self.vbar_op = torch.empty_like(self.kbar_op)
        self.out = torch.empty(T, p.c.num_q_heads, 128, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(T, p.c.num_q_heads, dtype=torch.float32, device=dev)


def run_layer(p: Problem, q, k_pages, v_pages, alpha: float, sink_blocks: int, window_blocks: int, bufs: Buffers,
              flags: int = FP_MEAN_CORRECTION, with_lse: bool = True, stream=None):
    """fp_select followed by fp_attention on one stream."""
    fp_select(p, q, k_pages, v_pages, alpha, sink_blocks, window_blocks, bufs.csr_cu, bufs.csr_idx, bufs.kbar,
              bufs.vbar, bufs.kbar_op, bufs.vbar_op, bufs.workspace, stream)
    fp_attention(p, q, k_pages, v_pages, bufs.csr_cu, bufs.csr_idx, bufs.kbar_op, bufs.vbar_op, flags, bufs.out,
                 bufs.lse if with_lse else None, bufs.workspace, stream)
    return bufs
