"""bench.py's own accounting against the oracle and the library's sizing (CPU).

The bench reports executed and dense-equivalent FLOPs from its own enumeration of segments; it must enumerate
exactly the segments the library launches and the oracle defines.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from block_sparse_long_mean_gb300 import binding as B  # noqa: E402
from block_sparse_long_mean_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("lengths,hq,hkv,kv_lengths", [
    ([2048], 4, 1, None), ([300, 0, 129, 1000], 8, 2, None), ([1], 16, 1, None),
    ([77, 200, 1, 0, 130], 8, 2, [300, 456, 129, 64, 130]), ([5], 4, 4, [1000]), ([640], 32, 4, [2000]),
])
def test_bench_segments_match_oracle_and_library(lengths, hq, hkv, kv_lengths):
    w = synth.make_workload("tiny_2k", device="cpu", lengths=lengths, hq=hq, hkv=hkv, kv_lengths=kv_lengths)
    seg = bench.segments_of(w)
    ref = oracle.segments(oracle.Problem.from_workload(w))
    np.testing.assert_array_equal(seg["D"], ref.D)
    assert len(seg["D"]) == B.fp_num_segments(B.Problem.from_workload(w))
    # every query row sits in exactly one tile per KV head
    g = hq // hkv
    assert int(seg["rows"].sum()) == hkv * g * sum(lengths)
    assert (seg["rows"] > 0).all() and (seg["rows"] <= 128).all()

