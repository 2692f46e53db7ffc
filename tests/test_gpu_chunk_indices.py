"""The varlen chunk bookkeeping on the GPU (gdr_chunk_indices through the C ABI) equals the plain
enumeration of oracle/chunk_index.py bit for bit: every (sequence, chunk) pair, the (-1, -1) rows after
the total, and the per-sequence chunk offsets (MindSpeed-Ops chunk_kda_bwd.md, input table: cu_seqlens
[N+1], chunk_indices [NT, 2])."""
import json
import os

import numpy as np
import pytest
import torch

from chunked_gated_delta_09_gb300 import ops
from oracle.chunk_index import enumerate_chunks

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "chunk_indices.json")


def _check(cu, BT, slack=3):
    cu = [int(x) for x in cu]
    idx_ref, off_ref = enumerate_chunks(cu, BT)
    max_chunks = cu[-1] // BT + (len(cu) - 1) + slack
    assert max_chunks >= len(idx_ref)
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    idx, off = ops.chunk_indices(cu_dev, BT, max_chunks)
    torch.cuda.synchronize()
    idx, off = idx.cpu().numpy(), off.cpu().numpy()
    want = np.full((max_chunks, 2), -1, dtype=np.int32)
    if idx_ref:
        want[:len(idx_ref)] = np.asarray(idx_ref, dtype=np.int32)
    assert idx.dtype == np.int32 and off.dtype == np.int32
    assert np.array_equal(idx, want), (cu, BT)
    assert np.array_equal(off, np.asarray(off_ref, dtype=np.int32)), (cu, BT)


def test_golden_cases_bit_exact():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        _check(c["cu_seqlens"], c["BT"])


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("BT", [16, 32, 64])
def test_random_lengths_with_empty_sequences_bit_exact(seed, BT):
    rng = np.random.default_rng(1000 * seed + BT)
    n = int(rng.integers(1, 40))
    lens = rng.integers(0, 300, size=n)
    lens[rng.random(n) < 0.3] = 0  # empty sequences
    cu = np.concatenate([[0], np.cumsum(lens)])
    _check(cu, BT)


def test_many_sequences_span_several_scan_tiles():
    """More sequences than one block of the kernel's scan (1024), lengths 0..130."""
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 131, size=2500)
    _check(np.concatenate([[0], np.cumsum(lens)]), 64)
