"""Plain enumeration of varlen chunk bookkeeping.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition (MindSpeed-Ops chunk_kda_bwd.md, input table: ``cu_seqlens`` [N+1] cumulative lengths and
``chunk_indices`` [NT, 2], NT = ceil(T / chunk_size)): the packed token axis holds N sequences, sequence
s covering tokens [cu[s], cu[s+1]).  Each sequence is cut into ceil(L_s / BT) chunks that never cross
its boundaries.  The chunks are listed sequence-major, chunk number ascending:
    chunk_indices[n] = (s, c)            the n-th chunk is chunk c of sequence s
    chunk_offsets[s] = number of chunks of all sequences before s   (chunk_offsets[N] = total)
"""
from __future__ import annotations


def enumerate_chunks(cu_seqlens, BT):
    """Return (chunk_indices as a list of (s, c) pairs, chunk_offsets as a list of N+1 ints)."""
    cu = [int(x) for x in cu_seqlens]
    indices = []
    offsets = [0]
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        n = (L + BT - 1) // BT
        for c in range(n):
            indices.append((s, c))
        offsets.append(offsets[-1] + n)
    return indices, offsets
