"""The backward's per-row workspace layout, checked on the CPU.

bwd_prep_kernel writes lse2 and delta for every row of a sequence's
128-row query blocks (rows past the sequence padded: lse2 = +inf,
delta = 0), sequence s starting at row offset

    off(s) = ((cu_q[s] + 3) & ~3) + 132 s

of each head's stripe, whose length (the head stride) is

    stride = (total_q + 132 num_seqs + 8 + 3) & ~3

floats; the dK/dV kernel bulk-copies 128 of those rows at a time and the
dQ kernel reads one per thread.  These tests restate the layout and check,
for random and edge-case length mixes, that every sequence's padded rows
start on a 16-byte boundary, never reach into the next sequence's rows,
and stay inside the stripe; and that the library's fa_bwd_workspace_bytes
is the two stripes (lse2, delta) of every head.
"""

import numpy as np
import pytest

BLOCK = 128


def seq_offset(q_start, s):
    return ((q_start + 3) & ~3) + 132 * s


def head_stride(total_q, num_seqs):
    return (total_q + 132 * num_seqs + 8 + 3) & ~3


def check_layout(lengths):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    n, total = len(lengths), int(cu[-1])
    stride = head_stride(total, n)
    prev_end = 0
    for s, L in enumerate(lengths):
        off = seq_offset(int(cu[s]), s)
        assert off % 4 == 0, "16-byte aligned (the bulk copies need it)"
        assert off >= prev_end, "overlaps the previous sequence's padded rows"
        end = off + -(-L // BLOCK) * BLOCK
        assert end <= stride, "past the head's stripe"
        prev_end = end
    return stride


@pytest.mark.parametrize("seed", range(30))
def test_random_mixes(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 200))
    check_layout(rng.integers(0, 3000, size=n).tolist())


@pytest.mark.parametrize("lengths", [
    [1], [128], [129], [0], [0, 0, 1], [1] * 500, [127, 1, 129, 255, 257], [3, 5, 7, 9, 11], [8192],
])
def test_edge_mixes(lengths):
    check_layout(lengths)


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_fwd_gb300 import _build
    import exact_tiled_attention_fwd_gb300 as F

    _build.build()
    F.load()
    return F


@pytest.mark.parametrize("num_seqs,total_q,H", [(1, 8192, 32), (16, 33822, 32), (3, 310, 2), (500, 1000, 7)])
def test_library_workspace_size(lib, num_seqs, total_q, H):
    assert lib.fa_bwd_workspace_bytes(num_seqs, total_q, H) == 2 * H * head_stride(total_q, num_seqs) * 4
