"""The varlen prefill's grid of (sequence, block) slots, checked on the CPU.

For fewer sequences than a CTA has threads, the contiguous varlen prefill
launches num_seqs + total_q // 256 slots per head instead of
max_seqlen / 256 blocks per sequence.  Sequence s owns the slots
[B_s, B_{s+1}), B_s = s + cu_q[s] // 256, and a CTA finds the sequence of
its slot y as the number of boundaries t in 1..num_seqs with B_t <= y
(one load of cu_q per thread and a block-wide count).  These tests restate
that mapping and check, by brute force over every slot, that for valid
offsets each Q block of each sequence gets exactly one slot and that the
launch holds no more slots than stated.  The kernel's own use of it is
tested on the GPU (tests/test_gpu_varlen.py).
"""

import numpy as np
import pytest

BLOCK_ROWS = 256  # two 128-row Q tiles per CTA


def slot_owner(cu_q, y):
    """(sequence, rank within its slots) of slot y, as a CTA computes it."""
    n = len(cu_q) - 1
    seq = sum(1 for t in range(1, n + 1) if t + cu_q[t] // BLOCK_ROWS <= y)
    if seq >= n:
        return None
    return seq, y - (seq + cu_q[seq] // BLOCK_ROWS)


def assignment(lengths):
    cu_q = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64).tolist()
    total = cu_q[-1]
    n_slots = len(lengths) + total // BLOCK_ROWS
    got = {}
    for y in range(n_slots):
        owner = slot_owner(cu_q, y)
        if owner is None:
            continue
        seq, rank = owner
        n_blocks = -(-lengths[seq] // BLOCK_ROWS)
        assert rank >= 0
        if rank < n_blocks:
            assert (seq, rank) not in got, "a block owns two slots"
            got[(seq, rank)] = y
    return got, n_slots


@pytest.mark.parametrize("seed", range(20))
def test_every_block_gets_one_slot(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    lengths = rng.integers(0, 5000, size=n).tolist()
    got, n_slots = assignment(lengths)
    want = {(s, r) for s, L in enumerate(lengths) for r in range(-(-L // BLOCK_ROWS))}
    assert set(got) == want
    assert n_slots == n + sum(lengths) // BLOCK_ROWS


@pytest.mark.parametrize("lengths", [
    [1], [255], [256], [257], [512], [0, 0, 0], [0, 300, 0], [256] * 7, [255, 1, 256, 257, 511, 513],
    [4096] * 16, [128, 4096], [1] * 383,
])
def test_edge_lengths(lengths):
    got, _ = assignment(lengths)
    want = {(s, r) for s, L in enumerate(lengths) for r in range(-(-L // BLOCK_ROWS))}
    assert set(got) == want


def test_slots_come_sequence_by_sequence():
    """Slots keep the sequences in order (the dispatch order the kernel's
    heaviest-first ordering within a sequence relies on)."""
    lengths = [700, 10, 3000, 256, 1]
    got, _ = assignment(lengths)
    by_slot = sorted((y, s) for (s, _), y in got.items())
    seqs = [s for _, s in by_slot]
    assert seqs == sorted(seqs)


def test_fewer_slots_than_the_old_grid_for_the_varlen_workload():
    """16 sequences of lengths U[128, 4096] (the varlen benchmark's recipe):
    the slot grid launches about half the CTAs of max_seqlen / 256 blocks
    per sequence."""
    from exact_tiled_attention_fwd_gb300 import workloads as W
    lengths = W.c4_lengths()
    _, n_slots = assignment(lengths)
    old = len(lengths) * -(-max(lengths) // BLOCK_ROWS)
    assert n_slots <= 0.6 * old
