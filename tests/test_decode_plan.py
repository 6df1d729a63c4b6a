"""The tensor-core decode's even division of the keys, checked on the CPU.

The plan kernel lays the 64-key blocks of every (sequence b, kv head) pair
end to end, b-major, and gives CTA c the blocks [c W, (c + 1) W), with

    W = max(ceil(total / grid), 8, ceil(m / (max_splits - 1)))

(m: the most blocks of one pair; max_splits: the partial slots the host
reserves per (sequence, head), ceil(max_seqlen / 512) + 1).  A pair starting
at block `start` with nb blocks has floor((start + nb - 1) / W) -
floor(start / W) + 1 segments, and segment s of it (CTA first + s) writes
slot s.  These tests restate that arithmetic and check, block by block,
that every block falls to exactly one CTA of the grid and that no pair ever
needs more slots than the workspace holds, for random and adversarial
length mixes.  The kernel itself is tested on the GPU
(tests/test_gpu_paged.py, tests/test_gpu_onehot_gather.py).
"""

import numpy as np
import pytest

BLOCK = 64
MIN_BLOCKS = 8


def host_max_splits(max_seqlen):
    return max(1, -(-max_seqlen // 512)) + 1


def host_grid(B, Hkv, max_seqlen, sms=152):
    blocks = B * Hkv * -(-max_seqlen // BLOCK)
    want = -(-blocks // MIN_BLOCKS)
    return max(1, min(want, 2 * sms))


def plan(seqlens, Hkv, grid, max_splits):
    nbs = [-(-L // BLOCK) for L in seqlens]
    total = Hkv * sum(nbs)
    m = max(nbs) if nbs else 0
    W = max(-(-total // grid), MIN_BLOCKS, -(-m // (max_splits - 1)))
    pairs = []  # (b, hk, start, nb, segments)
    run = 0
    for b, nb in enumerate(nbs):
        for hk in range(Hkv):
            start = run + hk * nb
            segs = 0 if nb == 0 else (start + nb - 1) // W - start // W + 1
            pairs.append((b, hk, start, nb, segs))
        run += Hkv * nb
    return W, total, pairs


def check(seqlens, Hkv, max_seqlen):
    grid = host_grid(len(seqlens), Hkv, max_seqlen)
    ms = host_max_splits(max_seqlen)
    W, total, pairs = plan(seqlens, Hkv, grid, ms)
    owner = np.full(total, -1, dtype=np.int64)
    for c in range(grid):
        lo, hi = c * W, min((c + 1) * W, total)
        if lo < hi:
            assert (owner[lo:hi] == -1).all(), "a block falls to two CTAs"
            owner[lo:hi] = c
    assert (owner >= 0).all(), "a block falls to no CTA of the grid"
    for b, hk, start, nb, segs in pairs:
        assert segs <= ms, (b, hk, nb, segs, ms)
        if nb:
            first = start // W
            cts = set(owner[start:start + nb].tolist())
            assert cts == set(range(first, first + segs)), "segments are the pair's CTAs, in order"


@pytest.mark.parametrize("seed", range(30))
def test_random_batches(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 300))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    max_seqlen = int(rng.integers(1, 20000))
    seqlens = rng.integers(0, max_seqlen + 1, size=B).tolist()
    check(seqlens, Hkv, max_seqlen)


@pytest.mark.parametrize("seqlens,Hkv,max_seqlen", [
    ([16384], 1, 16384),                    # one long pair: the slot bound sets W
    ([16384] + [1] * 500, 2, 16384),        # one long sequence among many tiny ones
    ([1] * 2500, 1, 1),                     # every pair one block
    ([0, 0, 5, 0], 2, 64),                  # empty sequences
    ([65, 64, 63, 129], 8, 129),            # block edges
    ([512, 513, 1024, 1025], 1, 1025),      # split-size edges of max_splits
    ([541_000 // 64 * 64], 2, 541_000),     # far past the grid's blocks
])
def test_edge_batches(seqlens, Hkv, max_seqlen):
    check(seqlens, Hkv, max_seqlen)


def test_benchmark_decode_batch():
    """The decode benchmark's lengths (64 sequences, U[512, 16384]) over 2
    kv heads: 304 CTAs of about 56 blocks each."""
    from exact_tiled_attention_fwd_gb300 import workloads as W_
    lens = W_.c5_lengths()
    check(lens, 2, max(lens))
    grid = host_grid(len(lens), 2, max(lens))
    W, total, _ = plan(lens, 2, grid, host_max_splits(max(lens)))
    assert grid == 304 and 50 <= W <= 60
