"""fa_paged_fwd_noalloc: paged decode that allocates nothing.

Some callers cannot hand this library a device workspace at the moment they
run attention: an engine that reserves all device memory at start-up and
gives none out later, a plugin that lives inside another runtime's memory
pool, or a decode loop that must never call cudaMalloc because an allocation
can stall the whole device.  fa_paged_fwd_noalloc keeps its split partials in
a fixed array inside the library instead.

These tests call it through the C-ABI and compare it with fa_paged_fwd (which
takes a caller workspace) and with the float64 oracle on the same inputs, for
two calls in a row with different batches, so the second call runs on
whatever the first one left in the shared array.  The capacity limit is
checked at its edge.  This file is named to be collected last.
"""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

# The fixed array holds 16 MiB; 256 bytes of it are kept back for the
# alignment of the (m, l) block, and every (sequence, head) pair needs
# (d + 2) * 4 bytes per split.  At d = 128: (16 MiB - 256) / 520 = 32,263.4.
MAX_PAIRS_D128 = 32263

pytestmark = pytest.mark.gpu


def _with_workspace(fa, pb, H, d, scale):
    B = pb.q.shape[0]
    o = torch.full_like(pb.q, float("nan"))
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = fa.fa_paged_workspace_size(B, H, d, pb.max_seqlen)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = fa.fa_paged_fwd(pb.q, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o, lse, B, H,
                         pb.k_cache.shape[2], d, 16, pb.num_pages, pb.block_table.shape[1], pb.max_seqlen,
                         scale, True, ws, ws_bytes)
    assert st == fa.FA_OK, fa.status_string(st)
    return o, lse


def _no_alloc(fa, pb, H, d, scale):
    B = pb.q.shape[0]
    o = torch.full_like(pb.q, float("nan"))
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    st = fa.fa_paged_fwd_noalloc(pb.q, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o, lse, B, H,
                                 pb.k_cache.shape[2], d, 16, pb.num_pages, pb.block_table.shape[1],
                                 pb.max_seqlen, scale, True)
    assert st == fa.FA_OK, fa.status_string(st)
    return o, lse


def _oracle_heads(pb, o, lse, heads, scale, what):
    """The float64 oracle on the given query heads of every sequence, each
    walking the real block_table over its kv head's slice of the real pool."""
    H = pb.q.shape[1]
    Hkv = pb.k_cache.shape[2]
    bt = pb.block_table.cpu().numpy()
    og, lg = f64(o), f64(lse)
    for h in heads:
        hk = h // (H // Hkv)
        O_ref, L_ref = oracle.attention_paged(f64(pb.q[:, h:h + 1]), f64(pb.k_cache[:, :, hk:hk + 1, :]),
                                              f64(pb.v_cache[:, :, hk:hk + 1, :]), bt, pb.lengths, 16, scale, True)
        assert_o_close(og[:, h:h + 1], O_ref, f"{what} h{h}")
        assert_lse_close(lg[:, h:h + 1], L_ref, f"{what} h{h}")


def test_no_alloc_matches_workspace_entry_point(fa):
    """Call 1: the full decode batch (B64 H32 d128, lengths U[512, 16384]);
    its partials need more than the fixed array at 512-token splits, so the
    call uses fewer, longer splits.  Call 2: a small ragged GQA batch that
    reuses the array.  Each is checked against fa_paged_fwd and against the
    oracle (sampled heads of the full batch, every head of the small one).
    Call 3 repeats call 1 and must match it bit for bit."""
    big = W.paged_inputs(W.c5_lengths(), 32, 128, 1239, "cuda", pool_on_device=True)
    small = W.paged_inputs([1, 17, 700, 33], 8, 64, 61, "cuda", Hkv=2, slack_pages=4)
    runs = [(big, 32, 128, (0, 17, 31)), (small, 8, 64, range(8))]
    first = None
    for i, (pb, H, d, heads) in enumerate(runs):
        scale = 1.0 / np.sqrt(d)
        o_ref, l_ref = _with_workspace(fa, pb, H, d, scale)
        o, l = _no_alloc(fa, pb, H, d, scale)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        assert_o_close(o, f64(o_ref), f"no-alloc call {i + 1}")
        assert_lse_close(l, f64(l_ref), f"no-alloc call {i + 1}")
        _oracle_heads(pb, o, l, heads, scale, f"no-alloc call {i + 1} vs oracle")
        if i == 0:
            first = (o.clone(), l.clone())
    o, l = _no_alloc(fa, big, 32, 128, 1.0 / np.sqrt(128))
    torch.cuda.synchronize()
    assert torch.equal(o, first[0]) and torch.equal(l, first[1])


def test_no_alloc_rejects_batches_beyond_the_array(fa):
    """B * H * (d + 2) * 4 bytes must fit the 16 MiB array minus 256 bytes:
    at d = 128, 32,264 (sequence, head) pairs are refused before any launch,
    however they are split between B and H."""
    A = 1 << 20  # never dereferenced: the size check comes first
    for B, H, Hkv in ((1, MAX_PAIRS_D128 + 1, 1), (1000, 33, 33), (8066, 4, 4)):
        st = fa.fa_paged_fwd_noalloc(A, A, A, A, A, A, None, B, H, Hkv, 128, 16, 10, 8, 100, 0.1, 1, 0)
        assert st == fa.FA_ERR_SCRATCH_CAPACITY, (B, H)
    assert "16 MiB" in fa.status_string(fa.FA_ERR_SCRATCH_CAPACITY)


def test_no_alloc_at_the_capacity_limit(fa):
    """Exactly 32,263 (sequence, head) pairs at d = 128 (B 419, H 77, 7 kv
    heads): the largest batch the array takes.  Short ragged lengths; the
    result matches fa_paged_fwd and the oracle on sampled heads."""
    B, H, Hkv, d = 419, 77, 7, 128
    assert B * H == MAX_PAIRS_D128
    lens = W.uniform_lengths(B, 1, 40, 62)
    pb = W.paged_inputs(lens, H, d, 62, "cuda", Hkv=Hkv, slack_pages=2)
    scale = 1.0 / np.sqrt(d)
    o_ref, l_ref = _with_workspace(fa, pb, H, d, scale)
    o, l = _no_alloc(fa, pb, H, d, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert_o_close(o, f64(o_ref), "no-alloc at the limit")
    assert_lse_close(l, f64(l_ref), "no-alloc at the limit")
    _oracle_heads(pb, o, l, (0, 40, 76), scale, "no-alloc at the limit vs oracle")
