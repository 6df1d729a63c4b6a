"""fa_paged_fwd_noalloc: paged decode that allocates nothing.

Some callers cannot hand this library a device workspace at the moment they
run attention: an engine that reserves all device memory at start-up and
gives none out later, a plugin that lives inside another runtime's memory
pool, or a decode loop that must never call cudaMalloc because an allocation
can stall the whole device.  fa_paged_fwd_noalloc keeps its split partials in
a fixed array inside the library instead.

These tests call it through the C-ABI and compare it with fa_paged_fwd (which
takes a caller workspace) on the same inputs, for two calls in a row with
different batches, so the second call runs on whatever the first one left in
the shared array.  This file is named to be collected last.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

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


def test_no_alloc_matches_workspace_entry_point(fa):
    """Call 1: the full decode batch (B64 H32 d128, lengths U[512, 16384]);
    its partials need more than the fixed array at 512-token splits, so the
    call uses fewer, longer splits.  Call 2: a small ragged GQA batch that
    reuses the array.  Call 3 repeats call 1 and must match it bit for bit."""
    big = W.paged_inputs(W.c5_lengths(), 32, 128, 1239, "cuda", pool_on_device=True)
    small = W.paged_inputs([1, 17, 700, 33], 8, 64, 61, "cuda", Hkv=2, slack_pages=4)
    runs = [(big, 32, 128), (small, 8, 64)]
    first = None
    for i, (pb, H, d) in enumerate(runs):
        scale = 1.0 / np.sqrt(d)
        o_ref, l_ref = _with_workspace(fa, pb, H, d, scale)
        o, l = _no_alloc(fa, pb, H, d, scale)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        assert_o_close(o, f64(o_ref), f"no-alloc call {i + 1}")
        assert_lse_close(l, f64(l_ref), f"no-alloc call {i + 1}")
        if i == 0:
            first = (o.clone(), l.clone())
    o, l = _no_alloc(fa, big, 32, 128, 1.0 / np.sqrt(128))
    torch.cuda.synchronize()
    assert torch.equal(o, first[0]) and torch.equal(l, first[1])


def test_no_alloc_rejects_batches_beyond_the_array(fa):
    """B * H * (d + 2) * 4 bytes must fit the 16 MiB array; one more (sequence,
    head) pair past that is refused before any launch."""
    A = 1 << 20  # never dereferenced: the size check comes first
    st = fa.fa_paged_fwd_noalloc(A, A, A, A, A, A, None, 1000, 33, 33, 128, 16, 10, 8, 100, 0.1, 1, 0)
    assert st == fa.FA_ERR_SCRATCH_CAPACITY
    assert "16 MiB" in fa.status_string(st)
