"""Paged decode (fa_paged_fwd) and the page gather against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


def run_paged(fa, pb, H, d, scale, causal=True):
    B = pb.q.shape[0]
    Hkv = pb.k_cache.shape[2]
    ps = pb.k_cache.shape[1]
    o = torch.full_like(pb.q, float("nan"))
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=pb.q.device)
    ws_bytes = fa.fa_paged_workspace_size(B, H, d, pb.max_seqlen)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=pb.q.device)
    st = fa.fa_paged_fwd(pb.q, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o, lse, B, H, Hkv, d, ps,
                         pb.num_pages, pb.block_table.shape[1], pb.max_seqlen, scale, causal, ws, ws_bytes)
    assert st == fa.FA_OK, fa.status_string(st)
    return o, lse


def check_full(fa, lengths, H, d, seed, Hkv=None, slack=3, page_size=16):
    pb = W.paged_inputs(lengths, H, d, seed, "cuda", Hkv=Hkv, slack_pages=slack, page_size=page_size)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_paged(fa, pb, H, d, scale)
    assert fa.fa_device_status() == fa.FA_OK
    O_ref, L_ref = oracle.attention_paged(f64(pb.q), f64(pb.k_cache), f64(pb.v_cache), pb.block_table.cpu().numpy(),
                                          lengths, page_size, scale, True)
    assert_o_close(o, O_ref, f"paged {lengths} page {page_size}")
    assert_lse_close(lse, L_ref, f"paged {lengths} page {page_size}")


@pytest.mark.parametrize("page_size", [32, 64, 128])
@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 128), (8, 2, 64), (32, 2, 128), (32, 4, 64)])
def test_page_sizes(fa, page_size, H, Hkv, d):
    """Pages of 32, 64 and 128 tokens: lengths below, at and just past a
    page, and across the 512- and 2048-token splits, on the CUDA-core split
    kernel (groups of 1 and 4) and the tensor-core decode (groups of 16 and
    8)."""
    lens = [1, page_size - 1, page_size, page_size + 1, 513, 2 * page_size + 7, 2049, 4500, 0]
    check_full(fa, lens, H, d, seed=40 + page_size + H + Hkv + d, Hkv=Hkv, page_size=page_size)


@pytest.mark.parametrize("d", [64, 128])
def test_short_and_ragged(fa, d):
    """seqlen below one page, exactly one page, one past, not a multiple of
    16, and a length spanning several splits."""
    check_full(fa, [1, 15, 16, 17, 100, 513, 1300, 2049], 4, d, seed=20 + d)


def test_empty_sequence(fa):
    """seqlen 0: O = 0 and LSE = -inf (no key is visible)."""
    check_full(fa, [0, 5, 0, 40], 2, 128, seed=21)


@pytest.mark.parametrize("H,Hkv,d", [(8, 2, 128), (8, 4, 128), (32, 2, 128), (16, 2, 64), (32, 2, 64),
                                     (6, 2, 64), (4, 4, 64), (12, 3, 128)])
def test_gqa_decode(fa, H, Hkv, d):
    """Query heads grouped over kv heads: the decode warps take 1, 2, 4 or 8
    heads of one group (groups of 2, 3, 4, 8, 16) and read each K/V row once
    for all of them."""
    check_full(fa, [700, 33, 1, 1500], H, d, seed=22 + H + Hkv, Hkv=Hkv)


@pytest.mark.parametrize("H,Hkv,d", [(32, 4, 128), (32, 2, 64), (32, 1, 128), (128, 1, 64), (160, 1, 128),
                                     (24, 2, 128), (48, 2, 64), (48, 1, 128), (64, 1, 128), (64, 1, 64),
                                     (256, 1, 64), (320, 1, 64)])
def test_tensor_core_decode(fa, H, Hkv, d):
    """Groups of 8 to 64 query heads decode on the tensor cores (the
    group's heads are the first rows of a Q tile; groups of 12, 24 and 48
    leave it part-used), in 2048-key splits merged by the combine step:
    empty, one-token, page-edge and multi-split lengths.  Groups of 128,
    160, 256 and 320 take the CUDA-core split kernel."""
    check_full(fa, [0, 1, 15, 16, 17, 700, 2048, 2049, 4500], H, d, seed=30 + H + Hkv + d, Hkv=Hkv)


def test_c5_sampled_heads(fa):
    """The full decode batch (B64, H32, d128, lengths U[512, 16384], random
    page permutation): every sequence, three sampled heads, each checked by
    the oracle walking the real block_table over that head's slice of the
    real pool."""
    lens = W.c5_lengths()
    H, d = 32, 128
    pb = W.paged_inputs(lens, H, d, 1239, "cuda", pool_on_device=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_paged(fa, pb, H, d, scale)
    assert fa.fa_device_status() == fa.FA_OK
    og, lg = f64(o), f64(lse)
    bt = pb.block_table.cpu().numpy()
    for h in (0, 13, 31):
        kp = f64(pb.k_cache[:, :, h:h + 1, :])
        vp = f64(pb.v_cache[:, :, h:h + 1, :])
        O_ref, L_ref = oracle.attention_paged(f64(pb.q[:, h:h + 1]), kp, vp, bt, lens, 16, scale, True)
        assert_o_close(og[:, h:h + 1], O_ref, f"C5 h{h}")
        assert_lse_close(lg[:, h:h + 1], L_ref, f"C5 h{h}")


@pytest.mark.parametrize("Hkv", [8, 2])
def test_c5_grouped_sampled_heads(fa, Hkv):
    """The full decode batch over 8 kv heads (4 query heads each, the
    CUDA-core grouped warps) and over 2 kv heads (16 each, the tensor-core
    path), as bench.py times them: every sequence, sampled query heads of
    several kv groups, checked by the oracle walking the real table over that
    kv head's slice of the real pool."""
    lens = W.c5_lengths()
    H, d = 32, 128
    pb = W.paged_inputs(lens, H, d, 1239 + Hkv, "cuda", Hkv=Hkv, pool_on_device=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_paged(fa, pb, H, d, scale)
    assert fa.fa_device_status() == fa.FA_OK
    og, lg = f64(o), f64(lse)
    bt = pb.block_table.cpu().numpy()
    for h in (0, 9, 16, 31):
        hk = h // (H // Hkv)
        kp = f64(pb.k_cache[:, :, hk:hk + 1, :])
        vp = f64(pb.v_cache[:, :, hk:hk + 1, :])
        O_ref, L_ref = oracle.attention_paged(f64(pb.q[:, h:h + 1]), kp, vp, bt, lens, 16, scale, True)
        assert_o_close(og[:, h:h + 1], O_ref, f"C5 Hkv{Hkv} h{h}")
        assert_lse_close(lg[:, h:h + 1], L_ref, f"C5 Hkv{Hkv} h{h}")


@pytest.mark.parametrize("page_size", [16, 64])
def test_gather_bit_exact(fa, page_size):
    """fa_paged_gather (a copy kernel sharing the decode kernel's chunk
    lookup) reads exactly the bytes the host walk of block_table selects."""
    lens = [1, 16, 17, 250, 999, 2048]
    pb = W.paged_inputs(lens, 4, 128, 23, "cuda", slack_pages=5, page_size=page_size)
    for cache in (pb.k_cache, pb.v_cache):
        out = torch.zeros((len(lens), pb.max_seqlen, 4, 128), dtype=torch.bfloat16, device="cuda")
        st = fa.fa_paged_gather(cache, pb.block_table, pb.seqlens, out, len(lens), 4, 128, page_size, pb.num_pages,
                                pb.block_table.shape[1], pb.max_seqlen)
        assert st == fa.FA_OK
        assert fa.fa_device_status() == fa.FA_OK
        host = cache.cpu().view(torch.int16).numpy()
        got = out.cpu().view(torch.int16).numpy()
        bt = pb.block_table.cpu().numpy()
        for b, L in enumerate(lens):
            ref = oracle.gather_paged_kv(host, bt[b], L, page_size)
            assert np.array_equal(got[b, :L], ref), f"seq {b}"


@pytest.mark.parametrize("H,Hkv", [(2, 2), (16, 2)])
def test_bad_block_table_entry(fa, H, Hkv):
    """An entry outside the pool (or negative) is skipped and reported; the
    other sequences are unaffected.  16 query heads per kv head take the
    tensor-core decode."""
    lens = [40, 40, 2100]
    pb = W.paged_inputs(lens, H, 64, 24, "cuda", Hkv=Hkv)
    bt = pb.block_table.clone()
    bt[1, 1] = pb.num_pages + 100
    bt[2, 130] = -7  # in the second 2048-key split
    pb2 = W.PagedBatch(pb.q, pb.k_cache, pb.v_cache, bt, pb.seqlens, pb.lengths, pb.max_seqlen, pb.num_pages)
    o, lse = run_paged(fa, pb2, H, 64, 0.125)
    assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX
    O_ref, L_ref = oracle.attention_paged(f64(pb.q), f64(pb.k_cache), f64(pb.v_cache), pb.block_table.cpu().numpy(),
                                          lens, 16, 0.125, True)
    assert_o_close(o[0:1], O_ref[0:1], "good sequence")
    assert_lse_close(lse[0:1], L_ref[0:1], "good sequence")
    assert np.all(np.isfinite(f64(o[1:])))


def test_seqlen_beyond_max_reported(fa):
    """A seqlens entry above max_seqlen is clamped to max_seqlen and reported,
    on the CUDA-core path and on the tensor-core path."""
    for H, Hkv in ((4, 4), (16, 2)):
        lens = [100, 300]
        pb = W.paged_inputs(lens, H, 64, 26, "cuda", Hkv=Hkv, slack_pages=4)
        bad = pb.seqlens.clone()
        bad[0] = pb.max_seqlen + 50
        pb2 = W.PagedBatch(pb.q, pb.k_cache, pb.v_cache, pb.block_table, bad, pb.lengths, pb.max_seqlen, pb.num_pages)
        o, lse = run_paged(fa, pb2, H, 64, 0.125)
        assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX
        O_ref, L_ref = oracle.attention_paged(f64(pb.q), f64(pb.k_cache), f64(pb.v_cache),
                                              pb.block_table.cpu().numpy(), lens, 16, 0.125, True)
        assert_o_close(o[1:2], O_ref[1:2], f"H{H}/{Hkv} good sequence")
        assert np.all(np.isfinite(f64(o)))


def test_deterministic(fa):
    pb = W.paged_inputs([3000, 17], 4, 128, 25, "cuda")
    o1, l1 = run_paged(fa, pb, 4, 128, 0.088)
    o2, l2 = run_paged(fa, pb, 4, 128, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,page_size", [(128, 16), (64, 32), (128, 128)])
def test_tensor_core_decode_many_items(fa, d, page_size):
    """The tensor-core decode's CTAs (two per SM) each take many
    (split, sequence, kv head) items from a counter: 420 sequences, most of
    them one or two 64-key blocks with a partly used last page, empty ones
    between them, and a few long enough for several splits, so items of every
    size follow each other within a CTA.  Checked element by element against
    the oracle; a second call on the same inputs gives the same bits, so the
    counter starts from zero on every call."""
    rng = np.random.default_rng(71 + d + page_size)
    lens = [int(x) for x in rng.integers(0, 140, size=420)]
    for i in range(0, 420, 37):
        lens[i] = 0
    lens[5], lens[200], lens[399] = 4200, 2049, 6000
    H, Hkv = 32, 2
    pb = W.paged_inputs(lens, H, d, 72 + d, "cuda", Hkv=Hkv, slack_pages=2, page_size=page_size)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_paged(fa, pb, H, d, scale)
    o2, lse2 = run_paged(fa, pb, H, d, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert torch.equal(o, o2) and torch.equal(torch.nan_to_num(lse, neginf=-1e30), torch.nan_to_num(lse2, neginf=-1e30))
    O_ref, L_ref = oracle.attention_paged(f64(pb.q), f64(pb.k_cache), f64(pb.v_cache), pb.block_table.cpu().numpy(),
                                          lens, page_size, scale, True)
    assert_o_close(o, O_ref, f"many items d{d} page {page_size}")
    assert_lse_close(lse, L_ref, f"many items d{d} page {page_size}")


def test_tensor_core_decode_large_batch(fa):
    """2,500 sequences on the tensor-core decode: the plan kernel's 1024
    threads each scan a run of three sequences' lengths (a path smaller
    batches never take), with empty sequences at run boundaries and a few
    long ones among many short ones."""
    rng = np.random.default_rng(91)
    lens = [int(x) for x in rng.integers(0, 70, size=2500)]
    for i in (0, 1, 2, 3, 1023, 1024, 2047, 2048, 2499):
        lens[i] = 0
    lens[7], lens[1500], lens[2498] = 3000, 1100, 2049
    check_full(fa, lens, 16, 128, seed=92, Hkv=1, slack=2, page_size=16)
