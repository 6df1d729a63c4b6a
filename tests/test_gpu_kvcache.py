"""store_kvcache and the paged varlen prefill (a chunk that continues a cached
prefix) against the float64 oracle, through the C-ABI."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu

PAGE = 16


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


# ----------------------------------------------------------------- store_kvcache


@pytest.mark.parametrize("d,Hkv,T", [(128, 8, 300), (64, 2, 1), (128, 1, 4096)])
def test_store_kvcache_bit_exact(fa, d, Hkv, T):
    num_pages = (T + PAGE - 1) // PAGE + 3
    g = torch.Generator().manual_seed(T + d)
    kc = W.randn_bf16((num_pages, PAGE, Hkv, d), 501).cuda()
    vc = W.randn_bf16((num_pages, PAGE, Hkv, d), 502).cuda()
    k = W.randn_bf16((T, Hkv, d), 503).cuda()
    v = W.randn_bf16((T, Hkv, d), 504).cuda()
    slots = torch.randperm(num_pages * PAGE, generator=g)[:T].to(torch.int32)
    slots[::7] = -1  # padding tokens are not stored
    kc0, vc0 = kc.cpu().view(torch.int16).numpy(), vc.cpu().view(torch.int16).numpy()
    st = fa.fa_store_kvcache(k, v, kc, vc, slots.cuda(), T, Hkv, d, PAGE, num_pages)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    ek, ev = oracle.store_kvcache(bits(k), bits(v), kc0, vc0, slots.numpy(), PAGE)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_store_kvcache_bad_slot_reported(fa):
    T, Hkv, d, num_pages = 8, 2, 64, 2
    kc = torch.zeros((num_pages, PAGE, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = W.randn_bf16((T, Hkv, d), 505).cuda()
    v = W.randn_bf16((T, Hkv, d), 506).cuda()
    slots = torch.tensor([0, 1, 2, num_pages * PAGE, 3, -1, 31, 10 ** 6], dtype=torch.int32)
    assert fa.fa_store_kvcache(k, v, kc, vc, slots.cuda(), T, Hkv, d, PAGE, num_pages) == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX
    assert fa.fa_device_status() == fa.FA_OK  # cleared
    ek, ev = oracle.store_kvcache(bits(k), bits(v), np.zeros((num_pages, PAGE, Hkv, d), np.int16),
                                  np.zeros((num_pages, PAGE, Hkv, d), np.int16),
                                  np.where((slots.numpy() >= num_pages * PAGE), -1, slots.numpy()), PAGE)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_store_kvcache_empty(fa):
    kc = torch.zeros((1, PAGE, 1, 64), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    sl = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fa.fa_store_kvcache(z, z, kc, kc, sl, 0, 1, 64, PAGE, 1) == fa.FA_OK


# ----------------------------------------------------------------- paged varlen prefill


def run_paged(fa, b, H, Hkv, d, scale, causal):
    total_q = int(b.cu_q[-1])
    ps = b.k_cache.shape[1]
    o = torch.full((total_q, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, total_q), float("nan"), dtype=torch.float32, device="cuda")
    st = fa.fa_varlen_paged_fwd(b.q, b.k_cache, b.v_cache, o, lse, b.cu_q, b.cu_k, b.block_table,
                                len(b.lengths_q), b.max_q, b.max_k, total_q, H, Hkv, d, ps, b.num_pages,
                                b.block_table.shape[1], scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    return o, lse


def check_paged(fa, lq, lk, H, Hkv, d, causal, seed, scale=None, page_size=PAGE):
    b = W.chunk_inputs(lq, lk, H, d, seed, "cuda", Hkv=Hkv, slack_pages=2, page_size=page_size)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o, lse = run_paged(fa, b, H, Hkv, d, scale, causal)
    O_ref, L_ref = oracle.attention_varlen_paged(f64(b.q), b.k_cache.float().cpu().numpy(),
                                                 b.v_cache.float().cpu().numpy(), b.cu_q.cpu().numpy(),
                                                 b.cu_k.cpu().numpy(), b.block_table.cpu().numpy(), page_size, scale,
                                                 causal)
    what = f"lq{lq} lk{lk} H{H}/{Hkv} d{d} c{causal} page {page_size}"
    assert_o_close(o, O_ref, what)
    assert_lse_close(lse, L_ref, what)


def test_bench_chunk_full_size(fa):
    """The continuation chunk bench.py times (16 sequences, cached context
    U[512, 8192] + new tokens U[256, 2048], H32 d128, causal, pool on the
    device): every query row of three sequences on two heads, against the
    oracle's attention over keys gathered by its own host page walk."""
    lq, lk = W.chunk_lengths()
    H, d = W.CHUNK["H"], W.CHUNK["d"]
    b = W.chunk_inputs(lq, lk, H, d, 1240, "cuda", stale=0.0, pool_on_device=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_paged(fa, b, H, H, d, scale, True)
    og, lg = f64(o), f64(lse)
    cu = b.cu_q.cpu().numpy()
    bt = b.block_table.cpu().numpy()
    for s in (int(np.argmax(lk)), int(np.argmin(lq)), 7):
        a = int(cu[s])
        for h in (4, 29):
            kh = b.k_cache[:, :, h:h + 1].float().cpu().numpy()
            vh = b.v_cache[:, :, h:h + 1].float().cpu().numpy()
            K = oracle.gather_paged_kv(kh, bt[s], lk[s], PAGE)[:, 0]
            Vv = oracle.gather_paged_kv(vh, bt[s], lk[s], PAGE)[:, 0]
            O_ref, L_ref = oracle.attention_rows(f64(b.q[a:a + lq[s], h]), K, Vv, scale, True,
                                                 rows=np.arange(lq[s]), Lq=lq[s])
            assert_o_close(og[a:a + lq[s], h], O_ref, f"chunk s{s} h{h}")
            assert_lse_close(lg[h, a:a + lq[s]], L_ref, f"chunk s{s} h{h}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_continuation_chunks(fa, d, causal):
    """Chunks of new tokens after cached prefixes of ragged length (the tail
    slots of every last page hold NaN, which must never reach O)."""
    lk = [300, 129, 1000, 17, 16, 700]
    lq = [40, 129, 257, 1, 16, 128]
    check_paged(fa, lq, lk, 4, 2, d, causal, seed=21 + d)


@pytest.mark.parametrize("page_size", [32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
def test_continuation_chunks_page_sizes(fa, page_size, d):
    """Pages of 32, 64 and 128 tokens (one TMA box per page and panel; at
    128 a page is a whole key block): ragged chunks, partly used last pages
    holding NaN."""
    lk = [300, 129, 1000, 17, 16, 700, 2 * page_size + 3]
    lq = [40, 129, 257, 1, 16, 128, page_size]
    check_paged(fa, lq, lk, 4, 2, d, True, seed=51 + d + page_size, page_size=page_size)
    check_paged(fa, lq, lk, 4, 4, d, False, seed=52 + d + page_size, page_size=page_size)


@pytest.mark.parametrize("d", [64, 128])
def test_first_chunk_through_pages(fa, d):
    """Lq == Lk: a first chunk whose K/V were stored in the pool first."""
    lens = [1, 15, 16, 17, 255, 256, 257, 600]
    check_paged(fa, lens, lens, 2, 2, d, True, seed=31 + d)


def test_bad_page_entry_reported(fa):
    b = W.chunk_inputs([8], [100], 2, 64, 41, "cuda", stale=0.0)
    b.block_table[0, 2] = b.num_pages + 5  # tokens 32..47 point outside the pool
    total_q = int(b.cu_q[-1])
    o = torch.empty((total_q, 2, 64), dtype=torch.bfloat16, device="cuda")
    st = fa.fa_varlen_paged_fwd(b.q, b.k_cache, b.v_cache, o, None, b.cu_q, b.cu_k, b.block_table, 1, b.max_q,
                                b.max_k, total_q, 2, 2, 64, PAGE, b.num_pages, b.block_table.shape[1], 0.125, 1)
    assert st == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX


def test_chunked_prefill_equals_full_prefill(fa):
    """The engine flow of the page's data-flow section: store each chunk's
    K/V with store_kvcache, then attend through the page table.  Two chunks of
    one sequence give the same O/LSE as one unsplit varlen prefill."""
    H, Hkv, d, L, L1 = 4, 2, 128, 700, 300
    q, k, v, cu, _ = W.varlen_inputs([L], H, d, 51, "cuda", Hkv=Hkv)
    O_full, lse_full = fa.attention_varlen(q, k, v, cu, cu, L, L, causal=True)
    num_pages = (L + PAGE - 1) // PAGE + 4
    kc = torch.full((num_pages, PAGE, Hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    pages = torch.randperm(num_pages, generator=torch.Generator().manual_seed(52))[: (L + PAGE - 1) // PAGE]
    bt = pages.to(torch.int32)[None].cuda()
    outs, lses = [], []
    for a, e in ((0, L1), (L1, L)):
        slots = torch.tensor([int(pages[t // PAGE]) * PAGE + t % PAGE for t in range(a, e)], dtype=torch.int32)
        fa.store_kvcache(k[a:e], v[a:e], kc, vc, slots.cuda())
        cq = torch.tensor([0, e - a], dtype=torch.int32, device="cuda")
        ck = torch.tensor([0, e], dtype=torch.int32, device="cuda")
        o, lse = fa.attention_varlen_paged(q[a:e], kc, vc, cq, ck, bt, e - a, e, causal=True)
        outs.append(o)
        lses.append(lse)
    assert fa.fa_device_status() == fa.FA_OK
    O_ref, L_ref = oracle.attention_varlen(f64(q), f64(k), f64(v), cu.cpu().numpy(), cu.cpu().numpy(),
                                           1.0 / np.sqrt(d), True)
    assert_o_close(torch.cat(outs), O_ref, "chunked")
    assert_lse_close(torch.cat(lses, dim=1), L_ref, "chunked")
    diff = (torch.cat(outs).float() - O_full.float()).abs().max().item()
    assert diff <= 2e-2, diff
