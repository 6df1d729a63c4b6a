"""Packed variable-length prefill (fa_varlen_fwd) against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


def run_varlen(fa, q, k, v, cq, ck, lq, lk, scale, causal):
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((H, total_q), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_varlen_fwd(q, k, v, o, lse, cq, ck, len(lq), max(lq), max(lk), total_q, total_k, H, Hkv, d,
                          scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    return o, lse


def check_full(fa, lq, H, d, causal, seed, lk=None, Hkv=None):
    lk = lq if lk is None else lk
    q, k, v, cq, ck = W.varlen_inputs(lq, H, d, seed, "cuda", lengths_k=lk, Hkv=Hkv)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_varlen(fa, q, k, v, cq, ck, lq, lk, scale, causal)
    O_ref, L_ref = oracle.attention_varlen(f64(q), f64(k), f64(v), cq.cpu().numpy(), ck.cpu().numpy(), scale, causal)
    assert_o_close(o, O_ref, f"varlen {lq} c{causal}")
    assert_lse_close(lse, L_ref, f"varlen {lq} c{causal}")


def test_page_example(fa):
    """Two sequences of lengths 3 and 4: cu_seqlens [0, 3, 7] (dlog.com.cn
    page §3.3)."""
    for causal in (False, True):
        check_full(fa, [3, 4], 2, 64, causal, seed=3)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_mix(fa, d, causal):
    """1-token sequences, tile-straddling sequences, exact tile multiples."""
    check_full(fa, [1, 130, 2, 64, 257, 128, 3, 1, 511], 3, d, causal, seed=11 + d)


def test_gqa_varlen(fa):
    check_full(fa, [100, 300, 5], 8, 128, True, seed=12, Hkv=2)


@pytest.mark.parametrize("causal", [False, True])
def test_q_shorter_than_k(fa, causal):
    """Prefix continuation shape: each sequence's queries are its last Lq
    tokens, keys are all Lk; causal is bottom-right aligned."""
    check_full(fa, [1, 37, 128, 200], 2, 128, causal, seed=13, lk=[5, 300, 129, 1000])


def test_q_longer_than_k(fa):
    """Lq > Lk with causal: the first Lq - Lk rows see no key (O = 0,
    LSE = -inf), including a whole tile of such rows."""
    check_full(fa, [300, 20], 2, 64, True, seed=14, lk=[40, 3])


@pytest.mark.parametrize("causal", [False, True])
def test_zero_length_sequences(fa, causal):
    """Sequences with no queries are skipped; a sequence whose queries see no
    key (Lk = 0) gets O = 0 and LSE = -inf."""
    check_full(fa, [0, 5, 0, 130, 7], 2, 64, causal, seed=17, lk=[3, 0, 0, 200, 7])


def test_c4_sampled(fa):
    """16 sequences, lengths U[128, 4096], H32 d64, causal: the full-size
    launch bench-style, sampled rows of every sequence and head."""
    lens = W.c4_lengths()
    H, d = 32, 64
    q, k, v, cq, ck = W.varlen_inputs(lens, H, d, 1238, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = run_varlen(fa, q, k, v, cq, ck, lens, lens, scale, True)
    og, lg = f64(o), f64(lse)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    cu = cq.cpu().numpy()
    rng = np.random.default_rng(4)
    for s, L in enumerate(lens):
        a = int(cu[s])
        rows = np.unique(np.concatenate([[0, L - 1, min(127, L - 1), min(128, L - 1)], rng.choice(L, 6)]))
        for h in range(0, H, 3):
            O_ref, L_ref = oracle.attention_rows(f64(qc[a + rows, h]), f64(kc[a:a + L, h]), f64(vc[a:a + L, h]),
                                                 scale, True, rows=rows, Lq=L)
            assert_o_close(og[a + rows, h], O_ref, f"C4 s{s} h{h}")
            assert_lse_close(lg[h, a + rows], L_ref, f"C4 s{s} h{h}")


def test_c4_whole_sequences(fa):
    """The full-size C4 launch: every row of the longest and the shortest
    sequence, on three heads, against the oracle's naive causal attention of
    that sequence alone."""
    lens = W.c4_lengths()
    H, d = 32, 64
    q, k, v, cq, ck = W.varlen_inputs(lens, H, d, 1238, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = run_varlen(fa, q, k, v, cq, ck, lens, lens, scale, True)
    og, lg = f64(o), f64(lse)
    cu = cq.cpu().numpy()
    for s in (int(np.argmax(lens)), int(np.argmin(lens))):
        a, L = int(cu[s]), lens[s]
        for h in (0, 13, 31):
            O_ref, L_ref = oracle.attention_head(f64(q[a:a + L, h]), f64(k[a:a + L, h]), f64(v[a:a + L, h]), scale,
                                                 True)
            assert_o_close(og[a:a + L, h], O_ref, f"C4 whole s{s} h{h}")
            assert_lse_close(lg[h, a:a + L], L_ref, f"C4 whole s{s} h{h}")


def test_varlen_equals_dense_per_sequence(fa):
    """The GPU's varlen result for a sequence equals its dense result."""
    lens = [200, 77]
    q, k, v, cq, ck = W.varlen_inputs(lens, 2, 128, 15, "cuda")
    o, lse = run_varlen(fa, q, k, v, cq, ck, lens, lens, 0.1, True)
    a, b = 0, 200
    od = torch.empty((1, 200, 2, 128), dtype=torch.bfloat16, device="cuda")
    st = fa.fa_fwd(q[None, a:b].contiguous(), k[None, a:b].contiguous(), v[None, a:b].contiguous(), od, None,
                   1, 2, 2, 200, 128, 0.1, 1)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(od[0], o[a:b])


def test_bad_cu_seqlens_reported(fa):
    """A sequence longer than max_seqlen is reported, not computed past."""
    lens = [10, 300]
    q, k, v, cq, ck = W.varlen_inputs(lens, 1, 64, 16, "cuda")
    o = torch.zeros_like(q)
    st = fa.fa_varlen_fwd(q, k, v, o, None, cq, ck, 2, 128, 128, 310, 310, 1, 1, 64, 0.125, 0)
    assert st == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX
    assert fa.fa_device_status() == fa.FA_OK  # cleared


@pytest.mark.parametrize("causal", [False, True])
def test_bad_sequence_without_slots_reported(fa, causal):
    """Offsets [0, 300, 100, 310]: the middle sequence has a negative length,
    so the launch's (sequence, block) slots give it none; it is still
    reported, and the first sequence is still computed."""
    lens = [300, 10]
    q, k, v, cq, ck = W.varlen_inputs(lens, 2, 64, 17, "cuda")
    bad = torch.tensor([0, 300, 100, 310], dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q)
    st = fa.fa_varlen_fwd(q, k, v, o, None, bad, bad, 3, 512, 512, 310, 310, 2, 2, 64, 0.125, int(causal))
    assert st == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_ERR_DEVICE_INDEX
    assert fa.fa_device_status() == fa.FA_OK  # cleared
    o_ref, _ = run_varlen(fa, q[:300], k[:300], v[:300], cq[:2], ck[:2], [300], [300], 0.125, causal)
    torch.cuda.synchronize()
    # rows 100.. are also the third sequence's (offsets 100..310), so only
    # rows 0..99 are the first sequence's alone
    assert torch.equal(o[:100], o_ref[:100]), "sequence 0 differs"


@pytest.mark.parametrize("causal", [False, True])
def test_many_sequences(fa, causal):
    """400 sequences of 1 to 300 tokens: more sequences than a CTA has
    threads, so the launch keeps one block per (sequence, Q block) of the
    longest sequence."""
    rng = np.random.default_rng(23)
    lens = rng.integers(1, 301, size=400).tolist()
    check_full(fa, lens, 2, 64, causal, seed=24)
