"""Dense prefill (fa_fwd) against the float64 oracle, through the C-ABI."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


def run_dense(fa, q, k, v, scale, causal):
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    return o, lse


def check_full(fa, B, N, H, d, causal, seed, Hkv=None, scale=None):
    q, k, v = W.dense_inputs(B, N, H, d, seed, "cuda", Hkv=Hkv)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o, lse = run_dense(fa, q, k, v, scale, causal)
    O_ref, L_ref = oracle.attention_dense(f64(q), f64(k), f64(v), scale, causal)
    assert_o_close(o, O_ref, f"B{B} N{N} H{H} d{d} c{causal}")
    assert_lse_close(lse, L_ref, f"B{B} N{N} H{H} d{d} c{causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_c1(fa, causal):
    """B1 H1 N256 d64 (the single-head configuration; also run causal)."""
    check_full(fa, 1, 256, 1, 64, causal, seed=1234)


@pytest.mark.parametrize("causal", [False, True])
def test_c2_full(fa, causal):
    """B4 H16 N2048 d128, every output against the oracle."""
    check_full(fa, 4, 2048, 16, 128, causal, seed=1235)


def sampled_rows(N, rng, n_rand=48):
    fixed = [0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = set(r for r in fixed if 0 <= r < N)
    rows.update(rng.choice(N, size=min(n_rand, N), replace=False).tolist())
    return np.array(sorted(rows))


@pytest.mark.parametrize("causal", [False, True])
def test_c3_sampled(fa, causal):
    """B1 H32 N8192 d128 at full size (the launch bench.py times): sampled
    rows of every head against the oracle, computed row by row (rows are
    independent, so a sampled row is checked exactly as in the full run)."""
    B, N, H, d = 1, 8192, 32, 128
    q, k, v = W.dense_inputs(B, N, H, d, 1236, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = run_dense(fa, q, k, v, scale, causal)
    rng = np.random.default_rng(7 + causal)
    og, lg = f64(o), f64(lse)
    qh, kh, vh = q[0].cpu(), k[0].cpu(), v[0].cpu()
    for h in range(H):
        rows = sampled_rows(N, rng, n_rand=24)
        O_ref, L_ref = oracle.attention_rows(f64(qh[rows, h]), f64(kh[:, h]), f64(vh[:, h]), scale, causal,
                                             rows=rows, Lq=N)
        assert_o_close(og[0, rows, h], O_ref, f"C3 h{h}")
        assert_lse_close(lg[0, h, rows], L_ref, f"C3 h{h}")


@pytest.mark.parametrize("causal", [False, True])
def test_c3_whole_heads(fa, causal):
    """B1 H32 N8192 d128 at full size: every row of two heads (one in each
    causal head group of 8) against the oracle's naive attention of the head."""
    B, N, H, d = 1, 8192, 32, 128
    q, k, v = W.dense_inputs(B, N, H, d, 1236, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = run_dense(fa, q, k, v, scale, causal)
    og, lg = f64(o), f64(lse)
    for h in (3, 30):
        O_ref, L_ref = oracle.attention_head(f64(q[0, :, h]), f64(k[0, :, h]), f64(v[0, :, h]), scale, causal)
        assert_o_close(og[0, :, h], O_ref, f"C3 whole head {h} c{causal}")
        assert_lse_close(lg[0, h], L_ref, f"C3 whole head {h} c{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 63, 65, 127, 129, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(fa, N, d, causal):
    """Lengths around the 128-row tile: one row, partial tiles, a tile plus
    one, and a long ragged tail; two batches so a tail tile's rows reach into
    the next batch's tokens (which must be masked out)."""
    check_full(fa, 2, N, 2, d, causal, seed=100 + N + d)


@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 1)])
def test_gqa(fa, H, Hkv):
    check_full(fa, 2, 300, H, 128, True, seed=55, Hkv=Hkv)
    check_full(fa, 1, 200, H, 64, False, seed=56, Hkv=Hkv)


def test_head_groups(fa):
    """Causal d = 128 hands out (block, head) pairs in groups of 8 heads:
    12 heads make one full group and one of 4, over two batches."""
    check_full(fa, 2, 700, 12, 128, True, seed=58)
    check_full(fa, 2, 700, 12, 128, True, seed=59, Hkv=4)


def test_triton_tutorial_shape(fa):
    """The [2, 4, 1024, 64] case the yulong.wang page checks its kernel on."""
    check_full(fa, 2, 1024, 4, 64, False, seed=0)


def test_scale_not_default(fa):
    check_full(fa, 1, 333, 2, 128, True, seed=9, scale=0.37)
    check_full(fa, 1, 333, 2, 64, False, seed=10, scale=0.02)


def test_large_scores_rescale(fa):
    """Scores whose row max keeps growing along the keys force the lazy
    rescale of O in tensor memory: q = 4 * ones, keys scaled up with the key
    index, so each new block raises the max by far more than 2^8."""
    B, N, H, d = 1, 1024, 2, 64
    q = torch.full((B, N, H, d), 0.25, dtype=torch.bfloat16)
    ramp = torch.linspace(0.0, 8.0, N).reshape(1, N, 1, 1)
    k = (torch.ones((B, N, H, d)) * ramp).to(torch.bfloat16)
    v = W.randn_bf16((B, N, H, d), 77)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        o, lse = run_dense(fa, q, k, v, 1.0, causal)
        O_ref, L_ref = oracle.attention_dense(f64(q), f64(k), f64(v), 1.0, causal)
        assert_o_close(o, O_ref, f"ramp c{causal}")
        assert_lse_close(lse, L_ref, f"ramp c{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("top", [1.1, 0.0, -4.0])
def test_score_drift(fa, top, d):
    """Scores that drift along the keys by a set amount per 128-key block.

    top=1.1 raises the row max by about 3 log2 units per block: the row sum
    often exceeds 2^8 while the max stays within the exponent reference's
    bound (the exact path without a rescale), and every few blocks the bound
    is crossed (a rescale).  top=0 gives equal scores (P = 1 against the
    reference), top=-4 falling scores (later blocks underflow toward 0)."""
    B, N, H = 1, 1024, 2
    q = torch.full((B, N, H, d), 16.0 / d, dtype=torch.bfloat16)
    ramp = torch.linspace(0.0, top, N).reshape(1, N, 1, 1)
    k = (torch.ones((B, N, H, d)) * ramp).to(torch.bfloat16)
    v = W.randn_bf16((B, N, H, d), 78)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        o, lse = run_dense(fa, q, k, v, 1.0, causal)
        O_ref, L_ref = oracle.attention_dense(f64(q), f64(k), f64(v), 1.0, causal)
        assert_o_close(o, O_ref, f"drift {top} d{d} c{causal}")
        assert_lse_close(lse, L_ref, f"drift {top} d{d} c{causal}")


def test_lse_optional_and_deterministic(fa):
    q, k, v = W.dense_inputs(2, 700, 4, 128, 31, "cuda")
    o1 = torch.empty_like(q)
    o2 = torch.empty_like(q)
    assert fa.fa_fwd(q, k, v, o1, None, 2, 4, 4, 700, 128, 0.088, 1) == fa.FA_OK
    assert fa.fa_fwd(q, k, v, o2, None, 2, 4, 4, 700, 128, 0.088, 1) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2), "two runs differ"
    o3, _ = fa.attention(q, k, v, scale=0.088, causal=True)
    assert torch.equal(o1, o3)


@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned(fa, d):
    """An output buffer that starts 16 bytes past a 32-byte boundary (the
    API's alignment floor) takes the 16-byte store path: the same values as
    an aligned buffer, bit for bit, and the oracle's."""
    B, N, H = 1, 300, 3
    q, k, v = W.dense_inputs(B, N, H, d, 41, "cuda")
    scale = 1.0 / np.sqrt(d)
    o_al, lse_al = run_dense(fa, q, k, v, scale, True)
    assert o_al.data_ptr() % 32 == 0
    buf = torch.full((B * N * H * d + 8,), float("nan"), dtype=q.dtype, device=q.device)
    o_off = buf[8:].view(B, N, H, d)  # 16 bytes past the allocation's (256-byte aligned) start
    assert o_off.data_ptr() % 32 == 16
    lse_off = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd(q, k, v, o_off, lse_off, B, H, H, N, d, scale, True)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o_off, o_al)
    assert torch.equal(lse_off, lse_al)
    assert torch.isnan(buf[:8]).all(), "a store reached before the output"
    O_ref, L_ref = oracle.attention_dense(f64(q), f64(k), f64(v), scale, True)
    assert_o_close(o_off, O_ref, f"16-byte aligned o, d{d}")
