"""Backward pass (fa_bwd, fa_varlen_bwd) against the float64 oracle, through
the C-ABI.

O and LSE come from this library's forward on the same bf16 inputs (the
backward's contract); the oracle recomputes everything from q, k, v, dO in
float64.

Tolerance, per element, from the roundings the kernels make (u = 2^-9, the
bf16 unit roundoff; the bound below uses 2u = 2^-8 everywhere, and the test
allows twice the bound):
  * P^T and dS are rounded to bf16 before their products: relative u each;
  * delta_i = dO_i . O_i uses the forward's bf16 O, whose elements are off by
    at most u (|O| + P |V|) (its own P rounding and its output rounding);
  * P itself is recomputed from fp32 scores and the fp32 LSE (relative
    error ~1e-5, taken as 1e-5);
  * dQ, dK, dV are rounded to bf16 on output: relative u.
So, per head, with e_i = sum_d |dO_id| 2u (|O_id| + (P|V|)_id),
  err(dS_ij) <= 2u |dS_ij| + P_ij e_i
  |dV - ref| <= 2u (P^T |dO|) + 2u |dV|
  |dK - ref| <= scale (err(dS)^T |Q|) + 2u |dK|
  |dQ - ref| <= scale (err(dS) |K|) + 2u |dQ|
summed over the query heads of a kv head for dK and dV.  A dropped mask, a
wrong row or a missing term moves an element by O(P |dO|) or O(P |dP|),
far outside these bounds.
"""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import f64

pytestmark = pytest.mark.gpu

U2 = 2.0 ** -8


def head_bounds(q, k, v, do, scale, causal):
    """Error bounds of (dq, dk, dv) for one head, float64 [L, d] inputs."""
    O, _, _, P = oracle.attention_head(q, k, v, scale, causal, return_sp=True)
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    dP = do @ v.T
    delta = np.sum(do * O, axis=1)
    abs_ds = P * np.abs(dP - delta[:, None])
    e = np.sum(np.abs(do) * U2 * (np.abs(O) + P @ np.abs(v)), axis=1)
    err_ds = U2 * abs_ds + P * e[:, None] + 1e-5 * abs_ds
    bdv = U2 * (P.T @ np.abs(do)) + U2 * np.abs(dv)
    bdk = scale * (err_ds.T @ np.abs(q)) + U2 * np.abs(dk)
    bdq = scale * (err_ds @ np.abs(k)) + U2 * np.abs(dq)
    return (dq, dk, dv), (bdq, bdk, bdv)


def reference(q, k, v, do, cq, ck, scale, causal):
    """Oracle gradients and bounds for packed [total, heads, d] float64 inputs
    split by the boundary arrays (one sequence per entry)."""
    H, Hkv = q.shape[1], k.shape[1]
    g = H // Hkv
    ref = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
    bnd = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
    for s in range(len(cq) - 1):
        qs, ks = slice(int(cq[s]), int(cq[s + 1])), slice(int(ck[s]), int(ck[s + 1]))
        for h in range(H):
            r, b = head_bounds(q[qs, h], k[ks, h // g], v[ks, h // g], do[qs, h], scale, causal)
            ref[0][qs, h], bnd[0][qs, h] = r[0], b[0]
            for t in (1, 2):
                ref[t][ks, h // g] += r[t]
                bnd[t][ks, h // g] += b[t]
    return ref, bnd


def assert_grads_close(got, ref, bnd, what):
    for name, a, r, b in zip(("dq", "dk", "dv"), got, ref, bnd):
        a = f64(a).reshape(r.shape)
        assert np.all(np.isfinite(a)), f"{what} {name}: non-finite"
        err = np.abs(a - r)
        lim = 2.0 * b + 1e-6 * max(1e-30, float(np.abs(r).max(initial=0.0)))
        bad = err > lim
        if bad.any():
            idx = np.unravel_index(np.argmax(err - lim), err.shape)
            raise AssertionError(f"{what} {name}: {int(bad.sum())} of {err.size} outside the bound; worst at {idx}: "
                                 f"got {a[idx]:.6g} want {r[idx]:.6g} bound {lim[idx]:.3g}")


def run_dense(fa, B, N, H, Hkv, d, causal, seed):
    q, k, v = W.dense_inputs(B, N, H, d, seed, "cuda", Hkv=Hkv)
    do = W.randn_bf16((B, N, H, d), seed * 3 + 7, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.attention(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    return (q, k, v, do, scale), (dq, dk, dv)


@pytest.mark.parametrize("B,N,H,Hkv,d", [(2, 300, 4, 4, 128), (1, 517, 4, 2, 64), (3, 128, 2, 1, 128),
                                         (1, 1, 2, 2, 64), (1, 700, 2, 2, 128), (2, 257, 6, 3, 64),
                                         (2, 300, 12, 12, 128), (1, 400, 12, 4, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_backward(fa, B, N, H, Hkv, d, causal):
    (q, k, v, do, scale), got = run_dense(fa, B, N, H, Hkv, d, causal, seed=60 + N + d)
    flat = lambda t: f64(t).reshape(B * N, t.shape[2], d)
    cu = np.arange(B + 1) * N
    ref, bnd = reference(flat(q), flat(k), flat(v), flat(do), cu, cu, scale, causal)
    assert_grads_close([t.reshape(B * N, t.shape[2], d) for t in got], ref, bnd,
                       f"B{B} N{N} H{H}/{Hkv} d{d} c{causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward(fa, d, causal):
    """Ragged lengths, an empty query sequence, Lq < Lk (bottom-right causal:
    a chunk continuing a prefix) and Lq > Lk (leading rows see no key)."""
    lq = [1, 129, 300, 0, 64, 40, 257, 200]
    lk = [1, 129, 300, 5, 64, 300, 1000, 90]
    H, Hkv = 4, 2
    q, k, v, cq, ck = W.varlen_inputs(lq, H, d, 70 + d, "cuda", lengths_k=lk, Hkv=Hkv)
    do = W.randn_bf16(q.shape, 77 + d, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.attention_varlen(q, k, v, cq, ck, max(lq), max(lk), scale=scale, causal=causal)
    got = fa.attention_varlen_backward(q, k, v, o, lse, do, cq, ck, max(lq), max(lk), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    ref, bnd = reference(f64(q), f64(k), f64(v), f64(do), cq.cpu().numpy(), ck.cpu().numpy(), scale, causal)
    assert_grads_close(got, ref, bnd, f"varlen d{d} c{causal}")


def test_backward_deterministic(fa):
    """No atomics: two runs give the same bits."""
    B, N, H, d = 1, 1000, 4, 128
    q, k, v = W.dense_inputs(B, N, H, d, 81, "cuda", Hkv=2)
    do = W.randn_bf16((B, N, H, d), 82, "cuda")
    o, lse = fa.attention(q, k, v, causal=True)
    a = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    b = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_outputs_16_byte_aligned(fa, d):
    """dQ, dK and dV buffers 16 bytes past a 32-byte boundary (the API's
    alignment floor) take the 16-byte store path: the same bits as aligned
    buffers, and nothing written before them."""
    B, N, H = 1, 300, 4
    q, k, v = W.dense_inputs(B, N, H, d, 84, "cuda", Hkv=2)
    do = W.randn_bf16((B, N, H, d), 85, "cuda")
    o, lse = fa.attention(q, k, v, causal=True)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    bufs = [torch.full((x.numel() + 8,), float("nan"), dtype=x.dtype, device="cuda") for x in ref]
    dq, dk, dv = (b[8:].view(x.shape) for b, x in zip(bufs, ref))
    for x in (dq, dk, dv):
        assert x.data_ptr() % 32 == 16
    wsb = fa.fa_bwd_workspace_bytes(B, B * N, H)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    st = fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, wsb, B, H, 2, N, d, 1.0 / np.sqrt(d), 1)
    assert st == fa.FA_OK, fa.status_string(st)
    assert fa.fa_device_status() == fa.FA_OK
    torch.cuda.synchronize()
    for got, want, b in zip((dq, dk, dv), ref, bufs):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        assert torch.isnan(b[:8]).all(), "a store reached before the output"


def test_backward_workspace_too_small(fa):
    B, N, H, d = 1, 64, 2, 64
    q, k, v = W.dense_inputs(B, N, H, d, 83, "cuda")
    o, lse = fa.attention(q, k, v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, B * N, H) - 16, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = fa.fa_bwd(q, k, v, o, lse, q, dq, dk, dv, ws, ws.numel(), B, H, H, N, d, 0.125, 0)
    assert st == fa.FA_ERR_INVALID


@pytest.mark.parametrize("causal,heads", [(False, (5, 18)), (True, (0, 27))])
def test_backward_full_size_whole_heads(fa, causal, heads):
    """The launch bench.py times (B1 H32 N8192 d128): every element of two
    heads' dQ, dK and dV against the oracle's float64 gradients of those
    heads, within the per-element bound above.  Heads are independent
    (H = Hkv), so a head checked whole is checked exactly as in the full run."""
    B, N, H, d = 1, 8192, 32, 128
    q, k, v = W.dense_inputs(B, N, H, d, 1236, "cuda")
    do = W.randn_bf16_device((B, N, H, d), 1236 * 7 + 1, "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.attention(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for h in heads:
        ref, bnd = head_bounds(f64(q[0, :, h]), f64(k[0, :, h]), f64(v[0, :, h]), f64(do[0, :, h]), scale, causal)
        got = [t[0, :, h] for t in (dq, dk, dv)]
        assert_grads_close(got, ref, bnd, f"N8192 h{h} c{causal}")

