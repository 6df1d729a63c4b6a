"""Packed QKV / KV layouts against the float64 oracle, and bit for bit
against the unpacked entry points on the same values (the kernel is the same;
only the strides of the tensor maps differ)."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W
from gpu_helpers import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


def unpacked_dense(fa, q, k, v, scale, causal):
    B, N, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    assert fa.fa_fwd(q, k, v, o, lse, B, H, k.shape[2], N, d, scale, causal) == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_qkvpacked(fa, d, causal):
    B, N, H = 2, 333, 4
    q, k, v = W.dense_inputs(B, N, H, d, 61 + d, "cuda")
    qkv = torch.stack([q, k, v], dim=2).contiguous()
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.attention_qkvpacked(qkv, scale=scale, causal=causal)
    assert fa.fa_device_status() == fa.FA_OK
    O_ref, L_ref = oracle.attention_qkvpacked(f64(qkv), scale, causal)
    assert_o_close(o, O_ref, f"qkvpacked d{d} c{causal}")
    assert_lse_close(lse, L_ref, f"qkvpacked d{d} c{causal}")
    o2, lse2 = unpacked_dense(fa, q, k, v, scale, causal)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("d", [64, 128])
def test_kvpacked_gqa(fa, d):
    B, N, H, Hkv = 1, 517, 8, 2
    q, k, v = W.dense_inputs(B, N, H, d, 71 + d, "cuda", Hkv=Hkv)
    kv = torch.stack([k, v], dim=2).contiguous()
    scale = 1.0 / np.sqrt(d)
    for causal in (False, True):
        o, lse = fa.attention_kvpacked(q, kv, scale=scale, causal=causal)
        assert fa.fa_device_status() == fa.FA_OK
        O_ref, L_ref = oracle.attention_kvpacked(f64(q), f64(kv), scale, causal)
        assert_o_close(o, O_ref, f"kvpacked d{d} c{causal}")
        assert_lse_close(lse, L_ref, f"kvpacked d{d} c{causal}")
        o2, lse2 = unpacked_dense(fa, q, k, v, scale, causal)
        assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_varlen_packed(fa):
    lens_q, lens_k = [1, 200, 129, 64, 700], [1, 250, 129, 300, 700]
    H, Hkv, d = 4, 2, 128
    scale = 0.09
    # packed QKV: queries and keys share the lengths
    q, k, v, cu, _ = W.varlen_inputs(lens_q, H, d, 81, "cuda")
    qkv = torch.stack([q, k, v], dim=1).contiguous()
    T = q.shape[0]
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    assert fa.fa_varlen_qkvpacked_fwd(qkv, o, lse, cu, len(lens_q), max(lens_q), T, H, d, scale, 1) == fa.FA_OK
    assert fa.fa_device_status() == fa.FA_OK
    O_ref, L_ref = oracle.attention_varlen_qkvpacked(f64(qkv), cu.cpu().numpy(), scale, True)
    assert_o_close(o, O_ref, "varlen qkvpacked")
    assert_lse_close(lse, L_ref, "varlen qkvpacked")
    # packed KV with GQA and separate key lengths
    q, k, v, cq, ck = W.varlen_inputs(lens_q, H, d, 82, "cuda", lengths_k=lens_k, Hkv=Hkv)
    kv = torch.stack([k, v], dim=1).contiguous()
    o = torch.empty_like(q)
    lse = torch.empty((H, q.shape[0]), dtype=torch.float32, device="cuda")
    st = fa.fa_varlen_kvpacked_fwd(q, kv, o, lse, cq, ck, len(lens_q), max(lens_q), max(lens_k), q.shape[0],
                                   k.shape[0], H, Hkv, d, scale, 1)
    assert st == fa.FA_OK and fa.fa_device_status() == fa.FA_OK
    O_ref, L_ref = oracle.attention_varlen_kvpacked(f64(q), f64(kv), cq.cpu().numpy(), ck.cpu().numpy(), scale, True)
    assert_o_close(o, O_ref, "varlen kvpacked")
    assert_lse_close(lse, L_ref, "varlen kvpacked")
    o2, lse2 = fa.attention_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), scale=scale, causal=True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_qkvpacked_full_size_equals_unpacked(fa):
    """At the N=8192 d=128 H32 size the packed call reproduces the unpacked
    call bit for bit (the unpacked one is parity-checked against the oracle
    in test_gpu_prefill.py)."""
    B, N, H, d = 1, 8192, 32, 128
    q, k, v = W.dense_inputs(B, N, H, d, 1236, "cuda")
    qkv = torch.stack([q, k, v], dim=2).contiguous()
    for causal in (False, True):
        o, lse = fa.attention_qkvpacked(qkv, scale=1.0 / np.sqrt(d), causal=causal)
        o2, lse2 = unpacked_dense(fa, q, k, v, 1.0 / np.sqrt(d), causal)
        assert fa.fa_device_status() == fa.FA_OK
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
