"""Pins for the oracle's packed layouts (CPU only).  The packed tensors are
built here with np.stack from separately drawn Q, K, V, so each packed
function must equal the unpacked routine on those very tensors, bit for bit;
planted copies that read the wrong slot of the packed axis must fail."""

import numpy as np
import pytest

import oracle


def check_packed(qkv_fn, kv_fn, vqkv_fn, vkv_fn):
    fails = []
    rng = np.random.default_rng(201)
    B, S, H, Hkv, d = 2, 37, 4, 2, 8
    q, k, v = (rng.normal(size=(B, S, H, d)) for _ in range(3))
    kg, vg = (rng.normal(size=(B, S, Hkv, d)) for _ in range(2))
    for causal in (False, True):
        want = oracle.attention_dense(q, k, v, 0.3, causal)
        got = qkv_fn(np.stack([q, k, v], axis=2), 0.3, causal)
        if not all(np.array_equal(a, b) for a, b in zip(got, want)):
            fails.append(f"qkvpacked c{causal}")
        want = oracle.attention_dense(q, kg, vg, 0.3, causal)
        got = kv_fn(q, np.stack([kg, vg], axis=2), 0.3, causal)
        if not all(np.array_equal(a, b) for a, b in zip(got, want)):
            fails.append(f"kvpacked c{causal}")
    lens_q, lens_k = [3, 40, 1], [9, 40, 12]
    cq = np.concatenate([[0], np.cumsum(lens_q)])
    ck = np.concatenate([[0], np.cumsum(lens_k)])
    tq, tk = int(cq[-1]), int(ck[-1])
    q2, k2, v2 = (rng.normal(size=(tq, H, d)) for _ in range(3))
    kk, vv = (rng.normal(size=(tk, Hkv, d)) for _ in range(2))
    want = oracle.attention_varlen(q2, k2, v2, cq, cq, 0.3, True)
    got = vqkv_fn(np.stack([q2, k2, v2], axis=1), cq, 0.3, True)
    if not all(np.array_equal(a, b) for a, b in zip(got, want)):
        fails.append("varlen qkvpacked")
    want = oracle.attention_varlen(q2, kk, vv, cq, ck, 0.3, True)
    got = vkv_fn(q2, np.stack([kk, vv], axis=1), cq, ck, 0.3, True)
    if not all(np.array_equal(a, b) for a, b in zip(got, want)):
        fails.append("varlen kvpacked")
    return fails


def test_packed_pins():
    assert check_packed(oracle.attention_qkvpacked, oracle.attention_kvpacked, oracle.attention_varlen_qkvpacked,
                        oracle.attention_varlen_kvpacked) == []


def _swap_kv_qkv(qkv, scale, causal):
    return oracle.attention_dense(qkv[:, :, 0], qkv[:, :, 2], qkv[:, :, 1], scale, causal)


def _q_from_k(q, kv, scale, causal):
    return oracle.attention_dense(q, kv[:, :, 0], kv[:, :, 0], scale, causal)


def _wrong_axis(qkv, cu, scale, causal):
    # packed axis taken as the head axis
    return oracle.attention_varlen(qkv[:, :, 0].reshape(qkv.shape[0], 3, -1)[:, :, : qkv.shape[-1]][:, :1].repeat(
        qkv.shape[2], axis=1), qkv[:, 1], qkv[:, 2], cu, cu, scale, causal)


def _swap_kv_varlen(q, kv, cq, ck, scale, causal):
    return oracle.attention_varlen(q, kv[:, 1], kv[:, 0], cq, ck, scale, causal)


@pytest.mark.parametrize("which", ["swap_kv_qkv", "v_from_k", "wrong_axis", "swap_kv_varlen"])
def test_packed_mutant_is_caught(which):
    fns = [oracle.attention_qkvpacked, oracle.attention_kvpacked, oracle.attention_varlen_qkvpacked,
           oracle.attention_varlen_kvpacked]
    if which == "swap_kv_qkv":
        fns[0] = _swap_kv_qkv
    elif which == "v_from_k":
        fns[1] = _q_from_k
    elif which == "wrong_axis":
        fns[2] = _wrong_axis
    else:
        fns[3] = _swap_kv_varlen
    assert check_packed(*fns) != []
