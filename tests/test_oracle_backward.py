"""Pins for the oracle's backward pass (CPU only): attention_backward_head,
attention_backward_dense and attention_backward_varlen.

The checks never restate the chain rule the oracle uses.  They take the
function under test as an argument, so the planted-mistake copies at the end
of this file run through the very same checks and must fail one of them:

* central finite differences of L = sum(dO * O), with O from the forward
  oracle (pinned on its own elsewhere);
* torch's float64 autograd through its own attention routine, for the
  batched [B, N, H, d] layout, grouped kv heads (expanded for torch, whose
  autograd then sums each group) and varlen sequences with bottom-right
  causal masking;
* closed forms: with one key, O = v for every row, so dQ = dK = 0 and dV is
  the column sum of dO; since every row of dS sums to zero, the key gradients
  sum to zero over the keys and dQ does not change when one vector is added
  to every key.
"""

import numpy as np
import pytest
import torch

import oracle


def _fd_grads(q, k, v, do, scale, causal, h=1e-6):
    """Central differences of sum(dO * O) in every input entry."""
    def loss(q_, k_, v_):
        O, _ = oracle.attention_head(q_, k_, v_, scale, causal)
        return float(np.sum(do * O))

    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        for idx in np.ndindex(*g.shape):
            a = [x.copy() for x in args]
            a[which][idx] += h
            up = loss(*a)
            a[which][idx] -= 2 * h
            g[idx] = (up - loss(*a)) / (2 * h)
        grads.append(g)
    return grads


def check_backward(fn, fn_dense):
    """Return the list of pins that (fn, fn_dense) fail."""
    fails = []
    rng = np.random.default_rng(301)

    # Finite differences: non-causal, causal square, and bottom-right causal
    # with Lq > Lk (rows 0 and 1 see no key: their gradients are 0).
    for Lq, Lk, d, causal in ((5, 7, 3, False), (5, 5, 4, True), (6, 4, 3, True), (3, 9, 2, True)):
        q, k, v, do = (rng.normal(size=(n, d)) for n in (Lq, Lk, Lk, Lq))
        scale = 0.7
        got = fn(q, k, v, do, scale, causal)
        want = _fd_grads(q, k, v, do, scale, causal)
        for name, a, b in zip(("dq", "dk", "dv"), got, want):
            if not np.allclose(a, b, rtol=1e-6, atol=1e-7):
                fails.append(f"finite differences {name} Lq{Lq} Lk{Lk} causal={causal}")

    # One key: O = v for every row.
    q, do = rng.normal(size=(4, 3)), rng.normal(size=(4, 3))
    k, v = rng.normal(size=(1, 3)), rng.normal(size=(1, 3))
    dq, dk, dv = fn(q, k, v, do, 0.5, False)
    if not (np.allclose(dq, 0, atol=1e-14) and np.allclose(dk, 0, atol=1e-14)
            and np.allclose(dv, do.sum(axis=0, keepdims=True), atol=1e-14)):
        fails.append("single key")

    # Rows of dS sum to zero: sum_j dK_j = 0, and dQ is shift-invariant in K.
    q, k, v, do = (rng.normal(size=(n, 8)) for n in (33, 47, 47, 33))
    for causal in (False, True):
        dq, dk, _ = fn(q, k, v, do, 0.35, causal)
        if not np.allclose(dk.sum(axis=0), 0, atol=1e-12):
            fails.append(f"key gradients sum causal={causal}")
        dq2, _, _ = fn(q, k + rng.normal(size=(1, 8)), v, do, 0.35, causal)
        if not np.allclose(dq, dq2, atol=1e-12):
            fails.append(f"dq shift invariance causal={causal}")

    # Batched layout against torch's float64 autograd (bottom-right causal
    # via an explicit mask, since Lq == Lk here it is the lower triangle).
    B, N, H, d = 2, 37, 3, 16
    q, k, v, do = (rng.normal(size=(B, N, H, d)) for _ in range(4))
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
        mask = torch.ones(N, N, dtype=torch.bool).tril() if causal else None
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.25)
        out.backward(torch.tensor(do.transpose(0, 2, 1, 3)))
        got = fn_dense(q, k, v, do, 0.25, causal)
        for name, a, t in zip(("dq", "dk", "dv"), got, (tq, tk, tv)):
            if not np.allclose(a, t.grad.numpy().transpose(0, 2, 1, 3), rtol=1e-10, atol=1e-12):
                fails.append(f"torch autograd {name} causal={causal}")
    return fails


def test_backward_pins():
    assert check_backward(oracle.attention_backward_head, oracle.attention_backward_dense) == []


# ----------------------------------------------------------------- planted mistakes


def _mutant(kind):
    """A copy of the backward with one plausible mistake planted."""
    def head(q, k, v, do, scale, causal=False):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        Lq, Lk = q.shape[0], k.shape[0]
        vis = oracle.visible_mask(Lq, Lk, causal)
        if kind == "mask_ignored":
            vis = np.ones_like(vis)
        S = scale * (q @ k.T)
        Sm = np.where(vis, S, -np.inf)
        m = np.where(vis.any(axis=1), Sm.max(axis=1), 0.0)
        E = np.where(vis, np.exp(Sm - m[:, None]), 0.0)
        P = E / np.where(vis.any(axis=1), E.sum(axis=1), 1.0)[:, None]
        O = P @ v
        dP = do @ v.T
        D = np.sum(do * O, axis=1)
        if kind == "no_rowsum":
            D = np.zeros_like(D)
        if kind == "rowsum_of_dP":
            D = dP.sum(axis=1)
        dS = P * (dP - D[:, None])
        if kind == "sign":
            dS = -dS
        dv = P.T @ do if kind != "dv_from_dS" else dS.T @ do
        dq = scale * (dS @ k) if kind != "dq_unscaled" else dS @ k
        dk = scale * (dS.T @ q) if kind != "dk_from_do" else scale * (dS.T @ do)
        return dq, dk, dv

    def dense(q, k, v, do, scale, causal):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        B, N, H, d = q.shape
        out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
        for b in range(B):
            for h in range(H):
                hh = (h + 1) % H if kind == "head_mixup" else h
                g = head(q[b, :, h], k[b, :, hh], v[b, :, hh], do[b, :, h], scale, causal)
                for o, x in zip(out, g):
                    o[b, :, h] = x
        return out

    return head, dense


@pytest.mark.parametrize("kind", ["mask_ignored", "no_rowsum", "rowsum_of_dP", "sign", "dv_from_dS",
                                  "dq_unscaled", "dk_from_do", "head_mixup"])
def test_backward_mutant_is_caught(kind):
    assert check_backward(*_mutant(kind)) != []


# ----------------------------------------------------------------- grouped heads and varlen


def _torch_grads(q, k, v, do, scale, causal, group):
    """torch float64 autograd of one sequence [L, H, d]; the kv heads are
    expanded to the query heads, so autograd sums each group's gradients."""
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    Lq, Lk = q.shape[0], k.shape[0]
    mask = None
    if causal:
        mask = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(group, 0), tv.repeat_interleave(group, 0), attn_mask=mask, scale=scale)
    out.backward(torch.tensor(do.transpose(1, 0, 2)))
    return [t.grad.numpy().transpose(1, 0, 2) for t in (tq, tk, tv)]


def check_backward_wrappers(fn_dense, fn_varlen):
    """Return the list of pins that the grouped dense / varlen wrappers fail."""
    fails = []
    rng = np.random.default_rng(302)
    H, Hkv, d, scale = 6, 2, 8, 0.3
    # Grouped dense: every sequence against torch autograd.
    B, N = 2, 23
    q, do = rng.normal(size=(B, N, H, d)), rng.normal(size=(B, N, H, d))
    k, v = rng.normal(size=(B, N, Hkv, d)), rng.normal(size=(B, N, Hkv, d))
    for causal in (False, True):
        got = fn_dense(q, k, v, do, scale, causal)
        for b in range(B):
            want = _torch_grads(q[b], k[b], v[b], do[b], scale, causal, H // Hkv)
            for name, a, w in zip(("dq", "dk", "dv"), got, want):
                if not np.allclose(a[b], w, rtol=1e-10, atol=1e-12):
                    fails.append(f"grouped dense {name} causal={causal}")
    # Varlen with Lq <= Lk (bottom-right causal) and an empty sequence: each
    # sequence against torch autograd on its own rows; rows between
    # sequences' ends and the tensor end stay 0.
    lq, lk = [5, 0, 17, 9], [9, 4, 17, 30]
    cq = np.concatenate([[0], np.cumsum(lq)])
    ck = np.concatenate([[0], np.cumsum(lk)])
    q, do = rng.normal(size=(cq[-1], H, d)), rng.normal(size=(cq[-1], H, d))
    k, v = rng.normal(size=(ck[-1], Hkv, d)), rng.normal(size=(ck[-1], Hkv, d))
    for causal in (False, True):
        gq, gk, gv = fn_varlen(q, k, v, do, cq, ck, scale, causal)
        for s in range(len(lq)):
            qs, ks = slice(cq[s], cq[s + 1]), slice(ck[s], ck[s + 1])
            if lq[s] == 0:
                if not (np.all(gk[ks] == 0) and np.all(gv[ks] == 0)):
                    fails.append(f"varlen empty query sequence causal={causal}")
                continue
            want = _torch_grads(q[qs], k[ks], v[ks], do[qs], scale, causal, H // Hkv)
            for name, a, w in zip(("dq", "dk", "dv"), (gq[qs], gk[ks], gv[ks]), want):
                if not np.allclose(a, w, rtol=1e-10, atol=1e-12):
                    fails.append(f"varlen {name} seq{s} causal={causal}")
    return fails


def test_backward_wrapper_pins():
    assert check_backward_wrappers(oracle.attention_backward_dense, oracle.attention_backward_varlen) == []


def _wrapper_mutant(kind):
    def head_of(h, H, Hkv):
        return h % Hkv if kind == "group_modulo" else h // (H // Hkv)

    def dense(q, k, v, do, scale, causal):
        B, N, H, d = q.shape
        Hkv = k.shape[2]
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for h in range(H):
                hk = head_of(h, H, Hkv)
                a, bk, bv = oracle.attention_backward_head(q[b, :, h], k[b, :, hk], v[b, :, hk], do[b, :, h], scale,
                                                           causal)
                dq[b, :, h] = a
                if kind == "overwrite":
                    dk[b, :, hk], dv[b, :, hk] = bk, bv
                else:
                    dk[b, :, hk] += bk
                    dv[b, :, hk] += bv
        return dq, dk, dv

    def varlen(q, k, v, do, cq, ck, scale, causal):
        H, Hkv = q.shape[1], k.shape[1]
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for s in range(len(cq) - 1):
            qa, qb, ka, kb = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
            if kind == "top_left":  # causal aligned at the first key instead of the last
                kb = ka + min(kb - ka, qb - qa) if causal else kb
            for h in range(H):
                hk = head_of(h, H, Hkv)
                a, bk, bv = oracle.attention_backward_head(q[qa:qb, h], k[ka:kb, hk], v[ka:kb, hk], do[qa:qb, h],
                                                           scale, causal)
                dq[qa:qb, h] = a
                if kind == "overwrite":
                    dk[ka:kb, hk], dv[ka:kb, hk] = bk, bv
                else:
                    dk[ka:kb, hk] += bk
                    dv[ka:kb, hk] += bv
        return dq, dk, dv

    return dense, varlen


@pytest.mark.parametrize("kind", ["group_modulo", "overwrite", "top_left"])
def test_backward_wrapper_mutant_is_caught(kind):
    assert check_backward_wrappers(*_wrapper_mutant(kind)) != []
