"""Float64 CPU oracle for exact attention (the forward, and its backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes (the plain definition, no tiling, no fusion):

    S = scale * Q K^T            (dlog.com.cn "从标准 Attention 到 FlashAttention
                                  与分页执行", opening definition and its code)
    P = softmax(S, dim=-1)       (same page, §2.1 step two)
    O = P V                      (same page, §2.1 step three)
    LSE_i = log sum_j exp(S_ij)  (yulong.wang "L2.5 极致算子实战案例", §2.1:
                                  the forward writes O and the per-row
                                  logsumexp; natural log, written m + ln l)

All arithmetic is float64.  Inputs are whatever the caller passes (the tests
pass the very bf16 values the GPU sees, upcast exactly to float64).

Readings of points the pages leave open:

* scale is an explicit argument (the pages' 1/sqrt(d) is garbled on two of
  the three pages and omitted in the worked example);
* causal masking is bottom-right aligned: key j is visible to query i iff
  j <= i + (Lk - Lq).  With Lq == Lk this is the plain lower triangle with the
  diagonal; a single decode query sees every cached key;
* a row with no visible key has O = 0 and LSE = -inf;
* the paged KV pool is [num_pages, page_size, H, d]; logical token t of
  sequence b lives at page block_table[b][t // page_size], slot
  t % page_size.

Functions
---------
attention_head           naive single-head attention, materialises S and P
attention_rows           the same for a chosen subset of query rows
attention_head_blocked   the blocked online-softmax recurrence (invariant
                         check only; also returns the per-step (m, l) trace)
attention_dense          [B, N, H, d] batched multi-head wrapper
attention_varlen         packed [total, H, d] + cu_seqlens wrapper
attention_paged          single-query decode over a paged KV pool
store_kvcache            scatter of one step's K/V rows into the page pool
attention_qkvpacked      the packed layouts of the page's function table:
attention_kvpacked         QKV as [.., 3, H, d] or KV as [.., 2, Hkv, d],
attention_varlen_qkvpacked fixed-length or varlen; each slices the packed
attention_varlen_kvpacked  tensor and calls the routine above
attention_backward_head  gradients dQ, dK, dV of one head (the backward pass
attention_backward_dense   the pages describe: P recomputed from the saved
attention_backward_varlen  logsumexp, then the chain rule), and the batched
                           [B, N, H, d] and packed varlen wrappers (grouped
                           kv heads sum their query heads' dK, dV)
attention_varlen_paged   packed prefill whose K/V are read through the page
                         table (a chunk that continues a cached prefix)
gather_paged_kv          host walk of block_table (the bit-exact gather
                         reference)

Parity pins: every function here is pinned by tests under ``tests/``
(worked example, FA2 per-step table, closed forms, brute force, library
softmax/logsumexp, torch's float64 math SDPA, and the structural invariants).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "attention_head",
    "attention_rows",
    "attention_head_blocked",
    "attention_dense",
    "attention_varlen",
    "attention_paged",
    "attention_varlen_paged",
    "attention_qkvpacked",
    "attention_kvpacked",
    "attention_varlen_qkvpacked",
    "attention_varlen_kvpacked",
    "attention_backward_head",
    "attention_backward_dense",
    "attention_backward_varlen",
    "store_kvcache",
    "gather_paged_kv",
    "visible_mask",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def visible_mask(Lq: int, Lk: int, causal: bool, rows=None) -> np.ndarray:
    """Boolean [len(rows), Lk] mask of the keys each query row may attend to.

    Non-causal: every key.  Causal (bottom-right aligned): key j is visible
    to query i iff j <= i + (Lk - Lq).  The pages set ``causal=True`` for both
    the varlen prefill and the kv-cache decode call without defining the
    alignment (dlog.com.cn page, "v3 实际调用的两个函数"); bottom-right is the
    reading under which a decode query sees its whole history.
    """
    rows = np.arange(Lq) if rows is None else np.asarray(rows)
    if not causal:
        return np.ones((rows.shape[0], Lk), dtype=bool)
    j = np.arange(Lk)[None, :]
    return j <= (rows[:, None] + (Lk - Lq))


def attention_rows(q, k, v, scale: float, causal: bool, rows=None, Lq=None):
    """Naive attention for the query rows ``rows`` of one head.

    q: [len(rows), d] (the selected query rows), k, v: [Lk, d].
    ``Lq`` is the full query length (needed for the causal alignment); it
    defaults to the number of rows passed.  Returns (O [r, d], LSE [r]).

    Steps, in the order of the definition: S = scale * q k^T; masked entries
    are -inf; m = rowmax S; l = sum exp(S - m); P = exp(S - m) / l; O = P v;
    LSE = m + ln l.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    r = q.shape[0]
    Lk = k.shape[0]
    if Lq is None:
        Lq = r
    if rows is None:
        rows = np.arange(r)
    S = scale * (q @ k.T)  # [r, Lk]
    vis = visible_mask(Lq, Lk, causal, rows)
    S = np.where(vis, S, -np.inf)
    any_vis = vis.any(axis=1)
    m = np.where(any_vis, S.max(axis=1, initial=-np.inf), 0.0)
    E = np.where(vis, np.exp(S - m[:, None]), 0.0)
    l = E.sum(axis=1)
    safe_l = np.where(any_vis, l, 1.0)
    P = E / safe_l[:, None]
    O = P @ v
    O = np.where(any_vis[:, None], O, 0.0)
    lse = np.where(any_vis, m + np.log(safe_l), -np.inf)
    return O, lse


def attention_head(q, k, v, scale: float, causal: bool = False, return_sp: bool = False):
    """Naive single-head attention.  q: [Lq, d], k, v: [Lk, d].

    Materialises S and P ([Lq, Lk]) exactly as the pages' opening code does.
    Returns (O [Lq, d], LSE [Lq]) and, with ``return_sp``, also (S, P).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Lq, Lk = q.shape[0], k.shape[0]
    S = scale * (q @ k.T)
    vis = visible_mask(Lq, Lk, causal)
    Sm = np.where(vis, S, -np.inf)
    any_vis = vis.any(axis=1)
    m = np.where(any_vis, Sm.max(axis=1, initial=-np.inf), 0.0)
    E = np.where(vis, np.exp(Sm - m[:, None]), 0.0)
    l = E.sum(axis=1)
    safe_l = np.where(any_vis, l, 1.0)
    P = E / safe_l[:, None]
    O = np.where(any_vis[:, None], P @ v, 0.0)
    lse = np.where(any_vis, m + np.log(safe_l), -np.inf)
    if return_sp:
        return O, lse, Sm, P
    return O, lse


def attention_head_blocked(q, k, v, scale: float, causal: bool, block_m: int, block_n: int,
                           trace: list | None = None):
    """Blocked attention with the online-softmax recurrence, float64.

    This is the recurrence of dlog.com.cn "从标准 Attention 到 FlashAttention 与
    分页执行" §2.2 (and §2.3's FA2 form), written in its own notation: for each
    Q row block keep a running max m, running sum l and accumulator O; for
    each K/V block

        m_new = max(m, rowmax(S_ij))
        l     = l * exp(m - m_new) + rowsum(exp(S_ij - m_new))
        O     = O * exp(m - m_new) + exp(S_ij - m_new) @ V_j
        m     = m_new

    and finally O / l.  Start values are m = -inf, l = 0, O = 0.  The last
    block of either dimension is allowed to be short (the page's code assumes
    the block size divides N).  Rows that have seen no visible key yet keep
    m = -inf; their exp factors are taken as 0 (the guard the lqnn.cn page §5.1
    says an unguarded exp(m - m_new) lacks).

    If ``trace`` is a list, (m, l) of every row after every K/V block is
    appended to it as a tuple of arrays (the per-step table of §2.3).
    Used only as an invariant check: it must equal attention_head.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Lq, Lk, d = q.shape[0], k.shape[0], v.shape[1]
    O = np.zeros((Lq, d))
    lse = np.zeros(Lq)
    for i0 in range(0, Lq, block_m):
        i1 = min(i0 + block_m, Lq)
        rows = np.arange(i0, i1)
        Qi = q[i0:i1]
        m = np.full(i1 - i0, -np.inf)
        l = np.zeros(i1 - i0)
        Oi = np.zeros((i1 - i0, d))
        for j0 in range(0, Lk, block_n):
            j1 = min(j0 + block_n, Lk)
            Sij = scale * (Qi @ k[j0:j1].T)
            vis = visible_mask(Lq, Lk, causal, rows)[:, j0:j1]
            Sij = np.where(vis, Sij, -np.inf)
            m_new = np.maximum(m, Sij.max(axis=1, initial=-np.inf))
            seen = m_new > -np.inf
            ref = np.where(seen, m_new, 0.0)
            alpha = np.where(seen & (m > -np.inf), np.exp(np.where(m > -np.inf, m, 0.0) - ref), 0.0)
            Pij = np.where(vis, np.exp(Sij - ref[:, None]), 0.0)
            l = l * alpha + Pij.sum(axis=1)
            Oi = Oi * alpha[:, None] + Pij @ v[j0:j1]
            m = m_new
            if trace is not None:
                trace.append((m.copy(), l.copy()))
        seen = m > -np.inf
        safe_l = np.where(seen, l, 1.0)
        O[i0:i1] = np.where(seen[:, None], Oi / safe_l[:, None], 0.0)
        lse[i0:i1] = np.where(seen, m + np.log(safe_l), -np.inf)
    return O, lse


def attention_dense(q, k, v, scale: float, causal: bool):
    """Batched multi-head attention, layout [B, N, H, d] (the flash-attn
    fixed-length interface, dlog.com.cn page §3.1).

    k and v may have H_kv heads with H % H_kv == 0 (query head h reads kv head
    h // (H // H_kv), the grouping of the page's GQA section).
    Returns O [B, N, H, d] and LSE [B, H, N].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    g = H // Hkv
    O = np.zeros_like(q)
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o, s = attention_head(q[b, :, h], k[b, :, h // g], v[b, :, h // g], scale, causal)
            O[b, :, h] = o
            lse[b, h] = s
    return O, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool):
    """Packed variable-length attention (dlog.com.cn page §3.3).

    q: [total_q, H, d], k, v: [total_k, H_kv, d]; cu_seqlens_* are the int
    prefix sums (first 0, last = total).  Sequence s owns rows
    [cu[s], cu[s+1]); no token attends across sequences; causal applies inside
    each sequence with bottom-right alignment.  Each sequence is computed by
    the very same single-head routine on its slice, so the result equals
    per-sequence dense attention exactly.
    Returns O [total_q, H, d] and LSE [H, total_q].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    total_q, H, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    O = np.zeros_like(q)
    lse = np.full((H, total_q), -np.inf)
    for s in range(len(cq) - 1):
        qs, qe, ks, ke = cq[s], cq[s + 1], ck[s], ck[s + 1]
        if qe == qs:
            continue
        for h in range(H):
            o, l = attention_head(q[qs:qe, h], k[ks:ke, h // g], v[ks:ke, h // g], scale, causal)
            O[qs:qe, h] = o
            lse[h, qs:qe] = l
    return O, lse


def gather_paged_kv(cache, block_table_row, seqlen: int, page_size: int):
    """Walk one sequence's block_table row on the host and return its
    logical KV rows [seqlen, H, d], in token order.

    Token t is read from page block_table_row[t // page_size], slot
    t % page_size (the page pool plus per-sequence page table of the
    dlog.com.cn page's PagedAttention section).  Entries past the pages the
    sequence uses are never read.  A pure copy: no arithmetic.
    """
    cache = np.asarray(cache)
    out = np.empty((seqlen,) + cache.shape[2:], dtype=cache.dtype)
    for t in range(seqlen):
        page = int(block_table_row[t // page_size])
        out[t] = cache[page, t % page_size]
    return out


def attention_paged(q, k_cache, v_cache, block_table, seqlens, page_size: int, scale: float,
                    causal: bool = True):
    """Single-token decode over a paged KV pool (the kv-cache entry point of
    the dlog.com.cn page, §3.4 and "v3 实际调用的两个函数").

    q: [B, H, d] (the [B, 1, H, d] query with the unit axis dropped);
    k_cache, v_cache: [num_pages, page_size, H_kv, d]; block_table:
    [B, max_pages] ints; seqlens: [B].  The oracle first gathers each
    sequence's keys and values into contiguous arrays, then runs the dense
    single-head routine with one query row.  Under bottom-right alignment the
    one query (the newest token) sees all seqlens[b] keys, so ``causal`` does
    not change the result.
    Returns O [B, H, d] and LSE [B, H].
    """
    q = _f64(q)
    B, H, d = q.shape
    Hkv = np.asarray(k_cache).shape[2]
    g = H // Hkv
    O = np.zeros((B, H, d))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        kb = _f64(gather_paged_kv(k_cache, block_table[b], L, page_size))
        vb = _f64(gather_paged_kv(v_cache, block_table[b], L, page_size))
        for h in range(H):
            o, l = attention_head(q[b, h][None, :], kb[:, h // g], vb[:, h // g], scale, causal)
            O[b, h] = o[0]
            lse[b, h] = l[0]
    return O, lse



def store_kvcache(k, v, k_cache, v_cache, slot_mapping, page_size: int):
    """Write one step's key/value rows into the paged pool (the store_kvcache
    step of the dlog.com.cn page, "v3 attention 的一条完整数据流", step 3).

    k, v: [T, H_kv, d]; k_cache, v_cache: [num_pages, page_size, H_kv, d];
    slot_mapping: [T] ints.  Row i goes to flat slot slot_mapping[i], i.e.
    page slot // page_size, offset slot % page_size.  A negative slot marks a
    token that is not stored (padding); the pages leave this open and this is
    the reading taken.  Returns new arrays; the inputs are not modified.  A
    pure copy: no arithmetic.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    k, v = np.asarray(k), np.asarray(v)
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        page, off = divmod(int(slot), page_size)
        kc[page, off] = k[i]
        vc[page, off] = v[i]
    return kc, vc


def attention_varlen_paged(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, page_size: int,
                           scale: float, causal: bool):
    """Packed variable-length prefill whose keys and values live in the page
    pool (the prefill entry point with block_table, dlog.com.cn page "v3 实际
    调用的两个函数": a chunk that continues a cached prefix reads its K/V
    through block_table).

    q: [total_q, H, d] packed by cu_seqlens_q.  Sequence s has
    Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s] keys, the logical tokens
    0 .. Lk-1 of its pages (block_table[s]); its Lq queries are the newest Lq
    of those tokens, so with causal the bottom-right alignment applies (query
    i sees keys j <= i + Lk - Lq).  The oracle gathers each sequence's K/V on
    the host and runs the very routine attention_varlen uses on contiguous
    K/V, so the two agree exactly on the same rows.
    Returns O [total_q, H, d] and LSE [H, total_q].
    """
    q = _f64(q)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    total_q, H, d = q.shape
    Hkv = np.asarray(k_cache).shape[2]
    g = H // Hkv
    O = np.zeros_like(q)
    lse = np.full((H, total_q), -np.inf)
    for s in range(len(cq) - 1):
        qs, qe = cq[s], cq[s + 1]
        Lk = ck[s + 1] - ck[s]
        if qe == qs:
            continue
        kb = _f64(gather_paged_kv(k_cache, block_table[s], Lk, page_size))
        vb = _f64(gather_paged_kv(v_cache, block_table[s], Lk, page_size))
        for h in range(H):
            o, l = attention_head(q[qs:qe, h], kb[:, h // g], vb[:, h // g], scale, causal)
            O[qs:qe, h] = o
            lse[h, qs:qe] = l
    return O, lse


def attention_qkvpacked(qkv, scale: float, causal: bool):
    """Packed QKV, fixed length (flash_attn_qkvpacked_func in the dlog.com.cn
    page's function table, §3.2): qkv is [B, S, 3, H, d], index 0 of the
    packed axis is Q, 1 is K, 2 is V.  Slices and runs attention_dense."""
    qkv = np.asarray(qkv)
    return attention_dense(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], scale, causal)


def attention_kvpacked(q, kv, scale: float, causal: bool):
    """Packed KV with a separate Q (flash_attn_kvpacked_func, same table):
    q [B, S, H, d], kv [B, S, 2, Hkv, d] with K at index 0, V at index 1."""
    kv = np.asarray(kv)
    return attention_dense(q, kv[:, :, 0], kv[:, :, 1], scale, causal)


def attention_varlen_qkvpacked(qkv, cu_seqlens, scale: float, causal: bool):
    """Packed QKV, variable length (flash_attn_varlen_qkvpacked_func, §3.3):
    qkv is [total, 3, H, d]; queries and keys share cu_seqlens."""
    qkv = np.asarray(qkv)
    return attention_varlen(qkv[:, 0], qkv[:, 1], qkv[:, 2], cu_seqlens, cu_seqlens, scale, causal)


def attention_varlen_kvpacked(q, kv, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool):
    """Packed KV, variable length (flash_attn_varlen_kvpacked_func, §3.3):
    q [total_q, H, d], kv [total_k, 2, Hkv, d]."""
    kv = np.asarray(kv)
    return attention_varlen(q, kv[:, 0], kv[:, 1], cu_seqlens_q, cu_seqlens_k, scale, causal)


def attention_backward_head(q, k, v, do, scale: float, causal: bool = False):
    """Gradients of O = softmax(scale Q K^T) V for one head, given dO.

    The steps the pages give for the backward pass (the lqnn.cn FlashAttention
    article §2.3 and §4.3, the yulong.wang page §2.3): recompute S and P (here
    from the definition; the kernels use the forward's logsumexp), then apply
    the chain rule, subtracting the row sum in dS:
      dV = P^T dO
      dP = dO V^T
      dS = P * (dP - D),  D_i = sum_j P_ij dP_ij = sum_d dO_id O_id
           (the row sum subtracted in the softmax backward)
      dQ = scale dS K,   dK = scale dS^T Q
    Masked entries have P = 0, hence dS = 0.  A row with no visible key has
    O = 0 and contributes nothing.  q: [Lq, d], k, v: [Lk, d], do: [Lq, d].
    Returns (dq, dk, dv) in float64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Lq, Lk = q.shape[0], k.shape[0]
    _, _, _, P = attention_head(q, k, v, scale, causal, return_sp=True)
    vis = visible_mask(Lq, Lk, causal)
    P = np.where(vis, P, 0.0)
    O = P @ v
    dv = P.T @ do
    dP = do @ v.T
    D = np.sum(do * O, axis=1)
    dS = P * (dP - D[:, None])
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    return dq, dk, dv


def attention_backward_dense(q, k, v, do, scale: float, causal: bool):
    """Batched backward: q, do [B, N, H, d], k, v [B, N, Hkv, d].  Query
    head h reads kv head h // (H // Hkv), so a kv head's dK and dV are the
    sums over its query heads.  Returns dq, dk, dv (float64)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, N, H, d = q.shape
    g = H // k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            a, bk, bv = attention_backward_head(q[b, :, h], k[b, :, h // g], v[b, :, h // g], do[b, :, h], scale,
                                                causal)
            dq[b, :, h] = a
            dk[b, :, h // g] += bk
            dv[b, :, h // g] += bv
    return dq, dk, dv


def attention_backward_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool):
    """Packed varlen backward: q, do [total_q, H, d], k, v [total_k, Hkv, d];
    sequence s is rows cu[s]:cu[s+1] of each (bottom-right causal when the
    lengths differ).  Rows outside every sequence stay 0."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    H = q.shape[1]
    g = H // k.shape[1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cu_seqlens_q) - 1):
        qa, qb = int(cu_seqlens_q[s]), int(cu_seqlens_q[s + 1])
        ka, kb = int(cu_seqlens_k[s]), int(cu_seqlens_k[s + 1])
        for h in range(H):
            a, bk, bv = attention_backward_head(q[qa:qb, h], k[ka:kb, h // g], v[ka:kb, h // g], do[qa:qb, h],
                                                scale, causal)
            dq[qa:qb, h] = a
            dk[ka:kb, h // g] += bk
            dv[ka:kb, h // g] += bv
    return dq, dk, dv
