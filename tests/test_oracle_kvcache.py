"""Pins for the oracle's page-pool functions (CPU only): store_kvcache and
attention_varlen_paged.

Each check takes the function under test as an argument, so that the
planted-mistake copies at the end of this file run through the very same
checks and must fail at least one of them.  Nothing here restates the
oracle's own arithmetic: the checks use direct fancy indexing, the
contiguous varlen oracle, single-head attention on hand-cut key sets, and the
fact that a causal prefill split into chunks equals the unsplit one.
"""

import numpy as np
import pytest

import oracle

PAGE = 16


# ----------------------------------------------------------------- store


def check_store(store):
    """Return the list of store_kvcache pins that ``store`` fails."""
    fails = []
    rng = np.random.default_rng(101)
    num_pages, H, d = 6, 2, 4
    kc0 = rng.normal(size=(num_pages, PAGE, H, d))
    vc0 = rng.normal(size=(num_pages, PAGE, H, d))

    # A literal example: flat slot 37 with 16-token pages is page 2, slot 5;
    # slot 16 is page 1, slot 0; slot 15 is page 0, slot 15.
    k = np.arange(3 * H * d, dtype=np.float64).reshape(3, H, d) + 1000.0
    v = -k
    kc, vc = store(k, v, kc0, vc0, np.array([37, 16, 15]), PAGE)
    if not (np.array_equal(kc[2, 5], k[0]) and np.array_equal(kc[1, 0], k[1]) and np.array_equal(kc[0, 15], k[2])
            and np.array_equal(vc[2, 5], v[0])):
        fails.append("literal slots")

    # Round trip: rows scattered to a random permutation of slots come back,
    # bit for bit, from the host page walk over the pages they landed in.
    T = 40
    k = rng.normal(size=(T, H, d))
    v = rng.normal(size=(T, H, d))
    pages = rng.permutation(num_pages)[:3]
    slots = np.array([pages[t // PAGE] * PAGE + t % PAGE for t in range(T)])
    kc, vc = store(k, v, kc0, vc0, slots, PAGE)
    gk = oracle.gather_paged_kv(kc, pages, T, PAGE)
    gv = oracle.gather_paged_kv(vc, pages, T, PAGE)
    if not (np.array_equal(gk, k) and np.array_equal(gv, v)):
        fails.append("round trip")

    # Everything not addressed is unchanged; the inputs are not modified.
    touched = np.zeros((num_pages, PAGE), dtype=bool)
    touched[slots // PAGE, slots % PAGE] = True
    if not (np.array_equal(kc[~touched], kc0[~touched]) and np.array_equal(vc[~touched], vc0[~touched])):
        fails.append("untouched slots")
    kc_copy = kc0.copy()
    store(k, v, kc0, vc0, slots, PAGE)
    if not np.array_equal(kc0, kc_copy):
        fails.append("input modified")

    # Negative slots are skipped: the pool is unchanged.
    kc, vc = store(k[:4], v[:4], kc0, vc0, np.array([-1, -1, -5, -16]), PAGE)
    if not (np.array_equal(kc, kc0) and np.array_equal(vc, vc0)):
        fails.append("negative slots")
    return fails


def test_store_kvcache_pins():
    assert check_store(oracle.store_kvcache) == []


# ----------------------------------------------------------------- paged varlen


def _pool(rng, lens, H, d, slack=2):
    """A seeded pool holding every sequence's keys in a random permutation of
    pages; returns the pool, the table, and the contiguous rows (taken by
    direct indexing, not by the oracle's page walk)."""
    pages_per = [(L + PAGE - 1) // PAGE for L in lens]
    num_pages = sum(pages_per) + slack
    perm = rng.permutation(num_pages)
    bt = np.full((len(lens), max(pages_per) + 1), -3, dtype=np.int32)
    pos = 0
    for s, n in enumerate(pages_per):
        bt[s, :n] = perm[pos: pos + n]
        pos += n
    kc = rng.normal(size=(num_pages, PAGE, H, d))
    vc = rng.normal(size=(num_pages, PAGE, H, d))
    ks, vs = [], []
    for s, L in enumerate(lens):
        t = np.arange(L)
        ks.append(kc[bt[s, t // PAGE], t % PAGE])
        vs.append(vc[bt[s, t // PAGE], t % PAGE])
    return kc, vc, bt, ks, vs


def check_varlen_paged(fn):
    """Return the list of attention_varlen_paged pins that ``fn`` fails."""
    fails = []
    rng = np.random.default_rng(102)
    H, Hkv, d, scale = 4, 2, 8, 0.3
    lk = [37, 16, 100, 5]
    lq = [5, 16, 30, 1]  # chunks of new tokens at the end of each sequence
    kc, vc, bt, ks, vs = _pool(rng, lk, Hkv, d)
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = rng.normal(size=(int(cq[-1]), H, d))

    # Equals the contiguous varlen oracle on the gathered rows, exactly.
    kcat, vcat = np.concatenate(ks), np.concatenate(vs)
    for causal in (False, True):
        O, lse = fn(q, kc, vc, cq, ck, bt, PAGE, scale, causal)
        O2, lse2 = oracle.attention_varlen(q, kcat, vcat, cq, ck, scale, causal)
        if not (np.array_equal(O, O2) and np.array_equal(lse, lse2)):
            fails.append(f"contiguous equivalence causal={causal}")

    # Bottom-right causal, by hand: query i of a chunk of Lq sees the first
    # Lk - Lq + i + 1 keys.
    O, lse = fn(q, kc, vc, cq, ck, bt, PAGE, scale, True)
    for s in range(len(lk)):
        for i in (0, lq[s] - 1):
            row = cq[s] + i
            nvis = lk[s] - lq[s] + i + 1
            for h in (0, H - 1):
                o, l = oracle.attention_head(q[row, h][None], ks[s][:nvis, h // 2], vs[s][:nvis, h // 2], scale, False)
                if not (np.allclose(O[row, h], o[0], rtol=0, atol=1e-12) and abs(lse[h, row] - l[0]) < 1e-12):
                    fails.append(f"bottom-right s{s} i{i}")

    # A causal prefill split into two chunks equals the unsplit prefill: the
    # second chunk continues the first through the page table.
    L, L1 = 70, 29
    kc2, vc2, bt2, ks2, vs2 = _pool(rng, [L], Hkv, d)
    qf = rng.normal(size=(L, H, d))
    Of, lf = oracle.attention_varlen(qf, ks2[0], vs2[0], np.array([0, L]), np.array([0, L]), scale, True)
    Oa, la = fn(qf[:L1], kc2, vc2, np.array([0, L1]), np.array([0, L1]), bt2, PAGE, scale, True)
    Ob, lb = fn(qf[L1:], kc2, vc2, np.array([0, L - L1]), np.array([0, L]), bt2, PAGE, scale, True)
    if not (np.allclose(np.concatenate([Oa, Ob]), Of, rtol=0, atol=1e-12)
            and np.allclose(np.concatenate([la, lb], axis=1), lf, rtol=0, atol=1e-12)):
        fails.append("chunked prefill")
    return fails


def test_varlen_paged_pins():
    assert check_varlen_paged(oracle.attention_varlen_paged) == []


# ----------------------------------------------------------------- planted mistakes


def _store_mutant(kind):
    def store(k, v, k_cache, v_cache, slot_mapping, page_size):
        kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
        for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
            if slot < 0 and kind != "no_skip":
                continue
            if kind == "swapped":
                off, page = divmod(int(slot), page_size)
                page %= kc.shape[0]
                off %= page_size
            else:
                page, off = divmod(int(slot), page_size)
            if kind == "off_by_one":
                off = (off + 1) % page_size
            kc[page, off] = k[i]
            vc[page, off] = v[i] if kind != "v_from_k" else k[i]
        return kc, vc
    return store


@pytest.mark.parametrize("kind", ["swapped", "off_by_one", "no_skip", "v_from_k"])
def test_store_mutant_is_caught(kind):
    assert check_store(_store_mutant(kind)) != []


def _paged_mutant(kind):
    def fn(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, page_size, scale, causal):
        if kind == "top_left":
            # treat the chunk's queries as the first tokens of the sequence
            q = np.asarray(q, dtype=np.float64)
            H = q.shape[1]
            g = H // np.asarray(k_cache).shape[2]
            O = np.zeros_like(q)
            lse = np.full((H, q.shape[0]), -np.inf)
            for s in range(len(cu_seqlens_q) - 1):
                a, b = int(cu_seqlens_q[s]), int(cu_seqlens_q[s + 1])
                Lk = int(cu_seqlens_k[s + 1] - cu_seqlens_k[s])
                kb = oracle.gather_paged_kv(k_cache, block_table[s], Lk, page_size)
                vb = oracle.gather_paged_kv(v_cache, block_table[s], Lk, page_size)
                for h in range(H):
                    for i in range(b - a):
                        n = min(i + 1, Lk) if causal else Lk
                        o, l = oracle.attention_head(q[a + i, h][None], kb[:n, h // g], vb[:n, h // g], scale, False)
                        O[a + i, h], lse[h, a + i] = o[0], l[0]
            return O, lse
        if kind == "keys_from_q_lengths":
            return oracle.attention_varlen_paged(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_q, block_table,
                                                 page_size, scale, causal)
        if kind == "page_table_ignored":
            bt = np.tile(np.arange(block_table.shape[1], dtype=np.int32), (block_table.shape[0], 1))
            bt = np.minimum(bt, np.asarray(k_cache).shape[0] - 1)
            return oracle.attention_varlen_paged(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, bt, page_size,
                                                 scale, causal)
        raise AssertionError(kind)
    return fn


@pytest.mark.parametrize("kind", ["top_left", "keys_from_q_lengths", "page_table_ignored"])
def test_varlen_paged_mutant_is_caught(kind):
    assert check_varlen_paged(_paged_mutant(kind)) != []
