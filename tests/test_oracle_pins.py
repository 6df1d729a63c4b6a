"""The float64 oracle against its pins (CPU only)."""

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_CHECKS, load_golden


def head(q, k, v, scale, causal):
    return oracle.attention_head(q, k, v, scale, causal)


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_naive_oracle(check):
    check(head)


@pytest.mark.parametrize("bm,bn", [(1, 1), (7, 7), (3, 64), (64, 128), (128, 7), (10**6, 10**6)])
@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_blocked_oracle(check, bm, bn):
    """The blocked online-softmax form passes the same pins for any block."""
    check(lambda q, k, v, s, c: oracle.attention_head_blocked(q, k, v, s, c, bm, bn))


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_rows_oracle(check):
    """attention_rows on all rows is the same function."""
    check(lambda q, k, v, s, c: oracle.attention_rows(q, k, v, s, c))


def test_fa2_per_step_trace():
    """dlog.com.cn page §2.3 table: (m, l) of both rows after every K/V block
    with one key per block, to the printed 4 dp."""
    g = load_golden("fa2_trace.json")
    trace = []
    oracle.attention_head_blocked(g["Q"], g["K"], g["V"], 1.0, False, 2, 1, trace=trace)
    assert len(trace) == 4
    tol = g["printed_precision"] + 1e-12
    for step, (m, l) in enumerate(trace):
        for r, key in enumerate(("m_l_q0", "m_l_q1")):
            m_p, l_p = g[key][step]
            assert m[r] == m_p
            assert abs(l[r] - l_p) <= tol, (step, r, l[r], l_p)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(200, 200), (129, 300), (300, 129), (1, 77)])
def test_blocked_equals_naive(causal, Lq, Lk):
    rng = np.random.default_rng(Lq * 1000 + Lk + causal)
    q = rng.normal(size=(Lq, 64))
    k = rng.normal(size=(Lk, 64))
    v = rng.normal(size=(Lk, 64))
    O, lse = oracle.attention_head(q, k, v, 0.125, causal)
    for bm, bn in [(1, 7), (64, 64), (128, 128), (Lq, Lk)]:
        Ob, lb = oracle.attention_head_blocked(q, k, v, 0.125, causal, bm, bn)
        assert np.max(np.abs(O - Ob)) <= 1e-12
        fin = np.isfinite(lse)
        assert np.array_equal(fin, np.isfinite(lb))
        assert np.max(np.abs(lse[fin] - lb[fin]), initial=0) <= 1e-12


def test_rows_subset_matches_full():
    """Row independence: any subset of rows equals the same rows of the full
    computation (dlog.com.cn page §2.1)."""
    rng = np.random.default_rng(3)
    q = rng.normal(size=(50, 8))
    k = rng.normal(size=(50, 8))
    v = rng.normal(size=(50, 8))
    for causal in (False, True):
        O, lse = oracle.attention_head(q, k, v, 0.3, causal)
        rows = np.array([0, 7, 31, 49])
        Or, lr = oracle.attention_rows(q[rows], k, v, 0.3, causal, rows=rows, Lq=50)
        assert np.array_equal(Or, O[rows]) and np.array_equal(lr, lse[rows])


def test_dense_wrapper_layout():
    """[B, N, H, d] wrapper equals per-(b, h) single-head calls, bit for bit;
    LSE is laid out [B, H, N]."""
    rng = np.random.default_rng(5)
    B, N, H, d = 2, 33, 3, 8
    q, k, v = (rng.normal(size=(B, N, H, d)) for _ in range(3))
    O, lse = oracle.attention_dense(q, k, v, 0.2, True)
    for b in range(B):
        for h in range(H):
            o, l = oracle.attention_head(q[b, :, h], k[b, :, h], v[b, :, h], 0.2, True)
            assert np.array_equal(O[b, :, h], o) and np.array_equal(lse[b, h], l)


def test_dense_gqa_mapping():
    """H_kv < H: query head h reads kv head h // (H // H_kv)."""
    rng = np.random.default_rng(6)
    q = rng.normal(size=(1, 9, 4, 8))
    k = rng.normal(size=(1, 9, 2, 8))
    v = rng.normal(size=(1, 9, 2, 8))
    O, _ = oracle.attention_dense(q, k, v, 0.3, False)
    kk = np.repeat(k, 2, axis=2)
    vv = np.repeat(v, 2, axis=2)
    O2, _ = oracle.attention_dense(q, kk, vv, 0.3, False)
    assert np.array_equal(O, O2)


def test_varlen_equals_per_sequence_dense():
    """cu_seqlens example of the dlog.com.cn page §3.3 ([0, 3, 7]) plus a
    longer packed batch: every sequence equals dense attention on its slice,
    exactly, and no row attends across a boundary."""
    rng = np.random.default_rng(8)
    for lens in ([3, 4], [1, 130, 2, 64, 257]):
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T, H, d = int(cu[-1]), 2, 16
        q, k, v = (rng.normal(size=(T, H, d)) for _ in range(3))
        for causal in (False, True):
            O, lse = oracle.attention_varlen(q, k, v, cu, cu, 0.25, causal)
            assert lse.shape == (H, T)
            for s in range(len(lens)):
                a, b = cu[s], cu[s + 1]
                Od, ld = oracle.attention_dense(q[None, a:b], k[None, a:b], v[None, a:b], 0.25, causal)
                assert np.array_equal(O[a:b], Od[0]) and np.array_equal(lse[:, a:b], ld[0])
        # changing another sequence's keys does not change sequence 0
        k2 = k.copy()
        k2[cu[1]:] += 5.0
        O2, _ = oracle.attention_varlen(q, k2, v, cu, cu, 0.25, False)
        assert np.array_equal(O2[: cu[1]], oracle.attention_varlen(q, k, v, cu, cu, 0.25, False)[0][: cu[1]])


def _paged_setup(rng, B, H, d, lens, page, slack=3):
    pages_per = [(L + page - 1) // page for L in lens]
    num_pages = sum(pages_per) + slack
    perm = rng.permutation(num_pages)
    maxp = max(pages_per) + 2
    bt = np.full((B, maxp), -7, dtype=np.int32)  # junk past the used pages
    kc = rng.normal(size=(num_pages, page, H, d))
    vc = rng.normal(size=(num_pages, page, H, d))
    kk, vv = [], []
    pos = 0
    for b in range(B):
        bt[b, : pages_per[b]] = perm[pos: pos + pages_per[b]]
        pos += pages_per[b]
    for b in range(B):
        toks = np.arange(lens[b])
        kk.append(kc[bt[b, toks // page], toks % page])
        vv.append(vc[bt[b, toks // page], toks % page])
    return kc, vc, bt, kk, vv


def test_gather_bit_exact():
    """The host page walk returns exactly the rows direct fancy indexing
    selects (a copy, bit for bit)."""
    rng = np.random.default_rng(9)
    kc, vc, bt, kk, vv = _paged_setup(rng, 3, 2, 8, [1, 16, 45], 16)
    for b, L in enumerate([1, 16, 45]):
        g = oracle.gather_paged_kv(kc, bt[b], L, 16)
        assert g.dtype == kc.dtype and np.array_equal(g, kk[b])


def test_paged_equals_dense_on_ungathered():
    """Decode through block_table equals dense single-query attention on the
    contiguous keys, exactly; causal does not change a single newest-token
    query (bottom-right)."""
    rng = np.random.default_rng(10)
    lens = [1, 15, 16, 17, 100]
    B, H, d = len(lens), 2, 8
    kc, vc, bt, kk, vv = _paged_setup(rng, B, H, d, lens, 16)
    q = rng.normal(size=(B, H, d))
    for causal in (False, True):
        O, lse = oracle.attention_paged(q, kc, vc, bt, np.array(lens), 16, 0.35, causal)
        for b in range(B):
            for h in range(H):
                o, l = oracle.attention_head(q[b, h][None], kk[b][:, h], vv[b][:, h], 0.35, False)
                assert np.array_equal(O[b, h], o[0]) and lse[b, h] == l[0]
