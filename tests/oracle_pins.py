"""Pins for the float64 oracle: checks that tie it to things other than itself.

Each ``check_*`` takes a single-head attention implementation
``fn(q, k, v, scale, causal) -> (O, LSE)`` and raises AssertionError when the
implementation disagrees with what the pages or the mathematics fix.  The real
oracle must pass all of them (tests/test_oracle_pins.py); each deliberately
broken oracle in tests/test_oracle_mutants.py must fail at least one.

Sources of truth used here, none of which is the oracle's own formula:
  * the worked N=2, d=3 example and the FA2 per-step table of the dlog.com.cn
    page "从标准 Attention 到 FlashAttention 与分页执行" (§2.1, §2.3), stored
    under tests/golden/ with their citations;
  * closed forms (two-key softmax is a logistic function);
  * brute force in plain Python loops (math.exp, no numpy) on tiny inputs;
  * library routines: scipy.special.softmax / logsumexp and torch's float64
    math scaled_dot_product_attention on the CPU;
  * invariants: convex hull, shift of every score by c, joint permutation,
    constant values, identical keys, the first causal row.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- page values

def check_worked_example(fn):
    """The page's N=2, d=3 example (scale 1): printed P and O to 2 dp, plus
    the closed forms the printed values round: P[0,0] = 1/(1+e^3),
    P[1,0] = 1/(1+e^2), O[:,2] = 1 exactly (both V rows hold 1 there),
    LSE = 5 + ln(1+e^-3) and 3 + ln(1+e^-2)."""
    g = load_golden("worked_example.json")
    Q, K, V = (np.array(g[x], dtype=np.float64) for x in ("Q", "K", "V"))
    O, lse = fn(Q, K, V, g["scale"], False)
    tol = g["printed_precision"]
    P_printed = np.array(g["P_2dp"])
    O_printed = np.array(g["O_2dp"])
    # The page multiplies the rounded P by V (0.95 * 2 = 1.90), so the printed
    # O is exactly P_2dp @ V and differs from the true O by at most
    # tol * sum_j |V_jc| per column.
    assert np.max(np.abs(P_printed @ V - O_printed)) <= 1e-12
    bound = tol * np.abs(V).sum(axis=0)[None, :] + 1e-12
    assert np.all(np.abs(O - O_printed) <= bound), (O, O_printed)
    p00 = 1.0 / (1.0 + math.exp(3.0))
    p10 = 1.0 / (1.0 + math.exp(2.0))
    assert abs(p00 - P_printed[0, 0]) <= tol and abs(p10 - P_printed[1, 0]) <= tol
    # O row i = P[i,0] v0 + P[i,1] v1 with v0 = (1,0,1), v1 = (0,2,1)
    O_closed = np.array([[p00, 2 * (1 - p00), 1.0], [p10, 2 * (1 - p10), 1.0]])
    assert np.max(np.abs(O - O_closed)) <= 1e-12, (O, O_closed)
    lse_closed = np.array([5.0 + math.log1p(math.exp(-3.0)), 3.0 + math.log1p(math.exp(-2.0))])
    assert np.max(np.abs(lse - lse_closed)) <= 1e-12, (lse, lse_closed)


def check_fa2_final(fn):
    """Final O of the page's FA2 two-row table, to the printed 4 dp, and the
    row log-sum-exp implied by its last (m, l): LSE = m + ln l."""
    g = load_golden("fa2_trace.json")
    Q, K, V = (np.array(g[x], dtype=np.float64) for x in ("Q", "K", "V"))
    S = Q @ K.T
    assert np.array_equal(S[0], g["scores_q0"]) and np.array_equal(S[1], g["scores_q1"])
    O, lse = fn(Q, K, V, 1.0, False)
    tol = g["printed_precision"]
    assert np.max(np.abs(O - np.array(g["O_final"]))) <= tol + 1e-12, O
    for r, key in enumerate(("m_l_q0", "m_l_q1")):
        m, l = g[key][-1]
        assert abs(lse[r] - (m + math.log(l))) <= 1e-4, (lse, m, l)


# ------------------------------------------------------------ brute force

def brute_force(q, k, v, scale, causal):
    """Plain-Python attention on tiny inputs: explicit loops and math.exp."""
    Lq, d = len(q), len(q[0])
    Lk = len(k)
    O, L = [], []
    for i in range(Lq):
        scores = []
        for j in range(Lk):
            if causal and j > i + (Lk - Lq):
                continue
            s = 0.0
            for c in range(d):
                s += float(q[i][c]) * float(k[j][c])
            scores.append((j, scale * s))
        if not scores:
            O.append([0.0] * len(v[0]))
            L.append(-math.inf)
            continue
        top = max(s for _, s in scores)
        w = [(j, math.exp(s - top)) for j, s in scores]
        tot = sum(x for _, x in w)
        row = [0.0] * len(v[0])
        for j, x in w:
            for c in range(len(v[0])):
                row[c] += x / tot * float(v[j][c])
        O.append(row)
        L.append(top + math.log(tot))
    return np.array(O), np.array(L)


def check_brute_force(fn, seed=7):
    rng = _rng(seed)
    for trial in range(24):
        Lq = int(rng.integers(1, 6))
        Lk = int(rng.integers(1, 6))
        d = int(rng.integers(1, 5))
        dv = int(rng.integers(1, 4))
        causal = bool(trial % 2)
        scale = float(rng.uniform(0.2, 1.5))
        q = rng.normal(size=(Lq, d))
        k = rng.normal(size=(Lk, d))
        v = rng.normal(size=(Lk, dv))
        O, lse = fn(q, k, v, scale, causal)
        Ob, lb = brute_force(q.tolist(), k.tolist(), v.tolist(), scale, causal)
        assert np.max(np.abs(O - Ob)) <= 1e-12, (trial, O, Ob)
        fin = np.isfinite(lb)
        assert np.array_equal(np.isfinite(lse), fin), (lse, lb)
        assert np.max(np.abs(lse[fin] - lb[fin]), initial=0.0) <= 1e-12, (lse, lb)


# ------------------------------------------------------------ library routines

def check_scipy(fn, seed=11):
    """Row softmax and logsumexp from scipy (non-causal, random)."""
    from scipy.special import logsumexp, softmax

    rng = _rng(seed)
    q = rng.normal(size=(37, 16))
    k = rng.normal(size=(53, 16))
    v = rng.normal(size=(53, 8))
    scale = 0.25
    O, lse = fn(q, k, v, scale, False)
    S = scale * np.einsum("id,jd->ij", q, k)
    P = softmax(S, axis=1)
    assert np.max(np.abs(lse - logsumexp(S, axis=1))) <= 1e-12
    assert np.max(np.abs(O - np.einsum("ij,jc->ic", P, v))) <= 1e-12


def check_torch_sdpa(fn, seed=13):
    """torch's float64 math SDPA on the CPU (an independent implementation):
    non-causal with Lq != Lk, causal with Lq == Lk (torch's is_causal is the
    top-left triangle, which equals bottom-right only when Lq == Lk), and a
    bottom-right causal case through an explicit boolean mask."""
    import torch
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F

    rng = _rng(seed)
    cases = [(40, 70, 32, False), (64, 64, 16, True), (33, 33, 8, True)]
    for Lq, Lk, d, causal in cases:
        q = rng.normal(size=(Lq, d))
        k = rng.normal(size=(Lk, d))
        v = rng.normal(size=(Lk, d))
        scale = 1.0 / math.sqrt(d)
        O, _ = fn(q, k, v, scale, causal)
        with sdpa_kernel(SDPBackend.MATH):
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
                torch.from_numpy(v)[None, None], is_causal=causal, scale=scale)[0, 0].numpy()
        assert np.max(np.abs(O - ref)) <= 1e-12, (Lq, Lk, causal)
    # bottom-right alignment with Lq < Lk through an explicit mask
    Lq, Lk, d = 5, 12, 8
    q = rng.normal(size=(Lq, d))
    k = rng.normal(size=(Lk, d))
    v = rng.normal(size=(Lk, d))
    mask = np.arange(Lk)[None, :] <= (np.arange(Lq)[:, None] + (Lk - Lq))
    O, _ = fn(q, k, v, 0.5, True)
    with sdpa_kernel(SDPBackend.MATH):
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None], attn_mask=torch.from_numpy(mask)[None, None],
            scale=0.5)[0, 0].numpy()
    assert np.max(np.abs(O - ref)) <= 1e-12


# ------------------------------------------------------------ invariants

def check_convex_hull(fn, seed=17):
    """Each O coordinate lies between the min and max of the visible values."""
    rng = _rng(seed)
    for causal in (False, True):
        q = rng.normal(size=(31, 8))
        k = rng.normal(size=(31, 8))
        v = rng.normal(size=(31, 5))
        O, _ = fn(q, k, v, 0.7, causal)
        for i in range(31):
            vis = v[: i + 1] if causal else v
            assert np.all(O[i] >= vis.min(axis=0) - 1e-12) and np.all(O[i] <= vis.max(axis=0) + 1e-12), i


def check_shift(fn, seed=19):
    """Adding c_i to every score of row i leaves O unchanged and shifts LSE by
    c_i.  Realised with an extra feature: q' = [q, c/scale], k' = [k, 1]."""
    rng = _rng(seed)
    q = rng.normal(size=(9, 6))
    k = rng.normal(size=(14, 6))
    v = rng.normal(size=(14, 3))
    c = rng.normal(size=9) * 3
    scale = 0.4
    O, lse = fn(q, k, v, scale, False)
    O2, lse2 = fn(np.hstack([q, (c / scale)[:, None]]), np.hstack([k, np.ones((14, 1))]), v, scale, False)
    assert np.max(np.abs(O - O2)) <= 1e-12
    assert np.max(np.abs(lse2 - (lse + c))) <= 1e-12


def check_permutation(fn, seed=23):
    """Jointly permuting K and V rows (non-causal) changes nothing."""
    rng = _rng(seed)
    q = rng.normal(size=(7, 4))
    k = rng.normal(size=(19, 4))
    v = rng.normal(size=(19, 4))
    perm = rng.permutation(19)
    O, lse = fn(q, k, v, 1.0, False)
    O2, lse2 = fn(q, k[perm], v[perm], 1.0, False)
    assert np.max(np.abs(O - O2)) <= 1e-12 and np.max(np.abs(lse - lse2)) <= 1e-12


def check_constant_values_and_identical_keys(fn, seed=29):
    """Constant value rows give that row back.  Identical keys give the mean
    of V and LSE = s + ln(n), s the common score."""
    rng = _rng(seed)
    q = rng.normal(size=(6, 4))
    k = rng.normal(size=(10, 4))
    row = rng.normal(size=3)
    O, _ = fn(q, k, np.tile(row, (10, 1)), 0.9, False)
    assert np.max(np.abs(O - row[None, :])) <= 1e-12
    kr = rng.normal(size=4)
    K = np.tile(kr, (10, 1))
    V = rng.normal(size=(10, 3))
    O, lse = fn(q, K, V, 0.9, False)
    s = 0.9 * q @ kr
    assert np.max(np.abs(O - V.mean(axis=0)[None, :])) <= 1e-12
    assert np.max(np.abs(lse - (s + math.log(10)))) <= 1e-12


def check_causal_first_row(fn, seed=31):
    """Causal, Lq == Lk: row 0 sees only key 0, so O[0] = v0 and LSE[0] = s00;
    the last row sees every key, so it equals the non-causal last row."""
    rng = _rng(seed)
    q = rng.normal(size=(12, 5))
    k = rng.normal(size=(12, 5))
    v = rng.normal(size=(12, 4))
    O, lse = fn(q, k, v, 0.6, True)
    On, lsen = fn(q, k, v, 0.6, False)
    assert np.max(np.abs(O[0] - v[0])) <= 1e-12
    assert abs(lse[0] - 0.6 * float(q[0] @ k[0])) <= 1e-12
    assert np.max(np.abs(O[-1] - On[-1])) <= 1e-12 and abs(lse[-1] - lsen[-1]) <= 1e-12
    # row 1 is the two-key logistic mix of v0 and v1
    s0, s1 = 0.6 * float(q[1] @ k[0]), 0.6 * float(q[1] @ k[1])
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    assert np.max(np.abs(O[1] - ((1 - w1) * v[0] + w1 * v[1]))) <= 1e-12


def check_scale(fn, seed=37):
    """scale multiplies every score: (2q, scale) == (q, 2*scale); scale = 0
    gives the mean of V and LSE = ln Lk."""
    rng = _rng(seed)
    q = rng.normal(size=(5, 4))
    k = rng.normal(size=(8, 4))
    v = rng.normal(size=(8, 4))
    O1, l1 = fn(2 * q, k, v, 0.3, False)
    O2, l2 = fn(q, k, v, 0.6, False)
    assert np.max(np.abs(O1 - O2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12
    O0, l0 = fn(q, k, v, 0.0, False)
    assert np.max(np.abs(O0 - v.mean(axis=0))) <= 1e-12
    assert np.max(np.abs(l0 - math.log(8))) <= 1e-12


def check_empty_rows(fn):
    """Bottom-right causal with Lq > Lk: the first Lq - Lk rows see no key,
    so O = 0 and LSE = -inf; the rest see keys 0..i-(Lq-Lk)."""
    rng = _rng(41)
    q = rng.normal(size=(6, 3))
    k = rng.normal(size=(4, 3))
    v = rng.normal(size=(4, 3))
    O, lse = fn(q, k, v, 1.0, True)
    assert np.all(O[:2] == 0.0) and np.all(np.isneginf(lse[:2]))
    assert np.max(np.abs(O[2] - v[0])) <= 1e-12


ALL_CHECKS = [
    check_worked_example,
    check_fa2_final,
    check_brute_force,
    check_scipy,
    check_torch_sdpa,
    check_convex_hull,
    check_shift,
    check_permutation,
    check_constant_values_and_identical_keys,
    check_causal_first_row,
    check_scale,
    check_empty_rows,
]
