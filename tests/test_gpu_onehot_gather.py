"""Bit-exact checks of the page walks the product kernels run.

The paged entry points read keys and values through a page table (the
PagedAttention read of the dlog.com.cn page "从标准 Attention 到 FlashAttention
与分页执行", §3.4): token t of a sequence is slot t % page_size of page
block_table[t / page_size].  That read is a pure copy, so it must be exact.
A tolerance test cannot see one wrong key among thousands (its weight in O is
about 1 / L), so these tests make every checked output depend on exactly one
key:

* the key pool holds uniform signs (+1 / -1), so every score against a
  chosen key is an exact integer multiple of the query's factor;
* each query row is q = alpha * k_{t*} for a target token t* of its own, with
  alpha a power of two (exact in bf16).  Its score s* = alpha d scale beats
  every other visible key by at least 60 (natural log units; the test checks
  this on the oracle's S), so the oracle's P is one-hot to within e^-60 and
  its O rounded to bf16 is v_{t*} itself;
* the GPU's O row must then equal v_{t*} bit for bit, and its LSE the
  oracle's within 1e-3.

A wrong page, slot, head or row anywhere in the walk moves the target's score
off the maximum (O becomes another key's value or a mix) or reads the wrong
value row; a second copy of the target row read at another position doubles
its weight and moves the LSE by ln 2.  Either fails.

Targets cover page slots 0, 1, 15, 16, 17 (and the edges of larger pages),
the last tokens, the 128-key block edges, the 512- and 2048-token split
edges of the two decode kernels, and (on the smaller batches, over several
calls) one token of every page, which steps through every position of the
decode kernel's look-ahead ring.  Pages of 16, 32, 64 and 128 tokens are
covered.  In the paged prefill every key of every sequence is the target of
some query row, in one call.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MIN_GAP = 60.0  # natural-log units between the target's score and any other
LSE_ABS = 1e-3


def _alpha(d):
    # 16 * 128 / sqrt(128) = 181 and 32 * 64 / 8 = 256: the target's score;
    # random sign keys stay ~4.3 sqrt(d) below d, so the gap is > 100
    return 16.0 if d == 128 else 32.0


def _bits(t):
    """bf16 tensor -> int16 numpy (the raw bits), on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def _f64_rows(rows_i16):
    """int16 bf16 bits -> float64 numpy, exactly."""
    return torch.from_numpy(np.ascontiguousarray(rows_i16)).view(torch.bfloat16).to(torch.float64).numpy()


def _bf16_bits_of(x64):
    """float64 numpy -> bf16 bits (round to nearest even, through fp32; the
    values here sit within 1e-20 relative of a bf16 number, so the double
    rounding cannot matter)."""
    return torch.from_numpy(np.ascontiguousarray(x64)).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()


def _same_row(got, want, vstar):
    """Two output rows (bf16 bits) are equal bit for bit, except where the
    target value row is exactly zero (torch's normal draws give exact zeros
    about twice in ten million): there the result is the off-target
    remainder, below e^-60 times the largest value, and only its size is
    defined, so both sides must be below 1e-30 in magnitude (either sign of
    zero, or a denormal)."""
    zero = (vstar & 0x7FFF) == 0
    if not np.array_equal(got[~zero], want[~zero]):
        return False
    return bool(np.all(np.abs(_f64_rows(got[zero])) < 1e-30) and np.all(np.abs(_f64_rows(want[zero])) < 1e-30))


def special_positions(L, ps=16):
    """Page slots, block and split edges, and the last tokens of a sequence."""
    pts = {0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 127, 128, 129, 255, 256, 511, 512, 513, 1023, 1024, 1025,
           2047, 2048, 2049, 4095, 4096, 4097, 6143, 6144, 6145, L // 2, L - 17, L - 16, L - 15, L - 2, L - 1,
           ps - 1, ps, ps + 1, 2 * ps - 1, 2 * ps, 3 * ps + 5, L - ps, L - ps - 1}
    return sorted(p for p in pts if 0 <= p < L)


def every_page_positions(L, ps=16):
    """One token of every page, its slot stepping through the page."""
    return [p * ps + (p * 5) % ps for p in range((L + ps - 1) // ps) if p * ps + (p * 5) % ps < L]


def decode_targets(lengths, H, calls, every_page, ps=16):
    """targets[c][b][h] = the token query head h of sequence b aims at in
    call c: the special positions first, then (optionally) every page, cycling
    through the list."""
    out = []
    lists = []
    for L in lengths:
        lst = special_positions(L, ps)
        if every_page:
            lst = sorted(set(lst) | set(every_page_positions(L, ps)))
        lists.append(lst)
    for c in range(calls):
        out.append([[lst[(c * H + h) % len(lst)] if lst else -1 for h in range(H)] for lst in lists])
    return out, lists


def calls_needed(lists, H):
    return max(1, max((len(lst) + H - 1) // H for lst in lists))


class HostPool:
    """The page pool copied to the host once, as raw bf16 bits.  Each
    sequence's rows are gathered once by the oracle's host walk and kept as
    bits; the float64 copies are kept too for small batches (``keep_f64``)
    and made afresh per use for the full-size ones."""

    def __init__(self, pb, keep_f64=True, by_page=False):
        self.k = _bits(pb.k_cache)
        self.v = _bits(pb.v_cache)
        self.ps = pb.k_cache.shape[1]
        self.bt = pb.block_table.cpu().numpy()
        self.keep_f64 = keep_f64
        self.by_page = by_page
        self._bits = {}
        self._f64 = {}

    def _walk(self, cache, b, L):
        if not self.by_page or b < 2:
            return oracle.gather_paged_kv(cache, self.bt[b], L, self.ps)
        # The full-size pools: whole pages at once (the oracle's token walk
        # takes tens of microseconds a token there).  The same walk, checked
        # against the oracle's on the first two sequences below.
        n = (L + self.ps - 1) // self.ps
        return cache[self.bt[b, :n]].reshape((n * self.ps,) + cache.shape[2:])[:L]

    def check_walk(self, lengths):
        """The page-at-a-time walk equals the oracle's on sequences 2 and 3."""
        for b in (2, 3):
            if b < len(lengths):
                L = lengths[b]
                n = (L + self.ps - 1) // self.ps
                fast = self.k[self.bt[b, :n]].reshape((n * self.ps,) + self.k.shape[2:])[:L]
                assert np.array_equal(fast, oracle.gather_paged_kv(self.k, self.bt[b], L, self.ps))

    def seq(self, b, L):
        """(keys, values) of sequence b as bits [L, Hkv, d], then the same
        two as float64."""
        if b not in self._bits:
            self._bits[b] = (self._walk(self.k, b, L), self._walk(self.v, b, L))
        kb, vb = self._bits[b]
        if b in self._f64:
            return (kb, vb) + self._f64[b]
        f = (_f64_rows(kb), _f64_rows(vb))
        if self.keep_f64:
            self._f64[b] = f
        return (kb, vb) + f

    def key_f64(self, b, L, t, hk):
        """Key row t of kv head hk of sequence b, as float64."""
        if b not in self._bits:
            self.seq(b, L)
        return _f64_rows(self._bits[b][0][t, hk])


def build_decode_q(host, lengths, targets, H, Hkv, d):
    """q[b, h] = alpha * k_{t*} of kv head h / (H / Hkv), as bf16."""
    g = H // Hkv
    a = _alpha(d)
    q = np.zeros((len(lengths), H, d), dtype=np.float64)
    for b, L in enumerate(lengths):
        if L == 0:
            continue
        for h in range(H):
            q[b, h] = a * host.key_f64(b, L, targets[b][h], h // g)
    return torch.from_numpy(q).to(torch.bfloat16)


def check_decode(o, lse, host, q, lengths, targets, H, Hkv, d, what):
    """Oracle per (sequence, head); one-hot precondition; bit-exact O."""
    g = H // Hkv
    scale = 1.0 / math.sqrt(d)
    ob = _bits(o)
    lg = lse.detach().cpu().numpy().astype(np.float64)
    qf = q.to(torch.float64).numpy()
    for b, L in enumerate(lengths):
        if L == 0:
            assert np.all(ob[b] == 0), f"{what}: seq {b} (empty) O not zero"
            assert np.all(np.isneginf(lg[b])), f"{what}: seq {b} (empty) LSE not -inf"
            continue
        kb, vb, kf, vf = host.seq(b, L)
        for h in range(H):
            t = targets[b][h]
            hk = h // g
            O, lse_ref, S, P = oracle.attention_head(qf[b, h][None, :], kf[:, hk], vf[:, hk], scale, True,
                                                     return_sp=True)
            others = np.delete(S[0], t)
            gap = S[0, t] - (others.max() if others.size else -np.inf)
            assert gap >= MIN_GAP, f"{what}: precondition, seq {b} head {h} target {t}: gap {gap:.1f}"
            want = _bf16_bits_of(O[0])
            assert _same_row(want, want, vb[t, hk]) and _same_row(vb[t, hk], want, vb[t, hk]), \
                f"{what}: precondition, oracle O is not v[{t}]"
            got = ob[b, h]
            if not _same_row(got, want, vb[t, hk]):
                bad = int(np.sum(got != want))
                raise AssertionError(f"{what}: seq {b} (L={L}) head {h} target token {t} "
                                     f"(page entry {t // host.ps}, slot {t % host.ps}): {bad} of {d} O elements "
                                     f"differ")
            assert abs(lg[b, h] - lse_ref[0]) <= LSE_ABS, \
                f"{what}: seq {b} head {h} target {t}: LSE {lg[b, h]} vs {lse_ref[0]}"


def run_decode(fa, pb, q, H, Hkv, d, noalloc=False):
    B = q.shape[0]
    qd = q.to("cuda")
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    ps = pb.k_cache.shape[1]
    if noalloc:
        st = fa.fa_paged_fwd_noalloc(qd, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o, lse, B, H, Hkv, d,
                                     ps, pb.num_pages, pb.block_table.shape[1], pb.max_seqlen, scale, True)
    else:
        ws_bytes = fa.fa_paged_workspace_size(B, H, d, pb.max_seqlen)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        st = fa.fa_paged_fwd(qd, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o, lse, B, H, Hkv, d, ps,
                             pb.num_pages, pb.block_table.shape[1], pb.max_seqlen, scale, True, ws, ws_bytes)
    assert st == fa.FA_OK, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    return o, lse


# Lengths around pages, 128-key blocks and the 512 / 2048-token splits.
EDGE_LENGTHS = [1, 15, 16, 17, 33, 130, 511, 512, 513, 700, 2047, 2048, 2049, 4097, 5000, 0]


@pytest.mark.parametrize("H,Hkv,d", [
    (32, 32, 128),  # CUDA-core split kernel, one head per warp (G = 1)
    (32, 16, 128),  # G = 2
    (32, 8, 128),   # G = 4
    (32, 32, 64),
    (32, 8, 64),
    (32, 4, 128),   # 8 query heads per kv head: tensor-core decode
    (32, 2, 128),   # 16: tensor-core decode
    (32, 1, 64),    # 32: tensor-core decode, d = 64
])
def test_onehot_decode_every_page(fa, H, Hkv, d):
    """Every page of every sequence (one token each, slots stepping through
    0..15) plus the edge positions, over several calls."""
    pb = W.paged_inputs(EDGE_LENGTHS, H, d, 700 + H + Hkv + d, "cuda", Hkv=Hkv, slack_pages=5, k_signs=True)
    host = HostPool(pb)
    _, lists = decode_targets(EDGE_LENGTHS, H, 1, True)
    calls = calls_needed(lists, H)
    tg, _ = decode_targets(EDGE_LENGTHS, H, calls, True)
    covered = [set() for _ in EDGE_LENGTHS]
    for c in range(calls):
        q = build_decode_q(host, EDGE_LENGTHS, tg[c], H, Hkv, d)
        o, lse = run_decode(fa, pb, q, H, Hkv, d)
        check_decode(o, lse, host, q, EDGE_LENGTHS, tg[c], H, Hkv, d, f"H{H}/Hkv{Hkv} d{d} call {c}")
        for b, L in enumerate(EDGE_LENGTHS):
            if L:
                covered[b].update(tg[c][b])
    for b, L in enumerate(EDGE_LENGTHS):
        assert covered[b] == set(lists[b]), f"seq {b}: not every listed position was a target"


@pytest.mark.parametrize("page_size", [32, 64, 128])
@pytest.mark.parametrize("H,Hkv,d", [(32, 32, 128), (32, 8, 64), (32, 2, 128)])
def test_onehot_decode_page_sizes(fa, page_size, H, Hkv, d):
    """Pages of 32, 64 and 128 tokens: every page of every sequence and the
    page, block and split edges, through the CUDA-core split kernel (which
    walks a page in 16-token chunks) and the tensor-core decode (one TMA box
    per page and panel)."""
    pb = W.paged_inputs(EDGE_LENGTHS, H, d, 760 + page_size + Hkv + d, "cuda", Hkv=Hkv, slack_pages=3,
                        k_signs=True, page_size=page_size)
    host = HostPool(pb)
    _, lists = decode_targets(EDGE_LENGTHS, H, 1, True, page_size)
    calls = calls_needed(lists, H)
    tg, _ = decode_targets(EDGE_LENGTHS, H, calls, True, page_size)
    for c in range(calls):
        q = build_decode_q(host, EDGE_LENGTHS, tg[c], H, Hkv, d)
        o, lse = run_decode(fa, pb, q, H, Hkv, d)
        check_decode(o, lse, host, q, EDGE_LENGTHS, tg[c], H, Hkv, d, f"page {page_size} H{H}/Hkv{Hkv} call {c}")


@pytest.mark.parametrize("Hkv", [32, 8, 2])
def test_onehot_decode_full_batch(fa, Hkv):
    """The full decode batch (B64, H32, d128, lengths U[512, 16384], random
    page permutation, the pool drawn on the device) in the launch
    configurations bench.py times: 32 kv heads (one head per warp), 8 (four
    per warp) and 2 (tensor cores).  Each query head aims at a different
    special position of its sequence."""
    lens = W.c5_lengths()
    H, d = 32, 128
    pb = W.paged_inputs(lens, H, d, 1239 + 100 + Hkv, "cuda", Hkv=Hkv, pool_on_device=True, k_signs=True)
    host = HostPool(pb, keep_f64=False, by_page=True)
    host.check_walk(lens)
    tg, _ = decode_targets(lens, H, 1, False)
    q = build_decode_q(host, lens, tg[0], H, Hkv, d)
    o, lse = run_decode(fa, pb, q, H, Hkv, d)
    check_decode(o, lse, host, q, lens, tg[0], H, Hkv, d, f"C5 Hkv{Hkv}")


def test_onehot_decode_noalloc(fa):
    """The allocation-free decode (its own, longer splits) reads the same
    rows: one call over the edge lengths, checked against the oracle."""
    H, Hkv, d = 32, 8, 128
    pb = W.paged_inputs(EDGE_LENGTHS, H, d, 731, "cuda", Hkv=Hkv, slack_pages=5, k_signs=True)
    host = HostPool(pb)
    tg, _ = decode_targets(EDGE_LENGTHS, H, 1, False)
    q = build_decode_q(host, EDGE_LENGTHS, tg[0], H, Hkv, d)
    o, lse = run_decode(fa, pb, q, H, Hkv, d, noalloc=True)
    check_decode(o, lse, host, q, EDGE_LENGTHS, tg[0], H, Hkv, d, "noalloc")


def prefill_targets(Lq, Lk, H, causal):
    """targets[i][h] for query row i (absolute position Lk - Lq + i) of head
    h, such that every key 0 .. Lk-1 is the target of some (row, head).
    Keys are dealt from the last down to the (row, head) pairs from the last
    row down: the n-th key, Lk - 1 - n, goes to row Lq - 1 - n // H, which
    sees it (Lk - 1 - n <= Lk - 1 - n // H).  The pairs left over aim at a
    position derived from the row, always visible."""
    assert Lk <= Lq * H, "more keys than (row, head) pairs"
    tg = [[None] * H for _ in range(Lq)]
    for n in range(Lk):
        i, h = Lq - 1 - n // H, n % H
        t = Lk - 1 - n
        assert not causal or t <= i + Lk - Lq
        tg[i][h] = t
    for i in range(Lq):
        vis = (i + Lk - Lq + 1) if causal else Lk
        for h in range(H):
            if tg[i][h] is None:
                tg[i][h] = (i * 7 + h * 13) % vis
    return tg


@pytest.mark.parametrize("causal,lens_q,lens_k,H,Hkv,d,ps", [
    # whole prompts read through the page table: every key of every sequence
    (False, [1, 16, 17, 128, 129, 300, 1000, 2100], None, 2, 2, 128, 16),
    (True, [1, 16, 17, 128, 129, 300, 1000, 2100], None, 2, 2, 64, 16),
    # continuation chunks (bottom-right causal), grouped kv heads
    (True, [10, 200, 600, 1200, 1100], [40, 700, 2100, 4500, 4097], 4, 2, 128, 16),
    (True, [16, 100, 640], [17, 390, 2500], 4, 4, 64, 16),
    # larger pages: fewer, taller boxes
    (True, [10, 200, 600, 1100], [40, 700, 2100, 4097], 4, 2, 128, 32),
    (True, [10, 200, 600, 1100], [40, 700, 2100, 4097], 4, 2, 128, 64),
    (False, [1, 63, 64, 65, 129, 300, 1000], None, 2, 2, 64, 64),
    (True, [10, 200, 600, 1100], [40, 700, 2100, 4097], 4, 2, 128, 128),
    (True, [1, 127, 128, 129, 300, 1000], None, 2, 1, 64, 128),
])
def test_onehot_paged_prefill(fa, causal, lens_q, lens_k, H, Hkv, d, ps):
    """fa_varlen_paged_fwd (the TMA page boxes of the paged prefill): every
    key of every sequence is the target of some query row.  Unused slots of
    the pool hold NaN, so a stale row read as a key or value also fails."""
    lens_k = lens_q if lens_k is None else lens_k
    cb = W.chunk_inputs(lens_q, lens_k, H, d, 800 + H + d + int(causal) + ps, "cuda", Hkv=Hkv, slack_pages=3,
                        k_signs=True, page_size=ps)
    g = H // Hkv
    a = _alpha(d)
    scale = 1.0 / math.sqrt(d)
    kbits, vbits = _bits(cb.k_cache), _bits(cb.v_cache)
    bt = cb.block_table.cpu().numpy()
    cq = [int(x) for x in cb.cu_q.cpu()]
    total_q = cq[-1]
    q = np.zeros((total_q, H, d))
    seqs = []
    for s, (Lq, Lk) in enumerate(zip(lens_q, lens_k)):
        kb = oracle.gather_paged_kv(kbits, bt[s], Lk, ps)
        vb = oracle.gather_paged_kv(vbits, bt[s], Lk, ps)
        kf = _f64_rows(kb)
        tg = prefill_targets(Lq, Lk, H, causal)
        for i in range(Lq):
            for h in range(H):
                q[cq[s] + i, h] = a * kf[tg[i][h], h // g]
        seqs.append((kb, vb, kf, _f64_rows(vb), tg))
    qt = torch.from_numpy(q).to(torch.bfloat16)
    qd = qt.to("cuda")
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, total_q), float("nan"), dtype=torch.float32, device="cuda")
    st = fa.fa_varlen_paged_fwd(qd, cb.k_cache, cb.v_cache, o, lse, cb.cu_q, cb.cu_k, cb.block_table, len(lens_q),
                                cb.max_q, cb.max_k, total_q, H, Hkv, d, ps, cb.num_pages, cb.block_table.shape[1],
                                scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    ob = _bits(o)
    lg = lse.cpu().numpy().astype(np.float64)
    qf = qt.to(torch.float64).numpy()
    for s, (Lq, Lk) in enumerate(zip(lens_q, lens_k)):
        kb, vb, kf, vf, tg = seqs[s]
        covered = set()
        for h in range(H):
            hk = h // g
            rows = qf[cq[s]:cq[s] + Lq, h]
            O, lse_ref, S, _ = oracle.attention_head(rows, kf[:, hk], vf[:, hk], scale, causal, return_sp=True)
            want = _bf16_bits_of(O)
            for i in range(Lq):
                t = tg[i][h]
                covered.add(t)
                row = S[i].copy()
                row[t] = -np.inf
                gap = S[i, t] - row.max()
                assert gap >= MIN_GAP, f"precondition: seq {s} row {i} head {h}: gap {gap:.1f}"
                assert _same_row(vb[t, hk], want[i], vb[t, hk]), f"precondition: oracle O of row {i} is not v[{t}]"
            got = ob[cq[s]:cq[s] + Lq, h]
            bad_rows = np.array([i for i in range(Lq) if not _same_row(got[i], want[i], vb[tg[i][h], hk])],
                                dtype=np.int64)
            if bad_rows.size:
                i = int(bad_rows[0])
                t = tg[i][h]
                raise AssertionError(f"seq {s} (Lq={Lq}, Lk={Lk}) head {h}: {bad_rows.size} rows differ; first row "
                                     f"{i} aims at key {t} (page entry {t // ps}, slot {t % ps}, block {t // 128})")
            dl = np.abs(lg[h, cq[s]:cq[s] + Lq] - lse_ref)
            assert dl.max() <= LSE_ABS, f"seq {s} head {h}: LSE max-abs {dl.max():.3e}"
        assert covered == set(range(Lk)), f"seq {s}: some keys were never a target"


@pytest.mark.parametrize("causal", [False, True])
def test_onehot_varlen_contiguous(fa, causal):
    """The same check on the contiguous varlen prefill (128-row TMA tiles,
    ragged tails): every key of every sequence is some row's target."""
    lens = [1, 127, 128, 129, 255, 1000, 2049]
    H, d = 2, 128
    q0, k, v, cq_t, ck_t = W.varlen_inputs(lens, H, d, 901 + int(causal), "cpu")
    k = W.sign_bf16(tuple(k.shape), 902 + int(causal))
    a = _alpha(d)
    scale = 1.0 / math.sqrt(d)
    cq = [int(x) for x in cq_t]
    kf = k.to(torch.float64).numpy()
    vf = v.to(torch.float64).numpy()
    vb = _bits(v)
    q = np.zeros(tuple(q0.shape))
    tgs = []
    for s, L in enumerate(lens):
        tg = prefill_targets(L, L, H, causal)
        tgs.append(tg)
        for i in range(L):
            for h in range(H):
                q[cq[s] + i, h] = a * kf[cq[s] + tg[i][h], h]
    qt = torch.from_numpy(q).to(torch.bfloat16)
    total = cq[-1]
    o = torch.full((total, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, total), float("nan"), dtype=torch.float32, device="cuda")
    st = fa.fa_varlen_fwd(qt.to("cuda"), k.to("cuda"), v.to("cuda"), o, lse, cq_t.to("cuda"), ck_t.to("cuda"),
                          len(lens), max(lens), max(lens), total, total, H, H, d, scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    ob = _bits(o)
    qf = qt.to(torch.float64).numpy()
    for s, L in enumerate(lens):
        a0 = cq[s]
        for h in range(H):
            O, _, S, _ = oracle.attention_head(qf[a0:a0 + L, h], kf[a0:a0 + L, h], vf[a0:a0 + L, h], scale, causal,
                                               return_sp=True)
            want = _bf16_bits_of(O)
            for i in range(L):
                t = tgs[s][i][h]
                row = S[i].copy()
                row[t] = -np.inf
                assert S[i, t] - row.max() >= MIN_GAP
                assert _same_row(vb[a0 + t, h], want[i], vb[a0 + t, h])
            bad = [i for i in range(L) if not _same_row(ob[a0 + i, h], want[i], vb[a0 + tgs[s][i][h], h])]
            assert not bad, f"seq {s} head {h}: {len(bad)} rows differ, first {bad[0]}"
