"""Benchmark: exact attention forward on GB300 through the C-ABI.

One step = the whole hot path on the headline workloads, inputs resident in
device memory:
  1. dense prefill, B1 H32 N8192 d128, non-causal        (fa_fwd)
  2. the same, causal                                    (fa_fwd)
  3. packed varlen prefill, 16 sequences of U[128,4096]
     tokens, H32 d64, causal                             (fa_varlen_fwd)
  4. paged decode, B64 H32 d128, KV lengths U[512,16384],
     16-token pages in a random permutation              (fa_paged_fwd)
`value` is the prefill throughput in TFLOP/s (4 N^2 d per head, halved for
causal) over legs 1-2; leg 3 is reported in TFLOP/s (same convention, per
sequence) and leg 4 in GB/s of algorithmic bytes (every cached K/V byte
once, plus q, o, lse and the block_table).
L2 is flushed before every step: a 256 MiB buffer is written, then a second
256 MiB buffer is read, so that the step starts with none of its inputs in
L2 and without the flush's dirty lines still to write back (which would
otherwise land in the timed region as extra HBM traffic).  The decode pool
(~8.9 GB) is far larger than L2 anyway.

--impl reference times the float64 CPU oracle (a deliberately slow program)
on a bounded sample of the same workload instead.

For N > 1 (torchrun) each rank runs the same workload on its own GPU
(replicas: the forward has no exchange step); timings are max-reduced and
`value` counts the work of all ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % BF16 peak (N=8192,d=128); paged-decode KV GB/s"
C3 = dict(B=1, H=32, N=8192, d=128)
C5 = dict(B=64, H=32, d=128)
SEED_C3 = 1236
SEED_C4 = 1238
SEED_C5 = 1239
SEED_CHUNK = 1240
SEED_C1 = 1234
SEED_C2 = 1235
C1 = dict(B=1, H=1, N=256, d=64)
C2 = dict(B=4, H=16, N=2048, d=128)
WORKLOAD = ("dense prefill B1 H32 N8192 d128 non-causal + causal (fa_fwd), packed varlen prefill 16 x U[128,4096] "
            "tokens H32 d64 causal (fa_varlen_fwd), then paged decode B64 H32 d128, KV lengths uniform in "
            "[512,16384], 16-token pages in a seeded random permutation (fa_paged_fwd); then a prefix-cache "
            "continuation chunk, 16 sequences with cached context U[512,8192] + new tokens U[256,2048], H32 d128 "
            "causal: store the new K/V (fa_store_kvcache), attend through the page table (fa_varlen_paged_fwd), "
            "and the same shapes with contiguous K/V (fa_varlen_fwd) for comparison; then the dense N8192 non-causal "
            "prefill from one packed [B,N,3,H,d] QKV tensor (fa_qkvpacked_fwd)")
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# ncu captures of the current kernels: for prefill the mean of the N=8192
# non-causal and causal launches; for decode a 16-sequence capture scaled by
# cached tokens to the 64-sequence launch.  Set to None whenever a kernel
# changes after its capture.
PREFILL_TRAFFIC_BYTES = 251.3e6
DECODE_TRAFFIC_BYTES = 9.32e9


def prefill_flops(N, d, H, B, causal):
    f = 4.0 * N * N * d * H * B
    return f / 2 if causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    """The slowest rank's value (timing is max-reduced over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput of `world` replicas that each did flops_per_rank
    in at most ms_max milliseconds (weak scaling: the work grows with N)."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------------- oracle

_C3_HOST = {}


def run_cpu_oracle_sample(step: int, rows: int = 256):
    """The float64 oracle on `rows` query rows of one head of the headline
    prefill, non-causal and causal.  Returns (seconds, flops)."""
    import numpy as np

    import oracle
    from exact_tiled_attention_fwd_gb300 import workloads as W

    B, H, N, d = C3["B"], C3["H"], C3["N"], C3["d"]
    if not _C3_HOST:
        _C3_HOST["qkv"] = W.dense_inputs(B, N, H, d, SEED_C3, "cpu")
    q, k, v = _C3_HOST["qkv"]
    h = step % H
    rng = np.random.default_rng(step)
    sel = np.sort(rng.choice(N, size=rows, replace=False))
    qh = q[0, sel, h].float().numpy().astype(np.float64)
    kh = k[0, :, h].float().numpy().astype(np.float64)
    vh = v[0, :, h].float().numpy().astype(np.float64)
    scale = 1.0 / math.sqrt(d)
    t0 = time.perf_counter()
    oracle.attention_rows(qh, kh, vh, scale, False, rows=sel, Lq=N)
    oracle.attention_rows(qh, kh, vh, scale, True, rows=sel, Lq=N)
    dt = time.perf_counter() - t0
    flops = 4.0 * rows * N * d + 4.0 * float((sel + 1).sum()) * d
    return dt, flops


def cpu_baseline(budget_s: float = 20.0):
    secs, flops, n = 0.0, 0.0, 0
    while secs < budget_s and n < 2000:
        dt, f = run_cpu_oracle_sample(n)
        secs += dt
        flops += f
        n += 1
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} x 256 query rows of one head of the N=8192 d=128 prefill, non-causal and causal, "
                      f"float64 numpy (BLAS default threads), {secs:.1f} s of CPU work"}


def oracle_c1():
    """The float64 oracle on the whole single-head case (B1 H1 N256 d64)."""
    import numpy as np

    import oracle
    from exact_tiled_attention_fwd_gb300 import workloads as W

    q, k, v = W.dense_inputs(C1["B"], C1["N"], C1["H"], C1["d"], SEED_C1, "cpu")
    qh, kh, vh = (t[0, :, 0].float().numpy().astype(np.float64) for t in (q, k, v))
    ts = []
    for _ in range(5):
        t0 = time.perf_counter()
        oracle.attention_head(qh, kh, vh, 1.0 / math.sqrt(C1["d"]), False)
        ts.append(time.perf_counter() - t0)
    return {"us": statistics.median(ts) * 1e6, "sample": "the whole case, median of 5 runs", "cores": os.cpu_count()}


def oracle_c2_sample():
    """The float64 oracle on one whole head of the B4 H16 N2048 d128 prefill,
    non-causal and causal."""
    import numpy as np

    import oracle
    from exact_tiled_attention_fwd_gb300 import workloads as W

    q, k, v = W.dense_inputs(C2["B"], C2["N"], C2["H"], C2["d"], SEED_C2, "cpu")
    qh, kh, vh = (t[0, :, 0].float().numpy().astype(np.float64) for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.attention_head(qh, kh, vh, 1.0 / math.sqrt(C2["d"]), False)
    oracle.attention_head(qh, kh, vh, 1.0 / math.sqrt(C2["d"]), True)
    dt = time.perf_counter() - t0
    f = 4.0 * C2["N"] ** 2 * C2["d"] * 1.5
    return {"tflops": f / dt / 1e12, "s": dt, "sample": "head 0 of sequence 0, non-causal + causal",
            "cores": os.cpu_count()}


def reference_arm(args, world, rank):
    """--impl reference: the float64 oracle on the host cores."""
    if rank != 0:
        return
    for s in range(args.warmup):
        run_cpu_oracle_sample(10_000 + s)
    secs, flops = 0.0, 0.0
    for s in range(args.steps):
        dt, f = run_cpu_oracle_sample(s)
        secs += dt
        flops += f
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "each step: 256 query rows of one head, non-causal + causal"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "256 query rows of one head of the N=8192 d=128 prefill per step, "
                                   "non-causal and causal, float64 numpy"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours

def ours(args, world, rank, local):
    import torch

    import exact_tiled_attention_fwd_gb300 as F
    from exact_tiled_attention_fwd_gb300 import _build
    from exact_tiled_attention_fwd_gb300 import workloads as W

    _build.build()
    F.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    B, H, N, d = C3["B"], C3["H"], C3["N"], C3["d"]
    scale = 1.0 / math.sqrt(d)
    do_prefill = args.case in ("all", "prefill")
    do_varlen = args.case in ("all", "varlen")
    do_decode = args.case in ("all", "decode")
    do_chunk = args.case in ("all", "chunk")
    do_packed = args.case in ("all", "packed")
    do_bwd = args.case in ("all", "backward")
    do_small = args.case in ("all", "small")
    q, k, v = W.dense_inputs(B, N, H, d, SEED_C3, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    vl = W.c4_lengths() if do_varlen else [128]
    vH, vd = 32, 64
    vq, vk, vv, vcq, vck = W.varlen_inputs(vl, vH, vd, SEED_C4, dev)
    vo = torch.empty_like(vq)
    vlse = torch.empty((vH, vq.shape[0]), dtype=torch.float32, device=dev)
    lens = W.c5_lengths()[: args.decode_batch] if do_decode else [16]
    hkv5 = args.decode_hkv
    pb = W.paged_inputs(lens, C5["H"], C5["d"], SEED_C5, dev, Hkv=hkv5, pool_on_device=True)
    B5, H5, d5 = len(lens), C5["H"], C5["d"]
    o5 = torch.empty_like(pb.q)
    l5 = torch.empty((B5, H5), dtype=torch.float32, device=dev)
    ws_bytes = F.fa_paged_workspace_size(B5, H5, d5, pb.max_seqlen)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink[0])
    maxp = pb.block_table.shape[1]
    # prefix-cache continuation: store this chunk's K/V, then attend through
    # the page table; the same shapes through the contiguous varlen call are
    # timed beside it (the cost of paging)
    cl_q, cl_k = W.chunk_lengths(SEED_CHUNK) if do_chunk else ([16], [16])
    cH, cd = W.CHUNK["H"], W.CHUNK["d"]
    cb = W.chunk_inputs(cl_q, cl_k, cH, cd, SEED_CHUNK, dev, stale=0.0, pool_on_device=True)
    c_tq = int(cb.cu_q[-1])
    co = torch.empty((c_tq, cH, cd), dtype=torch.bfloat16, device=dev)
    clse = torch.empty((cH, c_tq), dtype=torch.float32, device=dev)
    cbt_h = cb.block_table.cpu()
    new_k = W.randn_bf16_device((c_tq, cH, cd), SEED_CHUNK * 5 + 1, dev)
    new_v = W.randn_bf16_device((c_tq, cH, cd), SEED_CHUNK * 5 + 2, dev)
    slots = []
    for s_, (lq_, lk_) in enumerate(zip(cl_q, cl_k)):
        slots += [int(cbt_h[s_, t // 16]) * 16 + t % 16 for t in range(lk_ - lq_, lk_)]
    c_slots = torch.tensor(slots, dtype=torch.int32, device=dev)
    # contiguous copies of every sequence's keys for the comparison leg
    ck_rows = torch.tensor([int(cbt_h[s_, t // 16]) * 16 + t % 16 for s_, lk_ in enumerate(cl_k) for t in range(lk_)],
                           dtype=torch.int64, device=dev)
    c_kc = cb.k_cache.view(-1, cH, cd)[ck_rows].contiguous()
    c_vc = cb.v_cache.view(-1, cH, cd)[ck_rows].contiguous()
    # the same chunk in a pool of 64-token pages (fewer, taller TMA boxes)
    cb64 = W.chunk_inputs(cl_q, cl_k, cH, cd, SEED_CHUNK + 64, dev, stale=0.0, pool_on_device=True, page_size=64)

    def prefill(causal):
        if not do_prefill:
            return
        st = F.fa_fwd(q, k, v, o, lse, B, H, H, N, d, scale, causal, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_fwd")

    def varlen():
        if not do_varlen:
            return
        st = F.fa_varlen_fwd(vq, vk, vv, vo, vlse, vcq, vck, len(vl), max(vl), max(vl), vq.shape[0], vk.shape[0],
                             vH, vH, vd, 1.0 / math.sqrt(vd), True, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_varlen_fwd")

    def decode():
        if not do_decode:
            return
        st = F.fa_paged_fwd(pb.q, pb.k_cache, pb.v_cache, pb.block_table, pb.seqlens, o5, l5, B5, H5, hkv5, d5, 16,
                            pb.num_pages, maxp, pb.max_seqlen, 1.0 / math.sqrt(d5), True, ws, ws_bytes, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_paged_fwd")

    qkv = torch.stack([q, k, v], dim=2).contiguous() if do_packed else q
    o_p = torch.empty_like(o)
    lse_p = torch.empty_like(lse)

    def packed():
        if not do_packed:
            return
        st = F.fa_qkvpacked_fwd(qkv, o_p, lse_p, B, H, N, d, scale, False, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_qkvpacked_fwd")

    # backward on the prefill shape: dO drawn once, O and LSE from the forward
    if do_bwd:
        dout = W.randn_bf16_device((B, N, H, d), SEED_C3 * 7 + 1, dev)
        bo_nc, bl_nc = F.attention(q, k, v, scale=scale, causal=False)
        bo_c, bl_c = F.attention(q, k, v, scale=scale, causal=True)
        g_q, g_k, g_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws_bytes = F.fa_bwd_workspace_bytes(B, B * N, H)
        bws = torch.empty(bws_bytes, dtype=torch.uint8, device=dev)

    def backward(causal):
        if not do_bwd:
            return
        bo, bl = (bo_c, bl_c) if causal else (bo_nc, bl_nc)
        st = F.fa_bwd(q, k, v, bo, bl, dout, g_q, g_k, g_v, bws, bws_bytes, B, H, H, N, d, scale, causal, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_bwd")

    # grouped-query decode on the same lengths: 8 kv heads (4 query heads per
    # kv head, the CUDA-core split kernel) and 2 kv heads (16 per kv head,
    # the tensor-core decode)
    do_gqa = args.case == "all"
    gqa = {}
    if do_gqa:
        for hkv_g in (8, 2):
            pg_ = W.paged_inputs(lens, C5["H"], C5["d"], SEED_C5 + hkv_g, dev, Hkv=hkv_g, pool_on_device=True)
            gws = F.fa_paged_workspace_size(B5, H5, d5, pg_.max_seqlen)
            gqa[hkv_g] = (pg_, torch.empty_like(pg_.q), torch.empty((B5, H5), dtype=torch.float32, device=dev),
                          torch.empty(gws, dtype=torch.uint8, device=dev), gws)

    def decode_gqa(hkv_g):
        if not do_gqa:
            return
        pg_, go, gl, gws_t, gws = gqa[hkv_g]
        st = F.fa_paged_fwd(pg_.q, pg_.k_cache, pg_.v_cache, pg_.block_table, pg_.seqlens, go, gl, B5, H5, hkv_g,
                            d5, 16, pg_.num_pages, pg_.block_table.shape[1], pg_.max_seqlen, 1.0 / math.sqrt(d5),
                            True, gws_t, gws, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_paged_fwd (grouped)")

    def store():
        if not do_chunk:
            return
        st = F.fa_store_kvcache(new_k, new_v, cb.k_cache, cb.v_cache, c_slots, c_tq, cH, cd, 16, cb.num_pages, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_store_kvcache")

    def chunk():
        if not do_chunk:
            return
        st = F.fa_varlen_paged_fwd(cb.q, cb.k_cache, cb.v_cache, co, clse, cb.cu_q, cb.cu_k, cb.block_table,
                                   len(cl_q), cb.max_q, cb.max_k, c_tq, cH, cH, cd, 16, cb.num_pages,
                                   cb.block_table.shape[1], 1.0 / math.sqrt(cd), True, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_varlen_paged_fwd")

    def chunk_page64():
        if not do_chunk:
            return
        st = F.fa_varlen_paged_fwd(cb64.q, cb64.k_cache, cb64.v_cache, co, clse, cb64.cu_q, cb64.cu_k,
                                   cb64.block_table, len(cl_q), cb64.max_q, cb64.max_k, c_tq, cH, cH, cd, 64,
                                   cb64.num_pages, cb64.block_table.shape[1], 1.0 / math.sqrt(cd), True, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_varlen_paged_fwd (64-token pages)")

    def chunk_contiguous():
        if not do_chunk:
            return
        st = F.fa_varlen_fwd(cb.q, c_kc, c_vc, co, clse, cb.cu_q, cb.cu_k, len(cl_q), cb.max_q, cb.max_k, c_tq,
                             c_kc.shape[0], cH, cH, cd, 1.0 / math.sqrt(cd), True, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_varlen_fwd (contiguous chunk)")

    # the single-head case (B1 H1 N256 d64, non-causal) and the batched MHA
    # prefill (B4 H16 N2048 d128, non-causal and causal)
    q1, k1, v1 = W.dense_inputs(C1["B"], C1["N"], C1["H"], C1["d"], SEED_C1, dev)
    o1 = torch.empty_like(q1)
    l1 = torch.empty((C1["B"], C1["H"], C1["N"]), dtype=torch.float32, device=dev)
    q2, k2, v2 = W.dense_inputs(C2["B"], C2["N"], C2["H"], C2["d"], SEED_C2, dev) if do_small else (q1, k1, v1)
    o2 = torch.empty_like(q2)
    l2 = torch.empty((q2.shape[0], q2.shape[2], q2.shape[1]), dtype=torch.float32, device=dev)

    def small_c1():
        if not do_small:
            return
        st = F.fa_fwd(q1, k1, v1, o1, l1, C1["B"], C1["H"], C1["H"], C1["N"], C1["d"], 1.0 / math.sqrt(C1["d"]),
                      False, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_fwd (B1 H1 N256 d64)")

    def small_c2(causal):
        if not do_small:
            return
        st = F.fa_fwd(q2, k2, v2, o2, l2, C2["B"], C2["H"], C2["H"], C2["N"], C2["d"], 1.0 / math.sqrt(C2["d"]),
                      causal, sp)
        if st != F.FA_OK:
            raise F.FAError(st, "fa_fwd (B4 H16 N2048 d128)")

    for _ in range(args.warmup):
        flush_l2()
        small_c1()
        small_c2(False)
        small_c2(True)
        prefill(False)
        prefill(True)
        varlen()
        decode()
        store()
        chunk()
        chunk_page64()
        chunk_contiguous()
        packed()
        backward(False)
        backward(True)
        decode_gqa(8)
        decode_gqa(2)
    torch.cuda.synchronize()
    st = F.fa_device_status(sp)
    if st != F.FA_OK:
        raise F.FAError(st, "warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)
    wall0 = time.perf_counter()
    for s in range(K):
        flush_l2()
        e = ev[s]
        e[0].record(stream)
        prefill(False)
        e[1].record(stream)
        prefill(True)
        e[2].record(stream)
        varlen()
        e[3].record(stream)
        decode()
        e[4].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()
    # The legs of the follow-up entry points (store, paged chunk, its
    # contiguous twin, packed QKV) are timed in a loop of their own after
    # the main one, so that their power draw does not change the clocks the
    # main legs run at.
    K2 = min(K, 100)
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(K2)]
    for s in range(K2):
        flush_l2()
        e = ev2[s]
        e[0].record(stream)
        store()
        e[1].record(stream)
        chunk()
        e[2].record(stream)
        chunk_contiguous()
        e[3].record(stream)
        packed()
        e[4].record(stream)
        flush_l2()
        e[5].record(stream)
        backward(False)
        e[6].record(stream)
        flush_l2()
        e[7].record(stream)
        chunk_page64()
        e[8].record(stream)
    # the causal backward and the grouped decodes in a pass of their own (a
    # flush sits between the legs)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K2)]
    for s in range(K2):
        flush_l2()
        ev3[s][0].record(stream)
        backward(True)
        ev3[s][1].record(stream)
        flush_l2()
        ev3[s][2].record(stream)
        decode_gqa(8)
        ev3[s][3].record(stream)
        flush_l2()
        ev3[s][4].record(stream)
        decode_gqa(2)
        ev3[s][5].record(stream)
    # the two small configurations in a pass of their own: C1 call by call
    # (its latency, the median of at least 20 calls), C2 with a flush
    # before each leg
    n1 = max(20, K2)
    ev1 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n1)]
    for s in range(n1):
        flush_l2()
        ev1[s][0].record(stream)
        small_c1()
        ev1[s][1].record(stream)
    ev4 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K2)]
    for s in range(K2):
        flush_l2()
        ev4[s][0].record(stream)
        small_c2(False)
        ev4[s][1].record(stream)
        flush_l2()
        ev4[s][2].record(stream)
        small_c2(True)
        ev4[s][3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    st = F.fa_device_status(sp)
    if st != F.FA_OK:
        raise F.FAError(st, "timed region")
    t_c1 = statistics.median(e[0].elapsed_time(e[1]) for e in ev1)
    t_c2 = sum(e[0].elapsed_time(e[1]) for e in ev4) / K2
    t_c2c = sum(e[2].elapsed_time(e[3]) for e in ev4) / K2
    t_c1, t_c2, t_c2c = (max_over_ranks(world, x) for x in (t_c1, t_c2, t_c2c))

    t_nc = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    t_c = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    t_var = sum(e[2].elapsed_time(e[3]) for e in ev) / K
    t_dec = sum(e[3].elapsed_time(e[4]) for e in ev) / K
    t_store = sum(e[0].elapsed_time(e[1]) for e in ev2) / K2
    t_chunk = sum(e[1].elapsed_time(e[2]) for e in ev2) / K2
    t_chunk_c = sum(e[2].elapsed_time(e[3]) for e in ev2) / K2
    t_packed = sum(e[3].elapsed_time(e[4]) for e in ev2) / K2
    t_bnc = sum(e[5].elapsed_time(e[6]) for e in ev2) / K2
    t_chunk64 = max_over_ranks(world, sum(e[7].elapsed_time(e[8]) for e in ev2) / K2)
    t_bc = sum(e[0].elapsed_time(e[1]) for e in ev3) / K2
    t_g8 = sum(e[2].elapsed_time(e[3]) for e in ev3) / K2
    t_g2 = sum(e[4].elapsed_time(e[5]) for e in ev3) / K2
    t_nc, t_c, t_var, t_dec, t_store, t_chunk, t_chunk_c, t_packed, t_bnc, t_bc, t_g8, t_g2 = (
        max_over_ranks(world, x)
        for x in (t_nc, t_c, t_var, t_dec, t_store, t_chunk, t_chunk_c, t_packed, t_bnc, t_bc, t_g8, t_g2))
    # continuation FLOPs, causal bottom-right, halved-square convention of
    # the varlen leg: 4 d H (Lq (Lk - Lq) + Lq^2 / 2) per sequence
    f_chunk = sum(4.0 * cd * cH * (lq_ * (lk_ - lq_) + lq_ * lq_ / 2) for lq_, lk_ in zip(cl_q, cl_k))
    store_bytes = 2.0 * 2 * c_tq * cH * cd * 2 + c_tq * 4  # K and V read + written, slot map
    f_var = sum(4.0 * L * L * vd * vH / 2 for L in vl)
    var_tflops = f_var / (t_var * 1e-3) / 1e12 if do_varlen else None
    f_nc = prefill_flops(N, d, H, B, False)
    f_c = prefill_flops(N, d, H, B, True)
    tflops = job_tflops(1, f_nc + f_c, t_nc + t_c)  # per replica; the job value multiplies by world
    kv_bytes = float(sum(lens)) * hkv5 * d5 * 2 * 2
    dec_bytes = kv_bytes + 2 * B5 * H5 * d5 * 2 + B5 * H5 * 4 + sum((L + 15) // 16 for L in lens) * 4
    gbs = dec_bytes / (t_dec * 1e-3) / 1e9
    peak_tf, peak_gbs, peak_src = load_peaks()

    def gqa_leg(hkv_g, t):
        # unique K/V bytes of the kv heads, plus q, o, LSE and table entries
        b_ = (float(sum(lens)) * hkv_g * d5 * 2 * 2 + 2 * B5 * H5 * d5 * 2 + B5 * H5 * 4
              + sum((L + 15) // 16 for L in lens) * 4)
        g_ = b_ / (t * 1e-3) / 1e9
        return {"ms": t, "gbs": g_, "frac_hbm": g_ / peak_gbs, "kv_heads": hkv_g, "query_heads_per_kv_head": H5 // hkv_g,
                "path": "cuda cores" if H5 // hkv_g < 8 else "tensor cores"}

    f_c1 = prefill_flops(C1["N"], C1["d"], C1["H"], C1["B"], False)
    f_c2 = prefill_flops(C2["N"], C2["d"], C2["H"], C2["B"], False)
    f_c2c = prefill_flops(C2["N"], C2["d"], C2["H"], C2["B"], True)
    if args.case != "all":
        if rank == 0:
            print(json.dumps({"case": args.case, "prefill_ms": [t_nc, t_c], "varlen_ms": t_var, "decode_ms": t_dec,
                              "c1_us": t_c1 * 1e3, "c2_ms": [t_c2, t_c2c],
                              "prefill_tflops": tflops if do_prefill else None, "varlen_tflops": var_tflops,
                              "decode_gbs": gbs if do_decode else None,
                              "chunk_ms": [t_store, t_chunk, t_chunk_c, t_chunk64],
                              "chunk_tflops": f_chunk / (t_chunk * 1e-3) / 1e12 if do_chunk else None,
                              "chunk_contiguous_tflops": f_chunk / (t_chunk_c * 1e-3) / 1e12 if do_chunk else None,
                              "store_gbs": store_bytes / (t_store * 1e-3) / 1e9 if do_chunk else None,
                              "qkvpacked_ms": t_packed,
                              "backward_ms": [t_bnc, t_bc],
                              "backward_tflops": [2.5 * f_nc / (t_bnc * 1e-3) / 1e12,
                                                  2.5 * f_c / (t_bc * 1e-3) / 1e12] if do_bwd else None}),
              flush=True)
        return

    # ---- end to end through the public API with pinned host buffers.  Each
    # step copies its q, k, v in, runs both prefill legs and copies O and LSE
    # of both back.  Steps are double-buffered over three streams (copy in,
    # compute, copy out), as a serving loop runs them, so one step's copies
    # overlap its neighbours' compute; every step still moves all of its bytes.
    E = max(4, min(K, 30))
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    bufs = []
    for _ in range(2):
        bufs.append({
            "q": torch.empty_like(q), "k": torch.empty_like(k), "v": torch.empty_like(v),
            "o": torch.empty_like(o), "l": torch.empty_like(lse), "oc": torch.empty_like(o), "lc": torch.empty_like(lse),
            "ho": torch.empty(o.shape, dtype=o.dtype).pin_memory(), "hl": torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
            "hoc": torch.empty(o.shape, dtype=o.dtype).pin_memory(), "hlc": torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
            "in": torch.cuda.Event(), "cmp": torch.cuda.Event(), "out": torch.cuda.Event(),
        })

    def e2e_step(i):
        bf = bufs[i % 2]
        s_in.wait_event(bf["cmp"])  # the buffer's previous compute has read its inputs
        with torch.cuda.stream(s_in):
            bf["q"].copy_(hq, non_blocking=True)
            bf["k"].copy_(hk, non_blocking=True)
            bf["v"].copy_(hv, non_blocking=True)
            bf["in"].record(s_in)
        stream.wait_event(bf["in"])
        stream.wait_event(bf["out"])  # the buffer's previous results have been copied out
        st1 = F.fa_fwd(bf["q"], bf["k"], bf["v"], bf["o"], bf["l"], B, H, H, N, d, scale, False, sp)
        st2 = F.fa_fwd(bf["q"], bf["k"], bf["v"], bf["oc"], bf["lc"], B, H, H, N, d, scale, True, sp)
        bf["cmp"].record(stream)
        s_out.wait_event(bf["cmp"])
        with torch.cuda.stream(s_out):
            bf["ho"].copy_(bf["o"], non_blocking=True)
            bf["hl"].copy_(bf["l"], non_blocking=True)
            bf["hoc"].copy_(bf["oc"], non_blocking=True)
            bf["hlc"].copy_(bf["lc"], non_blocking=True)
            bf["out"].record(s_out)
        if st1 or st2:
            raise F.FAError(st1 or st2, "fa_fwd (e2e)")

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(E):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(world, e0.elapsed_time(e1) / E)
    h2d = 3 * q.numel() * q.element_size()
    d2h = 2 * (o.numel() * o.element_size() + lse.numel() * lse.element_size())
    e2e_tflops = (f_nc + f_c) / (t_e2e * 1e-3) / 1e12

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": job_tflops(world, f_nc + f_c, t_nc + t_c),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": t_nc + t_c + t_var + t_dec,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every step: 256 MiB written, then 256 MiB read (no dirty flush lines left); decode pool 8.9 GB > L2",
                   "value_is": "prefill FLOPs / prefill time (legs 1-2), summed over ranks"},
        "pct_bf16_peak": tflops / peak_tf,
        "legs": {
            "prefill_noncausal": {"ms": t_nc, "tflops": f_nc / (t_nc * 1e-3) / 1e12},
            "prefill_causal": {"ms": t_c, "tflops": f_c / (t_c * 1e-3) / 1e12},
            "varlen_causal_d64": {"ms": t_var, "tflops": var_tflops, "frac_bf16_peak": var_tflops / peak_tf,
                                  "tokens": int(sum(vl))},
            "paged_decode": {"ms": t_dec, "gbs": gbs, "frac_hbm": gbs / peak_gbs, "kv_tokens": int(sum(lens))},
            "store_kvcache": {"ms": t_store, "gbs": store_bytes / (t_store * 1e-3) / 1e9,
                              "frac_hbm": store_bytes / (t_store * 1e-3) / 1e9 / peak_gbs, "tokens": c_tq},
            "paged_prefill_chunk": {"ms": t_chunk, "tflops": f_chunk / (t_chunk * 1e-3) / 1e12,
                                    "frac_bf16_peak": f_chunk / (t_chunk * 1e-3) / 1e12 / peak_tf,
                                    "new_tokens": c_tq, "cached_plus_new_tokens": int(sum(cl_k))},
            "paged_prefill_chunk_page64": {"ms": t_chunk64, "tflops": f_chunk / (t_chunk64 * 1e-3) / 1e12,
                                           "frac_bf16_peak": f_chunk / (t_chunk64 * 1e-3) / 1e12 / peak_tf,
                                           "vs_contiguous": t_chunk64 / t_chunk_c},
            "same_chunk_contiguous_kv": {"ms": t_chunk_c, "tflops": f_chunk / (t_chunk_c * 1e-3) / 1e12},
            "qkvpacked_noncausal": {"ms": t_packed, "tflops": f_nc / (t_packed * 1e-3) / 1e12,
                                    "frac_bf16_peak": f_nc / (t_packed * 1e-3) / 1e12 / peak_tf},
            # backward FLOPs by the usual count of 5 products (2.5x the
            # forward's); the kernels execute 7 (S and dP in both kernels)
            "backward_noncausal": {"ms": t_bnc, "tflops": 2.5 * f_nc / (t_bnc * 1e-3) / 1e12,
                                   "tflops_executed": 3.5 * f_nc / (t_bnc * 1e-3) / 1e12,
                                   "frac_bf16_peak_executed": 3.5 * f_nc / (t_bnc * 1e-3) / 1e12 / peak_tf},
            "backward_causal": {"ms": t_bc, "tflops": 2.5 * f_c / (t_bc * 1e-3) / 1e12,
                                "tflops_executed": 3.5 * f_c / (t_bc * 1e-3) / 1e12,
                                "frac_bf16_peak_executed": 3.5 * f_c / (t_bc * 1e-3) / 1e12 / peak_tf},
            "paged_decode_gqa_8kv": gqa_leg(8, t_g8),
            "paged_decode_gqa_2kv": gqa_leg(2, t_g2),
            "c1_single_head_B1H1N256d64": {"us": t_c1 * 1e3, "tflops": f_c1 / (t_c1 * 1e-3) / 1e12,
                                           "what": f"median of {n1} calls, each timed alone after an L2 flush; "
                                                   "latency-bound (16.8 MFLOP)"},
            "c2_noncausal_B4H16N2048d128": {"ms": t_c2, "tflops": f_c2 / (t_c2 * 1e-3) / 1e12,
                                            "frac_bf16_peak": f_c2 / (t_c2 * 1e-3) / 1e12 / peak_tf},
            "c2_causal_B4H16N2048d128": {"ms": t_c2c, "tflops": f_c2c / (t_c2c * 1e-3) / 1e12,
                                         "frac_bf16_peak": f_c2c / (t_c2c * 1e-3) / 1e12 / peak_tf},
        },
        "roofline": {"kernel": "prefill_kernel<128>", "bound": "tensor", "achieved": tflops, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": tflops / peak_tf, "traffic": PREFILL_TRAFFIC_BYTES,
                     "peak_source": f"{peak_src} bf16 dense (burst)"},
        "decode_roofline": {"kernel": "decode_split_kernel<128> + decode_combine_kernel<128>", "bound": "hbm",
                            "achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
                            "traffic": DECODE_TRAFFIC_BYTES, "peak_source": f"{peak_src} HBM copy"},
        "e2e": {"value": e2e_tflops * world, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "what": "prefill legs with q,k,v copied from pinned host memory and O, LSE copied back each step; "
                        "steps double-buffered over copy-in, compute and copy-out streams"},
        # main step: 2 prefill + varlen + decode split and combine; follow-ups:
        # store, chunk, contiguous twin, packed, 64-token chunk; two backwards of
        # 3 kernels; grouped decodes (CUDA-core split + combine, tensor-core
        # plan + decode + combine); C1; C2 non-causal and causal
        "gpu_launches": 5 * K + 5 * K2 + 6 * K2 + 5 * K2 + n1 + 2 * K2,
        "follow_up_legs": f"store_kvcache, paged_prefill_chunk (16- and 64-token pages), same_chunk_contiguous_kv, "
                          f"qkvpacked_noncausal, "
                          f"backward_(non)causal, paged_decode_gqa_8kv / _2kv and the C2 legs: {K2} steps of their "
                          f"own after the main timed loop, C1: {n1} calls; none in ms_per_step or value",
        "clocks": clk,
        "wall_s_timed": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_budget)
        line["legs"]["c1_single_head_B1H1N256d64"]["oracle"] = oracle_c1()
        line["legs"]["c2_noncausal_B4H16N2048d128"]["oracle"] = oracle_c2_sample()
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--case", choices=["all", "prefill", "varlen", "decode", "chunk", "packed", "backward", "small"],
                    default="all",
                    help="run only one leg (for profiling); prints a short line instead of the bench line")
    ap.add_argument("--decode-batch", type=int, default=64, help="sequences of the decode leg (profiling)")
    ap.add_argument("--decode-hkv", type=int, default=32,
                    help="kv heads of the decode leg (32 = plain multi-head; fewer = grouped queries, profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        reference_arm(args, world, rank)
        return
    world, rank, local = dist_setup()
    ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
