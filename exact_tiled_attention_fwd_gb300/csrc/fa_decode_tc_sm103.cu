// Paged single-token decode on the tensor cores for large query groups, as a
// persistent kernel over an even division of the keys.
//
// The group's query heads of one kv head are the rows of a query tile, so a
// 64-key block of the cache costs two small MMAs (the paged-attention decode
// of dlog.com.cn "从标准 Attention 到 FlashAttention 与分页执行" §3.4, with the
// split-KV of its FlashDecoding section):
//
//   S_j = Q K_j^T         tcgen05.mma (M 128, N 64, K d) -> TMEM
//   P_j = exp(S_j - m)    softmax warps, one thread per query head (row)
//   O  += P_j V_j         tcgen05.mma (M 128, N d, K 64) -> TMEM
//
// and each stretch of keys leaves its unnormalised O and (m, l) in the
// workspace for the combine kernel.  Every cached byte is read once, so the
// design is about keeping loads in flight:
//   - A CTA streams at a rate set by its own ring of K/V tiles (a tile is
//     reissued only once the MMA that read its slot's previous occupant is
//     done, so about two tiles per stream are in flight against the load
//     latency), whatever the other CTAs do.  The time of the launch is
//     therefore the largest number of blocks any CTA has, and the blocks are
//     divided evenly: two persistent CTAs per SM, CTA c takes blocks
//     [c W, (c + 1) W) of the sequence of all (sequence, kv head) pairs'
//     64-key blocks, crossing from pair to pair as segments (the division
//     that decode_tc_plan_kernel computes from seqlens).
//   - The producer streams K/V straight across segment boundaries; Q is
//     double-buffered, so the next segment's queries load while the current
//     one finishes; set-up and the first loads' latency are paid once per
//     CTA.
//   - S is double-buffered in TMEM by block parity (columns 0 and 64, O at
//     128), so the softmax of block j + 1 can start while P.V_j runs.
//
// Warp roles (256 threads, 2 CTAs per SM):
//   warp 0     TMA producer: walks the CTA's segments, publishes them, loads
//              Q and K/V
//   warp 1     allocates TMEM; issues every MMA
//   warps 2-3  idle
//   warps 4-7  softmax, one thread per row (TMEM lane); rows at or past the
//              group size hold no query head and skip the arithmetic
// Segment hand-off: a two-slot ring in shared memory, full/empty mbarriers.
// K/V ring positions, S buffers and the P tile's phases are counted over the
// CTA's whole run, so they continue across segments.
//
// Every wait is bounded in time (the library's convention): on expiry the
// error word records a timeout, the CTA's other warps see the abort flag,
// the producer drains its copies, the issuer waits for its MMAs, and TMEM is
// freed.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBN = kDecodeBlockN;     // keys per K/V block (64)
constexpr int kQRows = kDecodeQRows;   // query rows loaded per segment (64)
constexpr int kThreads = 256;
constexpr int kPlanThreads = 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may reach 2^8

// Shared memory.  The MMAs read 128 rows of Q and of P: rows 64-127 of a Q
// panel fall on the next panel, the other Q buffer or the P tile, and rows
// 64-127 of P on the first ring slot; they give output rows that are never
// stored.  (Smaller Q and P buffers for small groups, with the room given to
// a deeper ring, measured slower.)
template <int D>
struct DecSmem {
    static constexpr int kPanels = D / 64;
    static constexpr uint32_t kQPanel = kQRows * 128;     // 64 rows x 64 d
    static constexpr uint32_t kQTile = kQPanel * kPanels;
    static constexpr uint32_t kKVPanel = kBN * 128;       // 64 keys x 64 d
    static constexpr uint32_t kKVTile = kKVPanel * kPanels;
    static constexpr uint32_t kPTile = kQRows * 128;      // 64 rows x 64 keys
    static constexpr int kSlots = D == 128 ? 4 : 6;
    static constexpr uint32_t kQ = 0;                     // + buffer * kQTile
    static constexpr uint32_t kP = kQ + 2 * kQTile;
    static constexpr uint32_t kKV = kP + kPTile;          // + slot * kKVTile
    static constexpr uint32_t kBar = kKV + kSlots * kKVTile;
    static constexpr uint32_t kNumBars = 32;
    static constexpr uint32_t kSegs = kBar + kNumBars * 8;  // int[2][8]
    static constexpr uint32_t kTmemSlot = kSegs + 64;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    static constexpr uint32_t kDyn = kUsed + 1024;         // 1 KiB alignment slack
    static constexpr uint32_t kTmemCols = 256;              // S_even | S_odd | O
    static constexpr uint32_t kOCol = 128;
};

enum DecBar : uint32_t {
    D_Q_FULL = 0,       // + buffer
    D_Q_EMPTY = 2,      // + buffer: the segment's last S has read it
    D_SEG_FULL = 4,     // + slot
    D_SEG_EMPTY = 6,    // + slot: the issuer and the 4 softmax warps have read it
    D_S_FULL = 8,       // + S buffer
    D_S_FREE = 10,      // + S buffer: the softmax has read it
    D_P_FULL = 12,
    D_P_EMPTY = 13,     // the P.V that read the P tile is done
    D_O_FINAL = 14,     // the segment's last P.V is done
    D_O_FREE = 15,      // the softmax has read the segment's O
    D_MMA_DONE = 16,
    D_KV_FULL = 18,     // + slot (6)
    D_KV_EMPTY = 24,    // + slot (6)
    D_COUNT = 30,
};

// Position of K_j / V_j in a segment's load sequence K_0, K_1, V_0, K_2, V_1,
// ..., V_{n-1}.
__device__ __forceinline__ int pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int pos_v(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * n - 1; }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Keys of sequence b, clamped to [0, max_seqlen] as the combine step does
// (the plan kernel reports an out-of-range length).
__device__ __forceinline__ int seq_len(const DecodeTcParams& p, int b) {
    const int L = __ldg(p.seqlens + b);
    return L < 0 ? 0 : (L > p.max_seqlen ? p.max_seqlen : L);
}

// One segment: keys [kbeg, kbeg + Lk) of pair (b, hk), into partial slot s.
struct Seg {
    int b, hk, s;
    int kbeg;  // first key, a multiple of 64
    int Lk;    // keys in the segment, at least 1
    int L;     // keys of the sequence
    __device__ __forceinline__ int nblk() const { return (Lk + kBN - 1) / kBN; }
};

// Segment slot `k` of the hand-off ring, read after its full barrier.
__device__ __forceinline__ Seg read_seg(const volatile int* segs, int k) {
    Seg sg;
    sg.b = segs[k * 8 + 0];
    sg.hk = segs[k * 8 + 1];
    sg.s = segs[k * 8 + 2];
    sg.kbeg = segs[k * 8 + 3];
    sg.Lk = segs[k * 8 + 4];
    sg.L = segs[k * 8 + 5];
    return sg;
}

// The plan: prefix[b] (blocks of all pairs of the sequences before b,
// b-major), W = the blocks per CTA, and each pair's number of segments.  One
// CTA; each thread takes a contiguous run of sequences.
__global__ void __launch_bounds__(kPlanThreads) decode_tc_plan_kernel(const DecodeTcParams p) {
    grid_dependents_launch();  // the decode grid may set up while this runs
    __shared__ int warp_tot[kPlanThreads / 32];
    __shared__ int warp_max[kPlanThreads / 32];
    __shared__ int w_shared;
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const int per = (p.B + kPlanThreads - 1) / kPlanThreads;
    const int b0 = min(p.B, t * per), b1 = min(p.B, b0 + per);
    int sum = 0, mx = 0;
    for (int b = b0; b < b1; ++b) {
        const int raw = __ldg(p.seqlens + b);
        if (raw < 0 || raw > p.max_seqlen) atomicOr(p.err, FA_DEVERR_INDEX);
        const int nb = (seq_len(p, b) + kBN - 1) / kBN;
        sum += p.Hkv * nb;
        mx = max(mx, nb);
    }
    // exclusive scan of the threads' sums: within each warp, then over warps
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int wmax = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 31) warp_tot[warp] = incl;
    if (lane == 0) warp_max[warp] = wmax;
    __syncthreads();
    if (warp == 0) {
        const int v = warp_tot[lane];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        warp_tot[lane] = inc - v;  // blocks before warp `lane`'s sequences
        const int m = __reduce_max_sync(0xffffffffu, warp_max[lane]);
        if (lane == 31) {
            // Blocks per CTA: all blocks over the grid, at least
            // kDecodeTcMinBlocks, and enough that a pair of m blocks spans at
            // most max_splits CTAs (ceil(m / W) + 1 <= max_splits; the host
            // gives max_splits >= 2).
            int W = (inc + p.grid - 1) / p.grid;
            W = max(W, kDecodeTcMinBlocks);
            W = max(W, (m + p.max_splits - 2) / (p.max_splits - 1));
            w_shared = W;
            p.plan[0] = W;
            p.prefix[p.B] = inc;
        }
    }
    __syncthreads();
    const int W = w_shared;
    int run = warp_tot[warp] + incl - sum;  // blocks before sequence b0
    for (int b = b0; b < b1; ++b) {
        p.prefix[b] = run;
        const int nb = (seq_len(p, b) + kBN - 1) / kBN;
        for (int hk = 0; hk < p.Hkv; ++hk) {
            const int start = run + hk * nb;
            p.seg_ns[b * p.Hkv + hk] = nb == 0 ? 0 : (start + nb - 1) / W - start / W + 1;
        }
        run += p.Hkv * nb;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const DecodeTcParams p) {
    using L = DecSmem<D>;
    constexpr int kPanels = L::kPanels;
    constexpr int kSlots = L::kSlots;
    constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBN, false);  // B = K, K-major
    constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, true);    // B = V, MN-major

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](uint32_t id) { return sbase + L::kBar + id * 8; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    volatile int* segs = reinterpret_cast<volatile int*>(smem + L::kSegs);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_limit_ns;
    const float NEG_INF = -__int_as_float(0x7f800000);

    grid_dependents_launch();  // the combine grid may queue behind this one
    // ---- setup: barriers (thread 0), tensor memory (warp 1)
    if (threadIdx.x == 0) {
        for (int i = 0; i < D_COUNT; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(D_SEG_EMPTY + 0), 5);  // the issuer warp and the 4 softmax warps
        mbar_init(bar(D_SEG_EMPTY + 1), 5);
        mbar_init(bar(D_S_FREE + 0), 4);      // one arrive per softmax warp
        mbar_init(bar(D_S_FREE + 1), 4);
        mbar_init(bar(D_P_FULL), 4);
        mbar_init(bar(D_O_FREE), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

    // Register split: 256 threads launch with 128 each (two CTAs per SM); the
    // producer/MMA warp group drops to 56 and the softmax warps rise to 200.
    constexpr uint32_t kRegsLow = 56, kRegsHigh = 200;
    static_assert(128 * kRegsLow + 128 * kRegsHigh <= 128 * kThreads, "register split exceeds the launch");
    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0) {
            // ================= TMA producer =================
            // The whole warp runs the loop (its waits are warp-uniform); lane
            // 0 publishes segments and posts byte counts, and each of the
            // first boxes-per-block x panels lanes issues one box of a K/V
            // tile: a page, or the block's share of a page larger than the
            // block.  A box past the segment's keys, or from a bad table
            // entry, is loaded from just past the pool, where TMA fills zeros.
            const int page_rows = 1 << p.page_shift;
            const int box_rows = min(page_rows, kBN);
            const int bpb = kBN / box_rows;
            const int pg = lane / kPanels;  // this lane's box of a block
            const int pn = lane % kPanels;  // and panel
            const bool boxes = lane < bpb * kPanels;
            const uint64_t kv_policy = l2_evict_first_policy();  // K/V are read once
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            // This CTA's blocks [off, end) of the b-major sequence of all
            // pairs' blocks, and the sequence b holding block off (the largest
            // b with prefix[b] <= off).  The plan comes from the kernel ahead
            // of this one (launched as its programmatic dependent).
            grid_dependency_wait();
            const int W = p.plan[0];
            const int total = p.prefix[p.B];
            int off = static_cast<int>(blockIdx.x) * W;
            const int end = min(off + W, total);
            int b = 0;
            if (off < end) {
                int lo = 0, hi = p.B - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (p.prefix[mid] <= off) lo = mid; else hi = mid - 1;
                }
                b = lo;
            }
            bool ok = true;
            int n = 0;       // segments published
            int issued = 0;  // K/V loads issued: ring positions 0 .. issued - 1
            int qf0 = 0, qf1 = 0;  // Q loads issued per buffer
            while (ok) {
                // the next segment: blocks [off, min(end, the pair's last)) of
                // the pair holding block off
                Seg sg;
                sg.b = -1;
                if (off < end && !*abort_flag) {
                    while (p.prefix[b + 1] <= off) ++b;  // sequences with no block
                    const int base = p.prefix[b];
                    const int nb = (p.prefix[b + 1] - base) / p.Hkv;
                    const int local = off - base;
                    const int blk0 = local % nb;
                    const int blk1 = min(nb, blk0 + (end - off));
                    sg.b = b;
                    sg.hk = local / nb;
                    sg.s = static_cast<int>(blockIdx.x) - (base + sg.hk * nb) / W;
                    sg.L = seq_len(p, b);
                    sg.kbeg = blk0 * kBN;
                    sg.Lk = min(sg.L, blk1 * kBN) - sg.kbeg;
                    off += blk1 - blk0;
                }
                // publish segment n in slot n % 2 once segment n - 2 has been read there
                if (n >= 2) ok = warp_wait(bar(D_SEG_EMPTY + (n & 1)), ((n - 2) >> 1) & 1, abort_flag, p.err, lim);
                if (!ok) break;
                if (lane == 0) {
                    volatile int* dst = segs + (n & 1) * 8;
                    dst[0] = sg.b;
                    dst[1] = sg.hk;
                    dst[2] = sg.s;
                    dst[3] = sg.kbeg;
                    dst[4] = sg.Lk;
                    dst[5] = sg.L;
                    mbar_arrive(bar(D_SEG_FULL + (n & 1)));
                }
                __syncwarp();
                if (sg.b < 0) break;
                const int nblk = sg.nblk();
                const int pos = issued;  // ring position of this segment's first load
                // Q into buffer n % 2 once segment n - 2's last S has read it
                const int qb = n & 1;
                if (n >= 2) ok = warp_wait(bar(D_Q_EMPTY + qb), ((n - 2) >> 1) & 1, abort_flag, p.err, lim);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(D_Q_FULL + qb), L::kQTile);
#pragma unroll
                    for (int q = 0; q < kPanels; ++q)
                        tma_load_3d(sbase + L::kQ + qb * L::kQTile + q * L::kQPanel, &tm_q, bar(D_Q_FULL + qb), q * 64, 0,
                                    sg.b * p.H + sg.hk * p.group);
                }
                __syncwarp();
                if (qb) ++qf1; else ++qf0;
                // K/V.  Each lane's table entries are fetched four blocks ahead
                // of their first use (a table read takes about as long as a
                // block, so a one-block lookahead would pace the producer):
                // e0 .. e4 hold blocks j .. j + 4.
                const int* bt = p.block_table + static_cast<size_t>(sg.b) * p.max_pages;
                auto fetch = [&](int blk) {
                    const int key0 = blk * kBN + pg * box_rows;  // first key of the box, within the segment
                    return (boxes && blk < nblk && key0 < sg.Lk) ? __ldg(bt + ((sg.kbeg + key0) >> p.page_shift)) : -1;
                };
                int e0 = fetch(0), e1 = fetch(1), e2 = fetch(2), e3 = fetch(3), e4 = fetch(4);
                // ring position pos + lp <- K_j or V_j, this lane's box from page `page`
                auto load = [&](int lp, bool is_k, int j, int page) {
                    const int gp = pos + lp;
                    const int s = gp % kSlots;
                    // the slot's previous occupant (position gp - kSlots) has been consumed
                    if (gp >= kSlots) ok = ok && warp_wait(bar(D_KV_EMPTY + s), ((gp / kSlots) - 1) & 1, abort_flag, p.err, lim);
                    if (!ok) return;
                    if (lane == 0) mbar_arrive_expect_tx(bar(D_KV_FULL + s), L::kKVTile);
                    __syncwarp();
                    if (boxes) {
                        const void* map = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
                        const int key0 = j * kBN + pg * box_rows;
                        int row = p.num_pages << p.page_shift;
                        if (key0 < sg.Lk) {
                            if (page >= 0 && page < p.num_pages)
                                row = (page << p.page_shift) + ((sg.kbeg + key0) & (page_rows - 1));
                            else if (pn == 0 && is_k)
                                atomicOr(p.err, FA_DEVERR_INDEX);
                        }
                        tma_load_3d_hint(sbase + L::kKV + s * L::kKVTile + pn * L::kKVPanel + pg * box_rows * 128, map,
                                         bar(D_KV_FULL + s), pn * 64, sg.hk, row, kv_policy);
                    }
                    __syncwarp();
                    ++issued;
                };
                load(pos_k(0), true, 0, e0);
                for (int j = 0; ok && j < nblk; ++j) {
                    if (j + 1 < nblk) load(pos_k(j + 1), true, j + 1, e1);
                    load(pos_v(j, nblk), false, j, e0);
                    // block j is issued: rotate the entries
                    e0 = e1;
                    e1 = e2;
                    e2 = e3;
                    e3 = e4;
                    e4 = fetch(j + 5);
                }
                ++n;
            }
            // Drain: every copy this CTA issued lands before it exits.  Slot s
            // last held the largest position below `issued` that is s modulo
            // kSlots.
            if (lane == 0) {
#pragma unroll
                for (int s = 0; s < kSlots; ++s)
                    if (s < issued) mbar_wait_drain(bar(D_KV_FULL + s), (((issued - 1 - s) / kSlots)) & 1, lim);
                if (qf0 > 0) mbar_wait_drain(bar(D_Q_FULL + 0), (qf0 - 1) & 1, lim);
                if (qf1 > 0) mbar_wait_drain(bar(D_Q_FULL + 1), (qf1 - 1) & 1, lim);
            }
            __syncwarp();
        }
        else if (warp == 1) {
            // ================= MMA issuer =================
            // Per item: S_0 and S_1 once Q and their K tiles have landed; then
            // per block j: P.V_j once P_j is stored, and S_{j+2} into the S
            // buffer that S_j used once the softmax has read it.  The first
            // P.V of an item overwrites O, so it waits until the softmax has
            // read the previous item's O.  The issuer also zeroes the stale
            // rows of an item's last V tile.
            // Descriptor bases; a k-step only moves the start address, the low
            // field of the descriptor (addresses stay below 256 KiB, so the
            // addition never carries out of it).
            const uint64_t dq0 = sdesc_sw128(sbase + L::kQ, 16, 1024);
            const uint64_t dp = sdesc_sw128(sbase + L::kP, 16, 1024);
            const uint64_t dk = sdesc_sw128(sbase + L::kKV, 16, 1024);
            const uint64_t dv = sdesc_sw128(sbase + L::kKV, L::kKVPanel, 1024);
            const uint32_t t_o = tmem + L::kOCol;
            bool ok = true;
            bool issued_mma = false;
            int n = 0;    // items taken
            int g = 0;    // blocks before this item (S buffer and P phases)
            int pos = 0;  // ring position of this item's first load
            const int page_rows = 1 << p.page_shift;
            auto wait_pos = [&](int gp) {
                ok = ok && warp_wait(bar(D_KV_FULL + gp % kSlots), (gp / kSlots) & 1, abort_flag, p.err, lim);
            };
            // S buffer gb % 2 = Q (buffer qb) K^T, K at ring position gp
            auto issue_s = [&](int qb, int gb, int gp) {
                const int s = gp % kSlots;
                const uint64_t dq = dq0 + ((qb * L::kQTile) >> 4);
                const uint64_t b0 = dk + ((s * L::kKVTile) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t offa = ((kk >> 2) * L::kQPanel + (kk & 3) * 32) >> 4;
                        const uint32_t offb = ((kk >> 2) * L::kKVPanel + (kk & 3) * 32) >> 4;
                        mma_ss(tmem + (gb & 1) * kBN, dq + offa, b0 + offb, kIdescS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(D_S_FULL + (gb & 1)));
                    tc_commit(bar(D_KV_EMPTY + s));
                }
                __syncwarp();
                issued_mma = true;
            };
            // O (+)= P V, V at ring position gp
            auto issue_pv = [&](int gp, bool accumulate, bool last) {
                const int s = gp % kSlots;
                const uint64_t b0 = dv + ((s * L::kKVTile) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ss(t_o, dp + ((kk * 32) >> 4), b0 + ((kk * 16 * 128) >> 4), kIdescPV,
                               (accumulate || kk > 0) ? 1u : 0u);
                    tc_commit(bar(D_P_EMPTY));
                    tc_commit(bar(D_KV_EMPTY + s));
                    if (last) tc_commit(bar(D_O_FINAL));
                }
                __syncwarp();
            };
            auto release_q = [&](int qb) {
                if (elect_one()) tc_commit(bar(D_Q_EMPTY + qb));
                __syncwarp();
            };
            while (ok) {
                ok = warp_wait(bar(D_SEG_FULL + (n & 1)), (n >> 1) & 1, abort_flag, p.err, lim);
                if (!ok) break;
                const Seg sg = read_seg(segs, n & 1);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(D_SEG_EMPTY + (n & 1)));
                if (sg.b < 0) break;
                const int nblk = sg.nblk();
                // the sequence's last page is only partly used, and this
                // segment holds its last key: stale V rows to zero
                const bool v_tail = sg.kbeg + sg.Lk == sg.L && (sg.L & (page_rows - 1)) != 0;
                const int qb = n & 1;
                ok = warp_wait(bar(D_Q_FULL + qb), (n >> 1) & 1, abort_flag, p.err, lim);
                wait_pos(pos + pos_k(0));
                if (!ok) break;
                tc_fence_after();
                issue_s(qb, g, pos + pos_k(0));
                if (nblk > 1) {
                    wait_pos(pos + pos_k(1));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(qb, g + 1, pos + pos_k(1));
                }
                if (nblk <= 2) release_q(qb);
                for (int j = 0; ok && j < nblk; ++j) {
                    const int gb = g + j;
                    ok = warp_wait(bar(D_P_FULL), gb & 1, abort_flag, p.err, lim);
                    wait_pos(pos + pos_v(j, nblk));
                    if (j == 0 && n > 0) ok = ok && warp_wait(bar(D_O_FREE), (n - 1) & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    if (v_tail && j == nblk - 1) {
                        // Keys [L, roundup(L, page)) of the last V tile are
                        // stale pool slots: zero their rows before the last
                        // P.V (P is 0 there, but 0 times a non-finite stale
                        // value is not).
                        const int gp = pos + pos_v(j, nblk);
                        const int kb = sg.kbeg + j * kBN;  // the tile's first key
                        const int r_lo = sg.L - kb;
                        const int r_hi = min(((sg.L + page_rows - 1) & ~(page_rows - 1)) - kb, kBN);
                        const uint32_t base = sbase + L::kKV + (gp % kSlots) * L::kKVTile;
                        for (int e = lane; e < (r_hi - r_lo) * kPanels * 8; e += 32) {
                            const int chunk = e & 7;
                            const int q = (e >> 3) % kPanels;
                            const int rr = r_lo + (e >> 3) / kPanels;
                            st_shared_v4(base + q * L::kKVPanel + rr * 128 + chunk * 16, 0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    tc_fence_after();
                    issue_pv(pos + pos_v(j, nblk), j > 0, j == nblk - 1);
                    if (j + 2 < nblk) {
                        ok = warp_wait(bar(D_S_FREE + (gb & 1)), (gb >> 1) & 1, abort_flag, p.err, lim);
                        wait_pos(pos + pos_k(j + 2));
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(qb, gb + 2, pos + pos_k(j + 2));
                        if (j + 3 == nblk) release_q(qb);  // the item's last S
                    }
                }
                g += nblk;
                pos += 2 * nblk;
                ++n;
            }
            // Every MMA of this warp has finished before tensor memory is
            // released.
            if (issued_mma) {
                if (elect_one()) {
                    tc_commit(bar(D_MMA_DONE));
                    mbar_wait_drain(bar(D_MMA_DONE), 0, lim);
                }
                __syncwarp();
            }
        }
    } else {
        regs_inc<kRegsHigh>();
        // ================= softmax and the segments' partial results =================
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row of the tile == TMEM lane
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        // this row of the P tile (128-byte swizzle: chunk c of the row lands at
        // (c ^ (row % 8)) * 16); only rows below kQRows have one
        const uint32_t p_row = sbase + L::kP + static_cast<uint32_t>(r) * 128;
        const uint32_t p_sw = static_cast<uint32_t>(r & 7);
        const bool active = quarter * 32 < p.group;  // this warp holds query heads
        const bool valid = r < p.group;
        const float c = p.scale_log2;
        bool ok = true;
        int n = 0;  // items taken
        int g = 0;  // blocks before this item
        while (ok) {
            ok = warp_wait(bar(D_SEG_FULL + (n & 1)), (n >> 1) & 1, abort_flag, p.err, lim);
            if (!ok) break;
            const Seg sg = read_seg(segs, n & 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(D_SEG_EMPTY + (n & 1)));
            if (sg.b < 0) break;
            const int nblk = sg.nblk();
            float m_ref = NEG_INF;  // exponent reference (log2 units)
            float l = 0.f;
            for (int j = 0; ok && j < nblk; ++j) {
                const int gb = g + j;
                ok = warp_wait(bar(D_S_FULL + (gb & 1)), (gb >> 1) & 1, abort_flag, p.err, lim);
                if (!ok) break;
                uint32_t pk[kBN / 2];
                float alpha = 1.f;
                bool resc = false;
                if (active) {
                    tc_fence_after();
                    uint32_t u[kBN];
                    tmem_ld64(t_row + (gb & 1) * kBN, u);
                    // the scores are in registers: the issuer may reuse the buffer
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(D_S_FREE + (gb & 1)));
                    const int lim_c = sg.Lk - 1 - j * kBN;  // the segment's last key, within the block
                    if (lim_c < kBN - 1) {
#pragma unroll
                        for (int i = 0; i < kBN; ++i)
                            if (i > lim_c) u[i] = __float_as_uint(NEG_INF);
                    }
                    // the block's row maximum; the reference moves only when the
                    // maximum grows by more than kRescaleThreshold, so O is
                    // rarely rescaled (the reference cancels in O / l and
                    // returns in the LSE)
                    float mx0 = NEG_INF, mx1 = NEG_INF, mx2 = NEG_INF, mx3 = NEG_INF;
#pragma unroll
                    for (int i = 0; i < kBN; i += 8) {
                        mx0 = fmax3(mx0, __uint_as_float(u[i]), __uint_as_float(u[i + 1]));
                        mx1 = fmax3(mx1, __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]));
                        mx2 = fmax3(mx2, __uint_as_float(u[i + 4]), __uint_as_float(u[i + 5]));
                        mx3 = fmax3(mx3, __uint_as_float(u[i + 6]), __uint_as_float(u[i + 7]));
                    }
                    const float m_new = fmaxf(m_ref, fmax3(mx0, mx1, fmaxf(mx2, mx3)) * c);
                    resc = (m_ref != NEG_INF) && (m_new - m_ref > kRescaleThreshold);
                    alpha = resc ? ex2(m_ref - m_new) : 1.f;
                    if (resc || m_ref == NEG_INF) m_ref = m_new;
                    const float mu = m_ref == NEG_INF ? 0.f : m_ref;
                    // P = 2^(S c - mu) as bf16 pairs, and the row sum in fp32
                    const float2 c2 = make_float2(c, c);
                    const float2 nmu2 = make_float2(-mu, -mu);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < kBN / 2; ++i) {
                        const float2 x =
                            __ffma2_rn(make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])), c2, nmu2);
                        const float2 e = make_float2(ex2(x.x), ex2(x.y));
                        if (i & 1)
                            acc1 = __fadd2_rn(acc1, e);
                        else
                            acc0 = __fadd2_rn(acc0, e);
                        pk[i] = pack_bf16x2(e.x, e.y);
                    }
                    l = l * alpha + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
                } else {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(D_S_FREE + (gb & 1)));
                }
                // the P tile and O are free once the previous block's P.V is done
                if (gb > 0) ok = warp_wait(bar(D_P_EMPTY), (gb - 1) & 1, abort_flag, p.err, lim);
                if (!ok) break;
                if (active) {
                    if (__any_sync(0xffffffffu, resc)) {
                        tc_fence_after();
#pragma unroll
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t o[32];
                            tmem_ld32(t_row + L::kOCol + ch * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(t_row + L::kOCol + ch * 32, o);
                        }
                        tmem_st_wait();
                    }
                    if (r < kQRows) {
#pragma unroll
                        for (int cc = 0; cc < kBN / 8; ++cc)
                            st_shared_v4(p_row + ((static_cast<uint32_t>(cc) ^ p_sw) << 4), pk[4 * cc], pk[4 * cc + 1],
                                         pk[4 * cc + 2], pk[4 * cc + 3]);
                    }
                }
                // make the P rows visible to the tensor core, then publish
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(D_P_FULL));
            }
            if (!ok) break;
            // ---- the segment's unnormalised O and (m, l), log2 domain
            ok = warp_wait(bar(D_O_FINAL), n & 1, abort_flag, p.err, lim);
            if (!ok) break;
            tc_fence_after();
            if (active) {
                uint32_t o[D / 32][32];
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(t_row + L::kOCol + ch * 32, o[ch]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(D_O_FREE));  // the next segment's first P.V may overwrite O
                if (valid) {
                    const size_t slot =
                        (static_cast<size_t>(sg.b) * p.H + sg.hk * p.group + r) * p.max_splits + sg.s;
                    float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * D);
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[ch * 8 + i] = make_float4(__uint_as_float(o[ch][4 * i]), __uint_as_float(o[ch][4 * i + 1]),
                                                          __uint_as_float(o[ch][4 * i + 2]), __uint_as_float(o[ch][4 * i + 3]));
                    *reinterpret_cast<float2*>(p.ws_ml + slot * 2) = make_float2(l > 0.f ? m_ref : NEG_INF, l);
                }
            } else {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(D_O_FREE));
            }
            g += nblk;
            ++n;
        }
    }
    tc_fence_before();
    cta_sync(kThreads);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeTcParams& p,
                     cudaStream_t stream) {
    using L = DecSmem<D>;
    static_assert(L::kDyn <= 232448u, "shared memory budget");
    static_assert(2 * (L::kDyn + 1024) <= 233472u, "two CTAs per SM");
    static_assert(D_COUNT <= L::kNumBars && L::kSlots <= 6, "barrier block");
    static_assert(L::kOCol + D <= L::kTmemCols && 2 * kBN <= L::kOCol, "tensor memory columns");
    static_assert(L::kQTile % 1024 == 0 && L::kPTile % 1024 == 0, "swizzled tiles start on 1 KiB");
    static_assert(L::kQ + L::kQTile + (L::kPanels - 1) * L::kQPanel + 128 * 128 <= L::kBar &&
                      L::kP + 128 * 128 <= L::kBar,
                  "the MMAs' 128-row reads of Q and P stay in shared memory");
    auto kern = decode_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kDyn));
    if (e != cudaSuccess) return e;
    decode_tc_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the decode grid starts while the plan kernel runs; its producer waits
    // for the plan (grid_dependency_wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kDyn;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace

cudaError_t launch_decode_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, DecodeTcParams p,
                             int d, cudaStream_t stream) {
    // Two CTAs per SM, or fewer when even kDecodeTcMinBlocks blocks each
    // would leave some idle (an upper bound on the blocks: every sequence at
    // max_seqlen).
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(p.B) * p.Hkv * ((p.max_seqlen + kBN - 1) / kBN);
    const long long want = (blocks + kDecodeTcMinBlocks - 1) / kDecodeTcMinBlocks;
    p.grid = static_cast<int>(want < 2ll * sms ? (want < 1 ? 1 : want) : 2ll * sms);
    return d == 128 ? launch_d<128>(tq, tk, tv, p, stream) : launch_d<64>(tq, tk, tv, p, stream);
}

}  // namespace fa
