// Backward pass of exact attention for sm_103a.
//
// Given Q, K, V, the forward's O and LSE, and dO, compute
//
//   P    = exp(scale Q K^T - LSE)          recomputed, never stored
//   dV   = P^T dO
//   dP   = dO V^T
//   dS   = P * (dP - delta),   delta_i = dO_i . O_i   (the row sum)
//   dQ   = scale dS K,         dK = scale dS^T Q
//
// the recomputation scheme of the lqnn.cn FlashAttention article (§2.3: keep
// only O and the row statistics, recompute S and P in the backward; §4.3: the
// chain rule, with the row sum subtracted in dS) and the yulong.wang page
// §2.3 (P rebuilt from the saved logsumexp).
//
// Three launches on one stream:
//   bwd_prep_kernel   delta_i and the LSE in log2 units, into a padded fp32
//                     workspace (rows past a sequence: LSE +inf, delta 0, so
//                     their P is exactly 0 in the kernels below)
//   bwd_dkdv_kernel   one CTA per (128-key block, kv head, sequence): K_j and
//                     V_j stay in shared memory while every visible 128-row
//                     query block of every query head of the group streams
//                     past; dK_j and dV_j accumulate in tensor memory and are
//                     written once
//   bwd_dq_kernel     one CTA per (128-row query block, head, sequence): Q_i
//                     and dO_i stay in shared memory while the visible K/V
//                     blocks stream past; dQ_i accumulates in tensor memory
//                     and is written once.  It reads none of dK/dV, so it is
//                     launched to start in the dK/dV grid's tail
//                     (programmatic dependent launch) and waits for that
//                     grid only before its CTAs exit
// dQ is therefore never accumulated with atomics across key blocks (the
// article's §4.3 and §6.4 name those atomics as the cost to avoid, by
// keeping the dQ accumulation on chip and writing it once); the price is
// that S and dP are computed in both kernels (7 matrix products per block
// pair instead of 5).  The result is deterministic.
//
// Every product is a tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) with
// M = 128; operands are TMA-loaded 128-byte-swizzled tiles or, for dS, bf16
// pairs written back into tensor memory (the A-from-TMEM form).

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// Warps 0 and 2: TMA producers (one operand ring each); warps 1 and 3: MMA
// issuers (two issue streams); warps 4-11: compute.
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPanelBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(addr));
    return r;
}

// Descriptor offset (16-byte units) of k-step kk (16 elements of the
// contraction) in a K-major tile made of 64-column panels.
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
    return ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
}

// Sequence geometry shared by the three kernels.  Returns false (and flags
// the error word once) when a varlen entry is out of range.
struct Geom {
    int q_start, Lq, k_start, Lk;
};
__device__ __forceinline__ bool seq_geom(const BackwardParams& p, int seq, bool report, Geom& g) {
    if (p.cu_q != nullptr) {
        g.q_start = p.cu_q[seq];
        g.Lq = p.cu_q[seq + 1] - g.q_start;
        g.k_start = p.cu_k[seq];
        g.Lk = p.cu_k[seq + 1] - g.k_start;
        const bool bad = g.q_start < 0 || g.Lq < 0 || g.Lk < 0 || g.q_start + g.Lq > p.total_q ||
                         g.Lq > p.max_seqlen_q || g.Lk > p.max_seqlen_k || g.k_start < 0 ||
                         g.k_start + g.Lk > p.total_k;
        if (bad) {
            if (report) atomicOr(p.err, FA_DEVERR_INDEX);
            return false;
        }
    } else {
        g.q_start = seq * p.N;
        g.Lq = p.N;
        g.k_start = seq * p.N;
        g.Lk = p.N;
    }
    return true;
}


// Grid order of the two main kernels.  grid.x enumerates (block, head)
// pairs.  Causal: heads in groups of kHeadGroup, the blocks of a group
// heaviest first and the group's heads fastest, so the heaviest work of
// every group is handed out early (no head's heavy blocks are left for the
// last wave) while the CTAs resident at once cover only a few heads' operands
// in L2.  Measured at B1 H32 N8192 d128 causal: heads one after the other
// 1.34 ms, groups of 4 heads 1.30 ms, groups of 8 1.28 ms (all heads at once
// missed L2 on 3.5x the algorithmic bytes).  Non-causal: blocks fastest
// within a head.  blk_rank 0 is the heaviest block.
constexpr int kHeadGroup = 8;
template <bool CAUSAL>
__device__ __forceinline__ void grid_order(int x, int nblk, int nheads, int& blk_rank, int& head) {
    if (!CAUSAL) {
        blk_rank = x % nblk;
        head = x / nblk;
        return;
    }
    const int per = kHeadGroup * nblk;
    const int grp = x / per;
    const int gs = min(kHeadGroup, nheads - grp * kHeadGroup);
    const int rem = x - grp * per;
    blk_rank = rem / gs;
    head = grp * kHeadGroup + rem % gs;
}

// ============================================================== prep

// delta_i = sum_d dO_id O_id (fp32 sum of bf16 products) and lse2_i =
// LSE_i log2(e) for the rows of one (128-row block, head, sequence); padded
// rows of the block get delta 0 and lse2 +inf (also a row whose LSE is -inf,
// i.e. sees no key).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BackwardParams p) {
    constexpr int kLanes = D / 8;  // threads per row, 8 bf16 each
    constexpr int kRowsPerPass = 256 / kLanes;
    const int blk = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
    Geom g;
    if (!seq_geom(p, seq, blk == 0 && h == 0 && threadIdx.x == 0, g)) return;
    if (blk * kBlockM >= g.Lq) return;
    const long long lse_base = p.cu_q ? g.q_start : static_cast<long long>(seq) * p.H * p.N;
    float* lse2 = p.ws + h * p.ws_head_stride + bwd_ws_seq_offset(g.q_start, seq);
    float* delta = lse2 + p.H * p.ws_head_stride;
    const int sub = threadIdx.x % kLanes;
    const float INF = __int_as_float(0x7f800000);
    for (int rr = threadIdx.x / kLanes; rr < kBlockM; rr += kRowsPerPass) {
        const int row = blk * kBlockM + rr;
        float acc = 0.f;
        if (row < g.Lq) {
            const size_t off = (static_cast<size_t>(g.q_start + row) * p.H + h) * D + sub * 8;
            const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + off);
            const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + off);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(bf16lo_to_f32(av[e]), bf16lo_to_f32(bv[e]), acc);
                acc = fmaf(bf16hi_to_f32(av[e]), bf16hi_to_f32(bv[e]), acc);
            }
        }
#pragma unroll
        for (int m = kLanes / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (sub == 0) {
            float l2 = INF;
            if (row < g.Lq) {
                const float l = p.lse[lse_base + h * p.lse_head_stride + row];
                l2 = l == -INF ? INF : l * kLog2e;
            }
            lse2[row] = l2;
            delta[row] = row < g.Lq ? acc : 0.f;
        }
    }
}

// ============================================================== dK / dV

// One CTA: keys [128 j, 128 j + 128) of kv head hk.  Step n walks the
// (query head of the group, 128-row query block) pairs that see some key of
// the block.  Per step:
//
//   S^T  = K_j Q_n^T         SS, K-major both        -> TMEM [0, 128)
//   dP^T = V_j dO_n^T        SS, K-major both        -> TMEM [128, 256)
//   P^T  = 2^(S^T c - lse2)  compute warps           -> shared memory tile
//   dV  += P^T dO_n          SS, dO MN-major          -> TMEM [256, 256 + d)
//   dS^T = P^T (dP^T - delta) compute warps           -> bf16 pairs over dP^T
//   dK  += dS^T Q_n          TS (A from TMEM), Q MN-major -> TMEM [384, 384 + d)
//
// The compute warps own key rows (TMEM lanes): warp w covers lanes
// 32 (w % 4) .. + 31 and query columns 64 ((w - 4) / 4) .. + 63, so two
// threads share a key row.  Their dS^T bf16 pairs go to the first 32 of
// their own 64 dP^T columns, never into columns the other thread reads.
//
// Q_n and dO_n have rings of their own, each filled by its own producer
// thread (warp 0 and warp 2), so that neither waits behind the other's
// slot: a Q slot is freed by dK (the last product of a step), a dO slot
// by dV.  lse2 and delta of the step's 128 query rows travel with Q_n (one
// bulk copy each into a small buffer beside the Q slot); the compute warps
// read them from shared memory, and the slot is only freed after dK, i.e.
// after the compute warps have finished the step.
template <int D>
struct DkdvSmem {
    static constexpr uint32_t kTile = 128 * D * 2;      // a K, V, Q or dO tile
    static constexpr uint32_t kPTile = 128 * 128 * 2;   // P^T
    static constexpr int kSlots = D == 128 ? 2 : 4;     // per ring (Q, dO)
    static constexpr uint32_t kAux = 1024;              // lse2[128], delta[128] (fp32)
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + kTile;
    static constexpr uint32_t kP = kV + kTile;
    static constexpr uint32_t kQR = kP + kPTile;
    static constexpr uint32_t kDR = kQR + kSlots * kTile;
    static constexpr uint32_t kAuxR = kDR + kSlots * kTile;
    static constexpr uint32_t kBar = kAuxR + kSlots * kAux;
    static constexpr uint32_t kNumBars = 28;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    // No alignment slack: the kernel checks that the dynamic shared memory
    // starts on a 1024-byte boundary (the 128-byte swizzle atom) and reports
    // FA_DEVERR_LAYOUT otherwise.  At least 116 KiB so one CTA holds an SM.
    static constexpr uint32_t kDyn = kUsed > 118784u ? kUsed : 118784u;
};

enum DkdvBar : uint32_t {
    A_KV_FULL = 0,
    A_Q_FULL = 1,     // + slot (4): Q_n, lse2_n, delta_n
    A_Q_EMPTY = 5,    // + slot (4)
    A_DO_FULL = 9,    // + slot (4)
    A_DO_EMPTY = 13,  // + slot (4)
    A_S_FULL = 17,    // S^T_n in TMEM
    A_S_FREE = 18,    // compute warps have read S^T_n (8 arrivals)
    A_DP_FULL = 19,   // dP^T_n in TMEM
    A_P_FULL = 20,    // P^T_n in shared memory (8 arrivals)
    A_P_EMPTY = 21,   // dV += P^T_n dO_n done
    A_DS_FULL = 22,   // dS^T_n in TMEM (8 arrivals)
    A_DS_EMPTY = 23,  // dK += dS^T_n Q_n done
    A_DONE = 24,      // + issuer (2): its last product done (dK, dV final)
    A_DRAIN = 26,     // + issuer (2): own drain before tensor memory is freed
    A_COUNT = 28,
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BackwardParams p) {
    using L = DkdvSmem<D>;
    constexpr int kPanels = D / 64;
    constexpr int kSlots = L::kSlots;
    // The dQ kernel behind this one reads none of its results: it may start
    // on the SMs this grid's last wave leaves free.
    grid_dependents_launch();
    constexpr uint32_t kIdescT = idesc_bf16_f32(128, 128, false);  // S^T, dP^T
    constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, true);     // dV, dK

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err, FA_DEVERR_LAYOUT);
        return;
    }
    auto bar = [&](uint32_t id) { return sbase + L::kBar + id * 8; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // With causal masking the low key blocks see the most query blocks: block
    // rank r is key block r.
    int jb, hk;
    grid_order<CAUSAL>(static_cast<int>(blockIdx.x), p.num_k_blocks, p.Hkv, jb, hk);
    const int seq = blockIdx.z;
    Geom g;
    if (!seq_geom(p, seq, jb == 0 && hk == 0 && threadIdx.x == 0, g)) return;
    const int key0 = jb * kBlockN;
    if (key0 >= g.Lk) return;
    const int diag = g.Lk - g.Lq;  // key j visible to query i iff j <= i + diag
    const int nq = (g.Lq + kBlockM - 1) / kBlockM;
    // First query block with a row that sees a key of this block.
    int i_lo = 0;
    if (CAUSAL) {
        const int first_row = key0 - diag;  // smallest row that sees key0
        i_lo = first_row <= 0 ? 0 : first_row / kBlockM;
    }
    const int per_head = nq > i_lo ? nq - i_lo : 0;
    const int n_steps = per_head * p.group;
    const int rows_here = min(kBlockN, g.Lk - key0);

    if (n_steps == 0) {
        // No query sees these keys: dK = dV = 0.
        for (int e = threadIdx.x; e < rows_here * (D / 8); e += kThreads) {
            const int r = e / (D / 8), c = e % (D / 8);
            const size_t off = (static_cast<size_t>(g.k_start + key0 + r) * p.Hkv + hk) * D + c * 8;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dk) + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dv) + off) = make_uint4(0, 0, 0, 0);
        }
        return;
    }

    // step n -> (query head, query block)
    auto step_head = [&](int n) { return hk * p.group + n / per_head; };
    // Each CTA starts its walk over the query blocks at its own offset (its
    // key block index), so that the CTAs of one head, which run at the same
    // time, ask for different Q / dO tiles at any moment: a tile is fetched
    // from memory once and then read from L2 by the others.
    const int rot = per_head > 0 ? jb % per_head : 0;
    auto step_block = [&](int n) {
        const int m = n % per_head + rot;
        return i_lo + (m >= per_head ? m - per_head : m);
    };
    const float* ws_seq = p.ws + bwd_ws_seq_offset(g.q_start, seq);  // this sequence's lse2 / delta rows
    // Q_n (with lse2_n, delta_n) or dO_n into slot n % kSlots of its ring
    auto load_step = [&](bool is_q, int n) {
        const int s = n % kSlots;
        const uint32_t full = (is_q ? A_Q_FULL : A_DO_FULL) + s;
        const int hq = step_head(n), ib = step_block(n);
        mbar_arrive_expect_tx(bar(full), L::kTile + (is_q ? 1024u : 0u));
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn)
            tma_load_3d(sbase + (is_q ? L::kQR : L::kDR) + s * L::kTile + pn * kPanelBytes, is_q ? &tm_q : &tm_do,
                        bar(full), pn * 64, hq, g.q_start + ib * kBlockM);
        if (is_q) {
            const float* src = ws_seq + hq * p.ws_head_stride + ib * kBlockM;
            bulk_load_1d(sbase + L::kAuxR + s * L::kAux, src, 512, bar(full));
            bulk_load_1d(sbase + L::kAuxR + s * L::kAux + 512, src + p.H * p.ws_head_stride, 512, bar(full));
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < A_COUNT; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(A_S_FREE), 8);
        mbar_init(bar(A_P_FULL), 8);
        mbar_init(bar(A_DS_FULL), 8);
        *abort_flag = 0;
        fence_barrier_init();
        // The first loads need only the barriers: issue them now, so that they
        // overlap the tensor-memory allocation and the CTA barrier.  K and V,
        // then step 0's Q (with its lse2 / delta) and dO.
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_arrive_expect_tx(bar(A_KV_FULL), 2 * L::kTile);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn) {
            tma_load_3d(sbase + L::kK + pn * kPanelBytes, &tm_k, bar(A_KV_FULL), pn * 64, hk, g.k_start + key0);
            tma_load_3d(sbase + L::kV + pn * kPanelBytes, &tm_v, bar(A_KV_FULL), pn * 64, hk, g.k_start + key0);
        }
        load_step(true, 0);
        load_step(false, 0);
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    const uint64_t lim = p.wait_limit_ns;

    // 128 * 72 + 256 * 216 = 64,512 = 384 * 168 (the launch's registers).
    constexpr uint32_t kRegsLow = 72, kRegsHigh = 216;
    static_assert(128 * kRegsLow + 256 * kRegsHigh <= 168 * kThreads, "register split exceeds the launch");
    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0 || warp == 2) {
            // ================= TMA producers: warp 0 K, V, then Q_n (+ lse2,
            // delta); warp 2 dO_n =================
            const bool is_q = warp == 0;
            if (lane == 0) {
                const uint32_t ring_full = is_q ? A_Q_FULL : A_DO_FULL;
                const uint32_t ring_empty = is_q ? A_Q_EMPTY : A_DO_EMPTY;
                bool ok = true;
                // (K, V and step 0 were issued before the CTA barrier.)
                for (int n = 1; ok && n < n_steps; ++n) {
                    const int s = n % kSlots;
                    if (n >= kSlots) ok = mbar_wait(bar(ring_empty + s), ((n / kSlots) - 1) & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    load_step(is_q, n);
                }
                // Drain: every copy this thread issued lands before the CTA exits.
                if (is_q) mbar_wait_drain(bar(A_KV_FULL), 0, lim);
                for (int s = 0; s < kSlots && s < n_steps; ++s) {
                    const int last = s + ((n_steps - 1 - s) / kSlots) * kSlots;  // last step put in slot s
                    mbar_wait_drain(bar(ring_full + s), (last / kSlots) & 1, lim);
                }
            }
            __syncwarp();
        } else {
            // ================= MMA issuers: warp 1 S^T and dK (the Q ring),
            // warp 3 dP^T and dV (the dO ring).  Two issue streams keep the
            // tensor pipe fed while either one waits. =================
            const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
            const int who = warp == 1 ? 0 : 1;
            bool ok = warp_wait(bar(A_KV_FULL), 0, abort_flag, p.err, lim);
            auto slot_off = [&](int n) { return static_cast<uint32_t>(((n % kSlots) * L::kTile) >> 4); };
            if (who == 0) {
                const uint64_t dk_a = sdesc_sw128(sbase + L::kK, 16, 1024);
                const uint64_t q_k = sdesc_sw128(sbase + L::kQR, 16, 1024);             // Q as K-major B
                const uint64_t q_mn = sdesc_sw128(sbase + L::kQR, kPanelBytes, 1024);   // Q as MN-major B
                auto wait_q = [&](int n) {
                    ok = ok && warp_wait(bar(A_Q_FULL + n % kSlots), (n / kSlots) & 1, abort_flag, p.err, lim);
                };
                // S^T_n = K Q_n^T
                auto issue_s = [&](int n) {
                    const uint64_t b0 = q_k + slot_off(n);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(t_s, dk_a + kmajor_step(kk), b0 + kmajor_step(kk), kIdescT, kk > 0 ? 1u : 0u);
                        tc_commit(bar(A_S_FULL));
                    }
                    __syncwarp();
                };
                // dK += dS^T_n Q_n, dS^T from TMEM: queries 16 kk .. 16 kk + 15 are
                // 8 columns at 128 + 64 (kk / 4) + 8 (kk % 4)
                auto issue_dk = [&](int n) {
                    const uint64_t b0 = q_mn + slot_off(n);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 128 / 16; ++kk)
                            mma_ts(t_dk, t_dp + 64 * (kk >> 2) + 8 * (kk & 3), b0 + ((kk * 16 * 128) >> 4), kIdescG,
                                   (n > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(bar(A_DS_EMPTY));
                        tc_commit(bar(A_Q_EMPTY + n % kSlots));
                        if (n == n_steps - 1) tc_commit(bar(A_DONE));
                    }
                    __syncwarp();
                };
                wait_q(0);
                if (ok) issue_s(0);
                for (int n = 0; ok && n < n_steps; ++n) {
                    if (n + 1 < n_steps) {
                        // S^T_{n+1} overwrites S^T_n: the compute warps have read it.
                        ok = ok && warp_wait(bar(A_S_FREE), n & 1, abort_flag, p.err, lim);
                        wait_q(n + 1);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(n + 1);
                    }
                    ok = ok && warp_wait(bar(A_DS_FULL), n & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dk(n);
                }
            } else {
                const uint64_t dv_a = sdesc_sw128(sbase + L::kV, 16, 1024);
                const uint64_t dp_a = sdesc_sw128(sbase + L::kP, 16, 1024);
                const uint64_t do_k = sdesc_sw128(sbase + L::kDR, 16, 1024);
                const uint64_t do_mn = sdesc_sw128(sbase + L::kDR, kPanelBytes, 1024);
                auto wait_do = [&](int n) {
                    ok = ok && warp_wait(bar(A_DO_FULL + n % kSlots), (n / kSlots) & 1, abort_flag, p.err, lim);
                };
                // dP^T_n = V dO_n^T
                auto issue_dp = [&](int n) {
                    const uint64_t b0 = do_k + slot_off(n);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(t_dp, dv_a + kmajor_step(kk), b0 + kmajor_step(kk), kIdescT, kk > 0 ? 1u : 0u);
                        tc_commit(bar(A_DP_FULL));
                    }
                    __syncwarp();
                };
                // dV += P^T_n dO_n (dO_n as N = d x K = 128 queries, MN-major)
                auto issue_dv = [&](int n) {
                    const uint64_t b0 = do_mn + slot_off(n);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 128 / 16; ++kk)
                            mma_ss(t_dv, dp_a + kmajor_step(kk), b0 + ((kk * 16 * 128) >> 4), kIdescG,
                                   (n > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(bar(A_P_EMPTY));
                        tc_commit(bar(A_DO_EMPTY + n % kSlots));
                        if (n == n_steps - 1) tc_commit(bar(A_DONE + 1));
                    }
                    __syncwarp();
                };
                wait_do(0);
                if (ok) issue_dp(0);
                for (int n = 0; ok && n < n_steps; ++n) {
                    ok = ok && warp_wait(bar(A_P_FULL), n & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dv(n);
                    if (n + 1 < n_steps) {
                        // dP^T_{n+1} overwrites dS^T_n: dK has read it.
                        ok = ok && warp_wait(bar(A_DS_EMPTY), n & 1, abort_flag, p.err, lim);
                        wait_do(n + 1);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dp(n + 1);
                    }
                }
            }
            // Every MMA this warp issued has completed before tensor memory is freed.
            if (elect_one()) {
                tc_commit(bar(A_DRAIN + who));
                mbar_wait_drain(bar(A_DRAIN + who), 0, lim);
            }
            __syncwarp();
        }
        tc_fence_before();
        cta_sync(kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
        return;
    }

    regs_inc<kRegsHigh>();
    // ================= compute warps (4-11) =================
    const int half = (warp - 4) >> 2;    // query columns 64 half .. + 63
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // key row of the block == TMEM lane
    const int key = key0 + r;            // key within the sequence
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t c_s = 64 * half, c_dp = 128 + 64 * half;
    const uint32_t p_row = sbase + L::kP + half * kPanelBytes + r * 128;
    const uint32_t p_sw = static_cast<uint32_t>(r & 7);
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int n = 0; ok && n < n_steps; ++n) {
        const int ib = step_block(n);
        // lse2 / delta of this thread's 64 query columns (they landed with Q_n,
        // whose barrier S^T_n's product already waited on)
        const uint32_t aux = sbase + L::kAuxR + (n % kSlots) * L::kAux + 256 * half;
        if (!warp_wait(bar(A_S_FULL), n & 1, abort_flag, p.err, lim) ||
            !warp_wait(bar(A_Q_FULL + n % kSlots), (n / kSlots) & 1, abort_flag, p.err, lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // P^T = 2^(S^T c - lse2); causal: query q sees this key iff q >= key - diag,
        // i.e. local column cl < lo is masked (only near the diagonal).
        float2 pv[32];
        const int lo = CAUSAL ? key - diag - ib * kBlockM - 64 * half : -1;
        const bool masked = CAUSAL && __any_sync(0xffffffffu, lo > 0);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t w[32];
            tmem_ld32(t_row + c_s + 32 * ch, w);
            if (ch == 1) {
                // S^T_n is in registers: the issuer may overwrite its columns.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(A_S_FREE));
            }
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 l = ld_shared_f4(aux + 4 * (32 * ch + 4 * q4));
                const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(w[4 * q4]), __uint_as_float(w[4 * q4 + 1])),
                                             c2, make_float2(-l.x, -l.y));
                const float2 x1 = __ffma2_rn(
                    make_float2(__uint_as_float(w[4 * q4 + 2]), __uint_as_float(w[4 * q4 + 3])), c2,
                    make_float2(-l.z, -l.w));
                pv[16 * ch + 2 * q4] = make_float2(ex2(x0.x), ex2(x0.y));
                pv[16 * ch + 2 * q4 + 1] = make_float2(ex2(x1.x), ex2(x1.y));
            }
        }
        if (masked) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (2 * i < lo) pv[i].x = 0.f;
                if (2 * i + 1 < lo) pv[i].y = 0.f;
            }
        }
        // dV of step n-1 has read the P^T tile.
        if (n > 0 && !warp_wait(bar(A_P_EMPTY), (n - 1) & 1, abort_flag, p.err, lim)) {
            ok = false;
            break;
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const uint32_t addr = p_row + ((static_cast<uint32_t>(cc) ^ p_sw) << 4);
            st_shared_v4(addr, pack_bf16x2(pv[4 * cc].x, pv[4 * cc].y), pack_bf16x2(pv[4 * cc + 1].x, pv[4 * cc + 1].y),
                         pack_bf16x2(pv[4 * cc + 2].x, pv[4 * cc + 2].y), pack_bf16x2(pv[4 * cc + 3].x, pv[4 * cc + 3].y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(A_P_FULL));
        // dS^T = P^T (dP^T - delta), as bf16 pairs over this thread's dP^T columns.
        if (!warp_wait(bar(A_DP_FULL), n & 1, abort_flag, p.err, lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t pk[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t w[32];
            tmem_ld32(t_row + c_dp + 32 * ch, w);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 dl = ld_shared_f4(aux + 512 + 4 * (32 * ch + 4 * q4));
                const int i = 16 * ch + 2 * q4;
                const float2 a = __fmul2_rn(pv[i], __fadd2_rn(make_float2(__uint_as_float(w[4 * q4]),
                                                                          __uint_as_float(w[4 * q4 + 1])),
                                                              make_float2(-dl.x, -dl.y)));
                const float2 b = __fmul2_rn(pv[i + 1], __fadd2_rn(make_float2(__uint_as_float(w[4 * q4 + 2]),
                                                                              __uint_as_float(w[4 * q4 + 3])),
                                                                  make_float2(-dl.z, -dl.w)));
                pk[i] = pack_bf16x2(a.x, a.y);
                pk[i + 1] = pack_bf16x2(b.x, b.y);
            }
        }
        tmem_st32(t_row + c_dp, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(A_DS_FULL));
    }
    // ---- epilogue: dV and scale dK -> bf16, this thread's d / 2 columns of its key row
    if (ok) ok = warp_wait(bar(A_DONE), 0, abort_flag, p.err, lim) && warp_wait(bar(A_DONE + 1), 0, abort_flag, p.err, lim);
    if (ok) {
        tc_fence_after();
        const bool store = r < rows_here;
        const size_t off = (static_cast<size_t>(g.k_start + key) * p.Hkv + hk) * D + half * (D / 2);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t col = (which == 0 ? 256u : 384u) + half * (D / 2);
            const float mul = which == 0 ? 1.f : p.scale;
            uint16_t* dst = static_cast<uint16_t*>(which == 0 ? p.dv : p.dk) + off;
            // 32-byte stores when the tensor is 32-byte aligned (a row share is
            // D bytes, so every row share is then aligned too)
            const bool v8 = (reinterpret_cast<uintptr_t>(which == 0 ? p.dv : p.dk) & 31u) == 0;
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
                uint32_t v[32];
                tmem_ld32(t_row + col + ch * 32, v);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
                if (store) {
                    if (v8) {
                        st_global_v8(dst + ch * 32, pk);
                        st_global_v8(dst + ch * 32 + 16, pk + 8);
                    } else {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    cta_sync(kThreads);
}

// ============================================================== dQ

// One CTA: query rows [128 i, 128 i + 128) of head h.  Step j walks the
// visible 128-key blocks of kv head h / group:
//
//   S    = Q_i K_j^T         SS, K-major both        -> TMEM S[j % 2]
//   dP   = dO_i V_j^T        SS, K-major both        -> TMEM [256, 384)
//   dS   = P (dP - delta),   P = 2^(S c - lse2)      -> bf16 pairs over S[j % 2]
//   dQ  += dS K_j            TS, K_j MN-major         -> TMEM [384, 384 + d)
//
// S is double-buffered ([0, 128) and [128, 256)) so that S_{j+1} is computed
// while the compute warps still work on step j; a buffer is reused once the
// dQ product that read its dS has completed.  K_j and V_j have rings of
// their own: K_j is read by the first and the last product of a step, V_j
// only by dP, so V slots turn over much sooner.
template <int D>
struct DqSmem {
    static constexpr uint32_t kTile = 128 * D * 2;
    static constexpr int kKSlots = D == 128 ? 3 : 4;
    static constexpr int kVSlots = D == 128 ? 2 : 4;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kDO = kQ + kTile;
    static constexpr uint32_t kKR = kDO + kTile;
    static constexpr uint32_t kVR = kKR + kKSlots * kTile;
    static constexpr uint32_t kBar = kVR + kVSlots * kTile;
    static constexpr uint32_t kNumBars = 32;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    static constexpr uint32_t kDyn = (kUsed + 1024) > 118784u ? (kUsed + 1024) : 118784u;
};

enum DqBar : uint32_t {
    B_QD_FULL = 0,    // Q_i and dO_i
    B_K_FULL = 1,     // + slot (4)
    B_K_EMPTY = 5,    // + slot (4)
    B_V_FULL = 9,     // + slot (4)
    B_V_EMPTY = 13,   // + slot (4)
    B_S_FULL = 17,    // + buffer (2)
    B_DP_FULL = 19,
    B_DP_FREE = 20,   // compute warps have read dP_j (8 arrivals)
    B_DS_FULL = 21,   // dS_j in TMEM (8 arrivals)
    B_DQ_DONE = 22,   // dQ += dS_j K_j done
    B_DQ_FINAL = 23,
    B_DRAIN = 24,     // + issuer (2)
    B_COUNT = 26,
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BackwardParams p) {
    using L = DqSmem<D>;
    constexpr int kPanels = D / 64;
    constexpr int kKS = L::kKSlots, kVS = L::kVSlots;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);  // S, dP
    constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, true);     // dQ

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](uint32_t id) { return sbase + L::kBar + id * 8; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // With causal masking the last query blocks see the most keys: block rank
    // r is query block num_q_blocks - 1 - r.
    const int seq = blockIdx.z;
    int rank, h;
    grid_order<CAUSAL>(static_cast<int>(blockIdx.x), p.num_q_blocks, p.H, rank, h);
    const int ib = CAUSAL ? (p.num_q_blocks - 1 - rank) : rank;
    const int hk = h / p.group;
    Geom g;
    // This grid may start while the dK/dV grid ahead of it still runs (it
    // reads none of dK/dV); every CTA waits for that grid before it exits, so
    // that the work behind this one in the stream finds dK and dV written.
    if (!seq_geom(p, seq, ib == 0 && h == 0 && threadIdx.x == 0, g)) {
        grid_dependency_wait();
        return;
    }
    const int row0 = ib * kBlockM;
    if (row0 >= g.Lq) {
        grid_dependency_wait();
        return;
    }
    const int diag = g.Lk - g.Lq;
    const int r_last = min(g.Lq, row0 + kBlockM) - 1;
    int n_steps = (g.Lk + kBlockN - 1) / kBlockN;
    if (CAUSAL) {
        const int max_key = r_last + diag;
        n_steps = max_key < 0 ? 0 : min(n_steps, max_key / kBlockN + 1);
    }
    const int rows_here = r_last - row0 + 1;
    // Step j reads key block kblock(j): each CTA starts its walk at its own
    // offset, so the CTAs of a head ask for different K / V tiles at once.
    const int rot = n_steps > 0 ? ib % n_steps : 0;
    auto kblock = [&](int j) {
        const int m = j + rot;
        return m >= n_steps ? m - n_steps : m;
    };
    if (n_steps == 0) {
        // No row of the block sees a key: dQ = 0.
        for (int e = threadIdx.x; e < rows_here * (D / 8); e += kThreads) {
            const int rr = e / (D / 8), cc = e % (D / 8);
            const size_t off = (static_cast<size_t>(g.q_start + row0 + rr) * p.H + h) * D + cc * 8;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + off) = make_uint4(0, 0, 0, 0);
        }
        grid_dependency_wait();
        return;
    }

    // K_j or V_j into slot j % slots of its ring
    auto load_kv = [&](bool is_k, int j) {
        const int sl = j % (is_k ? kKS : kVS);
        const uint32_t full = (is_k ? B_K_FULL : B_V_FULL) + sl;
        mbar_arrive_expect_tx(bar(full), L::kTile);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn)
            tma_load_3d(sbase + (is_k ? L::kKR : L::kVR) + sl * L::kTile + pn * kPanelBytes, is_k ? &tm_k : &tm_v,
                        bar(full), pn * 64, hk, g.k_start + kblock(j) * kBlockN);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(B_DP_FREE), 8);
        mbar_init(bar(B_DS_FULL), 8);
        *abort_flag = 0;
        fence_barrier_init();
        // The first loads need only the barriers: issue them now, so that they
        // overlap the tensor-memory allocation and the CTA barrier.  Q and dO,
        // then step 0's K and V.
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_arrive_expect_tx(bar(B_QD_FULL), 2 * L::kTile);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn) {
            tma_load_3d(sbase + L::kQ + pn * kPanelBytes, &tm_q, bar(B_QD_FULL), pn * 64, h, g.q_start + row0);
            tma_load_3d(sbase + L::kDO + pn * kPanelBytes, &tm_do, bar(B_QD_FULL), pn * 64, h, g.q_start + row0);
        }
        load_kv(true, 0);
        load_kv(false, 0);
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    const uint64_t lim = p.wait_limit_ns;

    constexpr uint32_t kRegsLow = 88, kRegsHigh = 208;
    static_assert(128 * kRegsLow + 256 * kRegsHigh <= 168 * kThreads, "register split exceeds the launch");
    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0 || warp == 2) {
            // ================= TMA producers: warp 0 Q, dO and the K ring;
            // warp 2 the V ring =================
            const bool is_k = warp == 0;
            if (lane == 0) {
                const int nslots = is_k ? kKS : kVS;
                const uint32_t full = is_k ? B_K_FULL : B_V_FULL, empty = is_k ? B_K_EMPTY : B_V_EMPTY;
                bool ok = true;
                // (Q, dO and step 0 were issued before the CTA barrier.)
                for (int j = 1; ok && j < n_steps; ++j) {
                    const int sl = j % nslots;
                    if (j >= nslots) ok = mbar_wait(bar(empty + sl), ((j / nslots) - 1) & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    load_kv(is_k, j);
                }
                // Drain: the last fill of every slot (and Q / dO).
                if (is_k) mbar_wait_drain(bar(B_QD_FULL), 0, lim);
                for (int sl = 0; sl < nslots && sl < n_steps; ++sl) {
                    const int last = sl + ((n_steps - 1 - sl) / nslots) * nslots;
                    mbar_wait_drain(bar(full + sl), (last / nslots) & 1, lim);
                }
            }
            __syncwarp();
        } else {
            // ================= MMA issuers: warp 1 S and dQ (the K ring),
            // warp 3 dP (the V ring) =================
            const int who = warp == 1 ? 0 : 1;
            const uint64_t dq_a = sdesc_sw128(sbase + L::kQ, 16, 1024);
            const uint64_t ddo_a = sdesc_sw128(sbase + L::kDO, 16, 1024);
            const uint64_t dk_b = sdesc_sw128(sbase + L::kKR, 16, 1024);
            const uint64_t dk_mn = sdesc_sw128(sbase + L::kKR, kPanelBytes, 1024);
            const uint64_t dv_b = sdesc_sw128(sbase + L::kVR, 16, 1024);
            const uint32_t t_dp = tmem + 256, t_dq = tmem + 384;
            bool ok = warp_wait(bar(B_QD_FULL), 0, abort_flag, p.err, lim);
            auto issue_s = [&](int j) {
                const int ks = j % kKS;
                ok = ok && warp_wait(bar(B_K_FULL + ks), (j / kKS) & 1, abort_flag, p.err, lim);
                if (!ok) return;
                tc_fence_after();
                const uint64_t b0 = dk_b + ((ks * L::kTile) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + 128 * (j & 1), dq_a + kmajor_step(kk), b0 + kmajor_step(kk), kIdescS,
                               kk > 0 ? 1u : 0u);
                    tc_commit(bar(B_S_FULL + (j & 1)));
                }
                __syncwarp();
            };
            auto issue_dp = [&](int j) {
                const int vs = j % kVS;
                ok = ok && warp_wait(bar(B_V_FULL + vs), (j / kVS) & 1, abort_flag, p.err, lim);
                if (!ok) return;
                tc_fence_after();
                const uint64_t b0 = dv_b + ((vs * L::kTile) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(t_dp, ddo_a + kmajor_step(kk), b0 + kmajor_step(kk), kIdescS, kk > 0 ? 1u : 0u);
                    tc_commit(bar(B_DP_FULL));
                    tc_commit(bar(B_V_EMPTY + vs));
                }
                __syncwarp();
            };
            // dQ += dS_j K_j: dS from S[j % 2], keys 16 kk .. + 15 at columns
            // 64 (kk / 4) + 8 (kk % 4); K_j as N = d x K = 128 keys (MN-major).
            auto issue_dq = [&](int j) {
                const int ks = j % kKS;
                const uint64_t b0 = dk_mn + ((ks * L::kTile) >> 4);
                const uint32_t a0 = tmem + 128 * (j & 1);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        mma_ts(t_dq, a0 + 64 * (kk >> 2) + 8 * (kk & 3), b0 + ((kk * 16 * 128) >> 4), kIdescQ,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar(B_DQ_DONE));
                    tc_commit(bar(B_K_EMPTY + ks));
                    if (j == n_steps - 1) tc_commit(bar(B_DQ_FINAL));
                }
                __syncwarp();
            };
            if (who == 0) {
                issue_s(0);
                for (int j = 0; ok && j < n_steps; ++j) {
                    if (j + 1 < n_steps) {
                        // S[(j+1) % 2] held dS_{j-1}: dQ of step j-1 has read it.
                        if (j >= 1) ok = ok && warp_wait(bar(B_DQ_DONE), (j - 1) & 1, abort_flag, p.err, lim);
                        issue_s(j + 1);
                    }
                    ok = ok && warp_wait(bar(B_DS_FULL), j & 1, abort_flag, p.err, lim);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dq(j);
                }
            } else {
                issue_dp(0);
                for (int j = 0; ok && j + 1 < n_steps; ++j) {
                    // dP_{j+1} overwrites dP_j: the compute warps have read it.
                    ok = ok && warp_wait(bar(B_DP_FREE), j & 1, abort_flag, p.err, lim);
                    // S_{j+1} goes through the tensor pipe first: the compute
                    // warps need it first, dP_{j+1} only after their exponentials.
                    ok = ok && warp_wait(bar(B_S_FULL + ((j + 1) & 1)), ((j + 1) >> 1) & 1, abort_flag, p.err, lim);
                    issue_dp(j + 1);
                }
            }
            if (elect_one()) {
                tc_commit(bar(B_DRAIN + who));
                mbar_wait_drain(bar(B_DRAIN + who), 0, lim);
            }
            __syncwarp();
        }
        tc_fence_before();
        cta_sync(kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
        grid_dependency_wait();
        return;
    }

    regs_inc<kRegsHigh>();
    // ================= compute warps (4-11) =================
    const int half = (warp - 4) >> 2;   // key columns 64 half .. + 63 of each block
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the block == TMEM lane
    const int row = row0 + r;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const long long woff = h * p.ws_head_stride + bwd_ws_seq_offset(g.q_start, seq) + row;
    const float lse2 = p.ws[woff];                              // padded rows: +inf
    const float delta = p.ws[woff + p.H * p.ws_head_stride];    // padded rows: 0
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 nl2 = make_float2(-lse2, -lse2);
    const float2 nd2 = make_float2(-delta, -delta);
    bool ok = true;
    for (int j = 0; ok && j < n_steps; ++j) {
        const uint32_t c_s = 128 * (j & 1) + 64 * half;
        if (!warp_wait(bar(B_S_FULL + (j & 1)), (j >> 1) & 1, abort_flag, p.err, lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t u[64];
        tmem_ld64(t_row + c_s, u);
        // keys past the sequence, and (causal) keys past row + diag, get P = 0
        // (only blocks that reach past the sequence end or the diagonal)
        const int kbase = kblock(j) * kBlockN + 64 * half;
        int lim_c = g.Lk - 1 - kbase;
        if (CAUSAL) lim_c = min(lim_c, row + diag - kbase);
        const bool masked = __any_sync(0xffffffffu, lim_c < 63);
        float2 pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])), c2, nl2);
            pv[i] = make_float2(ex2(x.x), ex2(x.y));
        }
        if (masked) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (2 * i > lim_c) pv[i].x = 0.f;
                if (2 * i + 1 > lim_c) pv[i].y = 0.f;
            }
        }
        if (!warp_wait(bar(B_DP_FULL), j & 1, abort_flag, p.err, lim)) {
            ok = false;
            break;
        }
        tc_fence_after();
        tmem_ld64(t_row + 256 + 64 * half, u);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DP_FREE));
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float2 ds = __fmul2_rn(pv[i], __fadd2_rn(make_float2(__uint_as_float(u[2 * i]),
                                                                        __uint_as_float(u[2 * i + 1])), nd2));
            pk[i] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st32(t_row + c_s, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DS_FULL));
    }
    if (ok) ok = warp_wait(bar(B_DQ_FINAL), 0, abort_flag, p.err, lim);
    if (ok) {
        tc_fence_after();
        const bool store = row <= r_last;
        uint16_t* dst = static_cast<uint16_t*>(p.dq) + (static_cast<size_t>(g.q_start + row) * p.H + h) * D +
                        half * (D / 2);
        const bool v8 = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;  // 32-byte stores
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch) {
            uint32_t v[32];
            tmem_ld32(t_row + 384 + half * (D / 2) + ch * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * p.scale, __uint_as_float(v[2 * i + 1]) * p.scale);
            if (store) {
                if (v8) {
                    st_global_v8(dst + ch * 32, pk);
                    st_global_v8(dst + ch * 32 + 16, pk + 8);
                } else {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
    }
    tc_fence_before();
    cta_sync(kThreads);
    grid_dependency_wait();
}

// ============================================================== launch

template <int D, bool CAUSAL>
cudaError_t launch_dc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const BackwardParams& p, cudaStream_t stream) {
    static_assert(DkdvSmem<D>::kDyn <= 232448u && DqSmem<D>::kDyn <= 232448u, "shared memory budget");
    static_assert(DkdvSmem<D>::kSlots <= 4 && DqSmem<D>::kKSlots <= 4 && DqSmem<D>::kVSlots <= 4, "barrier slots");
    const dim3 gp(p.num_q_blocks, p.H, p.num_seqs);
    bwd_prep_kernel<D><<<gp, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    auto ka = bwd_dkdv_kernel<D, CAUSAL>;
    e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(DkdvSmem<D>::kDyn));
    if (e != cudaSuccess) return e;
    ka<<<dim3(p.num_k_blocks * p.Hkv, 1, p.num_seqs), kThreads, DkdvSmem<D>::kDyn, stream>>>(tq, tk, tv, tdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // dQ needs only the prep kernel's lse2 / delta (complete before any dK/dV
    // CTA ran), so it is launched to start in the dK/dV grid's tail.
    auto kb = bwd_dq_kernel<D, CAUSAL>;
    e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(DqSmem<D>::kDyn));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_q_blocks * p.H, 1, p.num_seqs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = DqSmem<D>::kDyn;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kb, tq, tk, tv, tdo, p);
}

}  // namespace

cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BackwardParams& p, int d, bool causal,
                            cudaStream_t stream) {
    if (d == 128)
        return causal ? launch_dc<128, true>(tq, tk, tv, tdo, p, stream) : launch_dc<128, false>(tq, tk, tv, tdo, p, stream);
    return causal ? launch_dc<64, true>(tq, tk, tv, tdo, p, stream) : launch_dc<64, false>(tq, tk, tv, tdo, p, stream);
}

}  // namespace fa
