// Prefill forward (dense and varlen) for sm_103a: TMA-staged tiles, tcgen05
// MMA into tensor memory, one thread per query row for the online softmax.
//
// What one CTA computes: two tiles of kBlockM = 128 query rows (256 rows) of
// one (sequence, head), streaming the sequence's K/V in kBlockN = 128-key
// blocks (tiling, dlog.com.cn "从标准 Attention 到 FlashAttention 与分页执行"
// §2.1; the (Q block, batch*head) grid of the lqnn.cn page §4.4).  For every
// K/V block j and each tile t:
//
//   S^t_j = Q^t K_j^T                    tcgen05.mma, SMEM x SMEM -> TMEM (fp32)
//   m'    = max(m, rowmax(S^t_j scale))   softmax warps, one thread per row
//   P^t_j = exp(S^t_j scale - m)          -> bf16 rows into shared memory
//                                          (d = 128) or into TMEM behind O^t (d = 64)
//   l     = l exp(m_old - m) + rowsum P^t_j
//   O^t  += P^t_j V_j                     tcgen05.mma, SMEM (or TMEM) x SMEM -> TMEM
//
// and at the end O / l and lse = m + ln l (online softmax, same page §2.2).
// The two tiles share every K/V load.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: the K/V ring (its lane 0, thread 0, also
//                initialises the barriers and issues both Q tiles and, with
//                contiguous K/V, the first K block before the CTA barrier, so
//                that those loads overlap the TMEM allocation)
//   warp 1       allocates tensor memory; issues tile 0's tcgen05.mma
//   warp 2       issues tile 1's tcgen05.mma
//                (the whole warp runs the issue loop, with its waits and
//                descriptor arithmetic warp-uniform; one elected lane
//                executes each tcgen05.mma / commit, which keeps the
//                per-MMA issue cost low enough to feed the tensor core)
//   warp 3       idle
//   warps 4-7    softmax, correction and epilogue of tile 0
//   warps 8-11   the same for tile 1
// Warp w may only touch TMEM lanes 32*(w%4)..+31; within a softmax warp
// group, thread r of the group owns row r of its tile = TMEM lane r.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128) S^0   [128,256) S^1   [256,256+d) O^0   [384,384+d) O^1
//   (d = 64: P^t as bf16 pairs in the 64 columns behind O^t)
//
// Decoupled S and P.  P^t_j goes to its own shared-memory tile (128 rows x
// 128 keys, the K-major 128-byte-swizzled layout the MMA reads) or, at
// d = 64, to the TMEM columns behind O^t, never over S^t, so S^t's columns
// are free as soon as the softmax has read them.  The softmax signals that right after its tensor-memory load,
// and the issuer starts S^t_{j+1} while the softmax is still computing
// P^t_j.  Per tile the issue order is S_0, S_1, PV_0, S_2, PV_1, ...; the
// softmax warps of a tile therefore run block after block without waiting
// on the tensor core, and the tensor core works on both tiles' S and P.V
// products underneath.
//
// Shared memory: Q (two tiles), P (two tiles), and a ring of kSlots K/V
// tiles loaded in the order K_0, K_1, V_0, K_2, V_1, K_3, ... (K one block
// ahead of V, the order the MMAs consume them).  A slot is released per tile
// (one empty barrier per tile and slot, committed after that tile's MMAs
// that read it); the producer waits for every tile that read the slot's
// previous occupant.
//
// Rescaling: the exponent reference m is only moved when a row's max grows
// by more than kRescaleThreshold (log2 units); otherwise the old reference is
// kept and P may exceed 1 (at most 2^8).  The result is the same softmax
// (the reference cancels in O/l and is added back in the LSE); it saves the
// TMEM read-modify-write of O on almost every block.
//
// Masking: keys at or past the sequence end are -inf (tail of the last
// block); with causal, key j > i + (Lk - Lq) is -inf (bottom-right).  Blocks
// entirely above the diagonal are never loaded (tile skipping).  Query rows
// past the sequence end are computed on whatever rows TMA brought in but
// never stored.
//
// Epilogue: O^t / l to bf16, one row per thread, 32-byte stores when the
// output is 32-byte aligned; LSE per row.
//
// Variants (template parameters):
//   PAGED   K/V come through a page table: the producer issues one box of a
//           page's rows (16 to 128) per page and panel, each lane one box, the
//           table entries fetched a block ahead (prefill chunks that continue
//           a cached prefix).
//   SLOTS   contiguous varlen with fewer sequences than a CTA has threads:
//           the grid numbers (sequence, 256-row block) slots instead of
//           giving every sequence max_seqlen / 256 blocks (launch_t).
// Dispatch order (cta_unit): non-causal CTAs run the Q blocks of a head
// together; causal ones hand out the heaviest Q blocks first, at d = 128 in
// groups of 8 heads so that few heads' K/V are live in L2 at once.  Dense
// CTAs also prefetch into L2 the Q tiles of the CTA one wave later.

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kTiles = 2;  // Q tiles per CTA
constexpr float kRescaleThreshold = 8.0f;
constexpr float kPBound = 256.0f;  // 2^kRescaleThreshold: the largest P the reference allows
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kPanelBytes = 128 * 128;  // 128 rows x 64 bf16: a panel of a Q or P tile
constexpr int kMaxSlots = 6;

// Threads per CTA: 4 control warps and 4 softmax warps per Q tile.
constexpr int kThreads = 128 + kTiles * 128;

// Two Q tiles, 128-key K/V blocks, a 3-slot K/V ring at d = 128 (6 at
// d = 64), all 512 TMEM columns (S^0 | S^1 | O^0 | O^1), one CTA per SM.
template <int D>
struct PrefillSmem {
    static constexpr int kBN = kBlockN;                         // keys per K/V block
    static constexpr uint32_t kQTile = kBlockM * D * 2;         // one Q tile
    static constexpr uint32_t kQPanel = kBlockM * 128;          // one 64-column panel of it
    static constexpr uint32_t kKVTile = kBN * D * 2;            // one K or V tile
    static constexpr uint32_t kKVPanel = kBN * 128;             // one 64-column panel of it
    static constexpr uint32_t kPTile = kBlockM * kBN * 2;       // one P tile
    static constexpr int kSlots = D == 128 ? 3 : 6;             // K/V ring
    static constexpr uint32_t kQ = 0;                           // + t * kQTile
    static constexpr uint32_t kP = kQ + kTiles * kQTile;        // + t * kPTile
    static constexpr uint32_t kKV = kP + kTiles * kPTile;       // + slot * kKVTile
    static constexpr uint32_t kBar = kKV + kSlots * kKVTile;
    static constexpr uint32_t kNumBars = 40;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    // Requested dynamic size: 1 KiB alignment slack; a prefill CTA asks for
    // at least 116 KiB so that it has its SM (and the 512 TMEM columns) alone.
    static constexpr uint32_t kDyn = (kUsed + 1024) > 118784u ? (kUsed + 1024) : 118784u;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kOCol = 256;                      // O^t at kOCol + t * 128
    // At d = 64, O^t uses 64 of its 128 columns and P^t (128 keys as bf16
    // pairs) the other 64: the P.V product reads its A operand from TMEM.
    static constexpr bool kPInTmem = D == 64;
    static constexpr uint32_t kPColOff = 64;                    // P^t at O^t + kPColOff
};

enum BarId : uint32_t {
    B_Q_FULL = 0,     // + tile
    B_KV_FULL = 2,    // + slot
    B_KV_EMPTY = 8,   // + tile * kMaxSlots + slot
    B_S_FULL = 20,    // + tile: S^t_j is in TMEM
    B_S_FREE = 22,    // + tile: the softmax has read S^t_j
    B_P_FULL = 24,    // + tile: P^t_j is in shared memory
    B_P_EMPTY = 26,   // + tile: PV^t_j is done (P tile free, O^t current)
    B_O_FINAL = 28,   // + tile
    B_MMA_DONE = 30,  // + tile
    B_EXP_TURN = 32,  // + tile: the other tile has finished its exponentials
    B_V_TAIL = 34,    // paged: stale rows of the last V tile are zeroed
    B_COUNT = 35,
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Position of K_j / V_j in the load sequence K_0, K_1, V_0, K_2, V_1, ...,
// K_{n-1}, V_{n-2}, V_{n-1} (n = blocks the CTA streams).
__device__ __forceinline__ int pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int pos_v(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * n - 1; }

// Keys visible to some row of the tile [r0, r_last]: the number of BN-key
// K/V blocks the tile needs (0 if the tile has no valid row or sees no key).
template <bool CAUSAL, int BN>
__device__ __forceinline__ int tile_blocks(int r0, int r_last, int Lk, int diag) {
    if (r_last < r0) return 0;
    int n = (Lk + BN - 1) / BN;
    if (CAUSAL) {
        const int max_key = r_last + diag;
        n = max_key < 0 ? 0 : min(n, max_key / BN + 1);
    }
    return n;
}

// Work unit of grid position (x, y): a 256-row Q block and a head.
// Non-causal: grid (block, head), blocks fastest, so the CTAs resident at
// once cover few heads and their K/V stay in L2.  Causal: grid.x enumerates
// (block, head) pairs in groups of heads, the blocks of a group from the
// last (most keys) to the first and the group's heads fastest, so the heavy
// work of every group is handed out early.  At d = 128 a group is 8 heads,
// which keeps the K/V live at once within L2 (B1 H32 N8192: 0.353 -> 0.342
// ms against all heads at once).  At d = 64 every head's K/V fits in L2:
// grid (head, block from the last), all heads at once, balances better
// (0.301 against 0.308 ms).
template <int D, bool CAUSAL>
__device__ __forceinline__ void cta_unit(int x, int y, int nblk, int nheads, int& qb, int& h) {
    if (!CAUSAL) {
        qb = x;
        h = y;
        return;
    }
    if (D != 128) {  // grid (head, block from the last)
        h = x;
        qb = nblk - 1 - y;
        return;
    }
    constexpr int hg = 8;
    const int per = hg * nblk;
    const int grp = x / per;
    const int gs = min(hg, nheads - grp * hg);
    const int rem = x - grp * per;
    qb = nblk - 1 - rem / gs;
    h = grp * hg + rem % gs;
}

template <int D, bool CAUSAL, bool PAGED, bool SLOTS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using L = PrefillSmem<D>;
    constexpr int kBN = L::kBN;
    constexpr int kPanels = D / 64;
    constexpr int kSlots = L::kSlots;
    constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBN, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, true);
    constexpr bool kPInTmem = L::kPInTmem;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](uint32_t id) { return sbase + L::kBar + id * 8; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nblk = (p.num_q_blocks + kTiles - 1) / kTiles;  // Q blocks of kTiles tiles
    // Dispatch order: cta_unit above, grid.z the sequence; or, for a varlen
    // grid that numbers its (sequence, block) slots (SLOTS), the slot (grid.y
    // causal, grid.x otherwise) and the head (the other one).  Slots
    // [B_s, B_{s+1}) belong to sequence s, B_s = s + floor(cu_q[s] / 256):
    // at least ceil(Lq / 256) of them, sequence by sequence, so that no
    // launch holds max_seqlen / 256 blocks for every sequence.
    int seq = blockIdx.z;
    int qb = 0, h = 0;
    int slot_rank = 0;  // slot grids: the slot's rank among its sequence's slots
    if constexpr (SLOTS) {
        const int y = static_cast<int>(CAUSAL ? blockIdx.y : blockIdx.x);
        h = static_cast<int>(CAUSAL ? blockIdx.x : blockIdx.y);
        const int t = threadIdx.x;  // sequence boundary t (the host keeps num_seqs < kThreads)
        const int cq = t <= p.num_seqs ? p.cu_q[t] : 0;
        seq = __syncthreads_count(t >= 1 && t <= p.num_seqs && t + cq / (kBlockM * kTiles) <= y);
        if (blockIdx.x == 0 && blockIdx.y == 0 && t < p.num_seqs) {
            // This CTA checks every sequence's offsets, since a sequence with
            // bad ones may own no slot.
            const int q0 = cq, lq = p.cu_q[t + 1] - cq, k0 = p.cu_k[t], lk = p.cu_k[t + 1] - k0;
            if (q0 < 0 || lq < 0 || lk < 0 || q0 + lq > p.total_q || lq > p.max_seqlen_q || lk > p.max_seqlen_k ||
                (PAGED ? lk > (static_cast<long long>(p.max_pages) << p.page_shift) : (k0 < 0 || k0 + lk > p.total_k)))
                atomicOr(p.err, FA_DEVERR_INDEX);
        }
        if (seq >= p.num_seqs) return;  // past the last sequence's slots
        slot_rank = y - (seq + p.cu_q[seq] / (kBlockM * kTiles));
    } else {
        cta_unit<D, CAUSAL>(static_cast<int>(blockIdx.x), static_cast<int>(blockIdx.y), nblk, p.H, qb, h);
    }
    const int hk = h / p.group;

    // ---- sequence geometry (uniform over the CTA)
    int q_start, Lq, k_start, Lk;
    const int* bt_row = PAGED ? p.block_table + static_cast<size_t>(seq) * p.max_pages : nullptr;
    if (p.cu_q != nullptr) {
        q_start = p.cu_q[seq];
        Lq = p.cu_q[seq + 1] - q_start;
        k_start = p.cu_k[seq];
        Lk = p.cu_k[seq + 1] - k_start;
        const bool bad = q_start < 0 || Lq < 0 || Lk < 0 || q_start + Lq > p.total_q || Lq > p.max_seqlen_q ||
                         Lk > p.max_seqlen_k ||
                         (PAGED ? Lk > (static_cast<long long>(p.max_pages) << p.page_shift)
                                : (k_start < 0 || k_start + Lk > p.total_k));
        if (bad) {
            if (threadIdx.x == 0 && qb == 0) atomicOr(p.err, FA_DEVERR_INDEX);
            return;
        }
    } else {
        q_start = seq * p.N;
        Lq = p.N;
        k_start = seq * p.N;
        Lk = p.N;
    }
    if constexpr (SLOTS) {
        // the sequence's blocks in the slot order: the heaviest first under the
        // causal mask, in order otherwise; slots past them stay empty
        const int nb_seq = (Lq + kBlockM * kTiles - 1) / (kBlockM * kTiles);
        if (slot_rank < 0 || slot_rank >= nb_seq) return;
        qb = CAUSAL ? nb_seq - 1 - slot_rank : slot_rank;
    }
    const int row0 = qb * kBlockM * kTiles;
    if (row0 >= Lq) return;
    const int diag = Lk - Lq;  // causal: key j visible to row i iff j <= i + diag
    int r_last[kTiles], nb[kTiles];
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        r_last[t] = min(Lq, row0 + (t + 1) * kBlockM) - 1;
        nb[t] = tile_blocks<CAUSAL, kBN>(row0 + t * kBlockM, r_last[t], Lk, diag);
    }
    const int nmax = max(nb[0], nb[1]);
    // Paged keys whose last page is only partly used: the stale slots past Lk
    // are loaded with the page, and their V rows are zeroed before the last
    // P.V (P is 0 there, but 0 * a non-finite stale value would not be).
    const int page_rows = PAGED ? 1 << p.page_shift : 1;  // tokens per page
    const bool v_tail = PAGED && (Lk & (page_rows - 1)) != 0 && nmax > 0 && (Lk - 1) / kBN == nmax - 1;
    const long long lse_base = p.cu_q ? q_start : static_cast<long long>(seq) * p.H * p.N;
    const float NEG_INF = -__int_as_float(0x7f800000);

    // Rows of a tile that sees no key at all: O = 0, LSE = -inf.
    if (warp >= 4) {
        const int t = (warp - 4) >> 2;
        const int row = row0 + t * kBlockM + (warp & 3) * 32 + lane;
        if (nb[t] == 0 && row <= r_last[t]) {
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + (static_cast<size_t>(q_start + row) * p.H + h) * D);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0, 0, 0, 0);
            if (p.lse != nullptr) p.lse[lse_base + h * p.lse_head_stride + row] = NEG_INF;
        }
    }
    if (nmax == 0) return;

    // ---- setup: barriers (thread 0), tensor memory (warp 1)
    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), 1);
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(B_S_FREE + t), 4);  // one arrive per softmax warp
            mbar_init(bar(B_P_FULL + t), 4);
            mbar_init(bar(B_EXP_TURN + t), 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
        // The first loads need only the barriers: issue them now, so that they
        // overlap the tensor-memory allocation and the CTA barrier.  The Q
        // tiles, and with contiguous K/V the first K block (ring position 0,
        // slot 0, which no tile has read before).
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
            if (nb[t] == 0) continue;
            mbar_arrive_expect_tx(bar(B_Q_FULL + t), L::kQTile);
#pragma unroll
            for (int pn = 0; pn < kPanels; ++pn)
                tma_load_3d(sbase + L::kQ + t * L::kQTile + pn * L::kQPanel, &tm_q, bar(B_Q_FULL + t), pn * 64, h,
                            q_start + row0 + t * kBlockM);
        }
        if constexpr (!PAGED) {
            mbar_arrive_expect_tx(bar(B_KV_FULL + 0), L::kKVTile);
#pragma unroll
            for (int pn = 0; pn < kPanels; ++pn)
                tma_load_3d(sbase + L::kKV + pn * L::kKVPanel, &tm_k, bar(B_KV_FULL + 0), pn * 64, hk, k_start);
        }
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    const uint64_t lim = p.wait_limit_ns;

    // Register split: 384 threads launch with 168 each (64,512 in all); the
    // producer/MMA warp group drops and the two softmax groups rise, keeping
    // the sum: 128*72 + 2*128*216 = 128*56 + 2*128*224 = 64,512.  (The pair
    // per head dim is the one ptxas allocates without spilling.)
    constexpr uint32_t kRegsLaunch = 168;
    constexpr uint32_t kRegsLow = D == 128 ? 72 : 56;
    constexpr uint32_t kRegsHigh = D == 128 ? 216 : 224;
    static_assert(kRegsLaunch * kThreads <= 65536, "launch registers");
    static_assert(128 * kRegsLow + (kThreads - 128) * kRegsHigh <= kRegsLaunch * kThreads,
                  "register split exceeds the launch");
    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0) {
            // ================= TMA producer =================
            // (The Q tiles, and with contiguous K/V the first K block, were
            // issued before the CTA barrier.)
            // Per (tile, slot): whether the tile reads the slot's current
            // occupant, and the parity of how many occupants it has read.
            uint32_t used = 0, par = 0;  // bit t * kMaxSlots + slot
            int last_fill[kMaxSlots];
#pragma unroll
            for (int s = 0; s < kMaxSlots; ++s) last_fill[s] = -1;
            auto account = [&](int i, int j) {
                const int s = i % kSlots;
                last_fill[s] = i / kSlots;
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    const uint32_t bit = 1u << (t * kMaxSlots + s);
                    if (j < nb[t]) {
                        used |= bit;
                        par ^= bit;
                    } else {
                        used &= ~bit;
                    }
                }
            };
            if constexpr (!PAGED) {
                // Contiguous K/V: lane 0 runs the loop, two boxes per tile.
                if (lane == 0) {
                    bool ok = true;
                    auto load = [&](int i, bool is_k, int j) {
                        const int s = i % kSlots;
#pragma unroll
                        for (int t = 0; t < kTiles; ++t) {
                            const uint32_t bit = 1u << (t * kMaxSlots + s);
                            if (ok && (used & bit))  // wait until tile t released the previous occupant
                                ok = mbar_wait(bar(B_KV_EMPTY + t * kMaxSlots + s), ((par & bit) ? 0u : 1u),
                                               abort_flag, p.err, lim);
                        }
                        if (!ok) return;
                        mbar_arrive_expect_tx(bar(B_KV_FULL + s), L::kKVTile);
                        const void* map = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
#pragma unroll
                        for (int pn = 0; pn < kPanels; ++pn)
                            tma_load_3d(sbase + L::kKV + s * L::kKVTile + pn * L::kKVPanel, map, bar(B_KV_FULL + s),
                                        pn * 64, hk, k_start + j * kBN);
                        account(i, j);
                    };
                    account(pos_k(0), 0);  // K_0: issued before the CTA barrier
                    for (int j = 0; ok && j < nmax; ++j) {
                        if (j + 1 < nmax) load(pos_k(j + 1), true, j + 1);
                        load(pos_v(j, nmax), false, j);
                    }
                    // Every load of this CTA is issued: pull into L2 the Q tiles
                    // of the CTA one wave of SMs further in the grid, which is
                    // about the one that takes an SM when this CTA ends.
                    if (p.cu_q == nullptr) {
                        uint32_t nsm;
                        asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
                        const long long lin = blockIdx.x + static_cast<long long>(gridDim.x) *
                                                               (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z) +
                                              nsm;
                        if (lin < static_cast<long long>(gridDim.x) * gridDim.y * gridDim.z) {
                            const int bx = static_cast<int>(lin % gridDim.x);
                            const long long r2 = lin / gridDim.x;
                            const int by = static_cast<int>(r2 % gridDim.y);
                            const int bz = static_cast<int>(r2 / gridDim.y);
                            int qb2, h2;
                            cta_unit<D, CAUSAL>(bx, by, nblk, p.H, qb2, h2);
#pragma unroll
                            for (int t = 0; t < kTiles; ++t) {
                                const int rr = qb2 * kBlockM * kTiles + t * kBlockM;
                                if (rr >= p.N) continue;
#pragma unroll
                                for (int pn = 0; pn < kPanels; ++pn)
                                    asm volatile(
                                        "cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                                            reinterpret_cast<uint64_t>(&tm_q)),
                                        "r"(pn * 64), "r"(h2), "r"(bz * p.N + rr)
                                        : "memory");
                            }
                        }
                    }
                }
            } else {
                // Paged K/V: the whole warp runs the loop (its waits are
                // warp-uniform); lane 0 posts the slot's byte count and each
                // lane issues one box (box lane / kPanels of the block, panel
                // lane % kPanels), so one instruction issues a whole tile.  A
                // box is one page, or the block's share of a page larger than
                // the block (box_rows = min(page, kBN) rows, the tensor maps'
                // box height): 16 boxes at d = 128 with 16-token pages and
                // 128-key blocks, 2 with 128-token pages.  A page past the
                // sequence, or a bad table entry, is loaded from just past the
                // pool: TMA fills zeros there (and still counts the bytes).
                const int box_rows = min(page_rows, kBN);
                const int bpb = kBN / box_rows;             // boxes per block (each panel)
                const int pg = lane / kPanels;              // this lane's box of a block
                const int pn = lane % kPanels;              // and panel
                const bool boxes = lane < bpb * kPanels;
                const int* bt = bt_row;
                // Table entries are fetched one block ahead of their use: the
                // entries of blocks j and j + 1 are in flight at once, kept by
                // block parity.
                auto fetch = [&](int blk) {
                    const int key0 = blk * kBN + pg * box_rows;  // first key of the box
                    return (boxes && blk < nmax && key0 < Lk) ? __ldg(bt + (key0 >> p.page_shift)) : -1;
                };
                int ent0 = fetch(0), ent1 = fetch(1);
                bool ok = true;
                auto load = [&](int i, bool is_k, int j) {
                    const int s = i % kSlots;
#pragma unroll
                    for (int t = 0; t < kTiles; ++t) {
                        const uint32_t bit = 1u << (t * kMaxSlots + s);
                        if (ok && (used & bit))
                            ok = warp_wait(bar(B_KV_EMPTY + t * kMaxSlots + s), ((par & bit) ? 0u : 1u), abort_flag,
                                           p.err, lim);
                    }
                    if (!ok) return;
                    if (lane == 0) mbar_arrive_expect_tx(bar(B_KV_FULL + s), L::kKVTile);
                    __syncwarp();
                    if (boxes) {
                        const void* map = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
                        const int page = (j & 1) ? ent1 : ent0;
                        const int key0 = j * kBN + pg * box_rows;
                        int row = p.num_pages << p.page_shift;
                        if (key0 < Lk) {
                            if (page >= 0 && page < p.num_pages)
                                row = (page << p.page_shift) + (key0 & (page_rows - 1));
                            else if (pn == 0 && is_k)
                                atomicOr(p.err, FA_DEVERR_INDEX);
                        }
                        tma_load_3d(sbase + L::kKV + s * L::kKVTile + pn * L::kKVPanel + pg * box_rows * 128, map,
                                    bar(B_KV_FULL + s), pn * 64, hk, row);
                    }
                    __syncwarp();
                    account(i, j);
                };
                load(pos_k(0), true, 0);
                for (int j = 0; ok && j < nmax; ++j) {
                    if (j + 1 < nmax) load(pos_k(j + 1), true, j + 1);
                    load(pos_v(j, nmax), false, j);
                    // block j is done: its parity slot takes block j + 2
                    if (j & 1)
                        ent1 = fetch(j + 2);
                    else
                        ent0 = fetch(j + 2);
                }
            }
            // Drain: every copy this CTA issued lands before the CTA exits.
            if (lane == 0) {
#pragma unroll
                for (int s = 0; s < kMaxSlots; ++s)
                    if (s < kSlots && last_fill[s] >= 0) mbar_wait_drain(bar(B_KV_FULL + s), last_fill[s] & 1, lim);
#pragma unroll
                for (int t = 0; t < kTiles; ++t)
                    if (nb[t] > 0) mbar_wait_drain(bar(B_Q_FULL + t), 0, lim);
            }
            __syncwarp();
            if (PAGED && v_tail) {
                // The whole warp zeroes rows [Lk, roundup(Lk, page)) of the
                // last V tile once it has landed, then releases the last P.V.
                const int i_last = pos_v(nmax - 1, nmax);
                if (warp_wait(bar(B_KV_FULL + i_last % kSlots), (i_last / kSlots) & 1, abort_flag, p.err, lim)) {
                    const int kb = (nmax - 1) * kBN;
                    const int r_lo = Lk - kb;
                    const int r_hi = min(((Lk + page_rows - 1) & ~(page_rows - 1)) - kb, kBN);
                    const uint32_t base = sbase + L::kKV + (i_last % kSlots) * L::kKVTile;
                    for (int e = lane; e < (r_hi - r_lo) * kPanels * 8; e += 32) {
                        const int chunk = e & 7;
                        const int pn = (e >> 3) % kPanels;
                        const int r = r_lo + (e >> 3) / kPanels;
                        st_shared_v4(base + pn * L::kKVPanel + r * 128 + chunk * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_V_TAIL));
                }
            }
        } else if (warp == 1 || warp == 2) {
            // ================= MMA issuers (warp 1: tile 0, warp 2: tile 1) =================
            const int t = warp - 1;
            const int n_t = nb[t];
            if (n_t > 0) {
                // Descriptor bases; a k-step only moves the start address, which
                // is the low field of the descriptor (addresses stay < 256 KiB, so
                // the addition never carries out of it).
                const uint64_t dq = sdesc_sw128(sbase + L::kQ + t * L::kQTile, 16, 1024);
                const uint64_t dp = sdesc_sw128(sbase + L::kP + t * L::kPTile, 16, 1024);
                const uint64_t dk = sdesc_sw128(sbase + L::kKV, 16, 1024);
                const uint64_t dv = sdesc_sw128(sbase + L::kKV, L::kKVPanel, 1024);
                const uint32_t t_s = tmem + t * 128;
                const uint32_t t_o = tmem + L::kOCol + t * 128;
                bool ok = warp_wait(bar(B_Q_FULL + t), 0, abort_flag, p.err, lim);
                auto wait_item = [&](int i) {
                    ok = ok && warp_wait(bar(B_KV_FULL + i % kSlots), (i / kSlots) & 1, abort_flag, p.err, lim);
                };
                // S^t_j = Q^t K_j^T into the S^t columns.
                auto issue_s = [&](int j) {
                    const int s = pos_k(j) % kSlots;
                    const uint64_t b0 = dk + ((s * L::kKVTile) >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t offa = ((kk >> 2) * L::kQPanel + (kk & 3) * 32) >> 4;
                            const uint32_t offb = ((kk >> 2) * L::kKVPanel + (kk & 3) * 32) >> 4;
                            mma_ss(t_s, dq + offa, b0 + offb, kIdescS, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(B_S_FULL + t));
                        tc_commit(bar(B_KV_EMPTY + t * kMaxSlots + s));
                    }
                    __syncwarp();
                };
                // O^t += P^t_j V_j, P from shared memory, or at d = 64 from
                // TMEM (keys 16 kk .. 16 kk + 15 are 8 columns at O^t + 64 + 8 kk).
                auto issue_pv = [&](int j) {
                    const int s = pos_v(j, nmax) % kSlots;
                    const uint64_t b0 = dv + ((s * L::kKVTile) >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            if constexpr (kPInTmem) {
                                mma_ts(t_o, t_o + L::kPColOff + 8 * kk, b0 + ((kk * 16 * 128) >> 4), kIdescPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                            } else {
                                const uint32_t offp = ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
                                mma_ss(t_o, dp + offp, b0 + ((kk * 16 * 128) >> 4), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        tc_commit(bar(B_P_EMPTY + t));
                        tc_commit(bar(B_KV_EMPTY + t * kMaxSlots + s));
                        if (j == n_t - 1) tc_commit(bar(B_O_FINAL + t));
                    }
                    __syncwarp();
                };
                wait_item(pos_k(0));
                if (ok) issue_s(0);
                for (int j = 0; ok && j < n_t; ++j) {
                    if (j + 1 < n_t) {
                        // S^t_{j+1} overwrites S^t_j: wait until the softmax has read it.
                        ok = ok && warp_wait(bar(B_S_FREE + t), j & 1, abort_flag, p.err, lim);
                        wait_item(pos_k(j + 1));
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(j + 1);
                    }
                    ok = ok && warp_wait(bar(B_P_FULL + t), j & 1, abort_flag, p.err, lim);
                    wait_item(pos_v(j, nmax));
                    if (PAGED && v_tail && j == nmax - 1)
                        ok = ok && warp_wait(bar(B_V_TAIL), 0, abort_flag, p.err, lim);
                    if (!ok) break;
                    tc_fence_after();  // P in TMEM (d = 64) was written by the softmax threads
                    issue_pv(j);
                }
                // Every MMA of this warp has finished before tensor memory is
                // released.
                if (elect_one()) {
                    tc_commit(bar(B_MMA_DONE + t));
                    mbar_wait_drain(bar(B_MMA_DONE + t), 0, lim);
                }
                __syncwarp();
            }
        }
        // The producer/MMA warp group ends here: join the CTA, then the
        // allocating warp frees tensor memory.
        tc_fence_before();
        cta_sync(kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, L::kTmemCols);
        }
        return;
    } else {
        regs_inc<kRegsHigh>();
        // ================= softmax / correction / epilogue =================
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;       // row of the tile == TMEM lane
        const int r0 = row0 + t * kBlockM;
        const int row = r0 + r;                   // row within the sequence
        const int n_t = t == 0 ? nb[0] : nb[1];
        const int n_other = t == 0 ? nb[1] : nb[0];  // blocks of the other tile
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t s_col = t * 128;
        const uint32_t o_col = L::kOCol + t * 128;
        // this row of the P tile (128-byte swizzle: chunk c of a 128-byte
        // panel row lands at (c ^ (row % 8)) * 16)
        const uint32_t p_row = sbase + L::kP + t * L::kPTile + r * 128;
        const uint32_t p_sw = static_cast<uint32_t>(r & 7);
        const float c = p.scale_log2;
        float m_ref = NEG_INF;  // exponent reference (log2 units)
        float l = 0.f;
        bool ok = n_t > 0;
        for (int j = 0; ok && j < n_t; ++j) {
            if (!warp_wait(bar(B_S_FULL + t), j & 1, abort_flag, p.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t u[kBN];
            if constexpr (kBN == 128)
                tmem_ld128(t_row + s_col, u);
            else
                tmem_ld64(t_row + s_col, u);
            // S^t_j is in registers: the issuer may overwrite its columns.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_FREE + t));
            const int kbase = j * kBN;
            const bool need_mask = (kbase + kBN > Lk) || (CAUSAL && kbase + kBN - 1 > r0 + diag);
            if (need_mask) {
                int lim_c = Lk - 1 - kbase;
                if (CAUSAL) lim_c = min(lim_c, row + diag - kbase);
#pragma unroll
                for (int i = 0; i < kBN; ++i)
                    if (i > lim_c) u[i] = __float_as_uint(NEG_INF);
            }
            // The two tiles take turns on their exponentials (tile 1 block j
            // after tile 0 block j, tile 0 block j after tile 1 block j-1), so
            // the warps of one tile run their exponentials while the other
            // tile's warps on the same sub-partitions load, store and wait.
            {
                const int jo = t == 1 ? j : j - 1;
                if (jo >= 0 && jo < n_other && !warp_wait(bar(B_EXP_TURN + t), jo & 1, abort_flag, p.err, lim)) {
                    ok = false;
                    break;
                }
            }
            // P = 2^(S c - mu) as bf16 pairs and its row sum, kept in
            // registers until the P tile is free, so that the wait for the
            // previous P.V overlaps this work.
            uint32_t pk[kBN / 2];
            float2 acc0, acc1;
            auto exponentials = [&](float mu) {
                const float2 c2 = make_float2(c, c);
                const float2 nmu2 = make_float2(-mu, -mu);
                acc0 = make_float2(0.f, 0.f);
                acc1 = make_float2(0.f, 0.f);
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
            };
            // Usual case: the reference m_ref stands.  P is computed against it
            // without the row max; since every P is at most the row sum, a sum
            // of at most 2^kRescaleThreshold shows that no P exceeds the bound
            // and the block is done.  Otherwise (first block, a jump of the
            // max, or a sum that is merely large) the row max decides, as
            // below, and P is recomputed.
            float alpha = 1.f;
            bool resc = false;
            bool exact = m_ref == NEG_INF;
            if (!exact) {
                exponentials(m_ref);
                exact = !(((acc0.x + acc0.y) + (acc1.x + acc1.y)) <= kPBound);  // also catches inf / NaN
            }
            if (exact) {
                float mx0 = NEG_INF, mx1 = NEG_INF, mx2 = NEG_INF, mx3 = NEG_INF;
#pragma unroll
                for (int i = 0; i < kBN; i += 8) {
                    mx0 = fmax3(mx0, __uint_as_float(u[i]), __uint_as_float(u[i + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]));
                    mx2 = fmax3(mx2, __uint_as_float(u[i + 4]), __uint_as_float(u[i + 5]));
                    mx3 = fmax3(mx3, __uint_as_float(u[i + 6]), __uint_as_float(u[i + 7]));
                }
                const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * c;
                const float m_new = fmaxf(m_ref, m_blk);
                resc = (m_ref != NEG_INF) && (m_new - m_ref > kRescaleThreshold);
                alpha = resc ? ex2(m_ref - m_new) : 1.f;
                if (resc || m_ref == NEG_INF) m_ref = m_new;
                exponentials(m_ref == NEG_INF ? 0.f : m_ref);
            }
            l = l * alpha + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_EXP_TURN + (t ^ 1)));
            // PV^t_{j-1} must be done before the P tile is rewritten or O^t is
            // rescaled.  (PV^t_{j-2} is known done: it was issued before
            // S^t_j.)
            if (j > 0 && !warp_wait(bar(B_P_EMPTY + t), (j - 1) & 1, abort_flag, p.err, lim)) {
                ok = false;
                break;
            }
            if (__any_sync(0xffffffffu, resc)) {
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(t_row + o_col + ch * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(t_row + o_col + ch * 32, o);
                }
                tmem_st_wait();
            }
            if constexpr (kPInTmem) {
                // P as bf16 pairs into the TMEM columns behind O^t
#pragma unroll
                for (int ch = 0; ch < kBN / 64; ++ch) {
                    uint32_t part[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) part[i] = pk[32 * ch + i];
                    tmem_st32(t_row + o_col + L::kPColOff + 32 * ch, part);
                }
                tmem_st_wait();
                tc_fence_before();
            } else {
                // keys 8c .. 8c+7 are 16-byte chunk c % 8 of panel c / 8
#pragma unroll
                for (int cc = 0; cc < kBN / 8; ++cc) {
                    const uint32_t addr = p_row + (cc >> 3) * kPanelBytes + ((static_cast<uint32_t>(cc & 7) ^ p_sw) << 4);
                    st_shared_v4(addr, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                }
                // make the P rows visible to the tensor core
                fence_proxy_async_smem();
            }
            // publish
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + t));
        }
        // ---- epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
        if (ok) ok = warp_wait(bar(B_O_FINAL + t), 0, abort_flag, p.err, lim);
        if (ok) {
            tc_fence_after();
            const bool store = row <= r_last[t];
            const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;  // 32-byte stores
            const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
            uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(q_start + row) * p.H + h) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(t_row + o_col + ch * 32, o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                if (store) {
                    if (o_v8) {
                        // a row is D * 2 bytes, so every row start is 32-byte aligned too
                        st_global_v8(orow + ch * 32, pk);
                        st_global_v8(orow + ch * 32 + 16, pk + 8);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
            if (store && p.lse != nullptr) {
                float lg;
                asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l));
                p.lse[lse_base + h * p.lse_head_stride + row] = l > 0.f ? (m_ref + lg) * kLn2 : NEG_INF;
            }
        }
    }

    tc_fence_before();
    cta_sync(kThreads);
}

template <int D, bool CAUSAL, bool PAGED>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     cudaStream_t stream) {
    using L = PrefillSmem<D>;
    static_assert(L::kDyn <= 232448u, "shared memory budget");
    static_assert(L::kBN == kBlockN, "the host sizes K/V boxes from kBlockN");
    static_assert(L::kSlots <= kMaxSlots, "K/V ring");
    cudaError_t e;
    // Contiguous varlen with fewer sequences than a CTA has threads: number
    // the (sequence, block) slots (the causal d = 128 grid keeps its head
    // groups).  A kernel of its own, so that the other launches keep their
    // code.
    if constexpr (!PAGED && (!CAUSAL || D == 64)) {
        const long long slots = static_cast<long long>(p.num_seqs) + p.total_q / (kBlockM * kTiles);
        if (p.cu_q != nullptr && p.num_seqs < kThreads && slots <= (CAUSAL ? 65535 : 2147483647ll)) {
            auto ks = prefill_kernel<D, CAUSAL, PAGED, true>;
            e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kDyn));
            if (e != cudaSuccess) return e;
            const int n = static_cast<int>(slots);
            ks<<<CAUSAL ? dim3(p.H, n, 1) : dim3(n, p.H, 1), kThreads, L::kDyn, stream>>>(tq, tk, tv, p);
            return cudaGetLastError();
        }
    }
    auto kern = prefill_kernel<D, CAUSAL, PAGED, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kDyn));
    if (e != cudaSuccess) return e;
    const int nblk = (p.num_q_blocks + kTiles - 1) / kTiles;
    const dim3 grid = !CAUSAL ? dim3(nblk, p.H, p.num_seqs)
                              : (D == 128 ? dim3(nblk * p.H, 1, p.num_seqs) : dim3(p.H, nblk, p.num_seqs));
    kern<<<grid, kThreads, L::kDyn, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

template <int D, bool PAGED>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     bool causal, cudaStream_t stream) {
    return causal ? launch_t<D, true, PAGED>(tq, tk, tv, p, stream) : launch_t<D, false, PAGED>(tq, tk, tv, p, stream);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int d, bool causal, cudaStream_t stream) {
    const bool paged = p.block_table != nullptr;
    if (d == 128)
        return paged ? launch_d<128, true>(tq, tk, tv, p, causal, stream) : launch_d<128, false>(tq, tk, tv, p, causal, stream);
    return paged ? launch_d<64, true>(tq, tk, tv, p, causal, stream) : launch_d<64, false>(tq, tk, tv, p, causal, stream);
}

}  // namespace fa
