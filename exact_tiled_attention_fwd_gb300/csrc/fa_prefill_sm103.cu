// Prefill forward (dense and varlen) for sm_103a: TMA-staged tiles, tcgen05
// MMA into tensor memory, one thread per query row for the online softmax.
//
// What one CTA computes: one tile of kBlockM = 128 query rows of one
// (sequence, head), streaming the sequence's K/V in kBlockN = 128-key blocks
// (tiling, dlog.com.cn "从标准 Attention 到 FlashAttention 与分页执行" §2.1;
// the (Q block, batch*head) grid of the lqnn.cn page §4.4).  Per K/V block j:
//
//   S_j  = Q K_j^T                       tcgen05.mma, SMEM x SMEM -> TMEM (fp32)
//   m'   = max(m, rowmax(S_j * scale))    softmax warps, one thread per row
//   P_j  = exp(S_j * scale - m)           -> bf16, written back into TMEM
//   l    = l * exp(m_old - m) + rowsum P_j
//   O   += P_j V_j                        tcgen05.mma, TMEM x SMEM -> TMEM
//
// and at the end O / l and lse = m + ln l (online softmax, same page §2.2).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into a 2-slot ring
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma
//   warps 2..5  softmax + correction + epilogue; warp w owns TMEM lanes
//               32*(w%4) .. +31, i.e. query rows of the tile, one per thread
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)    S/P buffer 0     [128,256)  S/P buffer 1     [256,256+d) O
// P_j (bf16 pairs) overwrites the first 64 columns of its S buffer after the
// owning thread has read the whole S row.  S is double-buffered so the
// tensor core computes S_{j+1} while the softmax warps work on S_j.
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

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPanelBytes = 128 * 128;  // 128 rows x 64 bf16

template <int D>
struct PrefillSmem {
    static constexpr uint32_t kTile = kBlockM * D * 2;  // one Q, K or V tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kTile;
    static constexpr uint32_t kV = kTile * (1 + kStages);
    static constexpr uint32_t kBar = kTile * (1 + 2 * kStages);
    // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2],
    //           s_full[2], p_full[2], o_ready, o_final, mma_done
    static constexpr uint32_t kNumBars = 16;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    // Requested dynamic size: 1 KiB alignment slack, and at least 116 KiB so
    // that a single CTA occupies an SM (each CTA takes all 512 TMEM columns).
    static constexpr uint32_t kDyn = (kUsed + 1024) > 118784u ? (kUsed + 1024) : 118784u;
};

enum BarId : uint32_t {
    B_Q_FULL = 0,
    B_K_FULL = 1,   // +stage
    B_K_EMPTY = 3,  // +stage
    B_V_FULL = 5,   // +stage
    B_V_EMPTY = 7,  // +stage
    B_S_FULL = 9,   // +buffer
    B_P_FULL = 11,  // +buffer
    B_O_READY = 13,
    B_O_FINAL = 14,
    B_MMA_DONE = 15,
};

__device__ __forceinline__ float fmax3(float a, float b, float c) { return fmaxf(fmaxf(a, b), c); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using L = PrefillSmem<D>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kOCol = 256;
    constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](uint32_t id) { return sbase + L::kBar + id * 8; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int h = blockIdx.y;
    const int hk = h / p.group;
    const int qb = CAUSAL ? (p.num_q_blocks - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);

    // ---- sequence geometry (uniform over the CTA)
    int q_start, Lq, k_start, Lk;
    if (p.cu_q != nullptr) {
        q_start = p.cu_q[seq];
        Lq = p.cu_q[seq + 1] - q_start;
        k_start = p.cu_k[seq];
        Lk = p.cu_k[seq + 1] - k_start;
        const bool bad = q_start < 0 || Lq < 0 || k_start < 0 || Lk < 0 || q_start + Lq > p.total_q ||
                         k_start + Lk > p.total_k || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k;
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
    const int row0 = qb * kBlockM;
    if (row0 >= Lq) return;
    const int row_last = min(Lq, row0 + kBlockM) - 1;
    const int diag = Lk - Lq;  // causal: key j visible to row i iff j <= i + diag
    int nkv = (Lk + kBlockN - 1) / kBlockN;
    if (CAUSAL) {
        const int max_key = row_last + diag;
        nkv = max_key < 0 ? 0 : min(nkv, max_key / kBlockN + 1);
    }

    // Rows that see no key at all: O = 0, LSE = -inf (no tensor-core work).
    if (nkv == 0) {
        if (warp >= 2) {
            const int r = (warp & 3) * 32 + lane;
            const int row = row0 + r;
            if (row <= row_last) {
                uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                                       (static_cast<size_t>(q_start + row) * p.H + h) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0, 0, 0, 0);
                if (p.lse != nullptr) {
                    const long long base = p.cu_q ? q_start : static_cast<long long>(seq) * p.H * p.N;
                    p.lse[base + h * p.lse_head_stride + row] = -__int_as_float(0x7f800000);
                }
            }
        }
        return;
    }

    // ---- setup: barriers (thread 0), tensor memory (warp 1)
    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_FULL + b), 128);
        }
        mbar_init(bar(B_O_READY), 1);
        mbar_init(bar(B_O_FINAL), 1);
        mbar_init(bar(B_MMA_DONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
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

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(B_Q_FULL), L::kTile);
#pragma unroll
            for (int pn = 0; pn < kPanels; ++pn)
                tma_load_3d(sbase + L::kQ + pn * kPanelBytes, &tm_q, bar(B_Q_FULL), pn * 64, h, q_start + row0);
            int k_last[kStages], v_last[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) k_last[s] = v_last[s] = -1;
            for (int j = 0; j < nkv; ++j) {
                const int s = j % kStages;
                const int n = j / kStages;
                const int krow = k_start + j * kBlockN;
                if (n > 0 && !mbar_wait(bar(B_K_EMPTY + s), (n - 1) & 1, abort_flag, p.err, lim)) break;
                mbar_arrive_expect_tx(bar(B_K_FULL + s), L::kTile);
#pragma unroll
                for (int pn = 0; pn < kPanels; ++pn)
                    tma_load_3d(sbase + L::kK + s * L::kTile + pn * kPanelBytes, &tm_k, bar(B_K_FULL + s), pn * 64,
                                hk, krow);
                k_last[s] = n;
                if (n > 0 && !mbar_wait(bar(B_V_EMPTY + s), (n - 1) & 1, abort_flag, p.err, lim)) break;
                mbar_arrive_expect_tx(bar(B_V_FULL + s), L::kTile);
#pragma unroll
                for (int pn = 0; pn < kPanels; ++pn)
                    tma_load_3d(sbase + L::kV + s * L::kTile + pn * kPanelBytes, &tm_v, bar(B_V_FULL + s), pn * 64,
                                hk, krow);
                v_last[s] = n;
            }
            // Drain: every copy this CTA issued lands before the CTA exits.
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                if (k_last[s] >= 0) mbar_wait_drain(bar(B_K_FULL + s), k_last[s] & 1, lim);
                if (v_last[s] >= 0) mbar_wait_drain(bar(B_V_FULL + s), v_last[s] & 1, lim);
            }
            mbar_wait_drain(bar(B_Q_FULL), 0, lim);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            auto q_desc = [&](int kk) {
                return sdesc_sw128(sbase + L::kQ + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            };
            auto k_desc = [&](int s, int kk) {
                return sdesc_sw128(sbase + L::kK + s * L::kTile + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            };
            auto v_desc = [&](int s, int kk) {
                return sdesc_sw128(sbase + L::kV + s * L::kTile + kk * (16 * 128), kPanelBytes, 1024);
            };
            auto issue_pv = [&](int i) -> bool {
                const int s = i % kStages;
                const int b = i & 1;
                if (!mbar_wait(bar(B_P_FULL + b), (i >> 1) & 1, abort_flag, p.err, lim)) return false;
                if (!mbar_wait(bar(B_V_FULL + s), (i / kStages) & 1, abort_flag, p.err, lim)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts(tmem + kOCol, tmem + b * 128 + kk * 8, v_desc(s, kk), kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(B_V_EMPTY + s));
                tc_commit(bar(B_O_READY));
                return true;
            };
            bool ok = mbar_wait(bar(B_Q_FULL), 0, abort_flag, p.err, lim);
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j % kStages;
                const int b = j & 1;
                if (!mbar_wait(bar(B_K_FULL + s), (j / kStages) & 1, abort_flag, p.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + b * 128, q_desc(kk), k_desc(s, kk), kIdescS, kk > 0 ? 1u : 0u);
                tc_commit(bar(B_K_EMPTY + s));
                tc_commit(bar(B_S_FULL + b));
                if (j > 0) ok = issue_pv(j - 1);
            }
            if (ok) ok = issue_pv(nkv - 1);
            if (ok) tc_commit(bar(B_O_FINAL));
            // Every MMA has finished before tensor memory is released.
            tc_commit(bar(B_MMA_DONE));
            mbar_wait_drain(bar(B_MMA_DONE), 0, lim);
        }
        __syncwarp();
    } else {
        // ================= softmax / correction / epilogue =================
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row of the tile == TMEM lane
        const int row = row0 + r;           // row within the sequence
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const float c = p.scale_log2;
        const float NEG_INF = -__int_as_float(0x7f800000);
        float m_ref = NEG_INF;  // exponent reference (log2 units)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            const int b = j & 1;
            if (!warp_wait(bar(B_S_FULL + b), (j >> 1) & 1, abort_flag, p.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[kBlockN];
#pragma unroll
            for (int ch = 0; ch < kBlockN / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(t_row + b * 128 + ch * 32, u);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[ch * 32 + i] = __uint_as_float(u[i]);
            }
            const int kbase = j * kBlockN;
            const bool need_mask =
                (kbase + kBlockN > Lk) || (CAUSAL && kbase + kBlockN - 1 > row0 + diag);
            if (need_mask) {
                int lim_c = Lk - 1 - kbase;
                if (CAUSAL) lim_c = min(lim_c, row + diag - kbase);
#pragma unroll
                for (int i = 0; i < kBlockN; ++i)
                    if (i > lim_c) x[i] = NEG_INF;
            }
            float mx0 = NEG_INF, mx1 = NEG_INF, mx2 = NEG_INF, mx3 = NEG_INF;
#pragma unroll
            for (int i = 0; i < kBlockN; i += 8) {
                mx0 = fmax3(mx0, x[i], x[i + 1]);
                mx1 = fmax3(mx1, x[i + 2], x[i + 3]);
                mx2 = fmax3(mx2, x[i + 4], x[i + 5]);
                mx3 = fmax3(mx3, x[i + 6], x[i + 7]);
            }
            const float m_blk = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
            const float m_new = fmaxf(m_ref, m_blk);
            const bool resc = (m_ref != NEG_INF) && (m_new - m_ref > kRescaleThreshold);
            if (__any_sync(0xffffffffu, resc)) {
                // O must hold P_{j-1} V_{j-1} before it is rescaled.
                if (!warp_wait(bar(B_O_READY), (j - 1) & 1, abort_flag, p.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = resc ? ex2(m_ref - m_new) : 1.f;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t u[32];
                    tmem_ld32(t_row + kOCol + ch * 32, u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                    tmem_st32(t_row + kOCol + ch * 32, u);
                }
                tmem_st_wait();
            }
            if (resc) {
                l *= ex2(m_ref - m_new);
                m_ref = m_new;
            }
            if (m_ref == NEG_INF) m_ref = m_new;
            const float mu = (m_ref == NEG_INF) ? 0.f : m_ref;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ex2(fmaf(x[ch * 64 + 2 * i], c, -mu));
                    const float p1 = ex2(fmaf(x[ch * 64 + 2 * i + 1], c, -mu));
                    s0 += p0;
                    s1 += p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st32(t_row + b * 128 + ch * 32, pk);
            }
            l += s0 + s1;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + b));
        }
        // ---- epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
        if (ok) ok = warp_wait(bar(B_O_FINAL), 0, abort_flag, p.err, lim);
        if (ok) {
            tc_fence_after();
            const bool store = row <= row_last;
            const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
            uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(q_start + row) * p.H + h) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t u[32];
                tmem_ld32(t_row + kOCol + ch * 32, u);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(u[2 * i]) * inv, __uint_as_float(u[2 * i + 1]) * inv);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (store && p.lse != nullptr) {
                float lg;
                asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l));
                const long long base = p.cu_q ? q_start : static_cast<long long>(seq) * p.H * p.N;
                p.lse[base + h * p.lse_head_stride + row] = l > 0.f ? (m_ref + lg) * kLn2 : NEG_INF;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     cudaStream_t stream) {
    using L = PrefillSmem<D>;
    static_assert(L::kDyn <= 232448u, "shared memory budget");
    auto kern = prefill_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kDyn));
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_q_blocks, p.H, p.num_seqs);
    kern<<<grid, kThreads, L::kDyn, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int d, bool causal, cudaStream_t stream) {
    if (d == 128) return causal ? launch_t<128, true>(tq, tk, tv, p, stream) : launch_t<128, false>(tq, tk, tv, p, stream);
    return causal ? launch_t<64, true>(tq, tk, tv, p, stream) : launch_t<64, false>(tq, tk, tv, p, stream);
}

}  // namespace fa
