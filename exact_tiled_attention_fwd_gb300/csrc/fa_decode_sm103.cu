// Paged single-token decode for sm_103a: split-KV partial attention over the
// page pool, then a combine of the per-split results.
//
// The cache is a pool of pages of 16, 32, 64 or 128 tokens,
// [num_pages, page, Hkv, d]; token t of sequence b is page
// block_table[b][t / page], slot t % page (the paged KV read
// of the dlog.com.cn page "从标准 Attention 到 FlashAttention 与分页执行",
// §3.4 and its PagedAttention section).  Decode reads every cached byte once,
// so the kernel is bound by HBM bandwidth, not by arithmetic: no tensor cores.
// (Query groups of 8 or more heads per kv head decode on the tensor cores
// instead, in the prefill kernel's decode mode, and share the combine kernel
// below.)
//
// Split kernel: one warp per (sequence, split of split_tokens tokens, G query
// heads of one kv head).  A warp reads the split in chunks of 16 tokens (a
// page of 16, or a quarter of a 64-token page) with 16-byte loads; D/8 lanes
// hold one key row (lane group g, element chunk c), so one warp instruction
// reads 32/(D/8) whole rows, each a contiguous d*2-byte run.  The next
// chunk's K/V lines are prefetched into L2 while a chunk is computed.
// Scores are the chunk dot products summed across the row's lanes (xor
// shuffles; for G > 1 a halving reduction that leaves one whole score per
// lane); the running (m, l, o) follow the online-softmax recurrence of the
// same page §2.2 with the chunk as the block.  The split writes its
// unnormalised o and (m, l).
//
// Combine kernel: one warp per (sequence, head) merges the splits with the
// same rescale rule: M = max m_s, w_s = 2^(m_s - M), l = sum w_s l_s,
// O = sum w_s o_s / l, LSE = (M + log2 l) ln 2.
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDecodeWarps = 8;
// Warps per split CTA: eight heads' warps for plain multi-head decode (one
// page row of eight heads is contiguous), four for grouped queries, whose
// larger register count would otherwise leave one CTA, eight warps, per SM.
template <int G>
__host__ __device__ constexpr int split_warps() { return G == 1 ? 8 : 4; }

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ uint4 ldg_stream(const void* ptr) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}

// Offset (in elements) of pool row `row` (page * page size + slot), kv head
// hk, element 0.
__device__ __forceinline__ size_t paged_row_offset(int row, int Hkv, int hk, int d) {
    return (static_cast<size_t>(row) * Hkv + hk) * static_cast<size_t>(d);
}

// Pool row of the first token of 16-token chunk `ck` of sequence b (page
// block_table[b][ck * 16 >> shift], slot ck * 16 within it), or -1 (recorded
// as an index error) when the table entry is outside the pool.
__device__ __forceinline__ int lookup_chunk(const int* block_table, int max_pages, int num_pages, int shift, int b,
                                            int ck, unsigned int* err) {
    const int t = ck * kPageChunk;
    const int page = __ldg(block_table + static_cast<size_t>(b) * max_pages + (t >> shift));
    if (static_cast<unsigned>(page) >= static_cast<unsigned>(num_pages)) {
        atomicOr(err, FA_DEVERR_INDEX);
        return -1;
    }
    return (page << shift) + (t & ((1 << shift) - 1));
}

__device__ __forceinline__ int clamp_seqlen(int L, int max_seqlen, unsigned int* err, bool report) {
    if (L < 0 || L > max_seqlen) {
        if (report) atomicOr(err, FA_DEVERR_INDEX);
        return L < 0 ? 0 : max_seqlen;
    }
    return L;
}

__device__ __forceinline__ float dot8(const float (&q)[8], const uint4& k) {
    float s = q[0] * bf16lo_to_f32(k.x);
    s = fmaf(q[1], bf16hi_to_f32(k.x), s);
    s = fmaf(q[2], bf16lo_to_f32(k.y), s);
    s = fmaf(q[3], bf16hi_to_f32(k.y), s);
    s = fmaf(q[4], bf16lo_to_f32(k.z), s);
    s = fmaf(q[5], bf16hi_to_f32(k.z), s);
    s = fmaf(q[6], bf16lo_to_f32(k.w), s);
    s = fmaf(q[7], bf16hi_to_f32(k.w), s);
    return s;
}

__device__ __forceinline__ void axpy8(float (&o)[8], float p, const uint4& v) {
    o[0] = fmaf(p, bf16lo_to_f32(v.x), o[0]);
    o[1] = fmaf(p, bf16hi_to_f32(v.x), o[1]);
    o[2] = fmaf(p, bf16lo_to_f32(v.y), o[2]);
    o[3] = fmaf(p, bf16hi_to_f32(v.y), o[3]);
    o[4] = fmaf(p, bf16lo_to_f32(v.z), o[4]);
    o[5] = fmaf(p, bf16hi_to_f32(v.z), o[5]);
    o[6] = fmaf(p, bf16lo_to_f32(v.w), o[6]);
    o[7] = fmaf(p, bf16hi_to_f32(v.w), o[7]);
}

// One warp per (sequence, split, G query heads of one kv head).  With
// grouped-query attention the G heads share every K/V row the warp loads, so
// each row is read once per group instead of once per query head; G = 1 is
// plain multi-head attention.
template <int D, int G>
__global__ void __launch_bounds__(split_warps<G>() * 32) decode_split_kernel(const DecodeParams p) {
    grid_dependents_launch();  // the combine grid (its dependent) may queue behind this one
    constexpr int LPR = D / 8;         // lanes per key row
    constexpr int RPI = 32 / LPR;      // rows per warp load
    constexpr int NI = kPageChunk / RPI;  // loads per lane per chunk (K and V each)
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.z;
    const int h0 = (blockIdx.y * split_warps<G>() + warp) * G;  // first of this warp's heads
    const int split = blockIdx.x;
    if (h0 >= p.H) return;
    const int L = clamp_seqlen(__ldg(p.seqlens + b), p.max_seqlen, p.err, split == 0 && lane == 0);
    const int t0 = split * p.split_tokens;
    if (t0 >= L) return;
    const int t1 = min(L, t0 + p.split_tokens);
    const int hk = h0 / p.group;  // G divides the group, so all G heads share it
    const int g = lane / LPR;  // row group within a warp load
    const int c = lane % LPR;  // 8-element chunk of the row

    // q chunks, pre-multiplied by scale * log2(e) so scores are in log2 units
    float qf[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const uint4 qv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                         (static_cast<size_t>(b) * p.H + h0 + j) * D + c * 8);
        qf[j][0] = bf16lo_to_f32(qv.x) * p.scale_log2;
        qf[j][1] = bf16hi_to_f32(qv.x) * p.scale_log2;
        qf[j][2] = bf16lo_to_f32(qv.y) * p.scale_log2;
        qf[j][3] = bf16hi_to_f32(qv.y) * p.scale_log2;
        qf[j][4] = bf16lo_to_f32(qv.z) * p.scale_log2;
        qf[j][5] = bf16hi_to_f32(qv.z) * p.scale_log2;
        qf[j][6] = bf16lo_to_f32(qv.w) * p.scale_log2;
        qf[j][7] = bf16hi_to_f32(qv.w) * p.scale_log2;
    }
    const uint16_t* kc = static_cast<const uint16_t*>(p.k_cache);
    const uint16_t* vc = static_cast<const uint16_t*>(p.v_cache);
    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = neg_inf();
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    }

    // The chunk walk runs ahead of the loads: the K/V rows of the chunk
    // kAhead chunks on are pulled into L2 while this chunk is computed, and
    // table entries are fetched one chunk before that, so a chunk's loads find
    // their lines in L2 instead of waiting on a dependent table load and then
    // on HBM.  Grouped warps, which compute longer per chunk, look two chunks
    // ahead (measured 4.5% faster with 4 heads per warp, no gain for one).
    // Chunks never straddle a page: every page size is a multiple of 16.
    const int pg0 = t0 / kPageChunk;
    const int pg_end = (t1 + kPageChunk - 1) / kPageChunk;
    auto entry = [&](int pg) {
        return pg < pg_end ? lookup_chunk(p.block_table, p.max_pages, p.num_pages, p.page_shift, b, pg, p.err) : -1;
    };
    // L2 prefetch of one chunk of this warp's kv head: lane l takes the
    // 128-byte lines l * kPf .. l * kPf + kPf - 1 of the chunk's K lines
    // followed by its V lines (row = line / kLinesPerRow).
    constexpr int kLinesPerRow = D / 64;
    constexpr int kLinesPerPage = kPageChunk * kLinesPerRow;  // per tensor
    constexpr int kPf = 2 * kLinesPerPage / 32;               // prefetches per lane
    static_assert(kPf * 32 == 2 * kLinesPerPage, "chunk lines per lane");
    auto prefetch_page = [&](int row0) {
        if (row0 < 0) return;
#pragma unroll
        for (int x = 0; x < kPf; ++x) {
            const int line = lane * kPf + x;
            const int tl = line % kLinesPerPage;
            const uint16_t* a = (line < kLinesPerPage ? kc : vc) +
                                paged_row_offset(row0 + tl / kLinesPerRow, p.Hkv, hk, D) + (tl % kLinesPerRow) * 64;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
    };
    constexpr int kAhead = G == 1 ? 1 : 2;
    int ent[kAhead + 1];  // table entries of pages pg .. pg + kAhead
#pragma unroll
    for (int a = 0; a <= kAhead; ++a) ent[a] = entry(pg0 + a);
#pragma unroll
    for (int a = 1; a < kAhead; ++a) prefetch_page(ent[a]);
    for (int pg = pg0; pg < pg_end; ++pg) {
        const int prow = ent[0];  // pool row of the chunk's first token
#pragma unroll
        for (int a = 0; a < kAhead; ++a) ent[a] = ent[a + 1];
        if (prow < 0) {  // outside the pool: skipped (and reported by entry())
            ent[kAhead] = entry(pg + kAhead + 1);
            continue;
        }
        uint4 kv[NI], vv[NI];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const size_t off = paged_row_offset(prow + i * RPI + g, p.Hkv, hk, D) + c * 8;
            kv[i] = ldg_stream(kc + off);
        }
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const size_t off = paged_row_offset(prow + i * RPI + g, p.Hkv, hk, D) + c * 8;
            vv[i] = ldg_stream(vc + off);
        }
        prefetch_page(ent[kAhead - 1]);
        ent[kAhead] = entry(pg + kAhead + 1);
        if constexpr (G == 1) {
    #pragma unroll
            for (int j = 0; j < G; ++j) {
                float s[NI];
    #pragma unroll
                for (int i = 0; i < NI; ++i) s[i] = dot8(qf[j], kv[i]);
    #pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) {
    #pragma unroll
                    for (int i = 0; i < NI; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], off);
                }
                float mp = neg_inf();
    #pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int tok = pg * kPageChunk + i * RPI + g;
                    if (tok >= t1) s[i] = neg_inf();
                    mp = fmaxf(mp, s[i]);
                }
    #pragma unroll
                for (int off = LPR; off < 32; off <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, off));
                const float m_new = fmaxf(m[j], mp);
                const float mu = m_new == neg_inf() ? 0.f : m_new;
                const float alpha = ex2(m[j] - mu);  // m = -inf -> 0
                l[j] *= alpha;
    #pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] *= alpha;
    #pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const float pi = ex2(s[i] - mu);
                    l[j] += pi;
                    axpy8(acc[j], pi, vv[i]);
                }
                m[j] = m_new;
            }
        } else {
            // Grouped heads.  Each K/V chunk is unpacked to fp32 pairs once and
            // used by all G heads with packed fp32x2 arithmetic.  The row sums
            // of the partial dot products are reduced by halving: at each xor
            // level a lane keeps half of its values (the upper half if its
            // lane bit is set) and adds the partner's matching half, so after
            // log2(LPR) levels lane c of a row group holds the whole score of
            // row c / 2 of its group (lanes c and c ^ 1 hold the same row).
            float sc[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float sv[NI];
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const float2 k0 = make_float2(bf16lo_to_f32(kv[i].x), bf16hi_to_f32(kv[i].x));
                    const float2 k1 = make_float2(bf16lo_to_f32(kv[i].y), bf16hi_to_f32(kv[i].y));
                    const float2 k2 = make_float2(bf16lo_to_f32(kv[i].z), bf16hi_to_f32(kv[i].z));
                    const float2 k3 = make_float2(bf16lo_to_f32(kv[i].w), bf16hi_to_f32(kv[i].w));
                    float2 a = __fmul2_rn(make_float2(qf[j][0], qf[j][1]), k0);
                    a = __ffma2_rn(make_float2(qf[j][2], qf[j][3]), k1, a);
                    a = __ffma2_rn(make_float2(qf[j][4], qf[j][5]), k2, a);
                    a = __ffma2_rn(make_float2(qf[j][6], qf[j][7]), k3, a);
                    sv[i] = a.x + a.y;
                }
                int n = NI;
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) {
                    if (n > 1) {
                        const bool up = (c & off) != 0;
                        n >>= 1;
#pragma unroll
                        for (int k = 0; k < NI / 2; ++k) {
                            if (k < n) {
                                const float keep = up ? sv[k + n] : sv[k];
                                const float send = up ? sv[k] : sv[k + n];
                                sv[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                            }
                        }
                    } else {
                        sv[0] += __shfl_xor_sync(0xffffffffu, sv[0], off);
                    }
                }
                const int tok = pg * kPageChunk + (c >> 1) * RPI + g;
                sc[j] = tok < t1 ? sv[0] : neg_inf();
            }
            // Page maximum (lane pairs hold equal rows, so xor 1 is skipped),
            // then each lane's own row probability.
            float pl[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float mp = sc[j];
#pragma unroll
                for (int off = 2; off < 32; off <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, off));
                const float m_new = fmaxf(m[j], mp);
                const float mu = m_new == neg_inf() ? 0.f : m_new;
                const float alpha = ex2(m[j] - mu);  // m = -inf -> 0
                pl[j] = ex2(sc[j] - mu);
                l[j] = l[j] * alpha + ((c & 1) == 0 ? pl[j] : 0.f);  // each row once
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 o = __fmul2_rn(make_float2(acc[j][e], acc[j][e + 1]), a2);
                    acc[j][e] = o.x;
                    acc[j][e + 1] = o.y;
                }
                m[j] = m_new;
            }
            // O += p V: row i of this lane's group is held by lane g * LPR + 2 i.
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const float2 v0 = make_float2(bf16lo_to_f32(vv[i].x), bf16hi_to_f32(vv[i].x));
                const float2 v1 = make_float2(bf16lo_to_f32(vv[i].y), bf16hi_to_f32(vv[i].y));
                const float2 v2 = make_float2(bf16lo_to_f32(vv[i].z), bf16hi_to_f32(vv[i].z));
                const float2 v3 = make_float2(bf16lo_to_f32(vv[i].w), bf16hi_to_f32(vv[i].w));
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float pi = __shfl_sync(0xffffffffu, pl[j], g * LPR + 2 * i);
                    const float2 p2 = make_float2(pi, pi);
                    float2 o = __ffma2_rn(p2, v0, make_float2(acc[j][0], acc[j][1]));
                    acc[j][0] = o.x;
                    acc[j][1] = o.y;
                    o = __ffma2_rn(p2, v1, make_float2(acc[j][2], acc[j][3]));
                    acc[j][2] = o.x;
                    acc[j][3] = o.y;
                    o = __ffma2_rn(p2, v2, make_float2(acc[j][4], acc[j][5]));
                    acc[j][4] = o.x;
                    acc[j][5] = o.y;
                    o = __ffma2_rn(p2, v3, make_float2(acc[j][6], acc[j][7]));
                    acc[j][6] = o.x;
                    acc[j][7] = o.y;
                }
            }
        }
    }
    // Sum the row groups: chunks add.  With G = 1 every lane of a group holds
    // the group's l; with grouped heads each even lane holds its own row's
    // share, so l is summed over every lane.
#pragma unroll
    for (int j = 0; j < G; ++j) {
        if (G > 1) {
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], off);
        }
        const size_t slot = (static_cast<size_t>(b) * p.H + h0 + j) * p.max_splits + split;
        if (g == 0) {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * D + c * 8);
            dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
            dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
        }
        if (lane == 0) *reinterpret_cast<float2*>(p.ws_ml + slot * 2) = make_float2(m[j], l[j]);
    }
}

template <int D>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_combine_kernel(const DecodeParams p) {
    grid_dependency_wait();  // the partials of the kernel ahead (launched as its dependent)
    constexpr int EPL = D / 32;  // elements per lane
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x * kDecodeWarps + warp;
    if (bh >= p.B * p.H) return;
    const int b = bh / p.H;
    const int L = clamp_seqlen(__ldg(p.seqlens + b), p.max_seqlen, p.err, false);
    const int ns = p.seg_ns != nullptr ? __ldg(p.seg_ns + b * p.Hkv + (bh % p.H) / p.group)
                                       : (L + p.split_tokens - 1) / p.split_tokens;
    const size_t base = static_cast<size_t>(bh) * p.max_splits;
    float M = neg_inf();
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p.ws_ml[(base + s) * 2]);
    const float mu = M == neg_inf() ? 0.f : M;
    float l = 0.f;
    float o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + (base + s) * 2);
        const float w = ex2(ml.x - mu);
        l = fmaf(w, ml.y, l);
        const float* src = p.ws_o + (base + s) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, src[e], o[e]);
    }
    const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.o) + static_cast<size_t>(bh) * D + lane * EPL;
    if constexpr (EPL == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0] * inv, o[1] * inv);
    }
    if (lane == 0 && p.lse != nullptr) {
        float lg;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l));
        p.lse[bh] = l > 0.f ? (M + lg) * kLn2 : neg_inf();
    }
}

// Pure copy of every row the decode kernel would read, through the same
// chunk lookup and row offset.  grid = (16-token chunks of the longest
// sequence, B).
__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
    const int b = blockIdx.y;
    const int pg = blockIdx.x;
    const int L = clamp_seqlen(__ldg(p.seqlens + b), p.max_seqlen, p.err, pg == 0 && threadIdx.x == 0);
    if (pg * kPageChunk >= L) return;
    const int prow = lookup_chunk(p.block_table, p.max_pages, p.num_pages, p.page_shift, b, pg, p.err);
    if (prow < 0) return;
    const int chunks = p.d / 8;                    // 16-byte chunks per row
    const int per_tok = p.Hkv * chunks;
    const int ntok = min(kPageChunk, L - pg * kPageChunk);
    const uint16_t* src = static_cast<const uint16_t*>(p.cache);
    uint16_t* out = static_cast<uint16_t*>(p.out);
    for (int u = threadIdx.x; u < ntok * per_tok; u += blockDim.x) {
        const int slot = u / per_tok;
        const int hk = (u % per_tok) / chunks;
        const int cc = u % chunks;
        const uint4 val = ldg_stream(src + paged_row_offset(prow + slot, p.Hkv, hk, p.d) + cc * 8);
        const size_t t = static_cast<size_t>(pg) * kPageChunk + slot;
        *reinterpret_cast<uint4*>(out + ((static_cast<size_t>(b) * p.max_seqlen + t) * p.Hkv + hk) * p.d + cc * 8) = val;
    }
}

// store_kvcache: row i of this step's K and V goes to flat slot
// slot_mapping[i] of the page pool (page slot / page_size, offset
// slot % page_size, so with contiguous pages the slot is the row of the pool
// viewed as [num_pages * page_size, Hkv, d]).  A negative slot is skipped; a
// slot past the pool is skipped and reported.  Work is spread over 16-byte
// chunks, one chunk of K and the same chunk of V per thread and step.
__global__ void __launch_bounds__(256) store_kvcache_kernel(const StoreParams p) {
    const int chunks = p.Hkv * p.d / 8;
    const long long units = static_cast<long long>(p.T) * chunks;
    const uint16_t* ks = static_cast<const uint16_t*>(p.k);
    const uint16_t* vs = static_cast<const uint16_t*>(p.v);
    uint16_t* kd = static_cast<uint16_t*>(p.k_cache);
    uint16_t* vd = static_cast<uint16_t*>(p.v_cache);
    for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long t = u / chunks;
        const int c = static_cast<int>(u % chunks);
        const int slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (c == 0) atomicOr(p.err, FA_DEVERR_INDEX);
            continue;
        }
        const size_t src = static_cast<size_t>(t) * chunks * 8 + static_cast<size_t>(c) * 8;
        const size_t dst = static_cast<size_t>(slot) * chunks * 8 + static_cast<size_t>(c) * 8;
        const uint4 kv = ldg_stream(ks + src);
        const uint4 vv = ldg_stream(vs + src);
        *reinterpret_cast<uint4*>(kd + dst) = kv;
        *reinterpret_cast<uint4*>(vd + dst) = vv;
    }
}

// One CTA waits on a barrier nothing arrives on; the bounded wait must give
// up and record the timeout.
__global__ void wait_selftest_kernel(unsigned int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    mbar_wait(bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace

namespace {

template <int D, int G>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
    const int warps = (p.H + G - 1) / G;
    constexpr int kW = split_warps<G>();
    dim3 grid(p.max_splits, (warps + kW - 1) / kW, p.B);
    decode_split_kernel<D, G><<<grid, kW * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

// Query heads per warp: up to 4 heads of a kv group (the largest count that
// divides the group).  8 heads at d = 64 fit the registers too, but leave so
// few warps per SM that the loads stop overlapping (measured slower).
template <int D>
cudaError_t launch_split_grouped(const DecodeParams& p, cudaStream_t stream) {
    if (p.group % 4 == 0) return launch_split<D, 4>(p, stream);
    if (p.group % 2 == 0) return launch_split<D, 2>(p, stream);
    return launch_split<D, 1>(p, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream) {
    cudaError_t e = d == 128 ? launch_split_grouped<128>(p, stream) : launch_split_grouped<64>(p, stream);
    if (e != cudaSuccess) return e;
    return launch_decode_combine(p, d, stream);
}

cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream) {
    // launched as the programmatic dependent of the split kernel: its launch
    // overlaps that kernel's last CTAs, and it waits for the partials
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.B * p.H + kDecodeWarps - 1) / kDecodeWarps);
    cfg.blockDim = dim3(kDecodeWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (d == 128) return cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, p);
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
    dim3 grid((p.max_seqlen + kPageChunk - 1) / kPageChunk, p.B);
    gather_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_store_kvcache(const StoreParams& p, cudaStream_t stream) {
    const long long units = static_cast<long long>(p.T) * (p.Hkv * p.d / 8);
    const long long want = (units + 255) / 256;
    const int grid = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
    store_kvcache_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned int* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

// Fixed device scratch for fa_paged_fwd_noalloc: the split partials live in
// this file-scope array instead of a caller workspace.  Every device that
// loads the library holds kStaticScratchBytes of it until the process exits.
// Host code may not use the array's name as a device address; the address is
// looked up once per device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_paged_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};
}  // namespace

cudaError_t static_scratch(void** ptr, size_t* bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_paged_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    *bytes = kStaticScratchBytes;
    return cudaSuccess;
}

}  // namespace fa
