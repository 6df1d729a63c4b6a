// Internal declarations shared by the host API (fa_api.cu) and the kernel
// translation units.  Not part of the public ABI (that is include/fa.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

// Bits of the device error word.
#define FA_DEVERR_TIMEOUT 1u
#define FA_DEVERR_INDEX 2u
#define FA_DEVERR_LAYOUT 4u  // a kernel found its shared memory misaligned

namespace fa {

// Query rows per tile, keys per K/V block of the prefill kernel.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Keys per K/V block of the tensor-core decode.  The host sizes every K/V
// tensor-map box from kBlockN or this, so that no box is taller than the
// shared-memory slot it lands in.
constexpr int kDecodeBlockN = 64;

// Tokens per page of the paged KV cache: 16, 32, 64 or 128 (a power of two
// that divides the 128-key block).  Kernels take it as a shift.  The
// CUDA-core decode walks every page in chunks of kPageChunk tokens.
constexpr int kMinPageSize = 16;
constexpr int kMaxPageSize = 128;
constexpr int kPageChunk = 16;
inline bool page_size_ok(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps == 128; }
inline int page_shift(int ps) { return ps == 16 ? 4 : ps == 32 ? 5 : ps == 64 ? 6 : 7; }

struct PrefillParams {
    void* o;                 // bf16 [rows, H, d]
    float* lse;              // fp32, may be null
    const int* cu_q;         // varlen: int32 [num_seqs + 1]; null for dense
    const int* cu_k;
    int N;                   // dense: tokens per sequence (queries and keys)
    int num_seqs;            // dense: B
    int H, Hkv, group;       // group = H / Hkv
    int max_seqlen_q, max_seqlen_k;
    int total_q, total_k;    // rows of q/o and of k/v
    int num_q_blocks;        // ceil(max_seqlen_q / kBlockM)
    float scale_log2;        // scale * log2(e)
    long long lse_head_stride;  // N (dense, [B,H,N]) or total_q (varlen, [H,total])
    unsigned int* err;       // device error word
    unsigned long long wait_limit_ns;
    // Paged K/V (varlen only): when block_table is set, sequence s's keys are
    // the logical tokens 0 .. Lk-1 of its pages, token t at page
    // block_table[s * max_pages + (t >> page_shift)], slot t % page size, and
    // the K/V tensor maps view the pool [num_pages << page_shift, Hkv, d]
    // with boxes of one page.
    const int* block_table;
    int max_pages, num_pages;
    int page_shift;          // log2 of the page size
};

struct DecodeParams {
    const void* q;           // bf16 [B, H, d]
    const void* k_cache;     // bf16 [num_pages, page, Hkv, d]
    const void* v_cache;
    const int* block_table;  // int32 [B, max_pages]
    const int* seqlens;      // int32 [B]
    void* o;                 // bf16 [B, H, d]
    float* lse;              // fp32 [B, H], may be null
    float* ws_o;             // fp32 [B, H, max_splits, d] unnormalised partial O
    float* ws_ml;            // fp32 [B, H, max_splits, 2] partial (m, l), log2 domain
    const int* seg_ns;       // partials per (b, kv head) when set (the tensor-core
                             // decode's segments); else ceil(seqlens[b] / split_tokens)
    int B, H, Hkv, group;
    int num_pages, max_pages, max_seqlen;
    int split_tokens;        // tokens per split (multiple of kPageChunk)
    int max_splits;
    int page_shift;          // log2 of the page size
    float scale_log2;
    unsigned int* err;
};

// Grouped decode on the tensor cores, persistent, with the keys divided
// evenly ("stream-K"): the work is the sequence of 64-key blocks of every
// (sequence b, kv head) pair, b-major; decode_tc_plan_kernel writes prefix[b]
// = Hkv * (blocks of sequences before b) (prefix[B] = all blocks), the
// blocks per CTA W = plan[0], and per pair the number of CTAs its blocks fall
// to, seg_ns[b * Hkv + kv head].  CTA c then takes blocks [c W, (c + 1) W):
// each stretch of them within one pair is a segment, whose unnormalised O
// and (m, l) go to slot (b * H + kv head * group + row) * max_splits + s,
// s = c - (first CTA of the pair) (the DecodeParams layout), which the
// combine kernel merges.  q is viewed as [B * H, 1, d] and the K/V tensor
// maps as the pool [num_pages << page_shift, Hkv, d].
struct DecodeTcParams {
    const int* seqlens;      // int32 [B]
    const int* block_table;  // int32 [B, max_pages]
    float* ws_o;
    float* ws_ml;
    int* prefix;             // int32 [B + 1], written by the plan kernel
    int* seg_ns;             // int32 [B * Hkv], written by the plan kernel
    int* plan;               // int32 [1]: W
    unsigned int* err;
    int B, H, Hkv, group;
    int max_pages, num_pages, page_shift, max_seqlen;
    int max_splits;          // slots per (b, head): at least ceil(max blocks / kDecodeTcMinBlocks) + 1
    int grid;                // CTAs of the decode launch
    float scale_log2;
    unsigned long long wait_limit_ns;
};
// Each CTA of the tensor-core decode takes at least this many 64-key blocks
// (so a pair spans at most ceil(blocks / this) + 1 CTAs).
constexpr int kDecodeTcMinBlocks = 8;

struct GatherParams {
    const void* cache;
    const int* block_table;
    const int* seqlens;
    void* out;               // bf16 [B, max_seqlen, Hkv, d]
    int B, Hkv, d;
    int num_pages, max_pages, max_seqlen;
    int page_shift;          // log2 of the page size
    unsigned int* err;
};

// Kernel launchers (defined next to their kernels).
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int d, bool causal, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream);
// The combine step alone (after a split kernel that filled ws_o / ws_ml).
cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream);
cudaError_t launch_decode_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             DecodeTcParams p, int d, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned int* err, unsigned long long limit_ns, cudaStream_t stream);

struct StoreParams {
    const void* k;           // bf16 [T, Hkv, d]
    const void* v;
    void* k_cache;           // bf16 [num_pages * page_size, Hkv, d]
    void* v_cache;
    const int* slot_mapping; // int32 [T]
    int T, Hkv, d;
    long long num_slots;     // num_pages * page_size
    unsigned int* err;
};
cudaError_t launch_store_kvcache(const StoreParams& p, cudaStream_t stream);

// Backward pass (dense or varlen, multi-head or grouped-query).
//   q, o, dout, dq : bf16 [rows_q, H, d];  k, v, dk, dv : bf16 [rows_k, Hkv, d]
//   lse            : the forward's fp32 LSE ([B, H, N] dense, [H, total_q] varlen)
//   ws             : fp32 workspace, two arrays of H * ws_head_stride floats:
//                    [0] the LSE in log2 units and [1] delta_i = dO_i . O_i,
//                    sequence s's rows at bwd_ws_seq_offset(cu_q[s], s) of each
//                    head, padded to a multiple of kBlockM rows (+inf / 0)
struct BackwardParams {
    const void* o;
    const void* dout;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* ws;
    long long ws_head_stride;
    const int* cu_q;         // varlen: int32 [num_seqs + 1]; null for dense
    const int* cu_k;
    int N, num_seqs, H, Hkv, group;
    int max_seqlen_q, max_seqlen_k, total_q, total_k;
    int num_q_blocks, num_k_blocks;  // ceil(max_seqlen / 128)
    float scale, scale_log2;
    long long lse_head_stride;
    unsigned int* err;
    unsigned long long wait_limit_ns;
};

// First workspace row of sequence s (q_start = its first query row): a
// multiple of 4 floats (16 bytes), and far enough from sequence s-1's rows
// to hold them padded to kBlockM.
__host__ __device__ inline long long bwd_ws_seq_offset(long long q_start, int s) {
    return ((q_start + 3) & ~3ll) + 132ll * s;
}
inline long long bwd_ws_head_stride(long long total_q, int num_seqs) {
    return (total_q + 132ll * num_seqs + 8 + 3) & ~3ll;
}

// Prep (delta, log2 LSE), then the dK/dV and dQ kernels, on one stream.
cudaError_t launch_backward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BackwardParams& p, int d, bool causal,
                            cudaStream_t stream);

// Size of the fixed device scratch used by fa_paged_fwd_noalloc, and the
// per-device lookup of its address (first call on a device does the lookup).
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
cudaError_t static_scratch(void** ptr, size_t* bytes);

// Decode split sizing shared by the workspace query and the launch.
inline int decode_split_tokens(int /*max_seqlen*/) { return 512; }
// Query groups of at least this many heads per kv head decode on the tensor
// cores, over an even division of the keys (DecodeTcParams); their partials
// take one more slot per (sequence, head) than these splits.
constexpr int kDecodeTcMinGroup = 8;
// The tensor-core decode loads the group's query heads as the first
// kDecodeQRows rows of its query tile (the MMA reads 128 rows; the rows past
// the group read neighbouring shared memory and are never stored), so groups
// of up to this many heads decode there.
constexpr int kDecodeQRows = 64;
inline int decode_max_splits(int max_seqlen) {
    const int t = decode_split_tokens(max_seqlen);
    const int s = (max_seqlen + t - 1) / t;
    return s < 1 ? 1 : s;
}

}  // namespace fa
