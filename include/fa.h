/*
 * Exact tiled attention forward for GB300 (sm_103a): the C-ABI.
 *
 * Every entry point computes, for each (sequence, head, query row i),
 *
 *     O_i   = sum_j softmax_j(scale * q_i . k_j) v_j
 *     LSE_i = ln sum_j exp(scale * q_i . k_j)
 *
 * over the keys j visible to row i, without ever writing the score matrix S
 * or the probability matrix P to device memory: Q is cut into row blocks,
 * K/V are streamed in column blocks, and a running max m, running sum l and
 * accumulator O are rescaled by exp(m_old - m_new) for every block, with O/l
 * and m + ln l written at the end.  (Page "从标准 Attention 到 FlashAttention 与
 * 分页执行", dlog.com.cn: opening definition, §2.1 tiling, §2.2 online
 * softmax; page "L2.5 极致算子实战案例", yulong.wang: §2.1, O plus the per-row
 * logsumexp is what the forward writes.)
 *
 * Conventions shared by all entry points
 * --------------------------------------
 *  - Tensors are bf16 (q, k, v, o, caches) or fp32 (lse), row-major, dense,
 *    in DEVICE memory owned by the caller.  The library allocates nothing.
 *    Every pointer must be 16-byte aligned.
 *  - Accumulation is fp32; P is rounded to bf16 before the P.V product; O is
 *    stored as bf16 round-to-nearest-even; LSE is the natural log, fp32.
 *  - H is the number of query heads, Hkv the number of key/value heads,
 *    H % Hkv == 0; query head h reads kv head h / (H / Hkv) (grouped-query
 *    attention, the page's GQA section).  Hkv == H is plain multi-head.
 *  - d (head dim) must be 64 or 128, else FA_ERR_UNSUPPORTED.
 *  - scale multiplies q.k (callers pass 1/sqrt(d) for standard attention);
 *    it must be finite and > 0, else FA_ERR_INVALID.
 *  - causal = 1 masks with bottom-right alignment: key j is visible to query
 *    i iff j <= i + (Lk - Lq).  For Lq == Lk this is the lower triangle with
 *    the diagonal; a single decode query sees its whole cache.
 *  - A query row with no visible key gets O = 0 and LSE = -inf.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Launches are asynchronous; no entry point synchronises unless the
 *    environment variable FA_CHECKED=1 is set, in which case each call
 *    synchronises its stream and returns the device-side status.
 *  - Host-side validation runs before any launch and returns FA_ERR_INVALID
 *    or FA_ERR_UNSUPPORTED without touching the GPU.  Index arrays that live
 *    on the device (cu_seqlens, block_table, seqlens) are checked by the
 *    kernels: a bad entry is never dereferenced (it is skipped, or its page
 *    is read as zeros, as each entry point states) and is recorded in a
 *    device error word that fa_device_status() reports.  The outputs of a
 *    sequence with a bad entry are not meaningful; the other sequences are
 *    unaffected.
 *  - Every wait inside a kernel is bounded in time; on expiry the kernel
 *    records FA_ERR_TIMEOUT in the device error word, drains its own copies,
 *    frees its tensor memory and returns.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID = 1,      /* bad argument (null/unaligned pointer, size, scale) */
    FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d not in {64,128}) */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = 4,      /* a kernel wait ran out (device error word) */
    FA_ERR_DEVICE_INDEX = 5, /* a kernel saw a bad cu_seqlens/block_table entry */
    FA_ERR_SCRATCH_CAPACITY = 6 /* fa_paged_fwd_noalloc: B*H too large for its fixed scratch */
} fa_status;

/* Version of this ABI (bumped on any signature change). */
int fa_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char* fa_status_string(int status);

/*
 * Dense batched multi-head forward (the fixed-length interface of the
 * dlog.com.cn page, §3.1).
 *   q, o : [B, N, H, d]   bf16
 *   k, v : [B, N, Hkv, d] bf16
 *   lse  : [B, H, N]      fp32, may be NULL (then not written)
 * Queries and keys have the same length N, so causal is the plain lower
 * triangle.  B, N, H, Hkv >= 1.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int Hkv, int N, int d, float scale, int causal,
           void* stream);

/*
 * Packed variable-length forward (the varlen interface of the dlog.com.cn
 * page, §3.3): the tokens of num_seqs sequences are concatenated.
 *   q, o : [total_q, H, d]   bf16
 *   k, v : [total_k, Hkv, d] bf16
 *   cu_seqlens_q, cu_seqlens_k : int32 [num_seqs + 1], DEVICE memory, prefix
 *       sums of the per-sequence lengths (first 0, non-decreasing, last =
 *       total).  Sequence s owns query rows [cu_q[s], cu_q[s+1]) and key rows
 *       [cu_k[s], cu_k[s+1]); no row attends across sequences.  The two
 *       arrays may be the same pointer.
 *   max_seqlen_q, max_seqlen_k : upper bounds of the per-sequence lengths
 *       (sizes the launch; a longer sequence is reported as
 *       FA_ERR_DEVICE_INDEX and its excess rows are not computed).
 *   lse  : [H, total_q] fp32, may be NULL.
 */
int fa_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                  int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                  int H, int Hkv, int d, float scale, int causal, void* stream);

/*
 * Packed layouts (the qkvpacked / kvpacked rows of the dlog.com.cn page's
 * function table, §3.2 and §3.3): the result a single projection produces,
 * passed without splitting it.  O and LSE are laid out as in fa_fwd /
 * fa_varlen_fwd.
 *   fa_qkvpacked_fwd        qkv : [B, N, 3, H, d] bf16 (index 0 Q, 1 K, 2 V;
 *                                 H query and key/value heads)
 *   fa_kvpacked_fwd         q   : [B, N, H, d];  kv : [B, N, 2, Hkv, d]
 *                                 (index 0 K, 1 V)
 *   fa_varlen_qkvpacked_fwd qkv : [total, 3, H, d]; one cu_seqlens for Q and K
 *   fa_varlen_kvpacked_fwd  q   : [total_q, H, d]; kv : [total_k, 2, Hkv, d]
 * Same arguments, conventions and errors as fa_fwd / fa_varlen_fwd
 * otherwise.  The packed tensors are read in place, through strided tensor
 * maps: nothing is copied.
 */
int fa_qkvpacked_fwd(const void* qkv, void* o, float* lse, int B, int H, int N, int d,
                     float scale, int causal, void* stream);
int fa_kvpacked_fwd(const void* q, const void* kv, void* o, float* lse,
                    int B, int H, int Hkv, int N, int d, float scale, int causal, void* stream);
int fa_varlen_qkvpacked_fwd(const void* qkv, void* o, float* lse, const int* cu_seqlens,
                            int num_seqs, int max_seqlen, int total, int H, int d,
                            float scale, int causal, void* stream);
int fa_varlen_kvpacked_fwd(const void* q, const void* kv, void* o, float* lse,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                           int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                           int H, int Hkv, int d, float scale, int causal, void* stream);

/*
 * Packed variable-length prefill whose keys and values are read through a
 * page table (the prefill entry point with block_table of the dlog.com.cn
 * page, "v3 实际调用的两个函数": a chunk that continues a cached prefix reads
 * its K/V straight from the page pool).
 *   q, o : [total_q, H, d] bf16, packed by cu_seqlens_q as in fa_varlen_fwd
 *   k_cache, v_cache : [num_pages, page_size, Hkv, d] bf16, the whole pool
 *   cu_seqlens_q, cu_seqlens_k : int32 [num_seqs + 1], DEVICE.  Sequence s
 *       has Lq = cu_q[s+1] - cu_q[s] queries and Lk = cu_k[s+1] - cu_k[s]
 *       keys; its keys are the logical tokens 0 .. Lk-1 of its pages and its
 *       queries are the newest Lq of them, so with causal = 1 query i sees
 *       keys j <= i + Lk - Lq (bottom-right; Lq <= Lk is expected).
 *   block_table : int32 [num_seqs, max_pages_per_seq], DEVICE; token t of
 *       sequence s is page block_table[s][t / page_size], slot
 *       t % page_size.  Entries past ceil(Lk / page_size) are never read; an
 *       entry outside [0, num_pages) is treated as a page of zeros and
 *       reported as FA_ERR_DEVICE_INDEX.  Slots of a sequence's last page
 *       past Lk may hold anything (they are never used, even if not finite).
 *   max_seqlen_q, max_seqlen_k : bounds as in fa_varlen_fwd;
 *       max_pages_per_seq * page_size >= max_seqlen_k.
 *   lse : [H, total_q] fp32, may be NULL.
 * page_size is 16, 32, 64 or 128 (else FA_ERR_UNSUPPORTED); each page is
 * read as one TMA box per 64-element panel, so larger pages take fewer boxes
 * per 128-key block (16 at d = 128 with 16-token pages, 2 with 128-token
 * pages).  (num_pages + 1) * page_size must stay below 2^31.
 */
int fa_varlen_paged_fwd(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, const int* block_table,
                        int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q,
                        int H, int Hkv, int d, int page_size, int num_pages,
                        int max_pages_per_seq, float scale, int causal, void* stream);

/*
 * Write one step's key/value rows into the page pool (the store_kvcache step
 * of the dlog.com.cn page, "v3 attention 的一条完整数据流", step 3, which runs
 * before the attention call of the same step).
 *   k, v : [num_tokens, Hkv, d] bf16
 *   k_cache, v_cache : [num_pages, page_size, Hkv, d] bf16, modified in place
 *   slot_mapping : int32 [num_tokens], DEVICE; row i goes to flat slot
 *       slot_mapping[i], i.e. page slot / page_size, offset
 *       slot % page_size.  A negative slot means "do not store" (padding);
 *       a slot >= num_pages * page_size is skipped and reported as
 *       FA_ERR_DEVICE_INDEX.  Two rows with the same slot: one of them wins.
 * num_tokens may be 0 (nothing is launched).  Any page_size >= 1.
 */
int fa_store_kvcache(const void* k, const void* v, void* k_cache, void* v_cache,
                     const int* slot_mapping, int num_tokens, int Hkv, int d,
                     int page_size, int num_pages, void* stream);

/*
 * Bytes of device workspace fa_paged_fwd needs for these sizes (the split-KV
 * partial results and, for the tensor-core path, the plan of its work
 * division).  Returns 0 for invalid sizes.
 */
size_t fa_paged_workspace_size(int B, int H, int d, int max_seqlen);

/*
 * Single-token decode over a paged KV cache (the kv-cache interface of the
 * dlog.com.cn page, §3.4 and its PagedAttention section).
 *   q, o      : [B, H, d] bf16 (one new token per sequence)
 *   k_cache, v_cache : [num_pages, page_size, Hkv, d] bf16, the whole pool
 *   block_table : int32 [B, max_pages_per_seq], DEVICE; logical token t of
 *       sequence b is page block_table[b][t / page_size], slot
 *       t % page_size.  Entries past ceil(seqlens[b] / page_size) are never
 *       read.  An entry outside [0, num_pages) is reported as
 *       FA_ERR_DEVICE_INDEX; the CUDA-core path skips its page, the
 *       tensor-core path (groups of 8 or more, below) reads it as zeros.
 *   seqlens   : int32 [B], DEVICE; cached tokens per sequence, each in
 *       [0, max_seqlen] (0 gives O = 0, LSE = -inf).
 *   lse       : [B, H] fp32, may be NULL.
 *   workspace : DEVICE scratch of at least
 *       fa_paged_workspace_size(B, H, d, max_seqlen) bytes, 16-byte aligned;
 *       it need not be initialised.
 * page_size is 16, 32, 64 or 128 (else FA_ERR_UNSUPPORTED), and
 * (num_pages + 1) * page_size must stay below 2^31.  causal is accepted;
 * under bottom-right alignment it does not change a single newest-token
 * query.
 * Groups of 8 to 64 query heads per kv head (H / Hkv) run on the tensor
 * cores: the group's query heads are the rows of one query tile, the
 * 64-key blocks of all (sequence, kv head) pairs are divided evenly over
 * two persistent CTAs per SM, and each CTA's partial results are merged as
 * in the CUDA-core path (three kernels on `stream`: a plan of the division,
 * the decode, the merge).  Smaller and larger groups use the CUDA-core split
 * kernel and its merge.  The results agree within the same tolerance; the
 * workspace is the same.
 */
int fa_paged_fwd(const void* q, const void* k_cache, const void* v_cache,
                 const int* block_table, const int* seqlens, void* o, float* lse,
                 int B, int H, int Hkv, int d, int page_size, int num_pages,
                 int max_pages_per_seq, int max_seqlen, float scale, int causal,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_paged_fwd without a caller workspace.  The pages describe no such call:
 * it exists for callers that cannot allocate device memory at the point they
 * run attention -- for example an engine that reserves all device memory up
 * front and hands out none afterwards, a plugin that runs inside someone
 * else's memory pool, or a decode step that must never call cudaMalloc
 * because an allocation can synchronise the device.
 *
 * Same arguments, layouts and results as fa_paged_fwd, minus workspace and
 * workspace_bytes.  The split-KV partials go to one fixed 16 MiB device array
 * inside this library, which every GPU that loads the library keeps until
 * the process exits.  The keys are split into as few pieces as needed for the
 * partials, B * H * splits * (d + 2) floats, to fit; 256 bytes of the array
 * are kept back for alignment, so a batch with
 * B * H * (d + 2) * 4 > 16 MiB - 256 bytes returns FA_ERR_SCRATCH_CAPACITY
 * before any launch (d = 128: at most 32,263 (sequence, head) pairs; d = 64:
 * at most 63,549).  Every query group takes the CUDA-core split kernel here,
 * including groups of 8 or more query heads per kv head, which fa_paged_fwd
 * sends to the tensor cores; the results agree within the same tolerance.  Nothing in the array needs to start at
 * zero: every partial the combine step reads is written earlier in the same
 * call.  All calls in the process share the array, so two calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race and
 * both results are undefined; order them on one stream.  The first call on a
 * device looks the array's address up with cudaGetSymbolAddress, so make
 * that first call before capturing any stream into a graph.  The call itself
 * allocates nothing (no cudaMalloc, no allocating library routine).
 */
int fa_paged_fwd_noalloc(const void* q, const void* k_cache, const void* v_cache,
                         const int* block_table, const int* seqlens, void* o, float* lse,
                         int B, int H, int Hkv, int d, int page_size, int num_pages,
                         int max_pages_per_seq, int max_seqlen, float scale, int causal,
                         void* stream);

/*
 * Copy the cached rows every sequence's page walk selects:
 * out[b][t][hk][:] = cache[block_table[b][t/page_size]][t%page_size][hk][:] for
 * t < seqlens[b].  out is bf16 [B, max_seqlen, Hkv, d] in DEVICE memory;
 * rows t >= seqlens[b] are left untouched.  A debugging aid: a kernel of its
 * own that shares the decode kernel's page lookup and row offset, not the
 * decode kernels themselves (their reads are checked bit for bit through
 * fa_paged_fwd and fa_varlen_paged_fwd with one-hot queries).
 */
int fa_paged_gather(const void* cache, const int* block_table, const int* seqlens, void* out,
                    int B, int Hkv, int d, int page_size, int num_pages,
                    int max_pages_per_seq, int max_seqlen, void* stream);

/*
 * Backward pass: the gradients dQ, dK, dV of a loss with respect to the
 * inputs of the forward, given dO.  P is recomputed from the forward's LSE
 * (it is never stored), then
 *
 *     dV = P^T dO,   dP = dO V^T,   dS_ij = P_ij (dP_ij - delta_i),
 *     delta_i = dO_i . O_i,   dQ = scale dS K,   dK = scale dS^T Q
 *
 * (the recomputation and the row-sum term of the lqnn.cn FlashAttention
 * article, §2.3 and §4.3, and of the yulong.wang page, §2.3).  With grouped
 * query heads, dK and dV of a kv head sum over its H / Hkv query heads.
 * dQ is accumulated on chip per 128-row query block and written once (no
 * atomics): the result is deterministic.
 *
 *   q, o, dout, dq : [B, N, H, d]   bf16   (o and lse: this library's forward
 *   k, v, dk, dv   : [B, N, Hkv, d] bf16    output for the same q, k, v,
 *   lse            : [B, H, N]      fp32    scale and causal)
 *   workspace      : DEVICE memory of at least
 *                    fa_bwd_workspace_bytes(B, B * N, H) bytes, 16-byte
 *                    aligned, owned by the caller; its contents on entry do
 *                    not matter and are overwritten.
 * Rows whose LSE is -inf (no visible key) contribute nothing; keys that no
 * query sees get dK = dV = 0.  Every row of dq, dk, dv is written.  Launches
 * three kernels on `stream`.  Errors as for fa_fwd; a workspace smaller than
 * required is FA_ERR_INVALID.
 */
size_t fa_bwd_workspace_bytes(int num_seqs, int total_q, int H);

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
           int causal, void* stream);

/*
 * Varlen backward: the packed layouts of fa_varlen_fwd (q, o, dout, dq:
 * [total_q, H, d]; k, v, dk, dv: [total_k, Hkv, d]; lse: [H, total_q];
 * cu_seqlens_*: int32 DEVICE [num_seqs + 1]), workspace of
 * fa_bwd_workspace_bytes(num_seqs, total_q, H) bytes.  Bottom-right causal as
 * in the forward.  A bad cu_seqlens entry skips that sequence (its outputs
 * are left untouched) and is reported by fa_device_status().
 */
int fa_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* workspace,
                  size_t workspace_bytes, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                  int H, int Hkv, int d, float scale, int causal, void* stream);

/*
 * Synchronise the stream, read the device error word and return FA_OK,
 * FA_ERR_TIMEOUT or FA_ERR_DEVICE_INDEX (or FA_ERR_CUDA if the sync itself
 * failed).  clear != 0 resets the word afterwards.
 */
int fa_device_status(void* stream, int clear);

/*
 * Self-test of the bounded wait: launch one CTA that waits on a barrier no
 * one arrives on, with a limit of limit_ns nanoseconds.  The kernel must
 * give up, record FA_ERR_TIMEOUT in the device error word and return, so the
 * next fa_device_status() reports FA_ERR_TIMEOUT and the context stays
 * usable.  No counterpart on the pages: it exists to test the failure path
 * without faulting or hanging a GPU.
 */
int fa_selftest_wait_timeout(long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
