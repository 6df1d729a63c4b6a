// Host side of the C-ABI declared in include/fa.h: argument validation,
// TMA descriptor encoding, kernel launches and the device error word.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

// Device error word: kernels OR FA_DEVERR_* bits into it.
__device__ unsigned int g_fa_error_word;

namespace {

constexpr int kAbiVersion = 4;
constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};

bool env_flag(const char* name) {
    const char* v = std::getenv(name);
    return v != nullptr && v[0] != '\0' && v[0] != '0';
}

unsigned long long wait_limit_ns() {
    const char* v = std::getenv("FA_WAIT_LIMIT_NS");
    if (v != nullptr && v[0] != '\0') {
        const unsigned long long x = std::strtoull(v, nullptr, 10);
        if (x > 0) return x;
    }
    return 2000000000ull;  // 2 s: far longer than any launch this library makes
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resolve the driver entry point and this device's error-word address.
fa_status ensure_init(unsigned int** err_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (g_err_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_fa_error_word) != cudaSuccess) return FA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned int*>(ptr);
    }
    *err_out = g_err_ptr[dev];
    return FA_OK;
}

// 3-D view (d, heads, rows) of a [rows, heads, d] bf16 tensor; a box is 64
// elements of d (128 bytes, the swizzle span) x 1 head x box_rows rows (a
// 128-row tile, or one 16-token page of the paged pool).
// row_stride is in elements between consecutive rows (heads * d for a dense
// tensor, more for one slot of a packed [rows, 3 or 2, heads, d] tensor).
fa_status make_map(CUtensorMap* map, const void* base, int d, int heads, long long rows,
                   int box_rows = fa::kBlockM, long long row_stride = 0) {
    if (row_stride == 0) row_stride = static_cast<long long>(heads) * d;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(row_stride) * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

fa_status finish(cudaError_t e, cudaStream_t stream) {
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (env_flag("FA_CHECKED")) return static_cast<fa_status>(fa_device_status(stream, 1));
    return FA_OK;
}

bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

}  // namespace

extern "C" {

int fa_abi_version(void) { return kAbiVersion; }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID: return "FA_ERR_INVALID: bad argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: valid but not implemented";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait ran out";
        case FA_ERR_DEVICE_INDEX: return "FA_ERR_DEVICE_INDEX: bad cu_seqlens/seqlens/block_table entry";
        case FA_ERR_SCRATCH_CAPACITY:
            return "FA_ERR_SCRATCH_CAPACITY: B*H*(d+2)*4 bytes exceed the fixed 16 MiB decode scratch";
        default: return "unknown fa_status";
    }
}

}  // extern "C"

namespace {

// One operand of the prefill: its first element and the elements between
// consecutive rows (tokens).
struct Operand {
    const void* base;
    long long row_stride;
};

fa_status dense_impl(Operand q, Operand k, Operand v, void* o, float* lse, int B, int H, int Hkv, int N, int d,
                     float scale, int causal, void* stream) {
    if (!q.base || !k.base || !v.base || !o) return FA_ERR_INVALID;
    if (!aligned16(q.base) || !aligned16(k.base) || !aligned16(v.base) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID;
    if (B < 1 || H < 1 || Hkv < 1 || N < 1 || H % Hkv != 0 || !scale_ok(scale)) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * N;
    if (B > 65535 || H > 65535 || rows > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    CUtensorMap tq, tk, tv;
    if ((st = make_map(&tq, q.base, d, H, rows, fa::kBlockM, q.row_stride)) != FA_OK) return st;
    const int kv_box = fa::kBlockN;
    if ((st = make_map(&tk, k.base, d, Hkv, rows, kv_box, k.row_stride)) != FA_OK) return st;
    if ((st = make_map(&tv, v.base, d, Hkv, rows, kv_box, v.row_stride)) != FA_OK) return st;
    fa::PrefillParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = nullptr;
    p.cu_k = nullptr;
    p.N = N;
    p.num_seqs = B;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.max_seqlen_q = N;
    p.max_seqlen_k = N;
    p.total_q = static_cast<int>(rows);
    p.total_k = static_cast<int>(rows);
    p.num_q_blocks = (N + fa::kBlockM - 1) / fa::kBlockM;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse_head_stride = N;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the causal grid enumerates (256-row block, head) pairs in grid.x
    if (static_cast<long long>((p.num_q_blocks + 1) / 2) * H > 2147483647ll) return FA_ERR_UNSUPPORTED;
    return finish(fa::launch_prefill(tq, tk, tv, p, d, causal != 0, s), s);
}

fa_status varlen_impl(Operand q, Operand k, Operand v, void* o, float* lse, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q,
                      int total_k, int H, int Hkv, int d, float scale, int causal, void* stream) {
    if (!q.base || !k.base || !v.base || !o || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID;
    if (!aligned16(q.base) || !aligned16(k.base) || !aligned16(v.base) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_INVALID;
    if (num_seqs < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 ||
        max_seqlen_k < 1 || !scale_ok(scale))
        return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    CUtensorMap tq, tk, tv;
    if ((st = make_map(&tq, q.base, d, H, total_q, fa::kBlockM, q.row_stride)) != FA_OK) return st;
    const int kv_box = fa::kBlockN;
    if ((st = make_map(&tk, k.base, d, Hkv, total_k, kv_box, k.row_stride)) != FA_OK) return st;
    if ((st = make_map(&tv, v.base, d, Hkv, total_k, kv_box, v.row_stride)) != FA_OK) return st;
    fa::PrefillParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.N = 0;
    p.num_seqs = num_seqs;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.num_q_blocks = (max_seqlen_q + fa::kBlockM - 1) / fa::kBlockM;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse_head_stride = total_q;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the causal grid enumerates (256-row block, head) pairs in grid.x
    if (static_cast<long long>((p.num_q_blocks + 1) / 2) * H > 2147483647ll) return FA_ERR_UNSUPPORTED;
    return finish(fa::launch_prefill(tq, tk, tv, p, d, causal != 0, s), s);
}

// Slot `slot` of a packed [rows, n, heads, d] bf16 tensor.
Operand packed(const void* base, int slot, int n, int heads, int d) {
    if (base == nullptr || heads < 1 || d < 1) return Operand{base, 0};  // sizes are rejected by the caller
    return Operand{static_cast<const uint16_t*>(base) + static_cast<size_t>(slot) * heads * d,
                   static_cast<long long>(n) * heads * d};
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N, int d,
           float scale, int causal, void* stream) {
    return dense_impl(Operand{q, 0}, Operand{k, 0}, Operand{v, 0}, o, lse, B, H, Hkv, N, d, scale, causal, stream);
}

int fa_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q,
                  int total_k, int H, int Hkv, int d, float scale, int causal, void* stream) {
    return varlen_impl(Operand{q, 0}, Operand{k, 0}, Operand{v, 0}, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs,
                       max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal, stream);
}

int fa_qkvpacked_fwd(const void* qkv, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                     void* stream) {
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return dense_impl(packed(qkv, 0, 3, H, d), packed(qkv, 1, 3, H, d), packed(qkv, 2, 3, H, d), o, lse, B, H, H, N,
                      d, scale, causal, stream);
}

int fa_kvpacked_fwd(const void* q, const void* kv, void* o, float* lse, int B, int H, int Hkv, int N, int d,
                    float scale, int causal, void* stream) {
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return dense_impl(Operand{q, 0}, packed(kv, 0, 2, Hkv, d), packed(kv, 1, 2, Hkv, d), o, lse, B, H, Hkv, N, d,
                      scale, causal, stream);
}

int fa_varlen_qkvpacked_fwd(const void* qkv, void* o, float* lse, const int* cu_seqlens, int num_seqs,
                            int max_seqlen, int total, int H, int d, float scale, int causal, void* stream) {
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return varlen_impl(packed(qkv, 0, 3, H, d), packed(qkv, 1, 3, H, d), packed(qkv, 2, 3, H, d), o, lse,
                       cu_seqlens, cu_seqlens, num_seqs, max_seqlen, max_seqlen, total, total, H, H, d, scale, causal,
                       stream);
}

int fa_varlen_kvpacked_fwd(const void* q, const void* kv, void* o, float* lse, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q,
                           int total_k, int H, int Hkv, int d, float scale, int causal, void* stream) {
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return varlen_impl(Operand{q, 0}, packed(kv, 0, 2, Hkv, d), packed(kv, 1, 2, Hkv, d), o, lse, cu_seqlens_q,
                       cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale,
                       causal, stream);
}

int fa_varlen_paged_fwd(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, const int* block_table, int num_seqs,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int H, int Hkv, int d, int page_size,
                        int num_pages, int max_pages_per_seq, float scale, int causal, void* stream) {
    if (!q || !k_cache || !v_cache || !o || !cu_seqlens_q || !cu_seqlens_k || !block_table) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u))
        return FA_ERR_INVALID;
    if (num_seqs < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || total_q < 1 || max_seqlen_q < 1 || max_seqlen_k < 1 ||
        num_pages < 1 || max_pages_per_seq < 1 || !scale_ok(scale))
        return FA_ERR_INVALID;
    if (static_cast<long long>(max_pages_per_seq) * page_size < max_seqlen_k) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::page_size_ok(page_size)) return FA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
    // rows of the pool view, plus one page of zero fill past its end, must be
    // addressable by a 32-bit TMA coordinate
    if ((static_cast<long long>(num_pages) + 1) * page_size > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    const long long pool_rows = static_cast<long long>(num_pages) * page_size;
    CUtensorMap tq, tk, tv;
    if ((st = make_map(&tq, q, d, H, total_q)) != FA_OK) return st;
    // one box per page, or per block-sized share of a page taller than a block
    const int kv_box = page_size < fa::kBlockN ? page_size : fa::kBlockN;
    if ((st = make_map(&tk, k_cache, d, Hkv, pool_rows, kv_box)) != FA_OK) return st;
    if ((st = make_map(&tv, v_cache, d, Hkv, pool_rows, kv_box)) != FA_OK) return st;
    fa::PrefillParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.N = 0;
    p.num_seqs = num_seqs;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.total_q = total_q;
    p.total_k = 0;  // not used with a page table
    p.num_q_blocks = (max_seqlen_q + fa::kBlockM - 1) / fa::kBlockM;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse_head_stride = total_q;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();
    p.block_table = block_table;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.page_shift = fa::page_shift(page_size);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the causal grid enumerates (256-row block, head) pairs in grid.x
    if (static_cast<long long>((p.num_q_blocks + 1) / 2) * H > 2147483647ll) return FA_ERR_UNSUPPORTED;
    return finish(fa::launch_prefill(tq, tk, tv, p, d, causal != 0, s), s);
}

int fa_store_kvcache(const void* k, const void* v, void* k_cache, void* v_cache, const int* slot_mapping,
                     int num_tokens, int Hkv, int d, int page_size, int num_pages, void* stream) {
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return FA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return FA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 3u) return FA_ERR_INVALID;
    if (num_tokens < 0 || Hkv < 1 || num_pages < 1 || page_size < 1) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const long long num_slots = static_cast<long long>(num_pages) * page_size;
    if (num_slots > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (num_tokens == 0) return finish(cudaSuccess, s);
    fa::StoreParams p{};
    p.k = k;
    p.v = v;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.slot_mapping = slot_mapping;
    p.T = num_tokens;
    p.Hkv = Hkv;
    p.d = d;
    p.num_slots = num_slots;
    p.err = err;
    return finish(fa::launch_store_kvcache(p, s), s);
}

size_t fa_paged_workspace_size(int B, int H, int d, int max_seqlen) {
    if (B < 1 || H < 1 || max_seqlen < 0 || (d != 64 && d != 128)) return 0;
    // The larger of the two paths' layouts: the tensor-core path keeps one
    // more partial per (sequence, head) than the CUDA-core path's splits, and
    // its plan (prefix[B + 1], seg_ns[B * Hkv <= B * H], W).
    const size_t splits = static_cast<size_t>(fa::decode_max_splits(max_seqlen)) + 1;
    const size_t slots = static_cast<size_t>(B) * H * splits;
    size_t bytes = (slots * d * sizeof(float) + 255) & ~size_t(255);
    bytes += (slots * 2 * sizeof(float) + 255) & ~size_t(255);
    bytes += ((static_cast<size_t>(B) + 1 + static_cast<size_t>(B) * H + 4) * sizeof(int) + 255) & ~size_t(255);
    return bytes;
}

int fa_paged_fwd(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                 const int* seqlens, void* o, float* lse, int B, int H, int Hkv, int d, int page_size,
                 int num_pages, int max_pages_per_seq, int max_seqlen, float scale, int causal, void* workspace,
                 size_t workspace_bytes, void* stream) {
    (void)causal;  // a single newest-token query sees its whole cache either way
    if (!q || !k_cache || !v_cache || !block_table || !seqlens || !o || !workspace) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(workspace))
        return FA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return FA_ERR_INVALID;
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || num_pages < 1 || max_pages_per_seq < 1 || max_seqlen < 0 ||
        !scale_ok(scale))
        return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::page_size_ok(page_size)) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_pages_per_seq) * page_size < max_seqlen) return FA_ERR_INVALID;
    if ((static_cast<long long>(num_pages) + 1) * page_size > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    if (B > 65535) return FA_ERR_UNSUPPORTED;
    const size_t need = fa_paged_workspace_size(B, H, d, max_seqlen);
    if (need == 0 || workspace_bytes < need) return FA_ERR_INVALID;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    const int group = H / Hkv;
    if (group >= fa::kDecodeTcMinGroup && group <= fa::kDecodeQRows &&
        static_cast<long long>(B) * Hkv * ((max_seqlen + 63) / 64) < (1ll << 31)) {
        // Large query groups: the tensor-core decode (the group's query heads
        // are the rows of a Q tile), then the combine step.
        const long long pool_rows = static_cast<long long>(num_pages) * page_size;
        CUtensorMap tq, tk, tv;
        if ((st = make_map(&tq, q, d, 1, static_cast<long long>(B) * H, fa::kDecodeQRows)) != FA_OK) return st;
        // one box per page, or per 64-key block of a larger page
        const int box_rows = page_size < fa::kDecodeBlockN ? page_size : fa::kDecodeBlockN;
        if ((st = make_map(&tk, k_cache, d, Hkv, pool_rows, box_rows)) != FA_OK) return st;
        if ((st = make_map(&tv, v_cache, d, Hkv, pool_rows, box_rows)) != FA_OK) return st;
        // Partials: one more slot per (sequence, head) than the CUDA-core
        // path's splits (a pair's blocks span at most that many CTAs), then
        // the plan arrays.
        const int splits = fa::decode_max_splits(max_seqlen) + 1;
        const size_t slots = static_cast<size_t>(B) * H * splits;
        char* w = static_cast<char*>(workspace);
        float* ws_o = reinterpret_cast<float*>(w);
        w += (slots * d * sizeof(float) + 255) & ~size_t(255);
        float* ws_ml = reinterpret_cast<float*>(w);
        w += (slots * 2 * sizeof(float) + 255) & ~size_t(255);
        int* prefix = reinterpret_cast<int*>(w);
        int* seg_ns = prefix + B + 1;
        int* plan = seg_ns + static_cast<size_t>(B) * Hkv;
        fa::DecodeTcParams tp{};
        tp.seqlens = seqlens;
        tp.block_table = block_table;
        tp.ws_o = ws_o;
        tp.ws_ml = ws_ml;
        tp.prefix = prefix;
        tp.seg_ns = seg_ns;
        tp.plan = plan;
        tp.err = err;
        tp.B = B;
        tp.H = H;
        tp.Hkv = Hkv;
        tp.group = group;
        tp.max_pages = max_pages_per_seq;
        tp.num_pages = num_pages;
        tp.page_shift = fa::page_shift(page_size);
        tp.max_seqlen = max_seqlen;
        tp.max_splits = splits;
        tp.scale_log2 = scale * 1.4426950408889634f;
        tp.wait_limit_ns = wait_limit_ns();
        fa::DecodeParams p{};
        p.seqlens = seqlens;
        p.o = o;
        p.lse = lse;
        p.B = B;
        p.H = H;
        p.Hkv = Hkv;
        p.group = group;
        p.num_pages = num_pages;
        p.max_pages = max_pages_per_seq;
        p.max_seqlen = max_seqlen;
        p.split_tokens = fa::decode_split_tokens(max_seqlen);
        p.max_splits = splits;
        p.page_shift = fa::page_shift(page_size);
        p.ws_o = ws_o;
        p.ws_ml = ws_ml;
        p.seg_ns = seg_ns;
        p.scale_log2 = tp.scale_log2;
        p.err = err;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        cudaError_t e = fa::launch_decode_tc(tq, tk, tv, tp, d, s);
        if (e == cudaSuccess) e = fa::launch_decode_combine(p, d, s);
        return finish(e, s);
    }
    fa::DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table;
    p.seqlens = seqlens;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.num_pages = num_pages;
    p.max_pages = max_pages_per_seq;
    p.max_seqlen = max_seqlen;
    p.split_tokens = fa::decode_split_tokens(max_seqlen);
    p.max_splits = fa::decode_max_splits(max_seqlen);
    p.page_shift = fa::page_shift(page_size);
    const size_t slots = static_cast<size_t>(B) * H * p.max_splits;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((slots * d * sizeof(float) + 255) & ~size_t(255)));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(fa::launch_decode(p, d, s), s);
}

int fa_paged_fwd_noalloc(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                         const int* seqlens, void* o, float* lse, int B, int H, int Hkv, int d, int page_size,
                         int num_pages, int max_pages_per_seq, int max_seqlen, float scale, int causal,
                         void* stream) {
    (void)causal;
    if (!q || !k_cache || !v_cache || !block_table || !seqlens || !o) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return FA_ERR_INVALID;
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || num_pages < 1 || max_pages_per_seq < 1 || max_seqlen < 0 ||
        !scale_ok(scale))
        return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::page_size_ok(page_size)) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_pages_per_seq) * page_size < max_seqlen) return FA_ERR_INVALID;
    if ((static_cast<long long>(num_pages) + 1) * page_size > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    if (B > 65535) return FA_ERR_UNSUPPORTED;
    // Split the keys so that the per-split partials fit the fixed scratch:
    // each (sequence, head, split) slot takes d floats of O and two of (m, l).
    const size_t cap = fa::kStaticScratchBytes;
    const size_t per_split = static_cast<size_t>(B) * H * (static_cast<size_t>(d) + 2) * sizeof(float);
    if (per_split + 256 > cap) return FA_ERR_SCRATCH_CAPACITY;
    const int fit = static_cast<int>((cap - 256) / per_split);
    int splits = fa::decode_max_splits(max_seqlen);
    int split_tokens = fa::decode_split_tokens(max_seqlen);
    if (splits > fit) {
        split_tokens = (max_seqlen + fit - 1) / fit;
        split_tokens = (split_tokens + fa::kPageChunk - 1) / fa::kPageChunk * fa::kPageChunk;
        splits = (max_seqlen + split_tokens - 1) / split_tokens;
        if (splits < 1) splits = 1;
    }
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    if (fa::static_scratch(&scratch, &scratch_bytes) != cudaSuccess) return FA_ERR_CUDA;
    const size_t slots = static_cast<size_t>(B) * H * splits;
    const size_t o_bytes = (slots * d * sizeof(float) + 255) & ~size_t(255);
    if (o_bytes + slots * 2 * sizeof(float) > scratch_bytes) return FA_ERR_SCRATCH_CAPACITY;
    fa::DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table;
    p.seqlens = seqlens;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.num_pages = num_pages;
    p.max_pages = max_pages_per_seq;
    p.max_seqlen = max_seqlen;
    p.split_tokens = split_tokens;
    p.max_splits = splits;
    p.page_shift = fa::page_shift(page_size);
    p.ws_o = static_cast<float*>(scratch);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(fa::launch_decode(p, d, s), s);
}

int fa_paged_gather(const void* cache, const int* block_table, const int* seqlens, void* out, int B, int Hkv, int d,
                    int page_size, int num_pages, int max_pages_per_seq, int max_seqlen, void* stream) {
    if (!cache || !block_table || !seqlens || !out) return FA_ERR_INVALID;
    if (!aligned16(cache) || !aligned16(out)) return FA_ERR_INVALID;
    if (B < 1 || Hkv < 1 || num_pages < 1 || max_pages_per_seq < 1 || max_seqlen < 1) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::page_size_ok(page_size) || B > 65535) return FA_ERR_UNSUPPORTED;
    if ((static_cast<long long>(num_pages) + 1) * page_size > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_pages_per_seq) * page_size < max_seqlen) return FA_ERR_INVALID;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    fa::GatherParams p{};
    p.cache = cache;
    p.block_table = block_table;
    p.seqlens = seqlens;
    p.out = out;
    p.B = B;
    p.Hkv = Hkv;
    p.d = d;
    p.num_pages = num_pages;
    p.max_pages = max_pages_per_seq;
    p.max_seqlen = max_seqlen;
    p.page_shift = fa::page_shift(page_size);
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(fa::launch_gather(p, s), s);
}

int fa_device_status(void* stream, int clear) {
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    if (clear && word != 0) {
        if (cudaMemsetAsync(err, 0, sizeof(unsigned int), s) != cudaSuccess) return FA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (word & FA_DEVERR_TIMEOUT) return FA_ERR_TIMEOUT;
    if (word & FA_DEVERR_INDEX) return FA_ERR_DEVICE_INDEX;
    if (word & FA_DEVERR_LAYOUT) return FA_ERR_CUDA;
    return FA_OK;
}

int fa_selftest_wait_timeout(long long limit_ns, void* stream) {
    if (limit_ns <= 0 || limit_ns > 10000000000ll) return FA_ERR_INVALID;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fa::launch_wait_selftest(err, static_cast<unsigned long long>(limit_ns), s) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

}  // extern "C"

namespace {

// Shared body of fa_bwd and fa_varlen_bwd (cu_q == nullptr: dense).
fa_status backward_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        const int* cu_q, const int* cu_k, int num_seqs, int N, int max_seqlen_q, int max_seqlen_k,
                        int total_q, int total_k, int H, int Hkv, int d, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_INVALID;
    if (cu_q && ((reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u)))
        return FA_ERR_INVALID;
    if (num_seqs < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 ||
        max_seqlen_k < 1 || !scale_ok(scale))
        return FA_ERR_INVALID;
    if (workspace_bytes < fa_bwd_workspace_bytes(num_seqs, total_q, H)) return FA_ERR_INVALID;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
    // grid.x of the two main kernels enumerates (128-row block, head) pairs
    if (static_cast<long long>((max_seqlen_q + fa::kBlockM - 1) / fa::kBlockM) * H > 2147483647ll ||
        static_cast<long long>((max_seqlen_k + fa::kBlockN - 1) / fa::kBlockN) * Hkv > 2147483647ll)
        return FA_ERR_UNSUPPORTED;
    unsigned int* err = nullptr;
    fa_status st = ensure_init(&err);
    if (st != FA_OK) return st;
    CUtensorMap tq, tk, tv, tdo;
    if ((st = make_map(&tq, q, d, H, total_q)) != FA_OK) return st;
    if ((st = make_map(&tk, k, d, Hkv, total_k)) != FA_OK) return st;
    if ((st = make_map(&tv, v, d, Hkv, total_k)) != FA_OK) return st;
    if ((st = make_map(&tdo, dout, d, H, total_q)) != FA_OK) return st;
    fa::BackwardParams p{};
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.ws = static_cast<float*>(workspace);
    p.ws_head_stride = fa::bwd_ws_head_stride(total_q, num_seqs);
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.N = N;
    p.num_seqs = num_seqs;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.num_q_blocks = (max_seqlen_q + fa::kBlockM - 1) / fa::kBlockM;
    p.num_k_blocks = (max_seqlen_k + fa::kBlockN - 1) / fa::kBlockN;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse_head_stride = cu_q ? total_q : N;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(fa::launch_backward(tq, tk, tv, tdo, p, d, causal != 0, s), s);
}

}  // namespace

extern "C" {

size_t fa_bwd_workspace_bytes(int num_seqs, int total_q, int H) {
    if (num_seqs < 1 || total_q < 0 || H < 1) return 0;
    return 2 * static_cast<size_t>(H) * static_cast<size_t>(fa::bwd_ws_head_stride(total_q, num_seqs)) * sizeof(float);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
           float scale, int causal, void* stream) {
    if (B < 1 || N < 1) return FA_ERR_INVALID;
    const long long rows = static_cast<long long>(B) * N;
    if (rows > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    return backward_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, nullptr, nullptr, B, N, N, N,
                         static_cast<int>(rows), static_cast<int>(rows), H, Hkv, d, scale, causal, stream);
}

int fa_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q,
                  int total_k, int H, int Hkv, int d, float scale, int causal, void* stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID;
    return backward_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, cu_seqlens_q, cu_seqlens_k,
                         num_seqs, 0, max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal, stream);
}

}  // extern "C"
