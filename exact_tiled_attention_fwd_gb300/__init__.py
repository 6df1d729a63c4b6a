"""Python binding of the sm_103a exact-attention library (libfa_sm103.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C-ABI of include/fa.h.  The functions below carry the C
names (fa_fwd, fa_varlen_fwd, fa_paged_fwd, ...) and accept either raw device
addresses (ints) or torch tensors for the pointer arguments; ``stream`` may be
a torch.cuda.Stream, a raw cudaStream_t (int) or None (torch's current
stream).  Non-zero statuses are returned, not raised; the ``attention*``
helpers allocate outputs and raise FAError instead.

There is no CPU fallback: if the library is missing, loading raises.
"""

from __future__ import annotations

import ctypes
import math
import os

from ._build import LIB as LIB_PATH

FA_OK = 0
FA_ERR_INVALID = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_DEVICE_INDEX = 5
FA_ERR_SCRATCH_CAPACITY = 6

EXPORTS = (
    "fa_abi_version", "fa_status_string", "fa_fwd", "fa_varlen_fwd", "fa_paged_workspace_size",
    "fa_paged_fwd", "fa_paged_fwd_noalloc", "fa_paged_gather", "fa_device_status", "fa_selftest_wait_timeout",
    "fa_varlen_paged_fwd", "fa_store_kvcache", "fa_qkvpacked_fwd", "fa_kvpacked_fwd", "fa_varlen_qkvpacked_fwd",
    "fa_varlen_kvpacked_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_varlen_bwd",
)

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path: str | None = None):
    """Load (once) and return the ctypes handle of libfa_sm103.so."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_abi_version.restype = i
    lib.fa_abi_version.argtypes = []
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i]
    lib.fa_fwd.restype = i
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_varlen_fwd.restype = i
    lib.fa_varlen_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_paged_workspace_size.restype = sz
    lib.fa_paged_workspace_size.argtypes = [i, i, i, i]
    lib.fa_paged_fwd.restype = i
    lib.fa_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_paged_fwd_noalloc.restype = i
    lib.fa_paged_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_qkvpacked_fwd.restype = i
    lib.fa_qkvpacked_fwd.argtypes = [vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_kvpacked_fwd.restype = i
    lib.fa_kvpacked_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_varlen_qkvpacked_fwd.restype = i
    lib.fa_varlen_qkvpacked_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_varlen_kvpacked_fwd.restype = i
    lib.fa_varlen_kvpacked_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_varlen_paged_fwd.restype = i
    lib.fa_varlen_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_store_kvcache.restype = i
    lib.fa_store_kvcache.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.fa_paged_gather.restype = i
    lib.fa_paged_gather.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.fa_device_status.restype = i
    lib.fa_device_status.argtypes = [vp, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.fa_bwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
    lib.fa_varlen_bwd.restype = i
    lib.fa_varlen_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, i, i, i, i, i, i, i, i, f, i,
                                  vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()  # torch tensor


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_abi_version() -> int:
    return load().fa_abi_version()


def fa_status_string(status: int) -> str:
    return status_string(status)


def fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream=None) -> int:
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d, scale,
                         int(bool(causal)), _stream(stream))


def fa_varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k,
                  total_q, total_k, H, Hkv, d, scale, causal, stream=None) -> int:
    return load().fa_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                _ptr(cu_seqlens_k), num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                H, Hkv, d, scale, int(bool(causal)), _stream(stream))


def fa_qkvpacked_fwd(qkv, o, lse, B, H, N, d, scale, causal, stream=None) -> int:
    return load().fa_qkvpacked_fwd(_ptr(qkv), _ptr(o), _ptr(lse), B, H, N, d, scale, int(bool(causal)),
                                   _stream(stream))


def fa_kvpacked_fwd(q, kv, o, lse, B, H, Hkv, N, d, scale, causal, stream=None) -> int:
    return load().fa_kvpacked_fwd(_ptr(q), _ptr(kv), _ptr(o), _ptr(lse), B, H, Hkv, N, d, scale, int(bool(causal)),
                                  _stream(stream))


def fa_varlen_qkvpacked_fwd(qkv, o, lse, cu_seqlens, num_seqs, max_seqlen, total, H, d, scale, causal,
                            stream=None) -> int:
    return load().fa_varlen_qkvpacked_fwd(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(cu_seqlens), num_seqs, max_seqlen,
                                          total, H, d, scale, int(bool(causal)), _stream(stream))


def fa_varlen_kvpacked_fwd(q, kv, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k,
                           total_q, total_k, H, Hkv, d, scale, causal, stream=None) -> int:
    return load().fa_varlen_kvpacked_fwd(_ptr(q), _ptr(kv), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                         _ptr(cu_seqlens_k), num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                         H, Hkv, d, scale, int(bool(causal)), _stream(stream))


def fa_varlen_paged_fwd(q, k_cache, v_cache, o, lse, cu_seqlens_q, cu_seqlens_k, block_table, num_seqs,
                        max_seqlen_q, max_seqlen_k, total_q, H, Hkv, d, page_size, num_pages, max_pages_per_seq,
                        scale, causal, stream=None) -> int:
    return load().fa_varlen_paged_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(block_table), num_seqs,
                                      max_seqlen_q, max_seqlen_k, total_q, H, Hkv, d, page_size, num_pages,
                                      max_pages_per_seq, scale, int(bool(causal)), _stream(stream))


def fa_store_kvcache(k, v, k_cache, v_cache, slot_mapping, num_tokens, Hkv, d, page_size, num_pages,
                     stream=None) -> int:
    return load().fa_store_kvcache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), num_tokens,
                                   Hkv, d, page_size, num_pages, _stream(stream))


def fa_paged_workspace_size(B, H, d, max_seqlen) -> int:
    return load().fa_paged_workspace_size(B, H, d, max_seqlen)


def fa_paged_fwd(q, k_cache, v_cache, block_table, seqlens, o, lse, B, H, Hkv, d, page_size, num_pages,
                 max_pages_per_seq, max_seqlen, scale, causal, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_paged_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seqlens), _ptr(o),
                               _ptr(lse), B, H, Hkv, d, page_size, num_pages, max_pages_per_seq, max_seqlen,
                               scale, int(bool(causal)), _ptr(workspace), workspace_bytes, _stream(stream))


def fa_paged_fwd_noalloc(q, k_cache, v_cache, block_table, seqlens, o, lse, B, H, Hkv, d, page_size, num_pages,
                         max_pages_per_seq, max_seqlen, scale, causal, stream=None) -> int:
    return load().fa_paged_fwd_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seqlens),
                                       _ptr(o), _ptr(lse), B, H, Hkv, d, page_size, num_pages, max_pages_per_seq,
                                       max_seqlen, scale, int(bool(causal)), _stream(stream))


def fa_paged_gather(cache, block_table, seqlens, out, B, Hkv, d, page_size, num_pages, max_pages_per_seq,
                    max_seqlen, stream=None) -> int:
    return load().fa_paged_gather(_ptr(cache), _ptr(block_table), _ptr(seqlens), _ptr(out), B, Hkv, d, page_size,
                                  num_pages, max_pages_per_seq, max_seqlen, _stream(stream))


def fa_device_status(stream=None, clear=True) -> int:
    return load().fa_device_status(_stream(stream), int(bool(clear)))


def fa_bwd_workspace_bytes(num_seqs, total_q, H) -> int:
    return load().fa_bwd_workspace_bytes(num_seqs, total_q, H)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal,
           stream=None) -> int:
    return load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                         _ptr(workspace), workspace_bytes, B, H, Hkv, N, d, scale, int(bool(causal)), _stream(stream))


def fa_varlen_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, cu_seqlens_q, cu_seqlens_k,
                  num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal,
                  stream=None) -> int:
    return load().fa_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(workspace), workspace_bytes, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale,
                                int(bool(causal)), _stream(stream))


def fa_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return load().fa_selftest_wait_timeout(int(limit_ns), _stream(stream))


# ----------------------------------------------------------------- torch helpers

def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def _req(t, name, dtype):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attention(q, k, v, scale=None, causal=False, out=None, lse=None, return_lse=True, stream=None):
    """Dense forward.  q: [B, N, H, d], k, v: [B, N, Hkv, d] bf16 CUDA tensors.
    Returns (O [B, N, H, d] bf16, LSE [B, H, N] fp32)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name, torch.bfloat16)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d] matching q")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(fa_fwd(q, k, v, out, lse if return_lse else None, B, H, Hkv, N, d, scale, causal, stream), "fa_fwd")
    return out, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale=None, causal=False,
                     out=None, lse=None, stream=None):
    """Packed varlen forward.  q: [total_q, H, d], k, v: [total_k, Hkv, d] bf16;
    cu_seqlens_*: int32 CUDA [num_seqs + 1].  Returns (O, LSE [H, total_q])."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name, torch.bfloat16)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _req(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_varlen_fwd(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q.numel() - 1, max_seqlen_q,
                       max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal, stream)
    _check(st, "fa_varlen_fwd")
    return out, lse


def attention_paged(q, k_cache, v_cache, block_table, seqlens, max_seqlen, scale=None, causal=True, out=None,
                    lse=None, workspace=None, stream=None):
    """Paged decode.  q: [B, H, d]; caches: [num_pages, 16, Hkv, d] bf16;
    block_table: int32 [B, max_pages]; seqlens: int32 [B].
    Returns (O [B, H, d], LSE [B, H])."""
    import torch

    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _req(t, name, torch.bfloat16)
    _req(block_table, "block_table", torch.int32)
    _req(seqlens, "seqlens", torch.int32)
    B, H, d = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = fa_paged_workspace_size(B, H, d, max_seqlen)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = fa_paged_fwd(q, k_cache, v_cache, block_table, seqlens, out, lse, B, H, Hkv, d, page_size, num_pages,
                      block_table.shape[1], max_seqlen, scale, causal, workspace, workspace.numel(), stream)
    _check(st, "fa_paged_fwd")
    return out, lse


def store_kvcache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """Write this step's rows into the page pool.  k, v: [T, Hkv, d] bf16;
    caches: [num_pages, page_size, Hkv, d] bf16; slot_mapping: int32 [T]
    (flat slots, negative = skip).  Modifies the caches in place."""
    import torch

    for name, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache)):
        _req(t, name, torch.bfloat16)
    _req(slot_mapping, "slot_mapping", torch.int32)
    T, Hkv, d = k.shape
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    st = fa_store_kvcache(k, v, k_cache, v_cache, slot_mapping, T, Hkv, d, page_size, num_pages, stream)
    _check(st, "fa_store_kvcache")


def attention_varlen_paged(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q,
                           max_seqlen_k, scale=None, causal=True, out=None, lse=None, stream=None):
    """Packed varlen prefill reading K/V through a page table (a chunk that
    continues a cached prefix).  q: [total_q, H, d]; caches: [num_pages, 16,
    Hkv, d] bf16; cu_seqlens_q/k: int32 [num_seqs + 1]; block_table: int32
    [num_seqs, max_pages].  Returns (O [total_q, H, d], LSE [H, total_q])."""
    import torch

    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _req(t, name, torch.bfloat16)
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("block_table", block_table)):
        _req(t, name, torch.int32)
    total_q, H, d = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_varlen_paged_fwd(q, k_cache, v_cache, out, lse, cu_seqlens_q, cu_seqlens_k, block_table,
                             cu_seqlens_q.numel() - 1, max_seqlen_q, max_seqlen_k, total_q, H, Hkv, d, page_size,
                             num_pages, block_table.shape[1], scale, causal, stream)
    _check(st, "fa_varlen_paged_fwd")
    return out, lse


def attention_qkvpacked(qkv, scale=None, causal=False, out=None, lse=None, stream=None):
    """Packed QKV forward.  qkv: [B, N, 3, H, d] bf16.  Returns (O [B, N, H, d],
    LSE [B, H, N])."""
    import torch

    _req(qkv, "qkv", torch.bfloat16)
    B, N, three, H, d = qkv.shape
    if three != 3:
        raise ValueError("qkv must be [B, N, 3, H, d]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty((B, N, H, d), dtype=qkv.dtype, device=qkv.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=qkv.device) if lse is None else lse
    _check(fa_qkvpacked_fwd(qkv, out, lse, B, H, N, d, scale, causal, stream), "fa_qkvpacked_fwd")
    return out, lse


def attention_kvpacked(q, kv, scale=None, causal=False, out=None, lse=None, stream=None):
    """Packed KV forward.  q: [B, N, H, d], kv: [B, N, 2, Hkv, d] bf16."""
    import torch

    _req(q, "q", torch.bfloat16)
    _req(kv, "kv", torch.bfloat16)
    B, N, H, d = q.shape
    Hkv = kv.shape[3]
    if kv.shape != (B, N, 2, Hkv, d):
        raise ValueError("kv must be [B, N, 2, Hkv, d] matching q")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(fa_kvpacked_fwd(q, kv, out, lse, B, H, Hkv, N, d, scale, causal, stream), "fa_kvpacked_fwd")
    return out, lse


def attention_backward(q, k, v, o, lse, dout, scale=None, causal=False, workspace=None, stream=None):
    """Dense backward.  q, o, dout: [B, N, H, d]; k, v: [B, N, Hkv, d] bf16;
    lse: [B, H, N] fp32 from the forward.  Returns (dq, dk, dv) bf16."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _req(t, name, torch.bfloat16)
    _req(lse, "lse", torch.float32)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shapes: q, o, dout [B, N, H, d]; k, v [B, N, Hkv, d]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_bytes(B, B * N, H)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace.numel() * workspace.element_size(), B, H,
                Hkv, N, d, scale, causal, stream)
    _check(st, "fa_bwd")
    return dq, dk, dv


def attention_varlen_backward(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                              scale=None, causal=False, workspace=None, stream=None):
    """Varlen backward.  q, o, dout: [total_q, H, d]; k, v: [total_k, Hkv, d]
    bf16; lse: [H, total_q] fp32.  Returns (dq, dk, dv) bf16."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _req(t, name, torch.bfloat16)
    _req(lse, "lse", torch.float32)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _req(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    num_seqs = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_bytes(num_seqs, total_q, H)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = fa_varlen_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace.numel() * workspace.element_size(),
                       cu_seqlens_q, cu_seqlens_k, num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d,
                       scale, causal, stream)
    _check(st, "fa_varlen_bwd")
    return dq, dk, dv
