"""The C-ABI library on the CPU: it builds, loads, exports every function
include/fa.h declares, and refuses bad arguments before touching a GPU."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_fwd_gb300 import _build
    import exact_tiled_attention_fwd_gb300 as F

    _build.build()
    F.load()
    return F


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("fa_fwd", "fa_varlen_fwd", "fa_paged_fwd", "fa_paged_workspace_size", "fa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    handle = lib.load()
    missing = [n for n in declared_functions() if not hasattr(handle, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(lib.EXPORTS)


def test_python_binding_has_the_same_names(lib):
    for n in declared_functions():
        assert callable(getattr(lib, n)), n


def test_status_strings(lib):
    for code in range(6):
        assert lib.status_string(code).startswith("FA_")
    assert "unknown" in lib.status_string(99)
    assert lib.fa_abi_version() == 4


def test_validation_without_gpu(lib):
    """Every check below fails before any CUDA call, so it runs on a CPU machine."""
    A = 1 << 20  # a fake, 16-byte aligned address
    S = 0
    assert lib.fa_fwd(0, A, A, A, None, 1, 1, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A + 8, A, A, A, None, 1, 1, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, A + 4, 1, 1, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 0, 1, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 1, 1, 1, 0, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 1, 6, 4, 8, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 1, 1, 1, 8, 128, 0.0, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 1, 1, 1, 8, 128, float("nan"), 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_fwd(A, A, A, A, None, 1, 1, 1, 8, 96, 0.1, 0, S) == lib.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd(A, A, A, A, None, 1, 1, 1, 8, 80, 0.1, 0, S) == lib.FA_ERR_UNSUPPORTED
    assert lib.fa_varlen_fwd(A, A, A, A, None, 0, A, 1, 8, 8, 8, 8, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_varlen_fwd(A, A, A, A, None, A + 2, A, 1, 8, 8, 8, 8, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_varlen_fwd(A, A, A, A, None, A, A, 0, 8, 8, 8, 8, 1, 1, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    ws = lib.fa_paged_workspace_size(2, 4, 128, 100)
    assert ws > 0
    # page size not in {16, 32, 64, 128}, too-small workspace, too few pages
    # per sequence
    for ps in (8, 48, 256):
        assert lib.fa_paged_fwd(A, A, A, A, A, A, None, 2, 4, 4, 128, ps, 10, 8, 100, 0.1, 1, A, ws, S) == \
            lib.FA_ERR_UNSUPPORTED
        assert lib.fa_paged_fwd_noalloc(A, A, A, A, A, A, None, 2, 4, 4, 128, ps, 10, 8, 100, 0.1, 1, S) == \
            lib.FA_ERR_UNSUPPORTED
    assert lib.fa_paged_fwd(A, A, A, A, A, A, None, 2, 4, 4, 128, 16, 10, 8, 100, 0.1, 1, A, ws - 1, S) == \
        lib.FA_ERR_INVALID
    assert lib.fa_paged_fwd(A, A, A, A, A, A, None, 2, 4, 4, 128, 16, 10, 6, 100, 0.1, 1, A, ws, S) == \
        lib.FA_ERR_INVALID
    assert lib.fa_paged_fwd(A, A, A, 0, A, A, None, 2, 4, 4, 128, 16, 10, 8, 100, 0.1, 1, A, ws, S) == \
        lib.FA_ERR_INVALID
    assert lib.fa_selftest_wait_timeout(0, S) == lib.FA_ERR_INVALID
    # paged varlen prefill: null table, unaligned cu_seqlens, page size, too
    # few pages per sequence for max_seqlen_k, d
    vp = lib.fa_varlen_paged_fwd
    assert vp(A, A, A, A, None, A, A, 0, 2, 64, 200, 64, 4, 2, 128, 16, 30, 13, 0.1, 1, S) == lib.FA_ERR_INVALID
    assert vp(A, A, A, A, None, A + 2, A, A, 2, 64, 200, 64, 4, 2, 128, 16, 30, 13, 0.1, 1, S) == lib.FA_ERR_INVALID
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 200, 64, 4, 2, 128, 48, 30, 13, 0.1, 1, S) == lib.FA_ERR_UNSUPPORTED
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 200, 64, 4, 2, 128, 256, 30, 13, 0.1, 1, S) == lib.FA_ERR_UNSUPPORTED
    # 32-token pages: 7 pages per sequence hold only 224 < 250 keys
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 250, 64, 4, 2, 128, 32, 30, 7, 0.1, 1, S) == lib.FA_ERR_INVALID
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 200, 64, 4, 2, 128, 16, 30, 12, 0.1, 1, S) == lib.FA_ERR_INVALID
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 200, 64, 4, 3, 128, 16, 30, 13, 0.1, 1, S) == lib.FA_ERR_INVALID
    assert vp(A, A, A, A, None, A, A, A, 2, 64, 200, 64, 4, 2, 96, 16, 30, 13, 0.1, 1, S) == lib.FA_ERR_UNSUPPORTED
    # packed layouts: null tensors, d, GQA with packed QKV is not expressible
    assert lib.fa_qkvpacked_fwd(0, A, None, 1, 4, 8, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_qkvpacked_fwd(A, A, None, 1, 4, 8, 96, 0.1, 0, S) == lib.FA_ERR_UNSUPPORTED
    assert lib.fa_qkvpacked_fwd(A + 8, A, None, 1, 4, 8, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_kvpacked_fwd(A, 0, A, None, 1, 4, 2, 8, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_kvpacked_fwd(A, A, A, None, 1, 4, 3, 8, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_varlen_qkvpacked_fwd(A, A, None, 0, 1, 8, 8, 4, 128, 0.1, 0, S) == lib.FA_ERR_INVALID
    assert lib.fa_varlen_kvpacked_fwd(A, A, A, None, A, A, 1, 8, 8, 8, 8, 4, 2, 64, 0.0, 0, S) == lib.FA_ERR_INVALID
    # store_kvcache: null slot map, unaligned cache, negative token count, d
    sk = lib.fa_store_kvcache
    assert sk(A, A, A, A, 0, 8, 2, 128, 16, 4, S) == lib.FA_ERR_INVALID
    assert sk(A, A, A + 8, A, A, 8, 2, 128, 16, 4, S) == lib.FA_ERR_INVALID
    assert sk(A, A, A, A, A, -1, 2, 128, 16, 4, S) == lib.FA_ERR_INVALID
    assert sk(A, A, A, A, A, 8, 2, 96, 16, 4, S) == lib.FA_ERR_UNSUPPORTED


def test_workspace_size_monotone(lib):
    assert lib.fa_paged_workspace_size(0, 4, 128, 10) == 0
    assert lib.fa_paged_workspace_size(1, 4, 96, 10) == 0
    a = lib.fa_paged_workspace_size(64, 32, 128, 16384)
    b = lib.fa_paged_workspace_size(64, 32, 128, 16385)
    assert 0 < a <= b and a % 256 == 0
