"""The C-ABI library: it loads, exports every declared entry point, and its host-side
argument checks return the documented status codes (no CUDA call is reached)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_page_gb300 import build as b
    b.build()
    from sparse_kv_page_gb300 import locks as L
    return L


def _declared():
    with open(os.path.join(ROOT, "include", "locks.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"LOCKS_API\s+(?:const\s+char\s*\*|int)\s+(locks_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 14
    so = ctypes.CDLL(lib.library_path())
    for n in names:
        assert hasattr(so, n), n


def test_no_oracle_in_product():
    """The product package never imports or links the oracle."""
    pkg = os.path.join(ROOT, "sparse_kv_page_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    txt = f.read()
                assert "import oracle" not in txt and "locks_oracle" not in txt, fn


def test_status_strings_and_sizes(lib):
    assert lib.locks_version() >= 10000
    assert lib.locks_status_string(0) == "ok"
    assert "timed out" in lib.locks_status_string(-5)
    dims = lib.make_dims(2, 32, 8, 1000, 2000)
    assert lib.locks_k_cap(dims, 2048) == 128
    assert lib.locks_k_cap(dims, 15) == 1
    assert lib.locks_k_cap(lib.make_dims(1, 1, 1, 10, 10), 2048) == 10
    ws = lib.locks_workspace_size(dims, 2048)
    need = 2 * 32 * 1000 * 4 + 2 * 32 * 256 * 2 * 8 + 2 * 8 * 128 * 4 + 2 * 8 * 4   # scores, partials, selection
    assert lib.locks_lse_partials_size(dims) == 2 * 32 * 256 * 2 * 8
    assert need <= ws <= need + 5 * 256


def test_host_validation_codes(lib):
    L = lib
    so = L.load_library()
    S = L.locks_summaries_t(None, None, None, None)
    bad = L.make_dims(1, 4, 1, 16, 16)
    bad.head_dim = 64
    assert so.locks_score_pages(ctypes.byref(bad), None, S, None, None, None, None, None, 0, None) == L.LOCKS_ERR_UNSUPPORTED
    bad = L.make_dims(1, 6, 3, 16, 16)       # 3 kv heads: not built
    assert so.locks_score_pages(ctypes.byref(bad), None, S, None, None, None, None, None, 0, None) == L.LOCKS_ERR_UNSUPPORTED
    bad = L.make_dims(1, 64, 2, 16, 16)      # group 32 > 16
    assert so.locks_score_pages(ctypes.byref(bad), None, S, None, None, None, None, None, 0, None) == L.LOCKS_ERR_UNSUPPORTED
    bad = L.make_dims(1, 6, 4, 16, 16)       # 6 % 4 != 0
    assert so.locks_score_pages(ctypes.byref(bad), None, S, None, None, None, None, None, 0, None) == L.LOCKS_ERR_INVALID_ARG
    ok = L.make_dims(1, 4, 1, 16, 16)
    assert so.locks_score_pages(ctypes.byref(ok), None, S, None, None, None, None, None, 0, None) == L.LOCKS_ERR_INVALID_ARG
    assert so.locks_select_pages(ctypes.byref(ok), None, None, None, -16, None, None, None, None, 0, None) == \
        L.LOCKS_ERR_INVALID_ARG
    assert so.locks_decode_step(ctypes.byref(ok), None, None, None, S, None, None, 256, None, None, None, None,
                                None, None, 0, None) == L.LOCKS_ERR_WORKSPACE_TOO_SMALL
    assert so.locks_sparse_attention(ctypes.byref(ok), None, None, None, None, None, None, 0, None, None, None, 0,
                                     None) == L.LOCKS_ERR_INVALID_ARG
    assert so.locks_select_attend(ctypes.byref(ok), None, None, None, None, None, None, None, 256, None, None, None,
                                  None, None, 0, None) == L.LOCKS_ERR_INVALID_ARG
    assert so.locks_k_cap(None, 16, None) == L.LOCKS_ERR_INVALID_ARG
    empty = L.make_dims(0, 4, 1, 16, 16)     # nothing to do
    assert so.locks_score_pages(ctypes.byref(empty), None, S, None, None, None, None, None, 0, None) == L.LOCKS_OK
    assert so.locks_build_summaries(ctypes.byref(ok), None, None, 0, S, None, 0, None) == L.LOCKS_OK
    assert so.locks_build_summaries(ctypes.byref(ok), None, None, -1, S, None, 0, None) == L.LOCKS_ERR_INVALID_ARG
    for cl in (1, 4, 10, 32, -8):            # only 0 (automatic), 8, 12 and 16 are accepted
        assert so.locks_set_select_cluster(cl) == L.LOCKS_ERR_INVALID_ARG
    for cl in (8, 12, 16, 0):
        assert so.locks_set_select_cluster(cl) == L.LOCKS_OK


def test_noalloc_rejects_oversized_problems_on_the_host(lib):
    """The workspace-free decode step refuses, before any CUDA call, a problem whose
    scratch exceeds its fixed 36 MiB array (batch 5 x 32 heads x 1M tokens needs 40.6 MiB)."""
    so = lib.load_library()
    fn = so.locks_decode_step_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(lib.locks_dims_t), P, P, P, lib.locks_summaries_t, P, P, ctypes.c_int32, P, P, P]
    fn.restype = ctypes.c_int
    S = lib.locks_summaries_t(None, None, None, None)
    for dims, budget in ((lib.make_dims(5, 32, 2, 65536, 5 * 65536), 512),
                         (lib.make_dims(5, 32, 8, 65536, 5 * 65536), 2048)):
        assert lib.locks_workspace_size(dims, budget) > (36 << 20)
        assert fn(ctypes.byref(dims), None, None, None, S, None, None, budget, None, None, None) == \
            lib.LOCKS_ERR_WORKSPACE_TOO_SMALL
    assert lib.locks_workspace_size(lib.make_dims(4, 32, 8, 65536, 4 * 65536), 2048) <= (36 << 20)
    assert lib.locks_workspace_size(lib.make_dims(4, 32, 2, 65536, 4 * 65536), 512) <= (36 << 20)
