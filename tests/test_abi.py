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


def test_host_validation_of_tail_status_and_ablation_calls(lib):
    """Argument errors of the remaining entry points, each caught on the host before any
    CUDA call. The stand-in device address A is never dereferenced: every case below
    returns from the argument checks (the first check that can pass is never the last)."""
    L = lib
    so = L.load_library()
    A = 1 << 20                                    # 256-byte aligned stand-in address
    INV, TOO_SMALL, UNSUP, OK = (L.LOCKS_ERR_INVALID_ARG, L.LOCKS_ERR_WORKSPACE_TOO_SMALL,
                                 L.LOCKS_ERR_UNSUPPORTED, L.LOCKS_OK)
    dims = L.make_dims(1, 8, 2, 64, 64)
    empty = L.make_dims(0, 8, 2, 64, 64)
    big = 1 << 30

    # locks_select_attend_tail(dims, q, k, v, table, scores, partials, seq, tail, budget,
    #                          selected, n_selected, out, lse, workspace, bytes, stream)
    def sat(d, q=A, partials=None, budget=64, ws=None, nws=0):
        return so.locks_select_attend_tail(ctypes.byref(d), q, A, A, A, A, partials, A, A, budget, A, A, A, None,
                                           ws, nws, None)

    assert sat(dims, budget=-1) == INV
    assert sat(empty) == OK
    assert so.locks_select_attend_tail(ctypes.byref(dims), None, None, None, None, None, None, None, None, 64,
                                       None, None, None, None, None, 0, None) == INV
    assert sat(dims, q=A + 4) == INV                # q: 8-byte aligned at least
    assert sat(dims, partials=A + 8) == INV         # partials: 16-byte aligned
    assert sat(dims, ws=A + 16, nws=big) == INV     # workspace: 256-byte aligned
    assert sat(dims, ws=A, nws=100) == TOO_SMALL

    # locks_decode_step_tail(dims, q, k, v, summaries, table, seq, tail, budget, out, lse,
    #                        scores, selected, n_selected, workspace, bytes, stream)
    need = L.locks_workspace_size(dims, 64)
    good = L.locks_summaries_t(A, A, A, A)

    def dst(d, q=A, summ=None, budget=64, ws=A, nws=need):
        return so.locks_decode_step_tail(ctypes.byref(d), q, A, A, summ if summ is not None else good, A, A, A,
                                         budget, A, None, None, None, None, ws, nws, None)

    assert dst(dims, budget=-1) == INV
    assert dst(dims, ws=None, nws=0) == TOO_SMALL
    assert dst(dims, nws=need - 1) == TOO_SMALL
    assert dst(dims, ws=A + 64) == INV
    assert dst(empty, nws=L.locks_workspace_size(empty, 64)) == OK
    assert dst(dims, q=None) == INV
    assert dst(dims, q=A + 8) == INV                # q: 16-byte aligned for the fused step
    assert dst(dims, summ=L.locks_summaries_t(None, None, None, None)) == INV
    assert dst(dims, summ=L.locks_summaries_t(A, A, A, A + 4)) == INV      # scales: 8-byte aligned
    assert dst(dims, summ=L.locks_summaries_t(A + 8, A, A, A)) == INV      # mu: 16-byte aligned

    # device status word and the bounded-wait self test
    st = ctypes.c_int32(0)
    assert so.locks_get_device_status(None, ctypes.byref(st), None) == INV
    assert so.locks_get_device_status(A, None, None) == INV
    assert so.locks_clear_device_status(None, None) == INV
    assert so.locks_selftest_bounded_wait(None, 0, 0, None) == INV
    assert so.locks_selftest_bounded_wait(A + 16, big, 0, None) == INV
    assert so.locks_selftest_bounded_wait(A, 100, 0, None) == TOO_SMALL

    # ablation calls: the checks that come before the device query
    n = ctypes.c_size_t(0)
    assert so.locks_ablation_workspace_size(None, ctypes.byref(n)) == INV
    assert so.locks_ablation_workspace_size(ctypes.byref(dims), None) == INV
    bad = L.make_dims(1, 8, 2, 64, 64)
    bad.page_size = 32
    assert so.locks_exact_scores(ctypes.byref(bad), A, A, A, A, A, None, 0, None) == UNSUP
    assert so.locks_exact_scores(ctypes.byref(dims), A, None, A, A, A, None, 0, None) == INV
    assert so.locks_exact_scores(ctypes.byref(dims), A, A + 2, A, A, A, None, 0, None) == INV
    huge = L.make_dims(1, 8, 2, 64 * 65536, 64)     # more page blocks than one grid dimension holds
    assert so.locks_exact_scores(ctypes.byref(huge), A, A, A, A, A, None, 0, None) == UNSUP
    assert so.locks_variant_scores(ctypes.byref(dims), A, A, None, A, 8, 8, 4, 8, A, None, 0, None) == INV
    assert so.locks_shared_basis(ctypes.byref(dims), A, A, None, 8, A, None, None, 0, None) == INV
    assert so.locks_shared_scores(ctypes.byref(dims), A, None, A, A, A, 8, A, None, 0, None) == INV
