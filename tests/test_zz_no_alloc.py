"""The workspace-free decode step, for callers that cannot allocate device memory.

Engines that keep all of HBM for their own KV pool, or that cannot afford the
device synchronisation cudaMalloc may cause inside a decode loop, call
locks_decode_step_noalloc, whose scratch is a fixed 36 MiB array inside the
library. This file is collected last on purpose: if it fails, a run that stops
at the first failure has already run every other test. It calls the entry
point through the C ABI and checks that two calls in a row each reproduce the
regular locks_decode_step output exactly (both run the same two kernels on the
same inputs), at an ordinary size and at the largest table that still fits the
array, and that one size step beyond it is rejected.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 36 << 20


def _noalloc_fn():
    from sparse_kv_page_gb300 import build as b
    b.build()
    so = ctypes.CDLL(b.LIB_PATH)
    fn = so.locks_decode_step_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(L.locks_dims_t), P, P, P, L.locks_summaries_t, P, P, ctypes.c_int32, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _largest_fitting_pages(hq, hkv, budget):
    """The largest max_pages_per_seq (batch 1) whose workspace fits the array, and the
    next size up (which does not)."""
    def need(m):
        return L.locks_workspace_size(L.make_dims(1, hq, hkv, m, 1), budget)
    lo, hi = 1, 1 << 22
    assert need(lo) <= SCRATCH_BYTES < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if need(mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo, hi


def _run_pair(fn, pages_alloc, max_pages):
    """Builds a seeded problem of `pages_alloc` summarised pages per sequence inside a page
    table of width `max_pages`; returns (reference out, lse) from locks_decode_step and the
    two no-alloc calls' (out, lse)."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS["llama8b_128k"].scaled(pages=pages_alloc)
    inp = synth.make_decode_inputs(w)

    def up(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    table_np = np.zeros((w.batch, max_pages), np.int32)
    table_np[:, :w.pages] = inp.page_table
    q, kc, vc = up(inp.q), up(inp.k_cache), up(inp.v_cache)
    table, seq = up(table_np), up(inp.seq_pages)
    dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, max_pages, w.num_phys_pages)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, dev)
    ids = torch.arange(w.num_phys_pages, dtype=torch.int32, device=dev)
    L.locks_build_summaries(dims, kc, ids, w.num_phys_pages, summ)
    budget = 2048

    ws = L.alloc_workspace(dims, budget, dev)
    ref_out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=dev)
    ref_lse = torch.zeros((w.batch, w.num_q_heads), device=dev)
    L.locks_decode_step(dims, q, kc, vc, summ, table, seq, budget, ref_out, ws, lse=ref_lse)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == L.LOCKS_OK

    stream = torch.cuda.current_stream().cuda_stream
    got = []
    for _ in range(2):
        out = torch.full((w.batch, w.num_q_heads, 128), -1, dtype=torch.int16, device=dev)
        lse = torch.full((w.batch, w.num_q_heads), float("nan"), device=dev)
        rc = fn(ctypes.byref(dims), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), summ.c(), table.data_ptr(),
                seq.data_ptr(), budget, out.data_ptr(), lse.data_ptr(), stream)
        assert rc == L.LOCKS_OK, L.locks_status_string(rc)
        torch.cuda.synchronize()
        got.append((out.cpu().numpy(), lse.cpu().numpy()))
    return (ref_out.cpu().numpy(), ref_lse.cpu().numpy()), got


def test_noalloc_decode_step_equals_decode_step_twice():
    fn = _noalloc_fn()
    (ref_out, ref_lse), got = _run_pair(fn, 700, 700)
    for out, lse in got:
        assert np.array_equal(out, ref_out)
        assert np.array_equal(lse, ref_lse)


def test_noalloc_at_the_largest_fitting_table():
    """A page table just inside the array (its score table and partials fill ~36 MiB;
    300 pages summarised) runs and equals locks_decode_step; one size step more is
    rejected before anything is launched."""
    fn = _noalloc_fn()
    fit, over = _largest_fitting_pages(32, 8, 2048)
    need_fit = L.locks_workspace_size(L.make_dims(1, 32, 8, fit, 1), 2048)
    assert SCRATCH_BYTES - 512 <= need_fit <= SCRATCH_BYTES
    (ref_out, ref_lse), got = _run_pair(fn, 300, fit)
    for out, lse in got:
        assert np.array_equal(out, ref_out)
        assert np.array_equal(lse, ref_lse)
    dims = L.make_dims(1, 32, 8, over, 300)
    rc = fn(ctypes.byref(dims), None, None, None, L.locks_summaries_t(None, None, None, None), None, None, 2048,
            None, None, None)
    assert rc == L.LOCKS_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_size_limit_at_1m_context():
    """At 32 query heads and 1M tokens batch 4 fits the array (the 4 x 1M GLM-shaped
    workload included) and batch 5 is rejected before anything is launched."""
    fn = _noalloc_fn()
    for hkv, budget in ((8, 2048), (2, 512)):
        assert L.locks_workspace_size(L.make_dims(4, 32, hkv, 65536, 4 * 65536), budget) <= SCRATCH_BYTES
        dims = L.make_dims(5, 32, hkv, 65536, 5 * 65536)
        assert L.locks_workspace_size(dims, budget) > SCRATCH_BYTES
        rc = fn(ctypes.byref(dims), None, None, None, L.locks_summaries_t(None, None, None, None), None, None,
                budget, None, None, None)
        assert rc == L.LOCKS_ERR_WORKSPACE_TOO_SMALL
