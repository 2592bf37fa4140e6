"""The workspace-free decode step, for callers that cannot allocate device memory.

Engines that keep all of HBM for their own KV pool, or that cannot afford the
device synchronisation cudaMalloc may cause inside a decode loop, call
locks_decode_step_noalloc, whose scratch is a fixed array inside the library.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It calls the entry point
through the C ABI and checks that two calls in a row each reproduce the
regular locks_decode_step output (same tolerance as the other attention tests).
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

ATT_ABS = 2e-2


def _noalloc_fn():
    from sparse_kv_page_gb300 import build as b
    b.build()
    so = ctypes.CDLL(b.LIB_PATH)
    fn = so.locks_decode_step_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(L.locks_dims_t), P, P, P, L.locks_summaries_t, P, P, ctypes.c_int32, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_decode_step_matches_decode_step_twice():
    fn = _noalloc_fn()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS["llama8b_128k"].scaled(pages=700)
    inp = synth.make_decode_inputs(w)

    def up(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    q, kc, vc = up(inp.q), up(inp.k_cache), up(inp.v_cache)
    table, seq = up(inp.page_table), up(inp.seq_pages)
    dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, dev)
    ids = torch.arange(w.num_phys_pages, dtype=torch.int32, device=dev)
    L.locks_build_summaries(dims, kc, ids, w.num_phys_pages, summ)
    budget = 2048

    ws = L.alloc_workspace(dims, budget, dev)
    ref_out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=dev)
    ref_lse = torch.zeros((w.batch, w.num_q_heads), device=dev)
    L.locks_decode_step(dims, q, kc, vc, summ, table, seq, budget, ref_out, ws, lse=ref_lse)
    torch.cuda.synchronize()
    ref = synth.bf16_bits_to_f32(ref_out.cpu().numpy().view(np.uint16))

    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full((w.batch, w.num_q_heads, 128), -1, dtype=torch.int16, device=dev)
        lse = torch.full((w.batch, w.num_q_heads), float("nan"), device=dev)
        rc = fn(ctypes.byref(dims), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), summ.c(), table.data_ptr(),
                seq.data_ptr(), budget, out.data_ptr(), lse.data_ptr(), stream)
        assert rc == 0, L.locks_status_string(rc)
        torch.cuda.synchronize()
        got = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16))
        assert np.abs(got - ref).max() < ATT_ABS
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() < 1e-3


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    dims = L.make_dims(16, 32, 8, 65536, 16 * 65536)   # 16 x 32 x 65536 fp32 scores = 128 MiB > 36 MiB
    rc = fn(ctypes.byref(dims), None, None, None, L.locks_summaries_t(None, None, None, None), None, None, 2048,
            None, None, None)
    assert rc == L.LOCKS_ERR_WORKSPACE_TOO_SMALL
