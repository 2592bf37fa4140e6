"""Python binding of the LOCKS C ABI (include/locks.h).

Argument marshalling only: every function below calls the entry point of the
same name in ``liblocks_gb300.so`` with raw device pointers taken from torch
tensors, on torch's current CUDA stream unless a stream is given. Nothing here
computes any part of the method, and there is no fallback: if the library is
missing or a call fails, an exception is raised.

A decode step over a paged cache (bf16 bits held in int16 tensors)::

    dims = make_dims(B, Hq, Hkv, max_pages, num_phys)
    summ = Summaries.empty(num_phys, Hkv)                  # resident summaries
    locks_build_summaries(dims, k_cache, page_ids, n, summ)  # when pages fill
    ws = alloc_workspace(dims, budget_tokens)
    out = torch.empty((B, Hq, 128), dtype=torch.int16, device="cuda")
    locks_decode_step(dims, q, k_cache, v_cache, summ, page_table, seq_pages,
                      budget_tokens, out, ws)               # graph-capturable
    assert locks_get_device_status(ws) == LOCKS_OK

q is fp32 [B][Hq][128]; k_cache / v_cache are [num_phys][Hkv][16][128];
page_table int32 [B][max_pages]; seq_pages int32 [B] (full, summarised pages);
out receives bf16 bits [B][Hq][128].
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

from . import build as _build

PAGE = 16
D_HEAD = 128
RANK = 8

_STATUS = {
    0: "LOCKS_OK", -1: "LOCKS_ERR_INVALID_ARG", -2: "LOCKS_ERR_UNSUPPORTED",
    -3: "LOCKS_ERR_WORKSPACE_TOO_SMALL", -4: "LOCKS_ERR_CUDA", -5: "LOCKS_ERR_TIMEOUT",
    -6: "LOCKS_ERR_BAD_INDEX",
}
LOCKS_OK, LOCKS_ERR_INVALID_ARG, LOCKS_ERR_UNSUPPORTED = 0, -1, -2
LOCKS_ERR_WORKSPACE_TOO_SMALL, LOCKS_ERR_CUDA, LOCKS_ERR_TIMEOUT, LOCKS_ERR_BAD_INDEX = -3, -4, -5, -6


class LocksError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({_STATUS.get(status, 'unknown')})")
        self.status = status


class locks_dims_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_phys_pages", ctypes.c_int32)]


class locks_summaries_t(ctypes.Structure):
    _fields_ = [("mu", ctypes.c_void_p), ("basis", ctypes.c_void_p), ("coef", ctypes.c_void_p),
                ("scales", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the in-tree CUDA library; raise if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"LOCKS CUDA library not built: {path} (run __graft_entry__.build())")
            _build.build()
        lib = ctypes.CDLL(path)
        P, S, I32, U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64
        D = ctypes.POINTER(locks_dims_t)
        SUM = locks_summaries_t
        sig = {
            "locks_version": ([], ctypes.c_int),
            "locks_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "locks_k_cap": ([D, I32, ctypes.POINTER(I32)], ctypes.c_int),
            "locks_workspace_size": ([D, I32, ctypes.POINTER(S)], ctypes.c_int),
            "locks_lse_partials_size": ([D, ctypes.POINTER(S)], ctypes.c_int),
            "locks_build_summaries": ([D, P, P, I32, SUM, P, S, P], ctypes.c_int),
            "locks_score_pages": ([D, P, SUM, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_select_pages": ([D, P, P, P, I32, P, P, P, P, S, P], ctypes.c_int),
            "locks_sparse_attention": ([D, P, P, P, P, P, P, I32, P, P, P, S, P], ctypes.c_int),
            "locks_select_attend": ([D, P, P, P, P, P, P, P, I32, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_decode_step": ([D, P, P, P, SUM, P, P, I32, P, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_select_attend_tail": ([D, P, P, P, P, P, P, P, P, I32, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_decode_step_tail": ([D, P, P, P, SUM, P, P, P, I32, P, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_decode_step_noalloc": ([D, P, P, P, SUM, P, P, I32, P, P, P], ctypes.c_int),
            "locks_get_device_status": ([P, ctypes.POINTER(I32), P], ctypes.c_int),
            "locks_clear_device_status": ([P, P], ctypes.c_int),
            "locks_set_wait_limit_ns": ([U64], ctypes.c_int),
            "locks_set_select_cluster": ([ctypes.c_int32], ctypes.c_int),
            "locks_selftest_bounded_wait": ([P, S, U64, P], ctypes.c_int),
            "locks_ablation_workspace_size": ([D, ctypes.POINTER(S)], ctypes.c_int),
            "locks_exact_scores": ([D, P, P, P, P, P, P, S, P], ctypes.c_int),
            "locks_variant_scores": ([D, P, P, P, P, I32, I32, I32, I32, P, P, S, P], ctypes.c_int),
            "locks_shared_basis": ([D, P, P, P, I32, P, P, P, S, P], ctypes.c_int),
            "locks_shared_scores": ([D, P, P, P, P, P, I32, P, P, S, P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise LocksError(fn, status)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("LOCKS buffers must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------ dims, buffers

def make_dims(batch: int, num_q_heads: int, num_kv_heads: int, max_pages_per_seq: int,
              num_phys_pages: int) -> locks_dims_t:
    return locks_dims_t(batch, num_q_heads, num_kv_heads, D_HEAD, PAGE, RANK, max_pages_per_seq, num_phys_pages)


@dataclasses.dataclass
class Summaries:
    """Device summary arrays (torch-owned) in the library's layout."""

    mu: torch.Tensor       # int8  [num_phys][Hkv][128]
    basis: torch.Tensor    # uint8 [num_phys][Hkv][512]
    coef: torch.Tensor     # int8  [num_phys][Hkv][128]
    scales: torch.Tensor   # int16 (fp16 bits) [num_phys][Hkv][4]

    @staticmethod
    def empty(num_phys: int, num_kv_heads: int, device="cuda") -> "Summaries":
        return Summaries(torch.zeros((num_phys, num_kv_heads, 128), dtype=torch.int8, device=device),
                         torch.zeros((num_phys, num_kv_heads, 512), dtype=torch.uint8, device=device),
                         torch.zeros((num_phys, num_kv_heads, 128), dtype=torch.int8, device=device),
                         torch.zeros((num_phys, num_kv_heads, 4), dtype=torch.int16, device=device))

    def c(self) -> locks_summaries_t:
        return locks_summaries_t(_ptr(self.mu), _ptr(self.basis), _ptr(self.coef), _ptr(self.scales))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.mu, self.basis, self.coef, self.scales))


def locks_version() -> int:
    return load_library().locks_version()


def locks_status_string(status: int) -> str:
    return load_library().locks_status_string(status).decode()


def locks_k_cap(dims: locks_dims_t, budget_tokens: int) -> int:
    out = ctypes.c_int32(0)
    _check("locks_k_cap", load_library().locks_k_cap(ctypes.byref(dims), budget_tokens, ctypes.byref(out)))
    return out.value


def locks_workspace_size(dims: locks_dims_t, budget_tokens: int) -> int:
    out = ctypes.c_size_t(0)
    _check("locks_workspace_size",
           load_library().locks_workspace_size(ctypes.byref(dims), budget_tokens, ctypes.byref(out)))
    return out.value


def alloc_workspace(dims: locks_dims_t, budget_tokens: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace of locks_workspace_size bytes (torch allocations are 256-byte aligned)."""
    n = locks_workspace_size(dims, budget_tokens)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def _ws(workspace: Optional[torch.Tensor]):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


# ------------------------------------------------------------ entry points

def locks_build_summaries(dims, k_cache, phys_page_ids, n_pages, summaries: Summaries, workspace=None,
                          stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_build_summaries", load_library().locks_build_summaries(
        ctypes.byref(dims), _ptr(k_cache), _ptr(phys_page_ids), int(n_pages), summaries.c(), ws, nws,
        _stream(stream)))


def locks_lse_partials_size(dims: locks_dims_t) -> int:
    n = ctypes.c_size_t(0)
    _check("locks_lse_partials_size", load_library().locks_lse_partials_size(ctypes.byref(dims), ctypes.byref(n)))
    return int(n.value)


def lse_partials_shape(dims: locks_dims_t):
    """Shape of an fp32 tensor holding the optional LSE-partials buffer."""
    return (locks_lse_partials_size(dims) // 4,)


def locks_score_pages(dims, q, summaries: Summaries, page_table, seq_pages, scores, workspace=None,
                      stream=None, lse_partials=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_score_pages", load_library().locks_score_pages(
        ctypes.byref(dims), _ptr(q), summaries.c(), _ptr(page_table), _ptr(seq_pages), _ptr(scores),
        _ptr(lse_partials), ws, nws, _stream(stream)))


def locks_select_pages(dims, scores, seq_pages, budget_tokens, selected, n_selected, sel_keys=None,
                       workspace=None, stream=None, lse_partials=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_select_pages", load_library().locks_select_pages(
        ctypes.byref(dims), _ptr(scores), _ptr(lse_partials), _ptr(seq_pages), int(budget_tokens), _ptr(selected),
        _ptr(n_selected), _ptr(sel_keys), ws, nws, _stream(stream)))


def locks_sparse_attention(dims, q, k_cache, v_cache, page_table, selected, n_selected, k_cap, out, lse=None,
                           workspace=None, stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_sparse_attention", load_library().locks_sparse_attention(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(selected),
        _ptr(n_selected), int(k_cap), _ptr(out), _ptr(lse), ws, nws, _stream(stream)))


def locks_select_attend(dims, q, k_cache, v_cache, page_table, scores, seq_pages, budget_tokens, selected,
                        n_selected, out, lse=None, workspace=None, stream=None, lse_partials=None,
                        tail_tokens=None) -> None:
    """tail_tokens (int32 [batch], optional): tokens of each sequence's unfilled page
    (logical page seq_pages[b]), attended whole (locks_select_attend_tail)."""
    ws, nws = _ws(workspace)
    if tail_tokens is None:
        _check("locks_select_attend", load_library().locks_select_attend(
            ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(scores),
            _ptr(lse_partials), _ptr(seq_pages), int(budget_tokens), _ptr(selected), _ptr(n_selected), _ptr(out),
            _ptr(lse), ws, nws, _stream(stream)))
    else:
        _check("locks_select_attend_tail", load_library().locks_select_attend_tail(
            ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(scores),
            _ptr(lse_partials), _ptr(seq_pages), _ptr(tail_tokens), int(budget_tokens), _ptr(selected),
            _ptr(n_selected), _ptr(out), _ptr(lse), ws, nws, _stream(stream)))


def locks_decode_step(dims, q, k_cache, v_cache, summaries: Summaries, page_table, seq_pages, budget_tokens, out,
                      workspace, lse=None, scores=None, selected=None, n_selected=None, stream=None,
                      tail_tokens=None) -> None:
    """tail_tokens (int32 [batch], optional): tokens of each sequence's unfilled page
    (logical page seq_pages[b]), attended whole (locks_decode_step_tail)."""
    ws, nws = _ws(workspace)
    if tail_tokens is None:
        _check("locks_decode_step", load_library().locks_decode_step(
            ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), summaries.c(), _ptr(page_table),
            _ptr(seq_pages), int(budget_tokens), _ptr(out), _ptr(lse), _ptr(scores), _ptr(selected),
            _ptr(n_selected), ws, nws, _stream(stream)))
    else:
        _check("locks_decode_step_tail", load_library().locks_decode_step_tail(
            ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), summaries.c(), _ptr(page_table),
            _ptr(seq_pages), _ptr(tail_tokens), int(budget_tokens), _ptr(out), _ptr(lse), _ptr(scores),
            _ptr(selected), _ptr(n_selected), ws, nws, _stream(stream)))


def locks_decode_step_noalloc(dims, q, k_cache, v_cache, summaries: Summaries, page_table, seq_pages,
                              budget_tokens, out, lse=None, stream=None) -> None:
    """locks_decode_step with the library's fixed scratch array in place of a workspace, for
    callers that cannot allocate device memory (see include/locks.h)."""
    _check("locks_decode_step_noalloc", load_library().locks_decode_step_noalloc(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), summaries.c(), _ptr(page_table),
        _ptr(seq_pages), int(budget_tokens), _ptr(out), _ptr(lse), _stream(stream)))


def locks_get_device_status(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("locks_get_device_status",
           load_library().locks_get_device_status(_ptr(workspace), ctypes.byref(out), _stream(stream)))
    return out.value


def locks_clear_device_status(workspace, stream=None) -> None:
    _check("locks_clear_device_status", load_library().locks_clear_device_status(_ptr(workspace), _stream(stream)))


def locks_set_wait_limit_ns(ns: int) -> None:
    _check("locks_set_wait_limit_ns", load_library().locks_set_wait_limit_ns(int(ns)))


def locks_set_select_cluster(cluster: int) -> None:
    """Pins the cluster size (8, 12 or 16 CTAs) of launches that select pages; 0 = automatic."""
    _check("locks_set_select_cluster", load_library().locks_set_select_cluster(int(cluster)))


def locks_selftest_bounded_wait(workspace, limit_ns: int, stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_selftest_bounded_wait",
           load_library().locks_selftest_bounded_wait(ws, nws, int(limit_ns), _stream(stream)))


# --------------------------------------------------------------- ablations

def locks_ablation_workspace_size(dims: locks_dims_t) -> int:
    out = ctypes.c_size_t(0)
    _check("locks_ablation_workspace_size", load_library().locks_ablation_workspace_size(ctypes.byref(dims),
                                                                                       ctypes.byref(out)))
    return out.value


def alloc_ablation_workspace(dims: locks_dims_t, device="cuda") -> torch.Tensor:
    """A zeroed workspace of locks_ablation_workspace_size bytes."""
    return torch.zeros(max(locks_ablation_workspace_size(dims), 256), dtype=torch.uint8, device=device)


def locks_exact_scores(dims, q, k_cache, page_table, seq_pages, scores, workspace=None, stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_exact_scores", load_library().locks_exact_scores(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(page_table), _ptr(seq_pages), _ptr(scores), ws, nws,
        _stream(stream)))


def locks_variant_scores(dims, q, k_cache, page_table, seq_pages, rank, bits_mu, bits_v, bits_c, scores,
                         workspace=None, stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_variant_scores", load_library().locks_variant_scores(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(page_table), _ptr(seq_pages), int(rank), int(bits_mu),
        int(bits_v), int(bits_c), _ptr(scores), ws, nws, _stream(stream)))


def locks_shared_basis(dims, k_cache, page_table, seq_pages, rank, basis, workspace, eigvals=None,
                       stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_shared_basis", load_library().locks_shared_basis(
        ctypes.byref(dims), _ptr(k_cache), _ptr(page_table), _ptr(seq_pages), int(rank), _ptr(basis),
        _ptr(eigvals), ws, nws, _stream(stream)))


def locks_shared_scores(dims, q, k_cache, page_table, seq_pages, basis, rank, scores, workspace,
                        stream=None) -> None:
    ws, nws = _ws(workspace)
    _check("locks_shared_scores", load_library().locks_shared_scores(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(page_table), _ptr(seq_pages), _ptr(basis), int(rank),
        _ptr(scores), ws, nws, _stream(stream)))
