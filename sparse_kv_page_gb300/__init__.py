"""LOCKS decode step for GB300 (sm_103a): a CUDA library behind a C ABI.

The compute lives in ``liblocks_gb300.so`` (``csrc/``, declared in
``include/locks.h``); ``locks`` is its ctypes binding. Build with
``sparse_kv_page_gb300.build.build()``.
"""

from .locks import (LocksError, Summaries, alloc_ablation_workspace, alloc_workspace, library_path, load_library,
                    locks_ablation_workspace_size, locks_build_summaries, locks_clear_device_status,
                    locks_decode_step, locks_decode_step_noalloc, locks_dims_t, locks_exact_scores,
                    locks_get_device_status, locks_k_cap, locks_lse_partials_size, locks_score_pages,
                    locks_select_attend, locks_select_pages, locks_selftest_bounded_wait, locks_set_select_cluster,
                    locks_set_wait_limit_ns,
                    locks_shared_basis, locks_shared_scores, locks_sparse_attention, locks_status_string,
                    locks_summaries_t, locks_variant_scores, locks_version, locks_workspace_size, make_dims)

__all__ = [
    "LocksError", "Summaries", "alloc_ablation_workspace", "alloc_workspace", "locks_ablation_workspace_size",
    "locks_exact_scores", "locks_shared_basis", "locks_shared_scores", "locks_variant_scores", "library_path", "load_library", "locks_build_summaries",
    "locks_clear_device_status", "locks_decode_step", "locks_decode_step_noalloc", "locks_dims_t", "locks_get_device_status", "locks_k_cap",
    "locks_score_pages", "locks_select_attend", "locks_select_pages", "locks_selftest_bounded_wait",
    "locks_set_select_cluster", "locks_set_wait_limit_ns", "locks_sparse_attention", "locks_status_string", "locks_summaries_t",
    "locks_lse_partials_size", "locks_version", "locks_workspace_size", "make_dims",
]
