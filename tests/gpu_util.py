"""Helpers for the GPU parity tests: upload numpy inputs, call the C ABI, compare.

Contains no part of the method: uploads, downloads and a decoder of the
documented summary byte layout (used only to check invariants of what the
CUDA builder writes; the oracle never sees CUDA output).
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import synth
from sparse_kv_page_gb300 import locks as L

DEV = torch.device("cuda:0")


def t(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def upload_summaries(mu, basis, coef, scales, num_phys: int, hkv: int) -> L.Summaries:
    return L.Summaries(t(np.asarray(mu, np.int8).reshape(num_phys, hkv, 128)),
                       t(np.asarray(basis, np.uint8).reshape(num_phys, hkv, 512)),
                       t(np.asarray(coef, np.int8).reshape(num_phys, hkv, 128)),
                       t(np.asarray(scales, np.uint16).reshape(num_phys, hkv, 4)))


def download_summaries(s: L.Summaries):
    return (s.mu.cpu().numpy(), s.basis.cpu().numpy(), s.coef.cpu().numpy(),
            s.scales.cpu().numpy().view(np.uint16))


def bf16_out(x: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f32(x.cpu().numpy().view(np.uint16)).astype(np.float64)


def cosine(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    na = np.linalg.norm(a, axis=-1)
    nb = np.linalg.norm(b, axis=-1)
    return (a * b).sum(-1) / np.maximum(na * nb, 1e-30)


# ---------------------------------------------------------- layout decoder
# From the summary layout in include/locks.h (tests use it to read what the
# CUDA builder wrote).

def _dim_parts(d):
    s, w = d // 16, d % 16
    return s, w // 8, (w % 8) // 2, w % 2


def decode_layout(mu, basis, coef, scales):
    """bytes of n units -> (mu_hat [n,128], v_hat [n,128,8], c_hat [n,16,8]) float64."""
    mu = np.asarray(mu, np.int8).reshape(-1, 128)
    basis = np.asarray(basis, np.uint8).reshape(-1, 512)
    coef = np.asarray(coef, np.int8).reshape(-1, 128)
    sc = np.asarray(scales, np.uint16).reshape(-1, 4).view(np.float16).astype(np.float64)
    mu_off = np.zeros(128, np.int64)
    vb = np.zeros((128, 8), np.int64)
    vn = np.zeros((128, 8), np.int64)
    for d in range(128):
        s, h, tt, e = _dim_parts(d)
        mu_off[d] = 32 * tt + 4 * s + 2 * h + e
        p = 2 * (s % 2) + h + 4 * e
        for r in range(8):
            vb[d, r] = 64 * r + 16 * tt + 4 * (s // 2) + p // 2
            vn[d, r] = p % 2
    c_off = np.zeros((16, 8), np.int64)
    for i in range(16):
        for r in range(8):
            c_off[i, r] = 4 * (4 * (i % 8) + r // 2) + 2 * (i // 8) + r % 2
    mu_hat = mu[:, mu_off].astype(np.float64) * sc[:, 0:1]
    byte = basis[:, vb]
    nib = np.where(vn[None] == 1, byte >> 4, byte & 0xF).astype(np.int64)
    nib = np.where(nib >= 8, nib - 16, nib)
    v_hat = nib.astype(np.float64) * sc[:, 1][:, None, None]
    c_hat = coef[:, c_off].astype(np.float64) * sc[:, 2][:, None, None]
    return mu_hat, v_hat, c_hat


@dataclasses.dataclass
class DeviceProblem:
    dims: L.locks_dims_t
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor
    seq_pages: torch.Tensor


def device_problem(q, k_cache, v_cache, page_table, seq_pages, num_phys: Optional[int] = None) -> DeviceProblem:
    B, Hq, _ = q.shape
    Hkv = k_cache.shape[1]
    maxp = page_table.shape[1]
    nphys = k_cache.shape[0] if num_phys is None else num_phys
    dims = L.make_dims(B, Hq, Hkv, maxp, nphys)
    return DeviceProblem(dims, t(np.asarray(q, np.float32)), t(k_cache), t(v_cache),
                         t(np.asarray(page_table, np.int32)), t(np.asarray(seq_pages, np.int32)))


def check_selection(sel_gpu, n_gpu, sel_orc, n_orc, keys_orc, seq_pages, tol=1e-3):
    """The boundary rule: same count k; every page in the symmetric difference has an
    oracle key within tol of the oracle's k-th largest key; output ascending."""
    B, Hkv, _ = sel_orc.shape
    for b in range(B):
        for h in range(Hkv):
            k = int(n_orc[b, h])
            assert int(n_gpu[b, h]) == k, (b, h, int(n_gpu[b, h]), k)
            g = sel_gpu[b, h, :k]
            o = sel_orc[b, h, :k]
            assert np.all(np.diff(g) > 0), "GPU selection not strictly ascending"
            assert np.all((g >= 0) & (g < seq_pages[b]))
            if k == 0:
                continue
            kk = keys_orc[b, h, :seq_pages[b]].copy()
            kk[np.isnan(kk)] = -np.inf
            thr = np.sort(kk)[::-1][k - 1]
            diff = np.setxor1d(g, o)
            for j in diff:
                assert abs(kk[j] - thr) <= tol or (np.isinf(kk[j]) and np.isinf(thr)), \
                    (b, h, int(j), float(kk[j]), float(thr))
