"""Float64 CPU oracle of the LOCKS decode step.

TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers; the library's product path
never imports this package, and this package never imports the product.

The arithmetic lives in ``locks_oracle.c`` (plain C, float64, one unit at a
time); this module compiles it with gcc and marshals numpy arrays through
ctypes. Each function cites the LOCKS page passage it follows:

* build    - "How LOCKS works" / "Code" (wps.hkprog.org LOCKS post) and the
             gist.science summary, 2.1 (eigendecomposition of centred keys,
             int8 centroid, int4 rank-8 basis, int8 coefficients)
* score    - score formula of "How LOCKS works" / summary 2.2
* group    - summary 2.3 (mean of the estimated mass shares of a GQA group)
* select   - "Code": k = budget // 16 pages, indices sorted ascending
* attend   - "Code": scaled dot-product attention over the selected pages
* ablations - exact (read-all-keys) page scores (Korean gist.science summary,
             sections 1 and 3); rank / bit-width variants of the summary
             ("Caveats": int4 loses a few recall points, int2 collapses); a
             shared basis and its projected scores ("Why shared-basis sparse
             attention is structurally broken"; Proposition 1)

Parity unpinned: nothing here is unpinned; see tests/test_oracle_pins.py for
the checks that tie every function to the pages and to the mathematics.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "locks_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblocks_oracle.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

PAGE, D, R = 16, 128, 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (float64, no fast-math, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64, u16 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint16
            sig = {
                "lo_version": ([], i32),
                "lo_max_threads": ([], i32),
                "lo_set_threads": ([i32], None),
                "lo_bf16_to_f64": ([u16], f64),
                "lo_f16_to_f64": ([u16], f64),
                "lo_f64_to_f16": ([f64], u16),
                "lo_round_f16": ([f64], f64),
                "lo_jacobi_eig": ([i32, P, P, f64, i32], i32),
                "lo_build_unit_f64": ([P, i32, P, P, P, P], None),
                "lo_encode_unit": ([P, P, P, P, P, P, P], None),
                "lo_decode_unit": ([P, P, P, P, P, P, P], None),
                "lo_build_units": ([i64, P, P, P, P, P], None),
                "lo_score_unit": ([P, P, P, P, i32], f64),
                "lo_scores": ([i32, i32, i32, i32, P, P, P, P, P, P, P, P], None),
                "lo_scores_sampled": ([i32, i32, i32, i32, P, P, P, P, P, P, i64, P, P, P, P], None),
                "lo_group_keys": ([i32, i32, i32, i32, P, P, P, P], None),
                "lo_select": ([i32, i32, i32, P, P, i32, i32, P, P], None),
                "lo_attend": ([i32, i32, i32, i32, P, P, P, P, P, P, i32, P, P, P, P], None),
                "lo_exact_score_unit": ([P, P], f64),
                "lo_exact_scores": ([i32, i32, i32, i32, P, P, P, P, P], None),
                "lo_quant_dequant": ([P, i32, i32], None),
                "lo_variant_scores": ([i32, i32, i32, i32, P, P, P, P, i32, i32, i32, i32, P], None),
                "lo_shared_basis": ([i32, i32, i32, P, P, P, i32, P, P], None),
                "lo_shared_scores": ([i32, i32, i32, i32, P, P, P, P, P, i32, P], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _p(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return _load().lo_max_threads()


def set_threads(n: int) -> None:
    _load().lo_set_threads(int(n))


# ------------------------------------------------------------------ numbers

def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.lo_bf16_to_f64(int(x)) for x in b.ravel()]).reshape(b.shape)


def f16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.lo_f16_to_f64(int(x)) for x in b.ravel()]).reshape(b.shape)


def f64_to_f16(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.array([lib.lo_f64_to_f16(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


# ------------------------------------------------------------------- build

def jacobi_eig(a: np.ndarray, tol: float = 1e-14, max_sweeps: int = 100) -> Tuple[np.ndarray, np.ndarray, int]:
    """Cyclic Jacobi (Golub & Van Loan 8.5). Returns (eigenvalues, eigenvectors as columns, sweeps)."""
    n = a.shape[0]
    m = _c(a, np.float64).copy()
    v = np.zeros((n, n), dtype=np.float64)
    sweeps = _load().lo_jacobi_eig(n, _p(m), _p(v), tol, max_sweeps)
    return np.diag(m).copy(), v, sweeps


def build_unit_f64(k_bits: np.ndarray, rank: int = R):
    """Unquantised summary of one 16 x 128 bf16 key page: (mu, V [128][r], C [16][r], eigvals [16])."""
    k = _c(k_bits, np.uint16).reshape(PAGE, D)
    mu = np.zeros(D)
    basis = np.zeros((D, rank))
    coef = np.zeros((PAGE, rank))
    ev = np.zeros(PAGE)
    _load().lo_build_unit_f64(_p(k), rank, _p(mu), _p(basis), _p(coef), _p(ev))
    return mu, basis, coef, ev


def build_units(k_bits: np.ndarray):
    """Quantised summaries of n pages ([n][16][128] bf16) -> (mu, basis, coef, scales) byte arrays."""
    k = _c(k_bits, np.uint16).reshape(-1, PAGE, D)
    n = k.shape[0]
    mu = np.zeros((n, 128), np.int8)
    basis = np.zeros((n, 512), np.uint8)
    coef = np.zeros((n, 128), np.int8)
    scales = np.zeros((n, 4), np.uint16)
    _load().lo_build_units(n, _p(k), _p(mu), _p(basis), _p(coef), _p(scales))
    return mu, basis, coef, scales


def encode_unit(mu: np.ndarray, basis: np.ndarray, coef: np.ndarray):
    """Quantise and lay out one unit's float64 (mu [128], V [128][8], C [16][8])."""
    m, v, c = _c(mu, np.float64), _c(basis, np.float64), _c(coef, np.float64)
    om = np.zeros(128, np.int8)
    ob = np.zeros(512, np.uint8)
    oc = np.zeros(128, np.int8)
    osc = np.zeros(4, np.uint16)
    _load().lo_encode_unit(_p(m), _p(v), _p(c), _p(om), _p(ob), _p(oc), _p(osc))
    return om, ob, oc, osc


def decode_unit(mu: np.ndarray, basis: np.ndarray, coef: np.ndarray, scales: np.ndarray):
    """Dequantise one unit's bytes -> (mu_hat [128], V_hat [128][8], C_hat [16][8])."""
    m, b, c, s = _c(mu, np.int8), _c(basis, np.uint8), _c(coef, np.int8), _c(scales, np.uint16)
    om = np.zeros(D)
    ov = np.zeros((D, R))
    oc = np.zeros((PAGE, R))
    _load().lo_decode_unit(_p(m), _p(b), _p(c), _p(s), _p(om), _p(ov), _p(oc))
    return om, ov, oc


# ------------------------------------------------------------------- score

def score_unit(q: np.ndarray, mu: np.ndarray, basis: np.ndarray, coef: np.ndarray) -> float:
    """Page score from float64 summaries of any rank (basis [128][r], coef [16][r])."""
    rank = basis.shape[1]
    qq, m = _c(q, np.float64), _c(mu, np.float64)
    v, c = _c(basis, np.float64), _c(coef, np.float64)
    return _load().lo_score_unit(_p(qq), _p(m), _p(v), _p(c), rank)


def scores(q, mu, basis, coef, scales, page_table, seq_pages, num_kv_heads: int) -> np.ndarray:
    """[B][Hq][max_pages] float64 scores from summary bytes (NaN where j >= seq_pages[b])."""
    q = _c(q, np.float32)
    B, Hq, _ = q.shape
    table = _c(page_table, np.int32)
    maxp = table.shape[1]
    out = np.full((B, Hq, maxp), np.nan)
    _load().lo_scores(B, Hq, num_kv_heads, maxp, _p(q), _p(_c(mu, np.int8)), _p(_c(basis, np.uint8)),
                      _p(_c(coef, np.int8)), _p(_c(scales, np.uint16)), _p(table),
                      _p(_c(seq_pages, np.int32)), _p(out))
    return out


def scores_sampled(q, mu, basis, coef, scales, page_table, num_kv_heads: int, sb, sh, sj) -> np.ndarray:
    q = _c(q, np.float32)
    B, Hq, _ = q.shape
    table = _c(page_table, np.int32)
    sb, sh, sj = _c(sb, np.int32), _c(sh, np.int32), _c(sj, np.int32)
    out = np.zeros(sb.shape[0])
    _load().lo_scores_sampled(B, Hq, num_kv_heads, table.shape[1], _p(q), _p(_c(mu, np.int8)),
                              _p(_c(basis, np.uint8)), _p(_c(coef, np.int8)), _p(_c(scales, np.uint16)),
                              _p(table), sb.shape[0], _p(sb), _p(sh), _p(sj), _p(out))
    return out


# ----------------------------------------------------------- group, select

def group_keys(scores_: np.ndarray, seq_pages, num_kv_heads: int):
    """(keys [B][Hkv][max_pages], head_lse [B][Hq]) - log of the group-mean mass share."""
    s = _c(scores_, np.float64)
    B, Hq, maxp = s.shape
    keys = np.full((B, num_kv_heads, maxp), np.nan)
    lse = np.zeros((B, Hq))
    _load().lo_group_keys(B, Hq, num_kv_heads, maxp, _p(s), _p(_c(seq_pages, np.int32)), _p(keys), _p(lse))
    return keys, lse


def select(keys: np.ndarray, seq_pages, budget_tokens: int, k_cap: Optional[int] = None):
    """(selected [B][Hkv][k_cap] ascending, n_selected [B][Hkv]); unused slots are -1."""
    k = _c(keys, np.float64)
    B, Hkv, maxp = k.shape
    if k_cap is None:
        k_cap = max(1, min(budget_tokens // PAGE, maxp))
    sel = np.full((B, Hkv, k_cap), -1, np.int32)
    nsel = np.zeros((B, Hkv), np.int32)
    _load().lo_select(B, Hkv, maxp, _p(k), _p(_c(seq_pages, np.int32)), int(budget_tokens), int(k_cap),
                      _p(sel), _p(nsel))
    return sel, nsel


# ---------------------------------------------------------------- attention

def attend(q, k_cache, v_cache, page_table, selected, n_selected, seq_pages=None, tail_tokens=None):
    """(out [B][Hq][128] float64, lse [B][Hq]) over the selected pages, plus, when given,
    the tail_tokens[b] tokens without a summary yet: logical pages seq_pages[b],
    seq_pages[b] + 1, ... (16 tokens each, the last one partial)."""
    q = _c(q, np.float32)
    B, Hq, _ = q.shape
    kc, vc = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    Hkv = kc.shape[1]
    table = _c(page_table, np.int32)
    sel = _c(selected, np.int32)
    nsel = _c(n_selected, np.int32)
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    if tail_tokens is not None:
        sp, tt = _c(seq_pages, np.int32), _c(tail_tokens, np.int32)
        psp, ptt = _p(sp), _p(tt)
    else:
        psp = ptt = None
    _load().lo_attend(B, Hq, Hkv, table.shape[1], _p(q), _p(kc), _p(vc), _p(table), _p(sel), _p(nsel),
                      sel.shape[2], psp, ptt, _p(out), _p(lse))
    return out, lse


def decode_step(q, k_cache, v_cache, page_table, seq_pages, mu, basis, coef, scales, budget_tokens: int,
                tail_tokens=None):
    """The whole step in float64: scores -> group keys -> select -> attend (plus the
    tail_tokens tokens without a summary, attended whole, when given)."""
    Hkv = k_cache.shape[1]
    s = scores(q, mu, basis, coef, scales, page_table, seq_pages, Hkv)
    keys, lse_h = group_keys(s, seq_pages, Hkv)
    sel, nsel = select(keys, seq_pages, budget_tokens)
    out, lse = attend(q, k_cache, v_cache, page_table, sel, nsel, seq_pages, tail_tokens)
    return dict(scores=s, keys=keys, head_lse=lse_h, selected=sel, n_selected=nsel, out=out, lse=lse)


# --------------------------------------------------------------- ablations

def _cache_args(q, k_cache, page_table, seq_pages):
    q = _c(q, np.float32)
    kc = _c(k_cache, np.uint16)
    table = _c(page_table, np.int32)
    return q, kc, table, _c(seq_pages, np.int32)


def exact_score_unit(q, k_bits) -> float:
    """log sum_i exp(q . k_i / sqrt(d)) over one page's 16 bf16 keys."""
    return _load().lo_exact_score_unit(_p(_c(q, np.float64)), _p(_c(k_bits, np.uint16).reshape(PAGE, D)))


def exact_scores(q, k_cache, page_table, seq_pages) -> np.ndarray:
    """[B][Hq][max_pages] exact page scores from all keys (NaN where j >= seq_pages[b])."""
    q, kc, table, seq = _cache_args(q, k_cache, page_table, seq_pages)
    B, Hq, _ = q.shape
    out = np.full((B, Hq, table.shape[1]), np.nan)
    _load().lo_exact_scores(B, Hq, kc.shape[1], table.shape[1], _p(q), _p(kc), _p(table), _p(seq), _p(out))
    return out


def quant_dequant(x, bits: int) -> np.ndarray:
    """x dequantised from its symmetric absmax codes of `bits` bits (0 = unchanged)."""
    y = _c(x, np.float64).copy()
    _load().lo_quant_dequant(_p(y), y.size, int(bits))
    return y


def variant_scores(q, k_cache, page_table, seq_pages, rank: int, bits_mu: int, bits_v: int,
                   bits_c: int) -> np.ndarray:
    """[B][Hq][max_pages] scores of rank-`rank` summaries quantised to the given widths."""
    q, kc, table, seq = _cache_args(q, k_cache, page_table, seq_pages)
    B, Hq, _ = q.shape
    out = np.full((B, Hq, table.shape[1]), np.nan)
    _load().lo_variant_scores(B, Hq, kc.shape[1], table.shape[1], _p(q), _p(kc), _p(table), _p(seq),
                              int(rank), int(bits_mu), int(bits_v), int(bits_c), _p(out))
    return out


def shared_basis(k_cache, page_table, seq_pages, rank: int):
    """(basis [B][Hkv][rank][128], eigvals [B][Hkv][128]) of each sequence's key second moment."""
    kc = _c(k_cache, np.uint16)
    table = _c(page_table, np.int32)
    seq = _c(seq_pages, np.int32)
    B, Hkv = table.shape[0], kc.shape[1]
    basis = np.zeros((B, Hkv, rank, D))
    ev = np.zeros((B, Hkv, D))
    _load().lo_shared_basis(B, Hkv, table.shape[1], _p(kc), _p(table), _p(seq), int(rank), _p(basis), _p(ev))
    return basis, ev


def shared_scores(q, k_cache, page_table, seq_pages, basis) -> np.ndarray:
    """[B][Hq][max_pages] scores of the keys projected on the shared basis ([B][Hkv][rank][128])."""
    q, kc, table, seq = _cache_args(q, k_cache, page_table, seq_pages)
    w = _c(basis, np.float64)
    B, Hq, _ = q.shape
    out = np.full((B, Hq, table.shape[1]), np.nan)
    _load().lo_shared_scores(B, Hq, kc.shape[1], table.shape[1], _p(q), _p(kc), _p(table), _p(seq), _p(w),
                             w.shape[2], _p(out))
    return out
