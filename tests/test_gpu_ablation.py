"""GPU parity of the selector-ablation kernels against the float64 oracle.

Exact and shared-basis scores are compared elementwise. The summary variants
build an eigendecomposition in fp32 on the GPU and in fp64 in the oracle:
unquantised variants are compared on units whose spectrum has a gap at the
kept rank (elsewhere the rank-r subspace itself is not unique); quantised
variants also differ where the two precisions put a value on opposite sides
of a rounding boundary, so most units must agree closely and all within the
size of one code step's effect.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

from tests.gpu_util import DEV, t  # noqa: E402

EXACT_TOL = 1e-4     # fp32 dot products of 128 terms, hardware exp2/log2
LN16 = math.log(16.0)


def _pages(rng, n, rank=8, noise=0.05):
    out = []
    for _ in range(n):
        mu = 0.5 * rng.standard_normal(128)
        b = np.linalg.qr(rng.standard_normal((128, rank)))[0].T
        a = rng.standard_normal((16, rank)) * np.linspace(3.0, 0.5, rank)[None, :]
        out.append(mu[None, :] + a @ b + noise * rng.standard_normal((16, 128)))
    return synth.f32_to_bf16_bits(np.stack(out).astype(np.float32))


def _problem(seed, B=2, hkv=2, g=4, maxp=150, nphys=400, seq=None):
    rng = np.random.default_rng(seed)
    kc = _pages(rng, nphys * hkv).reshape(nphys, hkv, 16, 128)
    q = rng.standard_normal((B, hkv * g, 128)).astype(np.float32)
    table = np.stack([rng.permutation(nphys)[:maxp] for _ in range(B)]).astype(np.int32)
    seq = np.array(seq if seq is not None else [maxp, maxp // 2 + 3][:B], np.int32)
    return q, kc, table, seq


def _dev(q, kc, table, seq):
    B, hq, _ = q.shape
    dims = L.make_dims(B, hq, kc.shape[1], table.shape[1], kc.shape[0])
    return dims, t(q), t(kc), t(table), t(seq)


def _nan_scores(B, hq, maxp):
    return torch.full((B, hq, maxp), float("nan"), dtype=torch.float32, device=DEV)


@pytest.mark.parametrize("hkv,g", [(2, 4), (8, 1), (2, 16), (1, 5)])
def test_exact_scores_match_oracle(hkv, g):
    q, kc, table, seq = _problem(10 * hkv + g, hkv=hkv, g=g)
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    s = _nan_scores(*q.shape[:2], table.shape[1])
    ws = L.alloc_ablation_workspace(dims, DEV)
    L.locks_exact_scores(dims, qd, kd, td, sd, s, workspace=ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    got = s.cpu().numpy()
    ref = oracle.exact_scores(q, kc, table, seq)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "entries past seq_pages must not be written"
    assert np.nanmax(np.abs(got - ref)) < EXACT_TOL


def _oracle_eigs(kc, table, seq, hkv):
    """Per (b, kv head, j) the oracle's 16 eigenvalues of the centred Gram matrix."""
    B, maxp = table.shape
    ev = np.full((B, hkv, maxp, 16), np.nan)
    for b in range(B):
        for h in range(hkv):
            for j in range(seq[b]):
                ev[b, h, j] = oracle.build_unit_f64(kc[table[b, j], h])[3]
    return ev


VARIANTS = [
    # rank, bits (mu, V, C)
    (15, 0, 0, 0), (8, 0, 0, 0), (4, 0, 0, 0),
    (8, 8, 4, 8), (8, 8, 8, 8), (8, 8, 2, 8), (4, 8, 4, 8), (15, 8, 4, 8), (8, 8, 4, 4), (8, 2, 2, 2),
]


@pytest.mark.parametrize("rank,bmu,bv,bc", VARIANTS)
def test_variant_scores_match_oracle(rank, bmu, bv, bc):
    hkv, g = 2, 4
    q, kc, table, seq = _problem(100 + rank * 10 + bv, hkv=hkv, g=g, maxp=120, nphys=300)
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    s = _nan_scores(*q.shape[:2], table.shape[1])
    ws = L.alloc_ablation_workspace(dims, DEV)
    L.locks_variant_scores(dims, qd, kd, td, sd, rank, bmu, bv, bc, s, workspace=ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    got = s.cpu().numpy()
    ref = oracle.variant_scores(q, kc, table, seq, rank, bmu, bv, bc)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    # units (b, kv head, j) with a spectral gap at the kept rank (rank 15 keeps the whole span)
    ev = _oracle_eigs(kc, table, seq, hkv)
    if rank < 15:
        gap = ev[..., rank - 1] >= 1.3 * np.maximum(ev[..., rank], 1e-30)
    else:
        gap = ~np.isnan(ev[..., 0])
    assert gap[~np.isnan(ev[..., 0])].mean() >= 0.5
    unit_err = np.abs(got - ref).reshape(2, hkv, g, -1).max(axis=2)       # [B][Hkv][maxp]
    err = unit_err[gap]
    if bmu == bv == bc == 0:
        assert err.max() < 2e-3, err.max()
    else:
        step = {8: 0.05, 4: 0.2, 2: 1.5}[min(b for b in (bmu, bv, bc))]
        assert np.mean(err < 2e-3) >= 0.9, np.mean(err < 2e-3)
        assert err.max() < step, err.max()


def _shared_problem(seed, B=2, hkv=2, g=4, maxp=200, nphys=450, rank_shared=8, decay=0.8):
    """Keys = a strong shared rank-`rank_shared` component (distinct energies) + page-local noise."""
    rng = np.random.default_rng(seed)
    basis = [np.linalg.qr(rng.standard_normal((128, rank_shared)))[0].T for _ in range(hkv)]
    energy = 4.0 * decay ** np.arange(rank_shared)
    k = np.zeros((nphys, hkv, 16, 128))
    for h in range(hkv):
        coef = rng.standard_normal((nphys, 16, rank_shared)) * energy
        k[:, h] = coef @ basis[h] + 0.3 * rng.standard_normal((nphys, 16, 128))
    kc = synth.f32_to_bf16_bits(k.astype(np.float32))
    q = rng.standard_normal((B, hkv * g, 128)).astype(np.float32)
    table = np.stack([rng.permutation(nphys)[:maxp] for _ in range(B)]).astype(np.int32)
    seq = np.array([maxp, maxp // 3][:B], np.int32)
    return q, kc, table, seq


@pytest.mark.parametrize("rank,rank_shared,decay", [(4, 8, 0.8), (8, 8, 0.8), (16, 16, 0.88)])
def test_shared_basis_matches_oracle(rank, rank_shared, decay):
    q, kc, table, seq = _shared_problem(7 + rank, rank_shared=rank_shared, decay=decay)
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    B, hkv = table.shape[0], kc.shape[1]
    ws = L.alloc_ablation_workspace(dims, DEV)
    basis = torch.zeros((B, hkv, rank, 128), dtype=torch.float32, device=DEV)
    ev = torch.zeros((B, hkv, 128), dtype=torch.float32, device=DEV)
    L.locks_shared_basis(dims, kd, td, sd, rank, basis, ws, eigvals=ev)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    ob, oev = oracle.shared_basis(kc, table, seq, rank)
    gb, gev = basis.cpu().numpy().astype(np.float64), ev.cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(hkv):
            assert oev[b, h, rank - 1] >= 1.1 * oev[b, h, rank]
            pg = gb[b, h].T @ gb[b, h]
            po = ob[b, h].T @ ob[b, h]
            assert np.abs(pg - po).max() < 2e-3
            assert np.abs(gb[b, h] @ gb[b, h].T - np.eye(rank)).max() < 1e-4      # orthonormal rows
            top = oev[b, h, :16]
            assert np.abs(gev[b, h, :16] - top).max() <= 1e-4 * top[0]


def test_shared_scores_match_oracle_on_the_oracle_basis():
    q, kc, table, seq = _shared_problem(3)
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    ws = L.alloc_ablation_workspace(dims, DEV)
    for rank in (0, 8, 128):
        ob, _ = oracle.shared_basis(kc, table, seq, rank)
        s = _nan_scores(*q.shape[:2], table.shape[1])
        L.locks_shared_scores(dims, qd, kd, td, sd, t(ob.astype(np.float32)), rank, s, ws)
        torch.cuda.synchronize()
        got = s.cpu().numpy()
        ref = oracle.shared_scores(q, kc, table, seq, ob)
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        assert np.nanmax(np.abs(got - ref)) < EXACT_TOL, rank
        if rank == 0:
            assert np.nanmax(np.abs(got - LN16)) < 1e-5
    assert L.locks_get_device_status(ws) == 0


def test_ablation_bad_page_index_is_reported():
    q, kc, table, seq = _problem(5, maxp=40, nphys=60)
    table = table.copy()
    table[1, 3] = 60            # one past the pool
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    ws = L.alloc_ablation_workspace(dims, DEV)
    s = _nan_scores(*q.shape[:2], table.shape[1])
    L.locks_exact_scores(dims, qd, kd, td, sd, s, workspace=ws)
    assert L.locks_get_device_status(ws) == L.LOCKS_ERR_BAD_INDEX
    L.locks_clear_device_status(ws)
    L.locks_variant_scores(dims, qd, kd, td, sd, 8, 8, 4, 8, s, workspace=ws)
    assert L.locks_get_device_status(ws) == L.LOCKS_ERR_BAD_INDEX


def test_ablation_argument_errors():
    q, kc, table, seq = _problem(6, maxp=8, nphys=20)
    dims, qd, kd, td, sd = _dev(q, kc, table, seq)
    s = _nan_scores(*q.shape[:2], table.shape[1])
    for rank, bits in ((0, (8, 4, 8)), (16, (8, 4, 8)), (8, (1, 4, 8)), (8, (8, 9, 8))):
        with pytest.raises(L.LocksError):
            L.locks_variant_scores(dims, qd, kd, td, sd, rank, *bits, s)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)
    basis = torch.zeros((2, 2, 8, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(L.LocksError):
        L.locks_shared_basis(dims, kd, td, sd, 8, basis, small)
    with pytest.raises(L.LocksError):
        L.locks_shared_basis(dims, kd, td, sd, 129, basis, L.alloc_ablation_workspace(dims, DEV))


def test_ablation_harness_properties():
    """On a shortened benchmark workload: the exact selection holds the most mass any k pages
    can hold, rank 15 unquantised reproduces it, and the variant kernel at the shipped
    widths agrees with the shipped summary path."""
    from sparse_kv_page_gb300 import ablation as AB

    w = synth.WORKLOADS["ctx1m"].scaled(pages=1024)
    inp = synth.make_decode_inputs(w, with_values=False)
    dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages)
    kc = t(inp.k_cache)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, DEV)
    L.locks_build_summaries(dims, kc, torch.arange(w.num_phys_pages, dtype=torch.int32, device=DEV),
                            w.num_phys_pages, summ)
    rec = AB.run(dims, t(inp.q), kc, t(inp.page_table), t(inp.seq_pages), summ, 512, inp.carriers, DEV)
    rows = {r["selector"]: r for r in rec["rows"]}
    exact = rows["exact (reads every key)"]
    assert exact["recall"] == 1.0 and exact["carriers_kept"] >= 0.9
    for r in rec["rows"]:
        assert 0.0 <= r["recall"] <= 1.0 and 0.0 <= r["carriers_kept"] <= 1.0
        assert r["mass"] <= exact["mass"] + 1e-4, r
    assert rows["r15 unquantised"]["recall"] >= 0.99
    assert exact["eta"] == 0.0 and exact["mass_vs_exact"] == 1.0
    for r in rec["rows"]:
        if r["selector"].startswith("r") and r.get("bits") == [0, 0, 0]:
            # Theorem 1: an unquantised summary's selection keeps at least e^(-4 eta) of the best mass
            assert r["mass_vs_exact"] >= r["theorem1_bound"] - 1e-4, r
    assert rows["r15 unquantised"]["eta"] < 1e-3
    shipped = rows["r8 int8/int4/int8 (shipped summary, locks_score_pages)"]
    variant = rows["r8 int8/int4/int8 (variant kernel)"]
    assert abs(shipped["recall"] - variant["recall"]) <= 0.02
    assert shipped["recall"] >= 0.8
