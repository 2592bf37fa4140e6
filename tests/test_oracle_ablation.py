"""Pins of the oracle's ablation functions (exact scores, rank / bit-width
variants, shared basis and its projected scores) against closed forms, numpy /
LAPACK routes, hand-worked quantiser cases and the oracle's already-pinned
shipped-summary path.
"""

import math

import numpy as np
import pytest

import synth

LN16 = math.log(16.0)


def _bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def _keys(rng, n, rank=8, noise=0.05):
    """n pages of rank-`rank` keys plus noise, as bf16 bits [n][16][128]."""
    out = []
    for _ in range(n):
        mu = 0.5 * rng.standard_normal(128)
        b = np.linalg.qr(rng.standard_normal((128, rank)))[0].T
        a = rng.standard_normal((16, rank)) * np.linspace(3.0, 0.5, rank)[None, :]
        out.append(mu[None, :] + a @ b + noise * rng.standard_normal((16, 128)))
    return _bf16(np.stack(out))


def _spectral_page(rng, svals):
    """bf16 keys mu + U diag(svals) V^T with U orthonormal and centred (columns orthogonal to ones)."""
    n = len(svals)
    a = rng.standard_normal((16, n))
    u = np.linalg.qr(a - a.mean(0))[0]
    v = np.linalg.qr(rng.standard_normal((128, n)))[0]
    return _bf16(0.1 * rng.standard_normal(128)[None, :] + (u * svals) @ v.T)


def _cache(rng, nphys, hkv, rank=8):
    return _keys(rng, nphys * hkv, rank).reshape(nphys, hkv, 16, 128)


def _problem(rng, B=2, hkv=2, g=3, maxp=12, nphys=30):
    kc = _cache(rng, nphys, hkv)
    q = rng.standard_normal((B, hkv * g, 128)).astype(np.float32)
    table = np.stack([rng.permutation(nphys)[:maxp] for _ in range(B)]).astype(np.int32)
    seq = np.array([maxp, maxp - 5][:B], np.int32)
    return q, kc, table, seq


# ------------------------------------------------------------ exact scores

def test_exact_score_closed_forms(oracle_lib):
    rng = np.random.default_rng(1)
    q = rng.standard_normal(128)
    k = _bf16(rng.standard_normal(128))
    kf = synth.bf16_bits_to_f32(k).astype(np.float64)
    same = np.tile(k, (16, 1))
    assert abs(oracle_lib.exact_score_unit(q, same) - (q @ kf / math.sqrt(128) + LN16)) < 1e-12
    one = np.zeros((16, 128), np.uint16)
    one[0] = k
    assert abs(oracle_lib.exact_score_unit(q, one) - math.log(math.exp(q @ kf / math.sqrt(128)) + 15)) < 1e-12
    assert abs(oracle_lib.exact_score_unit(np.zeros(128), _keys(rng, 1)[0]) - LN16) < 1e-12


def test_exact_scores_follow_table_and_heads(oracle_lib):
    rng = np.random.default_rng(2)
    q, kc, table, seq = _problem(rng)
    s = oracle_lib.exact_scores(q, kc, table, seq)
    g = q.shape[1] // kc.shape[1]
    for b in range(2):
        assert np.all(np.isnan(s[b, :, seq[b]:]))
        for h in range(q.shape[1]):
            for j in range(seq[b]):
                want = oracle_lib.exact_score_unit(q[b, h].astype(np.float64), kc[table[b, j], h // g])
                assert s[b, h, j] == want


# ------------------------------------------------------------ quantiser

def test_quantiser_hand_worked_widths(oracle_lib):
    qd = oracle_lib.quant_dequant
    assert np.array_equal(qd([1.0, -0.4, 0.6, -1.0], 2), [1.0, 0.0, 1.0, -1.0])     # int2: codes {-1, 0, 1}
    assert np.array_equal(qd([3.0, -1.4, 1.6], 2), [3.0, 0.0, 3.0])
    assert np.array_equal(qd([7.0, -3.0, 1.0, 0.0], 4), [7.0, -3.0, 1.0, 0.0])       # int4: qmax 7
    assert np.array_equal(qd([127.0, -64.0, 0.5, 1.5], 8), [127.0, -64.0, 0.0, 2.0])  # int8: ties to even
    x = np.array([0.3, -0.2, 1e-3])
    assert np.array_equal(qd(x, 0), x)
    assert np.array_equal(qd(np.zeros(5), 4), np.zeros(5))


@pytest.mark.parametrize("bits,qmax", [(2, 1), (4, 7), (8, 127)])
def test_quantiser_codes_and_error_bound(oracle_lib, bits, qmax):
    rng = np.random.default_rng(bits)
    x = rng.standard_normal(2000) * 0.3
    y = oracle_lib.quant_dequant(x, bits)
    s = float(np.float16(np.abs(x).max() / qmax))     # numpy's own fp16 rounding
    codes = y / s
    assert np.allclose(codes, np.round(codes), atol=1e-9)
    assert np.abs(codes).max() <= qmax + 1e-9
    # within half a step, except where the clamp at qmax bites (fp16 rounding of the scale)
    err = np.abs(x - y)
    inside = np.abs(x) <= qmax * s
    assert err[inside].max() <= s / 2 * (1 + 1e-12)
    assert err.max() <= s


# ------------------------------------------------------------ variants

def test_variant_rank15_unquantised_is_exact(oracle_lib):
    """Sixteen centred keys span at most 15 directions: the rank-15 summary is the page."""
    rng = np.random.default_rng(3)
    for rank_keys in (8, 15):
        q, kc, table, seq = _problem(rng)
        kc = _cache(rng, kc.shape[0], kc.shape[1], rank=rank_keys)
        v = oracle_lib.variant_scores(q, kc, table, seq, 15, 0, 0, 0)
        e = oracle_lib.exact_scores(q, kc, table, seq)
        assert np.nanmax(np.abs(v - e)) < 1e-9


def test_variant_shipped_setting_is_the_product_summary(oracle_lib):
    rng = np.random.default_rng(4)
    q, kc, table, seq = _problem(rng)
    v = oracle_lib.variant_scores(q, kc, table, seq, 8, 8, 4, 8)
    mu, basis, coef, scales = oracle_lib.build_units(kc.reshape(-1, 16, 128))
    p = oracle_lib.scores(q, mu, basis, coef, scales, table, seq, kc.shape[1])
    assert np.nanmax(np.abs(v - p)) < 1e-12
    assert np.array_equal(np.isnan(v), np.isnan(p))


@pytest.mark.parametrize("rank", [1, 4, 8, 12])
def test_variant_unquantised_is_svd_truncation(oracle_lib, rank):
    """Eckart-Young: the rank-r summary reconstructs mu + the rank-r truncated SVD of D (numpy)."""
    rng = np.random.default_rng(10 + rank)
    q, kc, table, seq = _problem(rng, B=1, hkv=1, g=2, maxp=6, nphys=6)
    kc = np.stack([_spectral_page(rng, 20.0 * 1.5 ** -np.arange(15.0)) for _ in range(6)])[:, None]
    v = oracle_lib.variant_scores(q, kc, table, seq, rank, 0, 0, 0)
    for j in range(seq[0]):
        k = synth.bf16_bits_to_f32(kc[table[0, j], 0]).astype(np.float64)
        mu = k.mean(0)
        u, sv, vt = np.linalg.svd(k - mu, full_matrices=False)
        assert sv[rank - 1] > 1.05 * sv[rank]
        rec = mu + (u[:, :rank] * sv[:rank]) @ vt[:rank]
        for h in range(2):
            t = rec @ q[0, h].astype(np.float64) / math.sqrt(128)
            assert abs(v[0, h, j] - np.logaddexp.reduce(t)) < 1e-9


def test_variant_score_error_grows_as_width_shrinks(oracle_lib):
    """The direction the ablation reports: int8 basis < int4 < int2 in score error."""
    rng = np.random.default_rng(5)
    q, kc, table, seq = _problem(rng, B=1, hkv=2, g=4, maxp=40, nphys=40)
    e = oracle_lib.exact_scores(q, kc, table, seq)
    err = {b: np.nanmean(np.abs(oracle_lib.variant_scores(q, kc, table, seq, 8, 8, b, 8) - e)) for b in (8, 4, 2)}
    assert err[8] < err[4] < err[2]
    r_err = {r: np.nanmean(np.abs(oracle_lib.variant_scores(q, kc, table, seq, r, 0, 0, 0) - e)) for r in (4, 8)}
    assert r_err[8] < r_err[4]


# ------------------------------------------------------------ shared basis

def test_shared_basis_closed_form_axes(oracle_lib):
    """Keys along coordinate axes: M is diagonal, the basis is those axes by energy."""
    kc = np.zeros((3, 1, 16, 128), np.float32)
    energy = {17: 6.0, 5: 4.0, 99: 2.0, 64: 1.0}       # per-token magnitude on each axis
    t = 0
    for axis, a in energy.items():
        for _ in range(6):
            kc[t // 16, 0, t % 16, axis] = a if t % 2 else -a
            t += 1
    kb = _bf16(kc)
    table = np.arange(3, dtype=np.int32)[None]
    seq = np.array([3], np.int32)
    basis, ev = oracle_lib.shared_basis(kb, table, seq, 5)
    want_axes = [17, 5, 99, 64]
    for r, axis in enumerate(want_axes):
        row = np.zeros(128)
        row[axis] = 1.0
        assert np.allclose(basis[0, 0, r], row, atol=1e-12)
        assert abs(ev[0, 0, r] - 6 * energy[axis] ** 2) < 1e-9
    assert np.all(basis[0, 0, 4] == 0.0)               # no energy left for a fifth direction


def test_shared_basis_projector_matches_lapack(oracle_lib):
    rng = np.random.default_rng(6)
    kc = _cache(rng, 12, 2, rank=8)
    table = np.stack([rng.permutation(12)[:10] for _ in range(2)]).astype(np.int32)
    seq = np.array([10, 7], np.int32)
    for rank in (4, 8, 16):
        basis, ev = oracle_lib.shared_basis(kc, table, seq, rank)
        for b in range(2):
            for h in range(2):
                k = synth.bf16_bits_to_f32(kc[table[b, :seq[b]], h]).astype(np.float64).reshape(-1, 128)
                w, u = np.linalg.eigh(k.T @ k)
                assert w[-rank] > 1.01 * w[-rank - 1]
                top = u[:, ::-1][:, :rank]
                assert np.abs(basis[b, h].T @ basis[b, h] - top @ top.T).max() < 1e-8
                assert np.allclose(ev[b, h], w[::-1], rtol=1e-10, atol=1e-8 * w[-1])


def test_shared_scores_full_basis_is_exact_and_empty_basis_is_log16(oracle_lib):
    rng = np.random.default_rng(7)
    q, kc, table, seq = _problem(rng, maxp=12, nphys=30)
    kc = _cache(rng, 30, 2, rank=15)
    basis, _ = oracle_lib.shared_basis(kc, table, seq, 128)
    e = oracle_lib.exact_scores(q, kc, table, seq)
    assert np.nanmax(np.abs(oracle_lib.shared_scores(q, kc, table, seq, basis) - e)) < 1e-9
    empty = np.zeros((2, 2, 0, 128))
    s0 = oracle_lib.shared_scores(q, kc, table, seq, empty)
    assert np.nanmax(np.abs(s0 - LN16)) < 1e-12


def test_shared_scores_coordinate_projection(oracle_lib):
    """W = the first r axes: the score is the LSE of the truncated dot products."""
    rng = np.random.default_rng(8)
    q, kc, table, seq = _problem(rng, B=1, hkv=1, g=2, maxp=5, nphys=5)
    r = 24
    w = np.zeros((1, 1, r, 128))
    w[0, 0, np.arange(r), np.arange(r)] = 1.0
    s = oracle_lib.shared_scores(q, kc, table, seq, w)
    for j in range(5):
        k = synth.bf16_bits_to_f32(kc[table[0, j], 0]).astype(np.float64)
        for h in range(2):
            t = k[:, :r] @ q[0, h, :r].astype(np.float64) / math.sqrt(128)
            assert abs(s[0, h, j] - np.logaddexp.reduce(t)) < 1e-12


def test_proposition1_shared_projection_is_blind_to_its_null_space(oracle_lib):
    """Two pages that differ only in directions the shared basis does not span get the
    same shared score, however differently they answer the query; a page inside the
    null space scores log 16 for every query. The page-local summary sees the difference."""
    rng = np.random.default_rng(9)
    w = np.zeros((1, 1, 8, 128))
    w[0, 0, np.arange(8), np.arange(8)] = 1.0          # shared basis: axes 0..7
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    common = rng.standard_normal((16, 128)) * 0.3
    common[:, 8:] = 0.0
    content = np.zeros((16, 128))
    content[:, 8:] = 8.0 * q[0, 0, 8:] / np.linalg.norm(q[0, 0, 8:])   # aligned with head 0's query
    pages = np.stack([common + content, common - content, content])    # carrier, anti-carrier, null-space page
    kc = _bf16(pages)[:, None]
    table = np.arange(3, dtype=np.int32)[None]
    seq = np.array([3], np.int32)
    sh = oracle_lib.shared_scores(q, kc, table, seq, w)
    ex = oracle_lib.exact_scores(q, kc, table, seq)
    loc = oracle_lib.variant_scores(q, kc, table, seq, 8, 0, 0, 0)
    assert abs(sh[0, 0, 0] - sh[0, 0, 1]) < 1e-12
    assert np.abs(sh[0, :, 2] - LN16).max() < 1e-12
    assert ex[0, 0, 0] - ex[0, 0, 1] > 10.0
    assert loc[0, 0, 0] - loc[0, 0, 1] > 10.0
