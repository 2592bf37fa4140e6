"""Pins of the float64 oracle against what the LOCKS pages and mathematics fix.

None of these checks re-types the oracle's own formulas: each compares it with
an independent route (numpy / LAPACK, a closed form, brute force over all
subsets, a theorem's bound, numpy's own float16 rounding, hand-worked layout
positions).
"""

import itertools
import math

import numpy as np
import pytest

import synth

pytestmark = []


def _keys(rng, rank=8, noise=0.05, mu_std=0.5):
    mu = mu_std * rng.standard_normal(128)
    q, r = np.linalg.qr(rng.standard_normal((128, rank)))
    b = q.T
    a = rng.standard_normal((16, rank))
    k = mu[None, :] + a @ b + noise * rng.standard_normal((16, 128))
    return synth.f32_to_bf16_bits(k.astype(np.float32))


def _exact_page_lse(k_bits, q):
    k = synth.bf16_bits_to_f32(k_bits).astype(np.float64).reshape(16, 128)
    logits = k @ q.astype(np.float64) / math.sqrt(128.0)
    m = logits.max()
    return m + math.log(np.exp(logits - m).sum()), logits


# ---------------------------------------------------------------- numbers

def test_f16_rounding_matches_numpy(oracle_lib):
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 5, 3000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, -3.0e-6]),
    ])
    got = oracle_lib.f64_to_f16(vals)
    with np.errstate(over="ignore"):             # 65520 and 1e6 round to inf on purpose
        want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    back = oracle_lib.f16_to_f64(want)
    assert np.array_equal(back, want.view(np.float16).astype(np.float64))


def test_bf16_decode_matches_bit_shift(oracle_lib):
    rng = np.random.default_rng(6)
    bits = synth.f32_to_bf16_bits(rng.standard_normal(2000).astype(np.float32) * 7)
    assert np.array_equal(oracle_lib.bf16_to_f64(bits), synth.bf16_bits_to_f32(bits).astype(np.float64))


# ----------------------------------------------------------- Jacobi (P6)

@pytest.mark.parametrize("n", [2, 5, 16])
def test_jacobi_matches_lapack(oracle_lib, n):
    rng = np.random.default_rng(n)
    for trial in range(10):
        a = rng.standard_normal((n, n))
        a = a + a.T
        w, v, sweeps = oracle_lib.jacobi_eig(a)
        assert sweeps < 30
        order = np.argsort(-w)
        ref = np.linalg.eigvalsh(a)[::-1]
        assert np.allclose(w[order], ref, atol=1e-11 * np.abs(ref).max())
        assert np.allclose(a @ v, v * w[None, :], atol=1e-10 * np.abs(ref).max())
        assert np.allclose(v.T @ v, np.eye(n), atol=1e-12)


def test_build_subspace_matches_svd(oracle_lib):
    """P6: the rank-8 basis spans the top-8 right singular subspace of the centred keys."""
    rng = np.random.default_rng(11)
    for trial in range(20):
        kb = _keys(rng, rank=8 if trial % 2 else 4)
        mu, basis, coef, ev = oracle_lib.build_unit_f64(kb, 8)
        k = synth.bf16_bits_to_f32(kb).astype(np.float64)
        dev = k - k.mean(axis=0)
        assert np.allclose(mu, k.mean(axis=0), atol=1e-14)
        u, s, vh = np.linalg.svd(dev, full_matrices=False)
        assert np.allclose(ev[:16], np.concatenate([s ** 2, np.zeros(16 - s.size)])[:16],
                           atol=1e-9 * s[0] ** 2)
        # well separated spectrum -> same projector
        if s[7] / s[8] > 1.2:
            p_orc = basis @ basis.T
            p_ref = vh[:8].T @ vh[:8]
            assert np.linalg.norm(p_orc - p_ref) < 1e-8
        assert np.allclose(basis.T @ basis, np.eye(8), atol=1e-10)
        assert np.allclose(coef, dev @ basis, atol=1e-10)
        # sign convention: largest-magnitude entry of each column is positive
        for r in range(8):
            assert basis[np.argmax(np.abs(basis[:, r])), r] > 0


def test_rank_deficient_page(oracle_lib):
    """A page of 16 equal keys has D = 0: basis and coefficients are zero."""
    row = synth.f32_to_bf16_bits(np.random.default_rng(3).standard_normal(128).astype(np.float32))
    kb = np.tile(row, (16, 1))
    mu, basis, coef, ev = oracle_lib.build_unit_f64(kb, 8)
    assert np.all(basis == 0) and np.all(coef == 0)
    assert np.allclose(mu, synth.bf16_bits_to_f32(row))


# ------------------------------------------------------- score closed forms

@pytest.mark.parametrize("rank", [15, 16])
def test_full_rank_summary_gives_exact_page_lse(oracle_lib, rank):
    """P1: rank >= 15 summaries reproduce the centred keys, so the score is the exact
    log-sum-exp of q.k/sqrt(128) over the page (LOCKS score formula)."""
    rng = np.random.default_rng(100 + rank)
    for trial in range(30):
        kb = _keys(rng, rank=8, noise=0.3) if trial % 3 else synth.f32_to_bf16_bits(
            rng.standard_normal((16, 128)).astype(np.float32))
        q = rng.standard_normal(128) * (1 + trial % 4)
        mu, basis, coef, _ = oracle_lib.build_unit_f64(kb, rank)
        s = oracle_lib.score_unit(q, mu, basis, coef)
        ref, _ = _exact_page_lse(kb, q)
        assert abs(s - ref) < 1e-11 * max(1.0, abs(ref))


def test_score_bounds_and_constant_page(oracle_lib):
    """P2: max logit <= score <= max logit + ln 16; a page of equal keys scores
    q.mu_hat/sqrt(d) + ln 16 (sixteen equal logits)."""
    rng = np.random.default_rng(7)
    for _ in range(30):
        kb = _keys(rng, noise=0.5)
        q = rng.standard_normal(128) * 2
        mu, basis, coef, _ = oracle_lib.build_unit_f64(kb, 15)
        s = oracle_lib.score_unit(q, mu, basis, coef)
        _, logits = _exact_page_lse(kb, q)
        assert logits.max() - 1e-9 <= s <= logits.max() + math.log(16) + 1e-9
    row = rng.standard_normal(128).astype(np.float32)
    kb = np.tile(synth.f32_to_bf16_bits(row), (16, 1))
    mb, bb, cb, sb = oracle_lib.build_units(kb[None])
    mu_hat, v_hat, c_hat = oracle_lib.decode_unit(mb[0], bb[0], cb[0], sb[0])
    q = rng.standard_normal(128)
    s = oracle_lib.score_unit(q, mu_hat, v_hat, c_hat)
    assert abs(s - (q @ mu_hat / math.sqrt(128) + math.log(16))) < 1e-12


def test_sign_flip_invariance(oracle_lib):
    """P12: negating a (V[:, r], C[:, r]) pair leaves the score unchanged."""
    rng = np.random.default_rng(9)
    kb = _keys(rng)
    mu, basis, coef, _ = oracle_lib.build_unit_f64(kb, 8)
    q = rng.standard_normal(128)
    s0 = oracle_lib.score_unit(q, mu, basis, coef)
    for r in range(8):
        b2, c2 = basis.copy(), coef.copy()
        b2[:, r] *= -1
        c2[:, r] *= -1
        assert abs(oracle_lib.score_unit(q, mu, b2, c2) - s0) < 1e-12
    # a dropped coefficient term is visible (the pin is not vacuous)
    c3 = coef.copy()
    c3[:, 0] = 0
    assert abs(oracle_lib.score_unit(q, mu, basis, c3) - s0) > 1e-6


# ---------------------------------------------------------- quantiser (P8)

def test_quantise_round_trip(oracle_lib):
    rng = np.random.default_rng(12)
    for _ in range(20):
        kb = _keys(rng)
        mu, basis, coef, _ = oracle_lib.build_unit_f64(kb, 8)
        om, ob, oc, osc = oracle_lib.encode_unit(mu, basis, coef)
        mh, vh, ch = oracle_lib.decode_unit(om, ob, oc, osc)
        for x, xh, qmax, sbits in ((mu, mh, 127, osc[0]), (basis, vh, 7, osc[1]), (coef, ch, 127, osc[2])):
            s = float(np.array(sbits, np.uint16).view(np.float16))
            want_s = np.float16(np.abs(x).max() / qmax)
            assert s == float(want_s)
            codes = np.round(xh / s)
            assert np.all(np.abs(codes) <= qmax)
            unclamped = np.abs(x) <= qmax * s
            assert np.all(np.abs(x - xh)[unclamped] <= s / 2 + 1e-15)
            assert np.all(np.abs(x - xh)[~unclamped] <= np.abs(x[~unclamped]) - qmax * s + s / 2 + 1e-12)
        assert osc[3] == 0
    om, ob, oc, osc = oracle_lib.encode_unit(np.zeros(128), np.zeros((128, 8)), np.zeros((16, 8)))
    assert not om.any() and not ob.any() and not oc.any() and not osc.any()


def test_layout_positions_hand_worked(oracle_lib):
    """The documented byte layout, checked on hand-worked positions."""
    # basis: (d, r) -> (byte, nibble); worked from
    # byte = 64 r + 16 t + 4 (s/2) + p/2, p = 2 (s%2) + h + 4 e
    cases = {(0, 0): (0, 0), (1, 0): (2, 0), (8, 0): (0, 1), (9, 0): (2, 1), (16, 0): (1, 0),
             (2, 0): (16, 0), (32, 0): (4, 0), (127, 7): (64 * 7 + 16 * 3 + 4 * 3 + 3, 1), (0, 1): (64, 0)}
    for (d, r), (byte, nib) in cases.items():
        v = np.zeros((128, 8))
        v[d, r] = 1.0
        _, ob, _, osc = oracle_lib.encode_unit(np.zeros(128), v, np.zeros((16, 8)))
        want = np.zeros(512, np.uint8)
        want[byte] = 7 << (4 * nib)
        assert np.array_equal(ob, want), (d, r)
        v[d, r] = -1.0
        _, ob, _, _ = oracle_lib.encode_unit(np.zeros(128), v, np.zeros((16, 8)))
        assert ob[byte] == (9 << (4 * nib)), (d, r)  # -7 as a two's complement nibble
    # mu: d -> 32 t + 4 s + 2 h + e
    for d, off in {0: 0, 1: 1, 8: 2, 9: 3, 16: 4, 2: 32, 127: 32 * 3 + 4 * 7 + 2 + 1}.items():
        m = np.zeros(128)
        m[d] = 1.0
        om, _, _, _ = oracle_lib.encode_unit(m, np.zeros((128, 8)), np.zeros((16, 8)))
        want = np.zeros(128, np.int8)
        want[off] = 127
        assert np.array_equal(om, want), d
    # coef: (i, r) -> 4 (4 (i%8) + r/2) + 2 (i/8) + r%2
    for (i, r), off in {(0, 0): 0, (0, 1): 1, (8, 0): 2, (8, 1): 3, (0, 2): 4, (1, 0): 16,
                        (15, 7): 4 * (4 * 7 + 3) + 2 + 1}.items():
        c = np.zeros((16, 8))
        c[i, r] = -2.0
        _, _, oc, _ = oracle_lib.encode_unit(np.zeros(128), np.zeros((128, 8)), c)
        want = np.zeros(128, np.int8)
        want[off] = -127
        assert np.array_equal(oc, want), (i, r)


def test_summary_is_about_ten_percent():
    """P5: summary bytes / page K+V bytes ~ 10% (r = 8, page of 16, int8/int4/int8 + scales)."""
    summary = 128 * 1 + 128 * 8 // 2 + 16 * 8 * 1 + 4 * 2
    assert summary == 776
    kv = 2 * 16 * 128 * 2
    assert 0.09 < summary / kv < 0.11


# ------------------------------------------------- group keys, select (P3, P9)

def _exact_scores(keys_bits, q):
    """[Hq][P] exact page LSEs from numpy (K decoded independently)."""
    k = synth.bf16_bits_to_f32(keys_bits).astype(np.float64)  # [P][16][128]
    logits = np.einsum("pid,hd->hpi", k, q.astype(np.float64)) / math.sqrt(128)
    m = logits.max(axis=2, keepdims=True)
    return (m + np.log(np.exp(logits - m).sum(axis=2, keepdims=True)))[..., 0]


def _rank15_scores(oracle_lib, keys_bits, q):
    out = np.zeros((q.shape[0], keys_bits.shape[0]))
    for j in range(keys_bits.shape[0]):
        mu, basis, coef, _ = oracle_lib.build_unit_f64(keys_bits[j], 15)
        for h in range(q.shape[0]):
            out[h, j] = oracle_lib.score_unit(q[h], mu, basis, coef)
    return out


@pytest.mark.parametrize("g", [1, 2, 4])
def test_selection_brute_force(oracle_lib, g):
    """P3: with exact (rank-15) scores, the selected k pages maximise the captured
    group-mean mass share over all C(P, k) subsets (mass ranking, Lemma 1 setting)."""
    rng = np.random.default_rng(20 + g)
    for trial in range(6):
        P = 6 + trial
        k = 1 + trial % 4
        keys_bits = np.stack([_keys(rng, noise=0.4, mu_std=0.3 + 0.2 * trial) for _ in range(P)])
        q = rng.standard_normal((g, 128)).astype(np.float32)
        s = _rank15_scores(oracle_lib, keys_bits, q.astype(np.float64))
        exact = _exact_scores(keys_bits, q)
        assert np.allclose(s, exact, atol=1e-10)
        kk, lse = oracle_lib.group_keys(s[None], np.array([P], np.int32), 1)
        sel, nsel = oracle_lib.select(kk, np.array([P], np.int32), 16 * k)
        assert nsel[0, 0] == k
        chosen = sel[0, 0, :k]
        assert np.all(np.diff(chosen) > 0)
        share = np.exp(exact - np.log(np.exp(exact).sum(axis=1, keepdims=True))).mean(axis=0)
        best = max(share[list(c)].sum() for c in itertools.combinations(range(P), k))
        assert share[chosen].sum() >= best - 1e-12


def test_mass_shares_normalised_and_g1_ranking(oracle_lib):
    """P9: per head the estimated shares sum to 1; with g = 1 the key is s - L."""
    rng = np.random.default_rng(31)
    s = rng.standard_normal((2, 4, 50)) * 3
    seq = np.array([50, 37], np.int32)
    keys, lse = oracle_lib.group_keys(s, seq, 2)
    for b in range(2):
        P = seq[b]
        for h in range(4):
            assert abs(np.exp(s[b, h, :P] - lse[b, h]).sum() - 1.0) < 1e-12
        for kvh in range(2):
            m = np.exp(s[b, 2 * kvh:2 * kvh + 2, :P] - lse[b, 2 * kvh:2 * kvh + 2, None]).mean(axis=0)
            assert np.allclose(np.exp(keys[b, kvh, :P]), m, rtol=1e-12)
    k1, l1 = oracle_lib.group_keys(s[:, :1], seq, 1)
    assert np.allclose(k1[0, 0, :50], s[0, 0] - l1[0, 0], atol=1e-12)


def test_select_ties_nan_and_budget(oracle_lib):
    keys = np.array([[[1.0, 3.0, 3.0, np.nan, 2.0, 3.0, -np.inf, 0.5]]])
    seq = np.array([8], np.int32)
    sel, n = oracle_lib.select(keys, seq, 16 * 2)
    assert n[0, 0] == 2 and list(sel[0, 0]) == [1, 2]          # ties -> lower page id
    sel, n = oracle_lib.select(keys, seq, 16 * 4 + 15)          # budget not a multiple of 16
    assert n[0, 0] == 4 and list(sel[0, 0]) == [1, 2, 4, 5]
    sel, n = oracle_lib.select(keys, seq, 16 * 100)             # k capped at the page count
    assert n[0, 0] == 8 and list(sel[0, 0]) == list(range(8))
    sel, n = oracle_lib.select(keys, seq, 15, k_cap=1)          # budget below one page
    assert n[0, 0] == 0
    sel, n = oracle_lib.select(keys, seq, 16 * 7)               # NaN ranks with -inf, below 0.5
    assert list(sel[0, 0]) == [0, 1, 2, 3, 4, 5, 7]


# ------------------------------------------------------ coverage bound (P4)

@pytest.mark.parametrize("g", [1, 4])
def test_theorem1_coverage_bound(oracle_lib, g):
    """P4: unquantised rank-8 scores within eta of the exact page LSEs keep at least
    e^(-4 eta) (e^(-2 eta) for g = 1) of the best captured exact mass share."""
    rng = np.random.default_rng(40 + g)
    P, k = 40, 6
    for trial in range(3):
        keys_bits = np.stack([_keys(rng, rank=8 + (j % 3) * 2, noise=0.1 + 0.1 * trial) for j in range(P)])
        q = rng.standard_normal((g, 128)).astype(np.float32)
        approx = np.zeros((g, P))
        for j in range(P):
            mu, basis, coef, _ = oracle_lib.build_unit_f64(keys_bits[j], 8)
            for h in range(g):
                approx[h, j] = oracle_lib.score_unit(q[h].astype(np.float64), mu, basis, coef)
        exact = _exact_scores(keys_bits, q)
        eta = np.abs(approx - exact).max()
        assert eta > 0
        kk, _ = oracle_lib.group_keys(approx[None], np.array([P], np.int32), 1)
        sel, _ = oracle_lib.select(kk, np.array([P], np.int32), 16 * k)
        share = np.exp(exact - np.log(np.exp(exact).sum(axis=1, keepdims=True))).mean(axis=0)
        opt = np.sort(share)[::-1][:k].sum()
        got = share[sel[0, 0, :k]].sum()
        bound = math.exp(-(2 if g == 1 else 4) * eta)
        assert got >= bound * opt - 1e-12


# -------------------------------------------------------------- attention (P7)

def _dense_attention(q, k_bits, v_bits):
    k = synth.bf16_bits_to_f32(k_bits).astype(np.float64)
    v = synth.bf16_bits_to_f32(v_bits).astype(np.float64)
    logits = k @ q.astype(np.float64) / math.sqrt(128)
    m = logits.max()
    p = np.exp(logits - m)
    return (p[:, None] * v).sum(axis=0) / p.sum(), m + math.log(p.sum())


def test_attention_all_pages_is_dense_softmax(oracle_lib):
    """P7: selecting every page gives textbook softmax attention; k = 1 gives a
    16-token softmax; an empty selection gives zeros and lse = -inf."""
    rng = np.random.default_rng(50)
    B, Hq, Hkv, P = 2, 4, 2, 5
    kc = synth.f32_to_bf16_bits(rng.standard_normal((B * P, Hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((B * P, Hkv, 16, 128)).astype(np.float32))
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    table = rng.permutation(B * P).reshape(B, P).astype(np.int32)
    sel = np.tile(np.arange(P, dtype=np.int32), (B, Hkv, 1))
    nsel = np.full((B, Hkv), P, np.int32)
    out, lse = oracle_lib.attend(q, kc, vc, table, sel, nsel)
    for b in range(B):
        for h in range(Hq):
            kvh = h // 2
            kb = kc[table[b], kvh].reshape(-1, 128)
            vb = vc[table[b], kvh].reshape(-1, 128)
            o, l = _dense_attention(q[b, h], kb, vb)
            assert np.allclose(out[b, h], o, atol=1e-12) and abs(lse[b, h] - l) < 1e-12
    one = np.full((B, Hkv, 1), 3, np.int32)
    out1, _ = oracle_lib.attend(q, kc, vc, table, one, np.ones((B, Hkv), np.int32))
    o, _ = _dense_attention(q[1, 3], kc[table[1, 3], 1], vc[table[1, 3], 1])
    assert np.allclose(out1[1, 3], o, atol=1e-12)
    out0, lse0 = oracle_lib.attend(q, kc, vc, table, one, np.zeros((B, Hkv), np.int32))
    assert np.all(out0 == 0) and np.all(np.isneginf(lse0))


def test_attention_tail_page(oracle_lib):
    """Tokens without a summary yet (the page being filled, and filled pages whose
    summaries are still being built) are attended whole: the tail's t tokens join the
    selected pages' tokens in one softmax. Pinned against textbook softmax attention over
    that token set; t = 16 equals selecting that page; t = 0 is no tail; tails spanning
    several pages."""
    rng = np.random.default_rng(51)
    B, Hq, Hkv, P = 3, 4, 2, 6
    kc = synth.f32_to_bf16_bits(rng.standard_normal((B * P, Hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((B * P, Hkv, 16, 128)).astype(np.float32))
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    table = rng.permutation(B * P).reshape(B, P).astype(np.int32)
    seq = np.array([4, 5, 2], np.int32)          # full pages; the unfilled page is logical page seq[b]
    tail = np.array([7, 16, 1], np.int32)
    sel = np.zeros((B, Hkv, 2), np.int32)
    sel[:, :, 0], sel[:, :, 1] = 0, 1
    nsel = np.array([[2, 1], [2, 0], [1, 2]], np.int32)
    out, lse = oracle_lib.attend(q, kc, vc, table, sel, nsel, seq, tail)
    for b in range(B):
        for h in range(Hq):
            kvh = h // 2
            pages = [table[b, sel[b, kvh, i]] for i in range(nsel[b, kvh])]
            kb = [kc[p_, kvh] for p_ in pages] + [kc[table[b, seq[b]], kvh][:tail[b]]]
            vb = [vc[p_, kvh] for p_ in pages] + [vc[table[b, seq[b]], kvh][:tail[b]]]
            o, l = _dense_attention(q[b, h], np.concatenate(kb), np.concatenate(vb))
            assert np.allclose(out[b, h], o, atol=1e-12) and abs(lse[b, h] - l) < 1e-12
    # t = 16 on page seq[1] = selecting that page as well
    sel3 = np.concatenate([sel, np.full((B, Hkv, 1), 5, np.int32)], axis=2)
    for kvh in range(Hkv):
        sel3[1, kvh, nsel[1, kvh]] = seq[1]
    out3, lse3 = oracle_lib.attend(q, kc, vc, table, sel3, nsel + np.array([[0, 0], [1, 1], [0, 0]], np.int32))
    assert np.allclose(out3[1], out[1], atol=1e-12) and np.allclose(lse3[1], lse[1], atol=1e-12)
    # t = 0: the plain selection
    out0, lse0 = oracle_lib.attend(q, kc, vc, table, sel, nsel, seq, np.zeros(B, np.int32))
    outn, lsen = oracle_lib.attend(q, kc, vc, table, sel, nsel)
    assert np.array_equal(out0, outn) and np.array_equal(lse0, lsen)
    # a tail over several pages (filled pages whose summaries are not built yet, then a
    # partial one): textbook softmax over the selected pages' tokens and those tokens
    seq2 = np.array([1, 2, 0], np.int32)
    tail2 = np.array([16 + 5, 32, 48 + 16], np.int32)
    out2, lse2 = oracle_lib.attend(q, kc, vc, table, sel, nsel, seq2, tail2)
    for b in range(B):
        for h in range(Hq):
            kvh = h // 2
            pages = [table[b, sel[b, kvh, i]] for i in range(nsel[b, kvh])]
            kb = [kc[p_, kvh] for p_ in pages]
            vb = [vc[p_, kvh] for p_ in pages]
            for j in range((tail2[b] + 15) // 16):
                nt = min(16, tail2[b] - 16 * j)
                kb.append(kc[table[b, seq2[b] + j], kvh][:nt])
                vb.append(vc[table[b, seq2[b] + j], kvh][:nt])
            o, l = _dense_attention(q[b, h], np.concatenate(kb), np.concatenate(vb))
            assert np.allclose(out2[b, h], o, atol=1e-12) and abs(lse2[b, h] - l) < 1e-12


# -------------------------------------------------- whole step, carriers (P10)

def test_tiny_workload_keeps_carriers(oracle_lib):
    """P10 (an expectation of the generator, not a hard pin): the 4 planted
    carrier pages of the tiny workload rank inside the 16 selected pages."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_decode_inputs(w)
    mu, basis, coef, scales = oracle_lib.build_units(inp.k_cache.reshape(-1, 16, 128))
    r = oracle_lib.decode_step(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages,
                               mu, basis, coef, scales, w.budgets[0])
    sel = set(r["selected"][0, 0, :r["n_selected"][0, 0]].tolist())
    assert r["n_selected"][0, 0] == 16
    assert set(inp.carriers[0][0].tolist()) <= sel
