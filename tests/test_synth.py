"""The seeded input generator: deterministic, right shapes, the configured structure."""

import numpy as np

import synth


def test_deterministic_and_shapes():
    w = synth.WORKLOADS["tiny"]
    a = synth.make_decode_inputs(w)
    b = synth.make_decode_inputs(w)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.v_cache, b.v_cache)
    assert np.array_equal(a.q, b.q)
    assert a.k_cache.shape == (256, 1, 16, 128) and a.k_cache.dtype == np.uint16
    assert a.q.shape == (1, 1, 128) and a.q.dtype == np.float32
    assert a.page_table.shape == (1, 256) and np.array_equal(a.page_table[0], np.arange(256))
    assert len(a.carriers[0][0]) == 4


def test_low_rank_structure_and_carriers():
    w = synth.WORKLOADS["llama8b_128k"].scaled(pages=64)
    inp = synth.make_decode_inputs(w)
    k = synth.bf16_bits_to_f32(inp.k_cache).astype(np.float64)  # [P][Hkv][16][128]
    dev = k - k.mean(axis=2, keepdims=True)
    s = np.linalg.svd(dev[5, 3], compute_uv=False)
    assert s[7] > 2 * s[8] and s[8] < 1.0  # rank-8 page plus 0.05 N(0,1) noise in 128 dims
    g = w.group
    for kvh in range(w.num_kv_heads):
        qhat = inp.q[0, kvh * g:(kvh + 1) * g].sum(0)
        qhat /= np.linalg.norm(qhat)
        for p in inp.carriers[0][kvh]:
            mu = k[p, kvh].mean(axis=0)
            assert abs(mu @ qhat / np.linalg.norm(mu) - 0.8) < 0.05


def test_page_type_mix_and_shuffled_table():
    w = synth.WORKLOADS["ctx1m"].scaled(pages=1000)
    t = synth.page_types(w, 0, 0)
    assert (t == synth.PAGE_LOWRANK8).sum() == 700 and (t == synth.PAGE_LOWRANK4).sum() == 200
    w3 = synth.WORKLOADS["batch8_256k"].scaled(pages=32, batch=3)
    table = synth.make_page_table(w3)
    assert sorted(table.ravel().tolist()) == list(range(96))
    assert not np.array_equal(table.ravel(), np.arange(96))


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    got = synth.f32_to_bf16_bits(x)
    assert list(synth.bf16_bits_to_f32(got)) == [1.0, 1.0 + 2 ** -6, -2.5, 0.0]


def test_random_summaries_valid_codes():
    s = synth.random_summaries(10, 2, seed=3, extreme_fraction=0.3)
    lo = s.basis & 0xF
    hi = s.basis >> 4
    assert not np.any(lo == 8) and not np.any(hi == 8)
    assert s.mu.min() >= -127 and s.coef.min() >= -127
    sc = s.scales.view(np.float16).astype(np.float64)
    assert np.all(sc[..., :3] > 0) and np.all(sc[..., 3] == 0)


def test_parallel_generation_matches_serial():
    w = synth.WORKLOADS["batch8_256k"].scaled(pages=5000, batch=2)
    a = synth.make_decode_inputs(w)
    b = synth.make_decode_inputs(w, workers=3)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.v_cache, b.v_cache)
