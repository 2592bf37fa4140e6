"""Checks against numbers the LOCKS pages print (tests/golden/, each cited in its file)."""

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "locks_sketch_constants.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_sketch_budget_gives_128_pages(oracle_lib):
    """The sketch keeps budget // page = 128 pages, i.e. 2048 of 65536 tokens (3.1%)."""
    g = _golden()
    pages = g["seq_len"] // g["page_size"]
    keys = np.random.default_rng(0).standard_normal((1, 1, pages))
    sel, n = oracle_lib.select(keys, np.array([pages], np.int32), g["token_budget"])
    assert n[0, 0] == g["n_top_pages"]
    attended = int(n[0, 0]) * g["page_size"]
    assert attended == g["attended_tokens"]
    assert f"{100 * attended / g['seq_len']:.1f}" == g["attended_percent_one_decimal"]
    assert np.all(np.diff(sel[0, 0, :n[0, 0]]) > 0)  # the sketch sorts the chosen indices


def test_summary_fraction_about_ten_percent(oracle_lib):
    """int8 centroid + int4 rank-8 basis + int8 coefficients (+ fp16 scales) ~ 10% of page K/V."""
    g = _golden()
    mu, basis, coef, scales = oracle_lib.build_units(np.zeros((1, 16, 128), np.uint16))
    summary = mu.nbytes + basis.nbytes + coef.nbytes + scales.nbytes
    kv = 2 * g["page_size"] * g["d_head"] * 2
    assert abs(summary / kv - g["summary_fraction_of_page_kv"]) <= g["summary_fraction_tolerance"]
    assert basis.nbytes == g["d_head"] * g["rank"] // 2


def test_sketch_scale_is_inverse_sqrt_d(oracle_lib):
    """The sketch scales logits by d_head ** -0.5: a one-token-dominated page scores q.k/sqrt(128)."""
    g = _golden()
    q = np.zeros(128)
    q[0] = 1000.0
    mu = np.zeros(128)
    basis = np.zeros((128, 1))
    basis[0, 0] = 1.0
    coef = np.full((16, 1), -1.0)
    coef[5, 0] = 1.0
    s = oracle_lib.score_unit(q, mu, basis, coef)
    assert abs(s - 1000.0 * g["d_head"] ** -0.5) < 1e-9
    assert math.isclose(g["d_head"] ** -0.5, 1 / math.sqrt(128))
