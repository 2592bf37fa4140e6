"""GPU <-> oracle parity of every step of the LOCKS decode path, through the C ABI.

Tolerances (fixed by the method's acceptance bar): page scores within 1e-3
absolute on identical summary bytes; selected pages identical except pages whose
oracle key lies within 1e-3 of the k-th key; attention outputs within 2e-2
absolute and cosine >= 0.9995 per head (bf16 output).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

from tests.gpu_util import (DEV, bf16_out, check_selection, cosine, decode_layout, device_problem,  # noqa: E402
                            download_summaries, t, upload_summaries)

SCORE_TOL = 1e-3
ATT_ABS = 2e-2
ATT_COS = 0.9995


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_kv_page_gb300 import build as b
    b.build()
    oracle.build()
    L.load_library()
    torch.cuda.set_device(DEV)


def _gpu_scores(prob, summ, fill=float("nan")):
    B, Hq = prob.q.shape[:2]
    maxp = prob.page_table.shape[1]
    scores = torch.full((B, Hq, maxp), fill, dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_score_pages(prob.dims, prob.q, summ, prob.page_table, prob.seq_pages, scores, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    return scores.cpu().numpy().astype(np.float64)


# ------------------------------------------------------------------ scores

@pytest.mark.parametrize("wname", ["tiny", "llama8b_128k", "glm9b_4x1m"])
def test_scores_on_oracle_built_summaries(wname):
    w = synth.WORKLOADS[wname]
    if w.pages > 256:
        w = w.scaled(pages=300, batch=min(w.batch, 2))
    inp = synth.make_decode_inputs(w)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    summ = upload_summaries(mu, basis, coef, scales, w.num_phys_pages, w.num_kv_heads)
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    got = _gpu_scores(prob, summ)
    ref = oracle.scores(inp.q, mu, basis, coef, scales, inp.page_table, inp.seq_pages, w.num_kv_heads)
    err = np.abs(got - ref).max()
    assert err < SCORE_TOL, err


@pytest.mark.parametrize("hkv,g", [(1, 1), (1, 3), (2, 16), (4, 2), (8, 4), (8, 8), (2, 5), (1, 16)])
def test_scores_random_bytes_ragged_shuffled(hkv, g):
    rng = np.random.default_rng(100 * hkv + g)
    B, maxp = 3, 150
    nphys = 500
    summ_np = synth.random_summaries(nphys, hkv, seed=hkv * 31 + g, extreme_fraction=0.1)
    q = (rng.standard_normal((B, hkv * g, 128)) * rng.uniform(0.25, 4.0, (B, hkv * g, 1))).astype(np.float32)
    table = np.stack([rng.permutation(nphys)[:maxp] for _ in range(B)]).astype(np.int32)
    seq = np.array([150, 77, 1], np.int32)
    kc = np.zeros((nphys, hkv, 16, 128), np.uint16)
    prob = device_problem(q, kc, kc, table, seq)
    summ = upload_summaries(summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, nphys, hkv)
    got = _gpu_scores(prob, summ)
    ref = oracle.scores(q, summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, table, seq, hkv)
    for b in range(B):
        P = seq[b]
        err = np.abs(got[b, :, :P] - ref[b, :, :P]).max()
        assert err < SCORE_TOL, (b, err)
        assert np.all(np.isnan(got[b, :, P:])), "entries past seq_pages must not be written"


def test_scores_extreme_query_scale():
    """The per-head power-of-two pre-scale keeps the f16 hi/lo split exact for any q scale."""
    rng = np.random.default_rng(7)
    hkv, g, B, maxp = 2, 4, 1, 64
    summ_np = synth.random_summaries(maxp, hkv, seed=5)
    q = rng.standard_normal((B, hkv * g, 128)).astype(np.float32)
    q[0, 0] *= 3000.0
    q[0, 1] *= 1e-4
    q[0, 5] *= 70000.0     # beyond the f16 range before scaling
    table = np.arange(maxp, dtype=np.int32)[None]
    seq = np.array([maxp], np.int32)
    kc = np.zeros((maxp, hkv, 16, 128), np.uint16)
    got = _gpu_scores(device_problem(q, kc, kc, table, seq), upload_summaries(
        summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, maxp, hkv))
    ref = oracle.scores(q, summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, table, seq, hkv)
    rel = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert rel.max() < 2e-6 * 70000 / 1000 + 1e-4, rel.max()
    assert np.abs(got[0, [2, 3, 4, 6, 7]] - ref[0, [2, 3, 4, 6, 7]]).max() < SCORE_TOL


# --------------------------------------------------------------- selection

def _select_case(scores, seq, budget, hkv):
    B, Hq, maxp = scores.shape
    dims = L.make_dims(B, Hq, hkv, maxp, max(1, B * maxp))
    k_cap = L.locks_k_cap(dims, budget)
    s_dev = t(scores.astype(np.float32))
    seq_dev = t(seq.astype(np.int32))
    sel = torch.full((B, hkv, k_cap), -7, dtype=torch.int32, device=DEV)
    nsel = torch.full((B, hkv), -7, dtype=torch.int32, device=DEV)
    keys = torch.full((B, hkv, maxp), float("nan"), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_select_pages(dims, s_dev, seq_dev, budget, sel, nsel, keys, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    s64 = scores.astype(np.float32).astype(np.float64)
    okeys, _ = oracle.group_keys(s64, seq, hkv)
    osel, onsel = oracle.select(okeys, seq, budget, k_cap)
    return sel.cpu().numpy(), nsel.cpu().numpy(), keys.cpu().numpy(), osel, onsel, okeys


@pytest.mark.parametrize("g,hkv", [(1, 1), (4, 8), (16, 2), (3, 2)])
@pytest.mark.parametrize("budget", [0, 15, 16, 160, 2048, 100000])
def test_selection_parity(g, hkv, budget):
    rng = np.random.default_rng(g * 1000 + budget)
    B, maxp = 3, 1100
    scores = rng.standard_normal((B, hkv * g, maxp)) * 2.0
    scores[1, :, 100:160] = 1.25          # a block of exact ties
    seq = np.array([1100, 517, 3], np.int32)
    sel, n, keys, osel, on, okeys = _select_case(scores, seq, budget, hkv)
    check_selection(sel, n, osel, on, okeys, seq)
    for b in range(B):
        P = seq[b]
        assert np.abs(keys[b, :, :P] - okeys[b, :, :P]).max() < 1e-5
        assert np.all(np.isnan(keys[b, :, P:]))


def test_selection_exact_ties_take_lowest_ids():
    B, hkv, g, maxp = 1, 1, 1, 4000
    scores = np.zeros((B, g, maxp))
    scores[0, 0, ::7] = 1.0                 # 572 equal maxima, keep 32 of them
    seq = np.array([maxp], np.int32)
    sel, n, _, osel, on, _ = _select_case(scores, seq, 32 * 16, hkv)
    assert n[0, 0] == 32
    assert np.array_equal(sel[0, 0], np.arange(0, 7 * 32, 7))
    assert np.array_equal(sel[0, 0], osel[0, 0])


def test_selection_nan_scores_rank_last():
    B, hkv, g, maxp = 1, 1, 2, 300
    rng = np.random.default_rng(3)
    scores = rng.standard_normal((B, g, maxp))
    scores[0, :, 10] = np.nan
    seq = np.array([maxp], np.int32)
    sel, n, _, osel, on, okeys = _select_case(scores, seq, 299 * 16, hkv)
    assert 10 not in sel[0, 0, :n[0, 0]].tolist()


# --------------------------------------------------------------- attention

@pytest.mark.parametrize("g,hkv,n_list", [(1, 1, [0, 1, 5]), (4, 8, [16, 3, 40, 0, 1, 7, 9, 128]),
                                          (16, 2, [200, 31]), (5, 2, [64, 65])])
def test_attention_parity(g, hkv, n_list):
    rng = np.random.default_rng(g * 17 + hkv)
    B = max(1, len(n_list) // hkv)
    maxp = 260
    nphys = B * maxp + 5
    kc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    q = (rng.standard_normal((B, hkv * g, 128)) * 1.5).astype(np.float32)
    table = rng.permutation(nphys)[:B * maxp].reshape(B, maxp).astype(np.int32)
    k_cap = max(n_list + [1])
    sel = np.full((B, hkv, k_cap), -1, np.int32)
    nsel = np.zeros((B, hkv), np.int32)
    it = iter(n_list * (B * hkv))
    for b in range(B):
        for h in range(hkv):
            n = next(it)
            nsel[b, h] = n
            sel[b, h, :n] = np.sort(rng.choice(maxp, n, replace=False))
    prob = device_problem(q, kc, vc, table, np.full(B, maxp, np.int32))
    out = torch.zeros((B, hkv * g, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, hkv * g), dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_sparse_attention(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, t(sel), t(nsel), k_cap,
                             out, lse, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    ref, ref_lse = oracle.attend(q, kc, vc, table, sel, nsel)
    got = bf16_out(out)
    assert np.abs(got - ref).max() < ATT_ABS
    lse_g = lse.cpu().numpy()
    for b in range(B):
        for h in range(hkv * g):
            if nsel[b, h // g] == 0:
                assert np.all(got[b, h] == 0) and np.isneginf(lse_g[b, h])
            else:
                assert cosine(got[b, h], ref[b, h]) >= ATT_COS
                assert abs(lse_g[b, h] - ref_lse[b, h]) < 1e-3


def test_attention_all_pages_is_dense_attention():
    """Every page selected (the dense comparator's path, many pages per warp): the output
    is textbook softmax attention over all of each sequence's tokens."""
    rng = np.random.default_rng(41)
    B, hkv, g, maxp = 2, 2, 4, 1500
    seq = np.array([1500, 913], np.int32)
    nphys = B * maxp
    kc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    q = (rng.standard_normal((B, hkv * g, 128)) * 1.5).astype(np.float32)
    table = rng.permutation(nphys).reshape(B, maxp).astype(np.int32)
    sel = np.tile(np.arange(maxp, dtype=np.int32), (B, hkv, 1))
    nsel = np.repeat(seq[:, None], hkv, axis=1).astype(np.int32)
    prob = device_problem(q, kc, vc, table, seq)
    out = torch.zeros((B, hkv * g, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, hkv * g), dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_sparse_attention(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, t(sel), t(nsel), maxp,
                             out, lse, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    got = bf16_out(out)
    kf = synth.bf16_bits_to_f32(kc).astype(np.float64)
    vf = synth.bf16_bits_to_f32(vc).astype(np.float64)
    lse_g = lse.cpu().numpy()
    for b in range(B):
        phys = table[b, :seq[b]]
        for h in range(hkv * g):
            keys = kf[phys, h // g].reshape(-1, 128)
            vals = vf[phys, h // g].reshape(-1, 128)
            logits = keys @ q[b, h].astype(np.float64) / np.sqrt(128.0)
            m = logits.max()
            p = np.exp(logits - m)
            ref = (p @ vals) / p.sum()
            assert np.abs(got[b, h] - ref).max() < ATT_ABS
            assert cosine(got[b, h], ref) >= ATT_COS
            assert abs(lse_g[b, h] - (m + np.log(p.sum()))) < 1e-3


@pytest.mark.parametrize("B,hkv,g,maxp,seq", [(1, 1, 4, 8192, [8192]), (2, 1, 4, 3000, [3000, 70]),
                                              (1, 2, 16, 2048, [2048])])
def test_split_attention_matches_dense_and_unsplit(B, hkv, g, maxp, seq):
    """With a full workspace, long selections are split over several clusters per segment and
    merged through the workspace by the last cluster to arrive: the output is the textbook
    dense softmax, equals the unsplit launch up to the merge order, and repeats exactly."""
    rng = np.random.default_rng(43 + maxp)
    seq = np.array(seq, np.int32)
    nphys = B * maxp
    kc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    q = (rng.standard_normal((B, hkv * g, 128)) * 1.5).astype(np.float32)
    table = rng.permutation(nphys).reshape(B, maxp).astype(np.int32)
    sel = np.tile(np.arange(maxp, dtype=np.int32), (B, hkv, 1))
    nsel = np.repeat(seq[:, None], hkv, axis=1).astype(np.int32)
    prob = device_problem(q, kc, vc, table, seq)
    ws = L.alloc_workspace(prob.dims, maxp * 16, DEV)

    def run(workspace):
        out = torch.zeros((B, hkv * g, 128), dtype=torch.int16, device=DEV)
        lse = torch.zeros((B, hkv * g), dtype=torch.float32, device=DEV)
        L.locks_sparse_attention(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, t(sel), t(nsel),
                                 maxp, out, lse, workspace)
        torch.cuda.synchronize()
        return out, lse

    o1, l1 = run(ws)
    o2, l2 = run(ws)
    assert L.locks_get_device_status(ws) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o0, l0 = run(None)
    assert np.abs(bf16_out(o1) - bf16_out(o0)).max() < 1e-2
    assert np.abs(l1.cpu().numpy() - l0.cpu().numpy()).max() < 1e-4
    got, lse_g = bf16_out(o1), l1.cpu().numpy()
    kf = synth.bf16_bits_to_f32(kc).astype(np.float64)
    vf = synth.bf16_bits_to_f32(vc).astype(np.float64)
    for b in range(B):
        phys = table[b, :seq[b]]
        for h in range(hkv * g):
            keys = kf[phys, h // g].reshape(-1, 128)
            vals = vf[phys, h // g].reshape(-1, 128)
            logits = keys @ q[b, h].astype(np.float64) / np.sqrt(128.0)
            m = logits.max()
            p = np.exp(logits - m)
            ref = (p @ vals) / p.sum()
            assert np.abs(got[b, h] - ref).max() < ATT_ABS
            assert cosine(got[b, h], ref) >= ATT_COS
            assert abs(lse_g[b, h] - (m + np.log(p.sum()))) < 1e-3


# ----------------------------------------------------------- fused step

def _run_decode(w, inp, mu, basis, coef, scales, budget):
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    summ = upload_summaries(mu, basis, coef, scales, w.num_phys_pages, w.num_kv_heads)
    k_cap = L.locks_k_cap(prob.dims, budget)
    ws = L.alloc_workspace(prob.dims, budget, DEV)
    out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((w.batch, w.num_q_heads), device=DEV)
    scores = torch.full((w.batch, w.num_q_heads, w.pages), float("nan"), device=DEV)
    sel = torch.zeros((w.batch, w.num_kv_heads, k_cap), dtype=torch.int32, device=DEV)
    nsel = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=DEV)
    L.locks_decode_step(prob.dims, prob.q, prob.k_cache, prob.v_cache, summ, prob.page_table, prob.seq_pages, budget,
                        out, ws, lse=lse, scores=scores, selected=sel, n_selected=nsel)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    return dict(out=bf16_out(out), lse=lse.cpu().numpy(), scores=scores.cpu().numpy().astype(np.float64),
                selected=sel.cpu().numpy(), n_selected=nsel.cpu().numpy(), prob=prob, k_cap=k_cap)


def _attend_on(prob, k_cap, selected, n_selected):
    """locks_sparse_attention on a given selection (no workspace: one cluster per segment)."""
    B, Hq = prob.q.shape[0], prob.q.shape[1]
    src = np.asarray(selected, np.int32)
    padded = np.zeros(src.shape[:2] + (k_cap,), np.int32)
    padded[:, :, :min(k_cap, src.shape[2])] = src[:, :, :k_cap]
    sel = t(padded)
    nsel = t(np.asarray(n_selected, np.int32))
    out = torch.zeros((B, Hq, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, Hq), device=DEV)
    L.locks_sparse_attention(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, sel, nsel, k_cap,
                             out, lse)
    torch.cuda.synchronize()
    return bf16_out(out), lse.cpu().numpy()


@pytest.mark.parametrize("wname,pages,batch,budget", [("tiny", None, None, 256), ("llama8b_128k", 700, 1, 2048),
                                                      ("batch8_256k", 400, 3, 512), ("glm9b_4x1m", 600, 2, 512),
                                                      ("ctx1m", 900, 1, 2048)])
def test_decode_step_matches_oracle(wname, pages, batch, budget):
    _check_decode_step(wname, pages, batch, budget)


@pytest.fixture
def pin_cluster():
    """Pins the selection launches' cluster size for one test, restoring the automatic
    choice afterwards."""
    def pin(cl):
        L.locks_set_select_cluster(cl)
    yield pin
    L.locks_set_select_cluster(0)


@pytest.mark.parametrize("cluster", [8, 12, 16])
@pytest.mark.parametrize("g,hkv,budget", [(4, 8, 160), (16, 2, 2048), (1, 1, 16), (3, 2, 100000)])
def test_selection_parity_every_cluster_size(pin_cluster, cluster, g, hkv, budget):
    """Each cluster size the launcher may pick (12 CTAs: one per SM) selects the oracle's
    pages, on ragged sequences with a block of exact ties."""
    pin_cluster(cluster)
    rng = np.random.default_rng(7 * cluster + g + budget)
    B, maxp = 3, 2500
    scores = rng.standard_normal((B, hkv * g, maxp)) * 2.0
    scores[0, :, 700:760] = 0.5
    seq = np.array([2500, 1201, 11], np.int32)
    sel, n, keys, osel, on, okeys = _select_case(scores, seq, budget, hkv)
    check_selection(sel, n, osel, on, okeys, seq)
    for b in range(B):
        assert np.abs(keys[b, :, :seq[b]] - okeys[b, :, :seq[b]]).max() < 1e-5


@pytest.mark.parametrize("cluster", [8, 12, 16])
@pytest.mark.parametrize("wname,pages,batch,budget", [("ctx1m", 900, 1, 2048), ("glm9b_4x1m", 600, 2, 512),
                                                      ("ctx1m", 2400, 1, 8192)])
def test_decode_step_every_cluster_size(pin_cluster, cluster, wname, pages, batch, budget):
    """The fused step at each cluster size; budget 8192 keeps 512 pages per (sequence, kv
    head), more than a CTA's warps take in their first ring slots, so the attention refills
    slots behind the tiles the selection issued."""
    pin_cluster(cluster)
    _check_decode_step(wname, pages, batch, budget)


@pytest.mark.parametrize("cluster", [8, 12, 16])
def test_selection_candidates_concentrated_in_one_cta(pin_cluster, cluster):
    """The K largest keys all lie in the first CTA's page range, so that CTA publishes more
    candidates than its fixed gather slots (kCandCap / cluster) and every CTA regathers
    by offsets; the selection is still the oracle's."""
    pin_cluster(cluster)
    rng = np.random.default_rng(11 + cluster)
    B, hkv, g, maxp = 1, 2, 4, 3000
    scores = rng.standard_normal((B, hkv * g, maxp)) * 0.3
    scores[:, :, :200] += 6.0    # the first 200 pages (inside CTA 0's range at any cluster size) dominate
    seq = np.array([maxp], np.int32)
    budget = 150 * 16
    sel, n, keys, osel, on, okeys = _select_case(scores, seq, budget, hkv)
    check_selection(sel, n, osel, on, okeys, seq)
    assert np.all(sel[0, :, :150] < 200)


def _check_decode_step(wname, pages, batch, budget):
    w = synth.WORKLOADS[wname]
    if pages is not None:
        w = w.scaled(pages=pages, batch=batch)
    inp = synth.make_decode_inputs(w)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    ref = oracle.decode_step(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages, mu, basis, coef, scales,
                             budget)
    got = _run_decode(w, inp, mu, basis, coef, scales, budget)
    assert np.abs(got["scores"] - ref["scores"]).max() < SCORE_TOL
    check_selection(got["selected"], got["n_selected"], ref["selected"], ref["n_selected"], ref["keys"],
                    inp.seq_pages)
    # outputs are compared where the selection is the oracle's (differences may only be
    # boundary ties, which the check above has verified); most segments must qualify
    g = w.group
    same = np.array([[np.array_equal(got["selected"][b, h], ref["selected"][b, h]) for h in range(w.num_kv_heads)]
                     for b in range(w.batch)])
    assert same.mean() >= 0.75, same
    heads = np.repeat(same, g, axis=1)                      # [B][Hq]
    assert np.abs(got["out"] - ref["out"])[heads].max() < ATT_ABS
    assert cosine(got["out"], ref["out"])[heads].min() >= ATT_COS
    assert np.abs(got["lse"] - ref["lse"])[heads].max() < 1e-3
    # every segment, including those whose selection differs at the boundary: the fused
    # output is the attention over the fused step's own selection (the attention call on
    # it, up to the merge order: one bf16 step), and the attention call on the oracle's
    # selection reproduces the oracle's output
    sep_out, sep_lse = _attend_on(got["prob"], got["k_cap"], got["selected"], got["n_selected"])
    assert np.all(np.abs(sep_out - got["out"]) <= 2.0 ** -7 * np.maximum(np.abs(sep_out), np.abs(got["out"])) + 1e-6)
    assert np.abs(sep_lse - got["lse"]).max() < 1e-5
    orc_out, orc_lse = _attend_on(got["prob"], got["k_cap"], ref["selected"], ref["n_selected"])
    assert np.abs(orc_out - ref["out"]).max() < ATT_ABS
    assert cosine(orc_out, ref["out"]).min() >= ATT_COS
    assert np.abs(orc_lse - ref["lse"]).max() < 1e-3
    # carriers (planted pages aligned with the group query) are kept
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            kept = set(got["selected"][b, h, :got["n_selected"][b, h]].tolist())
            car = set(inp.carriers[b][h].tolist())
            assert len(car & kept) >= 0.75 * len(car)


def test_select_attend_equals_separate_calls():
    """The fused selection+attention kernel gives exactly the two separate calls' results."""
    w = synth.WORKLOADS["glm9b_4x1m"].scaled(pages=500, batch=2)
    inp = synth.make_decode_inputs(w)
    rng = np.random.default_rng(0)
    scores = t((rng.standard_normal((w.batch, w.num_q_heads, w.pages)) * 2).astype(np.float32))
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    budget = 512
    k_cap = L.locks_k_cap(prob.dims, budget)
    res = []
    for fused in (True, False):
        sel = torch.zeros((w.batch, w.num_kv_heads, k_cap), dtype=torch.int32, device=DEV)
        nsel = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=DEV)
        out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=DEV)
        lse = torch.zeros((w.batch, w.num_q_heads), device=DEV)
        if fused:
            L.locks_select_attend(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, scores,
                                  prob.seq_pages, budget, sel, nsel, out, lse)
            # the same through partials computed from these scores on the host (max, sum per 8 pages)
        else:
            L.locks_select_pages(prob.dims, scores, prob.seq_pages, budget, sel, nsel)
            L.locks_sparse_attention(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, sel, nsel,
                                     k_cap, out, lse)
        torch.cuda.synchronize()
        res.append((sel.clone(), nsel.clone(), out.clone(), lse.clone()))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)


def test_decode_step_graph_capture_replays_identically():
    w = synth.WORKLOADS["llama8b_128k"].scaled(pages=320)
    inp = synth.make_decode_inputs(w)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    summ = upload_summaries(mu, basis, coef, scales, w.num_phys_pages, w.num_kv_heads)
    budget = 1024
    ws = L.alloc_workspace(prob.dims, budget, DEV)
    out = torch.zeros((1, 32, 128), dtype=torch.int16, device=DEV)
    L.locks_decode_step(prob.dims, prob.q, prob.k_cache, prob.v_cache, summ, prob.page_table, prob.seq_pages, budget,
                        out, ws)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            L.locks_decode_step(prob.dims, prob.q, prob.k_cache, prob.v_cache, summ, prob.page_table, prob.seq_pages,
                                budget, out, ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


# -------------------------------------------------------------- builder

def _key_pages(rng, n):
    """A mix: low-rank 8, low-rank 4, isotropic, constant pages (D = 0) and a large-magnitude page."""
    pages = []
    for i in range(n):
        kind = i % 5
        if kind in (0, 1):
            r = 8 if kind == 0 else 4
            mu = 0.5 * rng.standard_normal(128)
            qm, _ = np.linalg.qr(rng.standard_normal((128, r)))
            k = mu + rng.standard_normal((16, r)) @ qm.T + 0.05 * rng.standard_normal((16, 128))
        elif kind == 2:
            k = rng.standard_normal((16, 128))
        elif kind == 3:
            k = np.tile(rng.standard_normal(128), (16, 1))
        else:
            k = 300.0 * rng.standard_normal((16, 128))
        pages.append(k)
    return synth.f32_to_bf16_bits(np.stack(pages).astype(np.float32))


@pytest.mark.parametrize("hkv,nphys", [(1, 41), (2, 41), (8, 41), (8, 90)])
def test_builder_invariants(hkv, nphys):
    """Up to 512 units the builder takes one unit per warp, above it two; both are covered."""
    rng = np.random.default_rng(hkv + nphys)
    keys = _key_pages(rng, nphys * hkv).reshape(nphys, hkv, 16, 128)
    ids = np.array([p for p in range(nphys) if p % 4 != 1], np.int32)   # some pages not listed
    dims = L.make_dims(1, hkv, hkv, nphys, nphys)
    summ = L.Summaries.empty(nphys, hkv, DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_build_summaries(dims, t(keys), t(ids), len(ids), summ, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    gmu, gb, gc, gs = download_summaries(summ)
    omu, ob, oc, osc = oracle.build_units(keys.reshape(-1, 16, 128))
    omu, ob, oc, osc = (x.reshape(nphys, hkv, -1) for x in (omu, ob, oc, osc))
    unlisted = np.setdiff1d(np.arange(nphys), ids)
    assert not gmu[unlisted].any() and not gb[unlisted].any() and not gs[unlisted].any()
    g_mu, g_v, g_c = decode_layout(gmu[ids], gb[ids], gc[ids], gs[ids])
    o_mu, o_v, o_c = decode_layout(omu[ids], ob[ids], oc[ids], osc[ids])
    kf = synth.bf16_bits_to_f32(keys[ids]).astype(np.float64).reshape(-1, 16, 128)
    # centroid: same code up to one step
    smu_g = gs[ids][..., 0].view(np.float16).astype(np.float64).reshape(-1)
    assert np.all(np.abs(g_mu - o_mu) <= 1.01 * smu_g[:, None] + 1e-12)
    for u in range(kf.shape[0]):
        dev = kf[u] - kf[u].mean(0)
        sv = np.linalg.svd(dev, compute_uv=False)
        best = (sv[:8] ** 2).sum()
        tot = (sv ** 2).sum()
        res_g = np.linalg.norm(dev - g_c[u] @ g_v[u].T) ** 2
        res_o = np.linalg.norm(dev - o_c[u] @ o_v[u].T) ** 2
        if tot == 0:
            assert res_g == 0 and not g_v[u].any() and not g_c[u].any()
            continue
        # the GPU summary reconstructs the page as well as the oracle's (both quantised)
        assert res_g <= res_o * 1.05 + 1e-3 * tot, (u, res_g, res_o, tot)
        assert res_g <= (tot - best) + 0.05 * tot
        gaps = sv[:8] / np.maximum(sv[1:9], 1e-30)
        if np.all(gaps ** 2 >= 1.5):
            # well-separated spectrum: each basis column agrees to within one int4 step
            step = gs[ids].reshape(-1, 4)[u, 1:2].view(np.float16).astype(np.float64)[0]
            assert np.abs(g_v[u] - o_v[u]).max() <= 1.01 * step + 1e-12, u


def _eta(q, keys, mu_hat, v_hat, c_hat):
    """max_i |q . (k_i - mu_hat - V_hat c_i)| / sqrt(d) per (head, unit): the reconstruction error
    that bounds |score(summary) - exact page LSE| (log-sum-exp is 1-Lipschitz in the max norm)."""
    rec = mu_hat[:, None, :] + np.einsum("uir,udr->uid", c_hat, v_hat)
    res = keys - rec                                       # [u, 16, 128]
    return np.abs(np.einsum("hd,uid->hui", q, res)).max(axis=2) / math.sqrt(128)


def test_builder_end_to_end_scores():
    """Scores from GPU-built summaries (GPU scorer) vs oracle-built summaries (oracle scorer).

    Pages with a clear eigengap at the rank-8 cut (lambda_8 / lambda_9 >= 1.5) have one
    correct summary: agree within 1e-2. Pages with a flat spectrum at the cut (rank-4 and
    isotropic pages) admit any near-top-8 subspace: there the two scores must both lie
    within their own reconstruction error of the exact page LSE, |ds| <= eta_gpu + eta_orc."""
    w = synth.WORKLOADS["ctx1m"].scaled(pages=400)
    inp = synth.make_decode_inputs(w)
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, DEV)
    ids = t(np.arange(w.num_phys_pages, dtype=np.int32))
    L.locks_build_summaries(prob.dims, prob.k_cache, ids, w.num_phys_pages, summ)
    got = _gpu_scores(prob, summ)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    ref = oracle.scores(inp.q, mu, basis, coef, scales, inp.page_table, inp.seq_pages, w.num_kv_heads)
    g = w.group
    keys = synth.bf16_bits_to_f32(inp.k_cache).astype(np.float64)      # [P][Hkv][16][128]
    g_mu, g_v, g_c = decode_layout(*download_summaries(summ))
    o_mu, o_v, o_c = decode_layout(mu, basis, coef, scales)
    n_sep = 0
    for kvh in range(w.num_kv_heads):
        units = np.arange(w.pages) * w.num_kv_heads + kvh
        kk = keys[:, kvh]
        qh = inp.q[0, kvh * g:(kvh + 1) * g].astype(np.float64)
        eta_g = _eta(qh, kk, g_mu[units], g_v[units], g_c[units])
        eta_o = _eta(qh, kk, o_mu[units], o_v[units], o_c[units])
        d = np.abs(got[0, kvh * g:(kvh + 1) * g] - ref[0, kvh * g:(kvh + 1) * g])
        assert np.all(d <= eta_g + eta_o + 1e-3)
        dev = kk - kk.mean(axis=1, keepdims=True)
        sv = np.linalg.svd(dev, compute_uv=False)
        sep = (sv[:, 7] / np.maximum(sv[:, 8], 1e-30)) ** 2 >= 1.5
        n_sep += int(sep.sum())
        assert np.all(d[:, sep] < 1e-2)
    assert n_sep > 0.5 * w.pages * w.num_kv_heads


# ------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_selftest_bounded_wait(ws, 5_000_000)   # 5 ms
    assert L.locks_get_device_status(ws) == L.LOCKS_ERR_TIMEOUT
    L.locks_clear_device_status(ws)
    assert L.locks_get_device_status(ws) == 0
    x = torch.ones(1000, device=DEV)
    assert float(x.sum()) == 1000.0   # the context is still usable


def test_bad_page_table_entry_is_reported_not_read():
    hkv, g, maxp = 2, 4, 40
    summ_np = synth.random_summaries(maxp, hkv, seed=9)
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, hkv * g, 128)).astype(np.float32)
    table = np.arange(maxp, dtype=np.int32)[None].copy()
    table[0, 13] = 10_000_000
    seq = np.array([maxp], np.int32)
    kc = np.zeros((maxp, hkv, 16, 128), np.uint16)
    prob = device_problem(q, kc, kc, table, seq)
    summ = upload_summaries(summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, maxp, hkv)
    scores = torch.zeros((1, hkv * g, maxp), device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_score_pages(prob.dims, prob.q, summ, prob.page_table, prob.seq_pages, scores, ws)
    assert L.locks_get_device_status(ws) == L.LOCKS_ERR_BAD_INDEX
    ok_table = table.copy()
    ok_table[0, 13] = 0
    ref = oracle.scores(q, summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, ok_table, seq, hkv)
    got = scores.cpu().numpy()
    assert np.abs(got - ref).max() < SCORE_TOL   # page 13 was read from page 0 instead


def test_selection_from_lse_partials_matches_full_scores():
    """The per-8-page LSE partials written by the scorer give the same normaliser, keys and
    selection as reducing the full score table (ragged lengths, several segment sizes)."""
    rng = np.random.default_rng(4)
    for hkv, g, maxp, seq_list in ((8, 4, 1003, [1003, 517]), (2, 16, 700, [700, 9]), (1, 1, 64, [64, 1])):
        nphys = 2 * maxp
        summ_np = synth.random_summaries(nphys, hkv, seed=g)
        q = rng.standard_normal((2, hkv * g, 128)).astype(np.float32)
        table = np.stack([rng.permutation(nphys)[:maxp] for _ in range(2)]).astype(np.int32)
        seq = np.array(seq_list, np.int32)
        kc = np.zeros((nphys, hkv, 16, 128), np.uint16)
        prob = device_problem(q, kc, kc, table, seq)
        summ = upload_summaries(summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, nphys, hkv)
        scores = torch.zeros((2, hkv * g, maxp), device=DEV)
        part = torch.zeros(L.lse_partials_shape(prob.dims), device=DEV)
        L.locks_score_pages(prob.dims, prob.q, summ, prob.page_table, prob.seq_pages, scores, lse_partials=part)
        for budget in (16, 160, 2048):
            k_cap = L.locks_k_cap(prob.dims, budget)
            res = []
            for use in (True, False):
                sel = torch.zeros((2, hkv, k_cap), dtype=torch.int32, device=DEV)
                nsel = torch.zeros((2, hkv), dtype=torch.int32, device=DEV)
                keys = torch.full((2, hkv, maxp), float("nan"), device=DEV)
                L.locks_select_pages(prob.dims, scores, prob.seq_pages, budget, sel, nsel, keys,
                                     lse_partials=part if use else None)
                torch.cuda.synchronize()
                res.append((sel.cpu().numpy(), nsel.cpu().numpy(), keys.cpu().numpy()))
            (s1, n1, k1), (s2, n2, k2) = res
            assert np.array_equal(n1, n2)
            for b in range(2):
                P = seq[b]
                assert np.abs(k1[b, :, :P] - k2[b, :, :P]).max() < 2e-6
            okeys, _ = oracle.group_keys(scores.cpu().numpy().astype(np.float64), seq, hkv)
            osel, on = oracle.select(okeys, seq, budget, k_cap)
            check_selection(s1, n1, osel, on, okeys, seq)
