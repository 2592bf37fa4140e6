"""Parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times (grid, cluster size and stage split follow the full dims).

The summaries are random valid bytes (every code in range) so no K is needed to
score; the oracle scores the same bytes in float64 over the whole table and makes
its own selection from its own scores. The key and selection stage is also run on
one seeded score table given to both sides. K and V are then filled (seeded) only
on the pages the oracle selected, the fused decode step runs, and the oracle
attends over its selection from a compacted copy of those pages. Nothing the GPU
computes is given to the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

from tests.gpu_util import DEV, bf16_out, check_selection, cosine, t, upload_summaries  # noqa: E402

SCORE_TOL = 1e-3
KEY_TOL_S2 = 2e-4   # same scores on both sides: fp32 log-sum-exp over up to 65,536 pages
KEY_TOL = 2e-3      # each side's keys from its own scores: plus the scores' error
ATT_ABS = 2e-2
ATT_COS = 0.9995


CASES = [(n, b) for n in ("llama8b_128k", "batch8_256k", "ctx1m", "glm9b_4x1m") for b in synth.WORKLOADS[n].budgets]


@pytest.mark.parametrize("wname,budget", CASES)
def test_full_size_decode_step(wname, budget):
    w = synth.WORKLOADS[wname]
    B, Hq, Hkv, P, nphys = w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages
    q = synth.make_queries(w)
    table = synth.make_page_table(w)
    seq = np.full(B, P, np.int32)
    summ_np = synth.random_summaries(nphys, Hkv, seed=w.seed_of(0) + 100)
    summ = upload_summaries(summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, nphys, Hkv)
    dims = L.make_dims(B, Hq, Hkv, P, nphys)
    ws = L.alloc_workspace(dims, budget, DEV)
    qd, td, sd = t(q), t(table), t(seq)

    # 1. scores (with the LSE partials, as in the decode step) against the oracle's full table
    scores = torch.empty((B, Hq, P), dtype=torch.float32, device=DEV)
    part = torch.empty(L.lse_partials_shape(dims), dtype=torch.float32, device=DEV)
    L.locks_score_pages(dims, qd, summ, td, sd, scores, workspace=ws, lse_partials=part)
    torch.cuda.synchronize()
    ref_s = oracle.scores(q, summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, table, seq, Hkv)
    assert np.abs(scores.cpu().numpy() - ref_s).max() < SCORE_TOL

    # 2. selection from those scores (with the partials, as the step does): the oracle
    #    selects from its own scores, so pages may differ only at the k-th key
    keys, _ = oracle.group_keys(ref_s, seq, Hkv)
    osel, on = oracle.select(keys, seq, budget)
    k_cap = L.locks_k_cap(dims, budget)
    sel = torch.zeros((B, Hkv, k_cap), dtype=torch.int32, device=DEV)
    nsel = torch.zeros((B, Hkv), dtype=torch.int32, device=DEV)
    gkeys = torch.empty((B, Hkv, P), dtype=torch.float32, device=DEV)
    L.locks_select_pages(dims, scores, sd, budget, sel, nsel, sel_keys=gkeys, workspace=ws, lse_partials=part)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    sel_np, nsel_np = sel.cpu().numpy(), nsel.cpu().numpy()
    check_selection(sel_np, nsel_np, osel, on, keys, seq)
    assert np.abs(gkeys.cpu().numpy() - keys).max() < KEY_TOL

    # 3. the key and selection stage alone, on one seeded score table given to both sides
    rng = np.random.default_rng(w.seed_of(0) + 300)
    rs = (rng.standard_normal((B, Hq, P)) * 2.0).astype(np.float32)
    rkeys, _ = oracle.group_keys(rs, seq, Hkv)
    rsel, rn = oracle.select(rkeys, seq, budget)
    L.locks_select_pages(dims, t(rs), sd, budget, sel, nsel, sel_keys=gkeys, workspace=ws)
    torch.cuda.synchronize()
    assert np.abs(gkeys.cpu().numpy() - rkeys).max() < KEY_TOL_S2
    check_selection(sel.cpu().numpy(), nsel.cpu().numpy(), rsel, rn, rkeys, seq, tol=KEY_TOL_S2)

    # 4. the whole fused step; K/V exist only on the pages the oracle selected (seeded values)
    kc = torch.zeros((nphys, Hkv, 16, 128), dtype=torch.int16, device=DEV)
    vc = torch.zeros_like(kc)
    comp_table = np.zeros((B, P), np.int32)
    kparts, vparts, n_comp = [], [], 0
    for b in range(B):
        pages = np.unique(osel[b][np.arange(osel.shape[2])[None, :] < on[b][:, None]])
        kb = synth.f32_to_bf16_bits(rng.standard_normal((len(pages), Hkv, 16, 128)).astype(np.float32))
        vb = synth.f32_to_bf16_bits(rng.standard_normal((len(pages), Hkv, 16, 128)).astype(np.float32))
        phys = torch.from_numpy(table[b, pages].astype(np.int64)).to(DEV)
        kc[phys] = t(kb)
        vc[phys] = t(vb)
        comp_table[b, pages] = n_comp + np.arange(len(pages), dtype=np.int32)
        kparts.append(kb)
        vparts.append(vb)
        n_comp += len(pages)
    out = torch.zeros((B, Hq, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, Hq), dtype=torch.float32, device=DEV)
    sel2 = torch.zeros_like(sel)
    nsel2 = torch.zeros_like(nsel)
    L.locks_decode_step(dims, qd, kc, vc, summ, td, sd, budget, out, ws, lse=lse, selected=sel2, n_selected=nsel2)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    # the step's selection is the one the separate calls made in 2.
    assert np.array_equal(sel2.cpu().numpy(), sel_np) and np.array_equal(nsel2.cpu().numpy(), nsel_np)
    ref_o, ref_l = oracle.attend(q, np.concatenate(kparts), np.concatenate(vparts), comp_table, osel, on)
    # outputs are compared on the (request, kv head) segments whose selection is the
    # oracle's; others differ only at the boundary key, which 2. has verified
    same = np.array([[np.array_equal(sel_np[b, h], osel[b, h]) for h in range(Hkv)] for b in range(B)])
    assert same.mean() >= 0.75, same
    heads = np.repeat(same, Hq // Hkv, axis=1)
    got = bf16_out(out)
    assert np.abs(got - ref_o)[heads].max() < ATT_ABS
    assert cosine(got, ref_o)[heads].min() >= ATT_COS
    assert np.abs(lse.cpu().numpy() - ref_l)[heads].max() < 1e-3
    # every segment, including those whose selection differs at the boundary: the attention
    # call on the step's own selection gives the step's output (up to the merge order: one
    # bf16 step), and on the oracle's selection the oracle's output
    for chosen, n_chosen, check in ((sel_np, nsel_np, "self"), (osel, on, "oracle")):
        padded = np.zeros((B, Hkv, k_cap), np.int32)
        padded[:, :, :min(k_cap, chosen.shape[2])] = chosen[:, :, :k_cap]
        o2 = torch.zeros((B, Hq, 128), dtype=torch.int16, device=DEV)
        l2 = torch.zeros((B, Hq), dtype=torch.float32, device=DEV)
        L.locks_sparse_attention(dims, qd, kc, vc, td, t(padded), t(np.asarray(n_chosen, np.int32)), k_cap, o2, l2)
        torch.cuda.synchronize()
        g2, l2n = bf16_out(o2), l2.cpu().numpy()
        if check == "self":
            assert np.all(np.abs(g2 - got) <= 2.0 ** -7 * np.maximum(np.abs(g2), np.abs(got)) + 1e-6)
            assert np.abs(l2n - lse.cpu().numpy()).max() < 1e-5
        else:
            assert np.abs(g2 - ref_o).max() < ATT_ABS
            assert cosine(g2, ref_o).min() >= ATT_COS
            assert np.abs(l2n - ref_l).max() < 1e-3


def test_full_size_dense_attention_split_over_clusters():
    """The dense comparator's launch at 1M context (8 segments, each split over several
    clusters and merged through the workspace, every one of 65,536 pages selected) against
    the oracle's attention over all 1M tokens of every head. K and V come from a pool of
    2,048 random pages that a pseudo-random page table maps every logical page onto."""
    rng = np.random.default_rng(77)
    B, Hq, Hkv, P, pool = 1, 32, 8, 65536, 2048
    kc = synth.f32_to_bf16_bits(rng.standard_normal((pool, Hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((pool, Hkv, 16, 128)).astype(np.float32))
    q = (rng.standard_normal((B, Hq, 128)) * 2.0).astype(np.float32)
    table = ((np.arange(P, dtype=np.int64) * 7919 + 13) % pool).astype(np.int32)[None]
    sel = np.tile(np.arange(P, dtype=np.int32), (B, Hkv, 1))
    nsel = np.full((B, Hkv), P, np.int32)
    dims = L.make_dims(B, Hq, Hkv, P, pool)
    ws = L.alloc_workspace(dims, 2048, DEV)              # the decode step's workspace, as in the bench
    out = torch.zeros((B, Hq, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, Hq), dtype=torch.float32, device=DEV)
    L.locks_sparse_attention(dims, t(q), t(kc), t(vc), t(table), t(sel), t(nsel), P, out, lse, ws)
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    ref_o, ref_l = oracle.attend(q, kc, vc, table, sel, nsel)
    got = bf16_out(out)
    assert np.abs(got - ref_o).max() < ATT_ABS
    assert cosine(got, ref_o).min() >= ATT_COS
    assert np.abs(lse.cpu().numpy() - ref_l).max() < 1e-3
