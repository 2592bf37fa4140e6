"""Parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times (grid, cluster size and stage split follow the full dims).

The summaries are random valid bytes (every code in range) so no K is needed to
score; the oracle scores the same bytes in float64 over the whole table and makes
its own selection from its own scores. K and V are then filled (seeded) only on
the pages the GPU selected, the full fused decode step runs, and the oracle
attends over the same pages from a compacted copy of them.
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
KEY_TOL_S2 = 2e-4   # fp32 log-sum-exp over up to 65,536 pages, hardware exp2/log2
KEY_TOL = 2e-3      # plus the scores' own error
ATT_ABS = 2e-2
ATT_COS = 0.9995


@pytest.mark.parametrize("wname", ["llama8b_128k", "batch8_256k", "ctx1m", "glm9b_4x1m"])
def test_full_size_decode_step(wname):
    w = synth.WORKLOADS[wname]
    budget = max(w.budgets)
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
    L.locks_score_pages(dims, qd, summ, td, sd, scores, ws, lse_partials=part)
    torch.cuda.synchronize()
    ref_s = oracle.scores(q, summ_np.mu, summ_np.basis, summ_np.coef, summ_np.scales, table, seq, Hkv)
    assert np.abs(scores.cpu().numpy() - ref_s).max() < SCORE_TOL

    # 2. selection: the oracle selects from its own scores
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
    # the keys alone: against the oracle's keys of the GPU's own scores (S2 in isolation),
    # then against the oracle's keys of its own scores (S1 and S2 together)
    gk = gkeys.cpu().numpy()
    own, _ = oracle.group_keys(scores.cpu().numpy(), seq, Hkv)
    assert np.abs(gk - own).max() < KEY_TOL_S2
    assert np.abs(gk - keys).max() < KEY_TOL

    # 3. the whole fused step; K/V exist only on the pages selected (seeded values)
    rng = np.random.default_rng(w.seed_of(0) + 200)
    kc = torch.zeros((nphys, Hkv, 16, 128), dtype=torch.int16, device=DEV)
    vc = torch.zeros_like(kc)
    comp_table = np.zeros((B, P), np.int32)
    kparts, vparts, n_comp = [], [], 0
    for b in range(B):
        pages = np.unique(sel_np[b][:, :k_cap][np.arange(k_cap)[None, :] < nsel_np[b][:, None]])
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
    assert torch.equal(sel2, sel) and torch.equal(nsel2, nsel)
    ref_o, ref_l = oracle.attend(q, np.concatenate(kparts), np.concatenate(vparts), comp_table, sel_np, nsel_np)
    got = bf16_out(out)
    assert np.abs(got - ref_o).max() < ATT_ABS
    assert cosine(got, ref_o).min() >= ATT_COS
    assert np.abs(lse.cpu().numpy() - ref_l).max() < 1e-3
