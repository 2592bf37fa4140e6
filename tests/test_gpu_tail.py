"""The unfilled last page of each sequence (no summary yet) is attended whole,
and a page that fills gets its summary from a one-page build off the decode
stream (page-fill refresh)."""
import numpy as np
import pytest

import oracle
import synth

import torch

from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

from tests.gpu_util import DEV, bf16_out, cosine, device_problem, t, upload_summaries  # noqa: E402

ATT_ABS = 2e-2
ATT_COS = 0.9995


def _random_problem(seed, B, hkv, g, maxp, nphys):
    rng = np.random.default_rng(seed)
    kc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    vc = synth.f32_to_bf16_bits(rng.standard_normal((nphys, hkv, 16, 128)).astype(np.float32))
    q = (rng.standard_normal((B, hkv * g, 128)) * 1.5).astype(np.float32)
    table = rng.permutation(nphys)[:B * maxp].reshape(B, maxp).astype(np.int32)
    return rng, q, kc, vc, table


@pytest.mark.parametrize("hkv,g,budget", [(2, 4, 160), (8, 4, 512), (2, 16, 64), (2, 4, 0)])
def test_select_attend_tail_matches_oracle(hkv, g, budget):
    """Fused selection + attention with tails of 0..64 tokens (up to 4 pages) equals the
    oracle's attention over the same selection plus the tail tokens."""
    B, maxp = 5, 300
    rng, q, kc, vc, table = _random_problem(7 * hkv + g, B, hkv, g, maxp, B * maxp + 3)
    seq = np.array([200, 299, 1, 57, 120], np.int32)
    tail = np.array([21, 16, 1, 0, 64], np.int32)   # up to 4 pages without a summary
    scores = t((rng.standard_normal((B, hkv * g, maxp)) * 2).astype(np.float32))
    prob = device_problem(q, kc, vc, table, seq)
    k_cap = L.locks_k_cap(prob.dims, budget)
    sel = torch.zeros((B, hkv, max(k_cap, 1)), dtype=torch.int32, device=DEV)
    nsel = torch.zeros((B, hkv), dtype=torch.int32, device=DEV)
    out = torch.zeros((B, hkv * g, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((B, hkv * g), dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    L.locks_select_attend(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, scores, prob.seq_pages,
                          budget, sel, nsel, out, lse, ws, tail_tokens=t(tail))
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    sel_np, nsel_np = sel.cpu().numpy(), nsel.cpu().numpy()
    ref, ref_lse = oracle.attend(q, kc, vc, table, sel_np, nsel_np, seq, tail)
    got = bf16_out(out)
    lse_g = lse.cpu().numpy()
    assert np.abs(got - ref).max() < ATT_ABS
    has = (np.repeat(nsel_np, g, axis=1) > 0) | (tail[:, None] > 0)       # [B][Hq]: any token attended
    assert cosine(got, ref)[has].min() >= ATT_COS
    assert np.abs(lse_g[has] - ref_lse[has]).max() < 1e-3
    assert np.all(got[~has] == 0) and np.all(np.isneginf(lse_g[~has]))
    # the tail changes the output wherever it has tokens
    plain, _ = oracle.attend(q, kc, vc, table, sel_np, nsel_np)
    for b in range(B):
        if tail[b] > 0 and nsel_np[b].min() > 0:
            assert np.abs(ref[b] - plain[b]).max() > 1e-3


def test_tail_page_garbage_rows_are_ignored():
    """Rows past the tail may hold anything (here NaN and Inf); the result only
    depends on the tail's first tokens."""
    B, hkv, g, maxp = 2, 2, 4, 64
    rng, q, kc, vc, table = _random_problem(3, B, hkv, g, maxp, B * maxp)
    seq = np.array([40, 63], np.int32)
    tail = np.array([5, 9], np.int32)
    kc_bad, vc_bad = kc.copy(), vc.copy()
    for b in range(B):
        p = table[b, seq[b]]
        kc_bad[p, :, tail[b]:] = 0x7FC0      # NaN
        vc_bad[p, :, tail[b]:] = 0x7F80      # +Inf
    scores = t(rng.standard_normal((B, hkv * g, maxp)).astype(np.float32))
    outs = []
    for k_, v_ in ((kc, vc), (kc_bad, vc_bad)):
        prob = device_problem(q, k_, v_, table, seq)
        sel = torch.zeros((B, hkv, 4), dtype=torch.int32, device=DEV)
        nsel = torch.zeros((B, hkv), dtype=torch.int32, device=DEV)
        out = torch.zeros((B, hkv * g, 128), dtype=torch.int16, device=DEV)
        L.locks_select_attend(prob.dims, prob.q, prob.k_cache, prob.v_cache, prob.page_table, scores,
                              prob.seq_pages, 64, sel, nsel, out, tail_tokens=t(tail))
        torch.cuda.synchronize()
        outs.append(bf16_out(out))
    assert np.isfinite(outs[1]).all()
    assert np.array_equal(outs[0], outs[1])


def test_decode_step_tail_matches_oracle():
    """The whole step with unfilled pages: scores and selection over the full pages,
    attention over the selection plus each tail."""
    w = synth.WORKLOADS["llama8b_128k"].scaled(pages=400, batch=2)
    inp = synth.make_decode_inputs(w)
    seq = inp.seq_pages.copy()
    seq[:] = [397, 250]                      # summarised pages; the tail follows them
    tail = np.array([27, 3], np.int32)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    budget = 2048
    ref = oracle.decode_step(inp.q, inp.k_cache, inp.v_cache, inp.page_table, seq, mu, basis, coef, scales, budget,
                             tail_tokens=tail)
    summ = upload_summaries(mu, basis, coef, scales, w.num_phys_pages, w.num_kv_heads)
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, seq)
    k_cap = L.locks_k_cap(prob.dims, budget)
    ws = L.alloc_workspace(prob.dims, budget, DEV)
    out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=DEV)
    lse = torch.zeros((w.batch, w.num_q_heads), dtype=torch.float32, device=DEV)
    sel = torch.zeros((w.batch, w.num_kv_heads, k_cap), dtype=torch.int32, device=DEV)
    nsel = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=DEV)
    L.locks_decode_step(prob.dims, prob.q, prob.k_cache, prob.v_cache, summ, prob.page_table, prob.seq_pages, budget,
                        out, ws, lse=lse, selected=sel, n_selected=nsel, tail_tokens=t(tail))
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0
    sel_np, nsel_np = sel.cpu().numpy(), nsel.cpu().numpy()
    assert np.array_equal(nsel_np, ref["n_selected"])
    # attention is checked on the GPU's own selection (selection parity is tested elsewhere)
    ref_out, ref_lse = oracle.attend(inp.q, inp.k_cache, inp.v_cache, inp.page_table, sel_np, nsel_np, seq, tail)
    got = bf16_out(out)
    assert np.abs(got - ref_out).max() < ATT_ABS
    assert cosine(got, ref_out).min() >= ATT_COS
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 1e-3
    same = np.mean([np.array_equal(sel_np[b, h], ref["selected"][b, h]) for b in range(w.batch)
                    for h in range(w.num_kv_heads)])
    assert same >= 0.75


def test_page_fill_refresh_loop():
    """Decode with a growing sequence: one token per step joins the tail; when a page
    fills, its summary is built on a second stream (one page) while the page stays in
    the tail, attended whole, for the next steps; once the build has completed the page
    leaves the tail and is scored and selectable like every other page."""
    w = synth.WORKLOADS["tiny"].scaled(pages=64, batch=1)
    inp = synth.make_decode_inputs(w)
    budget = 128                               # 8 pages
    prob = device_problem(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages)
    dims = prob.dims
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, DEV)
    n_full, n_tail = 40, 9                     # 40 summarised pages, 9 tokens into page 40
    ids = torch.from_numpy(inp.page_table[0, :n_full].copy()).to(DEV)
    L.locks_build_summaries(dims, prob.k_cache, ids, n_full, summ)
    torch.cuda.synchronize()
    ws = L.alloc_workspace(dims, budget, DEV)
    k_cap = L.locks_k_cap(dims, budget)
    side = torch.cuda.Stream()
    built_pages, pending = [], []              # pending: (page, event, step launched)
    for step in range(40):
        n_tail += 1                            # this step's token joins the tail
        if n_tail % 16 == 0:
            # page n_full + n_tail // 16 - 1 just filled: build its summary off the decode stream
            page = n_full + n_tail // 16 - 1
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                pid = torch.from_numpy(inp.page_table[0, page:page + 1].copy()).to(DEV)
                L.locks_build_summaries(dims, prob.k_cache, pid, 1, summ, stream=side)
                ev = torch.cuda.Event()
                ev.record(side)
            pending.append((page, ev, step))
        # a page leaves the tail once its build is done and it has been in flight 3 steps
        while pending and pending[0][0] == n_full and step - pending[0][2] >= 3:
            pending[0][1].synchronize()
            built_pages.append(n_full)
            pending.pop(0)
            n_full, n_tail = n_full + 1, n_tail - 16
        seq = t(np.array([n_full], np.int32))
        tail = t(np.array([n_tail], np.int32))
        out = torch.zeros((1, w.num_q_heads, 128), dtype=torch.int16, device=DEV)
        sel = torch.zeros((1, w.num_kv_heads, k_cap), dtype=torch.int32, device=DEV)
        nsel = torch.zeros((1, w.num_kv_heads), dtype=torch.int32, device=DEV)
        L.locks_decode_step(dims, prob.q, prob.k_cache, prob.v_cache, summ, prob.page_table, seq, budget, out, ws,
                            selected=sel, n_selected=nsel, tail_tokens=tail)
        torch.cuda.current_stream().synchronize()
        assert L.locks_get_device_status(ws) == 0
        sel_np, nsel_np = sel.cpu().numpy(), nsel.cpu().numpy()
        assert (sel_np[0, :, :nsel_np[0, 0]] < n_full).all()   # only summarised pages are selected
        ref, _ = oracle.attend(inp.q, inp.k_cache, inp.v_cache, inp.page_table, sel_np, nsel_np,
                               np.array([n_full], np.int32), np.array([n_tail], np.int32))
        assert np.abs(bf16_out(out) - ref).max() < ATT_ABS
    torch.cuda.synchronize()
    assert built_pages == [40, 41] and n_full == 42
    # the refreshed pages' summaries are the ones a full build gives
    full = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, DEV)
    ids = torch.from_numpy(inp.page_table[0, :n_full].copy()).to(DEV)
    L.locks_build_summaries(dims, prob.k_cache, ids, n_full, full)
    torch.cuda.synchronize()
    for p in built_pages:
        ph = int(inp.page_table[0, p])
        for a, b in ((summ.mu, full.mu), (summ.basis, full.basis), (summ.coef, full.coef),
                     (summ.scales, full.scales)):
            assert torch.equal(a[ph], b[ph])
