"""Selector ablations on the synthetic carriers.

For one decode configuration already resident on the GPU, every selector below
scores all pages through the library's C ABI, the same group-mean keys and
top-k (locks_select_pages) choose its pages, and the choice is compared with
the exact selection, the one that reads every key (gist.science Korean
summary, sections 1 and 3):

* recall        - |S n E| / |E| per (request, kv head), averaged;
* mass          - sum over the chosen pages of the exact group-mean attention
                  share (each segment's shares sum to 1), averaged; the exact
                  selection's own value is the most any k pages can hold;
* carriers_kept - fraction of the planted carrier pages chosen;
* eta           - the largest |score - exact score| over (head, page), with the
                  mean error and e^(-4 eta), the least share of the best attainable
                  mass Theorem 1 guarantees an unquantised summary's selection
                  (gist.science summary, section 3), beside mass_vs_exact, the share
                  actually kept.

Selectors: the shipped rank-8 int8/int4/int8 summary (built once, scored by
locks_score_pages), page-local summaries of other ranks and code widths
(locks_variant_scores; LOCKS post, "Caveats": int4 loses a few recall points,
int2 collapses), and shared bases built from the whole sequence
(locks_shared_basis + locks_shared_scores; LOCKS post, "Why shared-basis
sparse attention is structurally broken"; Proposition 1). Each row also gives
the scorer's device time (CUDA events, mean of a few calls after one warm-up).

Run: python -m sparse_kv_page_gb300.ablation --workload llama8b_128k
"""
from __future__ import annotations

import argparse
import json
import math
import os
from typing import Callable, Dict, List, Sequence

import numpy as np
import torch

from . import locks as L

# (name, rank, bits of mu, basis, coefficients; 0 = unquantised)
VARIANTS = [
    ("r8 int8/int4/int8 (variant kernel)", 8, 8, 4, 8),
    ("r4 int8/int4/int8", 4, 8, 4, 8),
    ("r15 int8/int4/int8", 15, 8, 4, 8),
    ("r8 basis int8", 8, 8, 8, 8),
    ("r8 basis int2", 8, 8, 2, 8),
    ("r8 all int2", 8, 2, 2, 2),
    ("r4 unquantised", 4, 0, 0, 0),
    ("r8 unquantised", 8, 0, 0, 0),
    ("r15 unquantised", 15, 0, 0, 0),
]
SHARED_RANKS = (8, 32)


def _time_us(fn: Callable[[], None], reps: int = 3) -> float:
    fn()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1000.0 / reps


def _membership(sel: torch.Tensor, nsel: torch.Tensor, pages: int) -> torch.Tensor:
    """bool [B][Hkv][pages]: page j is among the n_selected entries of sel."""
    k = sel.shape[2]
    valid = torch.arange(k, device=sel.device)[None, None, :] < nsel[..., None]
    idx = torch.where(valid, sel, torch.zeros_like(sel)).long()
    m = torch.zeros(sel.shape[:2] + (pages,), dtype=torch.int32, device=sel.device)
    m.scatter_add_(2, idx, valid.int())
    return m > 0


def carrier_mask(carriers: Sequence[Sequence[np.ndarray]], shape, device) -> torch.Tensor:
    m = torch.zeros(shape, dtype=torch.bool, device=device)
    for b, per_head in enumerate(carriers):
        for h, pages in enumerate(per_head):
            if len(pages):
                m[b, h, torch.as_tensor(np.asarray(pages), dtype=torch.long, device=device)] = True
    return m


def selection_metrics(mem: torch.Tensor, mem_exact: torch.Tensor, share: torch.Tensor, carriers: torch.Tensor,
                      scores: torch.Tensor, exact_scores: torch.Tensor, live: torch.Tensor) -> Dict:
    """The metrics of one selector against the exact selection.

    mem, mem_exact, carriers: bool [B][Hkv][P] (chosen pages, the exact selection's,
    the planted carriers); share: float64 [B][Hkv][P], each (request, kv head)'s exact
    group-mean attention shares (zero past the sequence); scores, exact_scores:
    [B][Hq][P] page scores of the selector and of the exact selector; live: bool
    [B][1][P], the sequence's pages.
    """
    n_e = mem_exact.sum(2).clamp(min=1).double()
    held = (share * mem).sum(2)
    err = torch.where(live, (scores - exact_scores).abs(), torch.zeros((), dtype=scores.dtype, device=scores.device))
    eta = float(err.max().item()) if err.numel() else 0.0
    n_live = int(live.sum().item()) * scores.shape[1]
    n_car = int(carriers.sum().item())
    return {"recall": round(float(((mem & mem_exact).sum(2).double() / n_e).mean().item()), 4),
            "mass": round(float(held.mean().item()), 4),
            "mass_vs_exact": round(float((held / (share * mem_exact).sum(2)).mean().item()), 4),
            "carriers_kept": round(float((mem & carriers).sum().item()) / max(n_car, 1), 4),
            "eta": round(eta, 4),
            "mean_score_err": round(float(err.sum().item()) / max(n_live, 1), 5),
            "theorem1_bound": round(math.exp(-4.0 * eta), 4)}


def run(dims, q, k_cache, page_table, seq_pages, summaries, budget: int, carriers, device,
        variants=VARIANTS, shared_ranks=SHARED_RANKS) -> Dict:
    """All selectors on one resident configuration; returns the ablation record."""
    B, hq, hkv, P = dims.batch, dims.num_q_heads, dims.num_kv_heads, dims.max_pages_per_seq
    k_cap = L.locks_k_cap(dims, budget)
    ws = L.alloc_workspace(dims, budget, device)
    aws = L.alloc_ablation_workspace(dims, device)
    scores = torch.empty((B, hq, P), dtype=torch.float32, device=device)
    sel = torch.empty((B, hkv, k_cap), dtype=torch.int32, device=device)
    nsel = torch.empty((B, hkv), dtype=torch.int32, device=device)
    keys = torch.empty((B, hkv, P), dtype=torch.float32, device=device)

    def select(with_keys: bool = False):
        L.locks_select_pages(dims, scores, seq_pages, budget, sel, nsel, sel_keys=keys if with_keys else None,
                             workspace=ws)
        return _membership(sel, nsel, P)

    # the exact selection and the exact attention shares
    def exact():
        L.locks_exact_scores(dims, q, k_cache, page_table, seq_pages, scores, workspace=aws)

    exact_us = _time_us(exact)
    exact()
    exact_scores = scores.clone()
    mem_e = select(with_keys=True)
    live = torch.arange(P, device=device)[None, None, :] < seq_pages.long()[:, None, None]
    share = torch.where(live, torch.exp(keys.double()), torch.zeros((), dtype=torch.float64, device=device))
    cmask = carrier_mask(carriers, (B, hkv, P), device)
    n_car = int(cmask.sum().item())

    def row(name: str, mem: torch.Tensor, us: float, **extra) -> Dict:
        # eta: the largest |score - exact score| over (head, page) (Theorem 1's error; the
        # selection keeps at least e^(-4 eta) of the best attainable mass, unquantised summaries)
        r = {"selector": name}
        r.update(selection_metrics(mem, mem_e, share, cmask, scores, exact_scores, live))
        r["score_us"] = round(us, 1)
        r.update(extra)
        return r

    k_bytes = int(seq_pages.long().sum().item()) * hkv * 16 * 128 * 2
    rows: List[Dict] = [row("exact (reads every key)", mem_e, exact_us,
                            GBps=round(k_bytes / (exact_us * 1e-6) / 1e9, 1))]

    def shipped():
        L.locks_score_pages(dims, q, summaries, page_table, seq_pages, scores, ws)

    us = _time_us(shipped)
    shipped()
    rows.append(row("r8 int8/int4/int8 (shipped summary, locks_score_pages)", select(), us))

    for name, rank, bm, bv, bc in variants:
        def var(rank=rank, bm=bm, bv=bv, bc=bc):
            L.locks_variant_scores(dims, q, k_cache, page_table, seq_pages, rank, bm, bv, bc, scores,
                                   workspace=aws)

        us = _time_us(var, reps=1)
        var()
        rows.append(row(name, select(), us, rank=rank, bits=[bm, bv, bc]))

    for rank in shared_ranks:
        basis = torch.empty((B, hkv, rank, 128), dtype=torch.float32, device=device)

        def build_basis(rank=rank, basis=basis):
            L.locks_shared_basis(dims, k_cache, page_table, seq_pages, rank, basis, aws)

        basis_us = _time_us(build_basis, reps=1)

        def shared(rank=rank, basis=basis):
            L.locks_shared_scores(dims, q, k_cache, page_table, seq_pages, basis, rank, scores, aws)

        us = _time_us(shared)
        shared()
        rows.append(row(f"shared basis r{rank}", select(), us, rank=rank, basis_us=round(basis_us, 1)))

    status = L.locks_get_device_status(aws)
    if status != 0:
        raise L.LocksError(f"ablation kernels reported {L.locks_status_string(status)}")
    return {"budget": budget, "segments": B * hkv, "k": k_cap, "carriers": n_car,
            "exact_mass": rows[0]["mass"], "rows": rows}


def main(argv=None) -> None:
    import synth

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="llama8b_128k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--budget", type=int, default=0, help="tokens (default: the workload's largest budget)")
    ap.add_argument("--pages", type=int, default=0, help="shorten every sequence to this many pages")
    args = ap.parse_args(argv)
    w = synth.WORKLOADS[args.workload]
    if args.pages:
        w = w.scaled(pages=args.pages)
    budget = args.budget or max(w.budgets)
    inp = synth.make_decode_inputs(w, with_values=False, workers=min(16, os.cpu_count() or 1))
    from . import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def up(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    q, kc, table, seq = up(inp.q), up(inp.k_cache), up(inp.page_table), up(inp.seq_pages)
    dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, dev)
    L.locks_build_summaries(dims, kc, torch.arange(w.num_phys_pages, dtype=torch.int32, device=dev),
                            w.num_phys_pages, summ)
    rec = run(dims, q, kc, table, seq, summ, budget, inp.carriers, dev)
    rec["workload"] = w.name
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
