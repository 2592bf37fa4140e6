"""A multi-layer decode step in one CUDA graph (the gist.science summary of the LOCKS paper,
2.4: the whole decode step of the model runs inside full CUDA graphs).

Four layers of the Llama-3.1-8B-shaped workload (shortened), each with its own seeded
query, K/V cache, page table and summaries (built by the oracle), are captured as four
locks_decode_step calls in one graph, each layer with its own workspace and outputs. After
replays, every layer's scores, selection and attention output are checked against the
oracle's decode step on that layer's inputs, and the replayed outputs equal the same calls
made eagerly. Nothing the GPU computes is given to the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from sparse_kv_page_gb300 import locks as L

pytestmark = pytest.mark.gpu

from tests.gpu_util import DEV, bf16_out, check_selection, cosine, t, upload_summaries  # noqa: E402

SCORE_TOL = 1e-3
ATT_ABS = 2e-2
ATT_COS = 0.9995
LAYERS = 4


def _layer(base, layer):
    w = dataclasses.replace(base, seeds=(100 + 7 * layer,), name=f"{base.name}-layer{layer}")
    inp = synth.make_decode_inputs(w)
    mu, basis, coef, scales = oracle.build_units(inp.k_cache.reshape(-1, 16, 128))
    return w, inp, (mu, basis, coef, scales)


def test_model_graph_layers_match_oracle_and_eager():
    base = synth.WORKLOADS["llama8b_128k"].scaled(pages=400)
    budget = 1024
    layers = [_layer(base, l) for l in range(LAYERS)]
    dev_layers = []
    for w, inp, (mu, basis, coef, scales) in layers:
        dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages)
        k_cap = L.locks_k_cap(dims, budget)
        dev_layers.append(dict(
            dims=dims, q=t(inp.q), kc=t(inp.k_cache), vc=t(inp.v_cache), table=t(inp.page_table),
            seq=t(inp.seq_pages), summ=upload_summaries(mu, basis, coef, scales, w.num_phys_pages, w.num_kv_heads),
            ws=L.alloc_workspace(dims, budget, DEV),
            out=torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=DEV),
            lse=torch.zeros((w.batch, w.num_q_heads), device=DEV),
            scores=torch.full((w.batch, w.num_q_heads, w.pages), float("nan"), device=DEV),
            sel=torch.zeros((w.batch, w.num_kv_heads, k_cap), dtype=torch.int32, device=DEV),
            nsel=torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=DEV)))

    def step_all():
        for d in dev_layers:
            L.locks_decode_step(d["dims"], d["q"], d["kc"], d["vc"], d["summ"], d["table"], d["seq"], budget,
                                d["out"], d["ws"], lse=d["lse"], scores=d["scores"], selected=d["sel"],
                                n_selected=d["nsel"])

    # eager reference of the same calls
    step_all()
    torch.cuda.synchronize()
    eager = [(d["out"].clone(), d["lse"].clone(), d["sel"].clone(), d["nsel"].clone(), d["scores"].clone())
             for d in dev_layers]
    for d in dev_layers:
        d["out"].zero_()
        d["lse"].zero_()
        d["sel"].zero_()
        d["nsel"].zero_()
        d["scores"].fill_(float("nan"))

    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step_all()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()

    for l, ((w, inp, (mu, basis, coef, scales)), d, e) in enumerate(zip(layers, dev_layers, eager)):
        assert L.locks_get_device_status(d["ws"]) == 0, l
        # replay equals eager
        for got, ref in zip((d["out"], d["lse"], d["sel"], d["nsel"], d["scores"]), e):
            assert torch.equal(got, ref), l
        # and the oracle's decode step on this layer's inputs
        ref = oracle.decode_step(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_pages, mu, basis, coef,
                                 scales, budget)
        scores = d["scores"].cpu().numpy().astype(np.float64)
        assert np.abs(scores - ref["scores"]).max() < SCORE_TOL, l
        sel, nsel = d["sel"].cpu().numpy(), d["nsel"].cpu().numpy()
        check_selection(sel, nsel, ref["selected"], ref["n_selected"], ref["keys"], inp.seq_pages)
        out, lse = bf16_out(d["out"]), d["lse"].cpu().numpy()
        same = np.array([[np.array_equal(sel[b, h], ref["selected"][b, h]) for h in range(w.num_kv_heads)]
                         for b in range(w.batch)])
        assert same.mean() >= 0.75, (l, same)
        heads = np.repeat(same, w.group, axis=1)
        assert np.abs(out - ref["out"])[heads].max() < ATT_ABS, l
        assert cosine(out, ref["out"])[heads].min() >= ATT_COS, l
        assert np.abs(lse - ref["lse"])[heads].max() < 1e-3, l
        # segments whose selection differs at the boundary: the attention call on the
        # oracle's selection reproduces the oracle's output
        k_cap = sel.shape[2]
        osel = np.zeros_like(sel)
        osel[:, :, :min(k_cap, ref["selected"].shape[2])] = ref["selected"][:, :, :k_cap]
        o2 = torch.zeros_like(d["out"])
        l2 = torch.zeros_like(d["lse"])
        L.locks_sparse_attention(d["dims"], d["q"], d["kc"], d["vc"], d["table"], t(osel),
                                 t(np.asarray(ref["n_selected"], np.int32)), k_cap, o2, l2)
        torch.cuda.synchronize()
        assert np.abs(bf16_out(o2) - ref["out"]).max() < ATT_ABS, l
        assert np.abs(l2.cpu().numpy() - ref["lse"]).max() < 1e-3, l
    # the layers really are different problems
    assert not torch.equal(dev_layers[0]["out"], dev_layers[1]["out"])
