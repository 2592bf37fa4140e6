"""Host logic of the selector-ablation harness (no GPU): selection membership
and the carrier mask, on CPU tensors."""
import numpy as np
import torch

from sparse_kv_page_gb300 import ablation as AB


def test_membership_ignores_unused_slots():
    # unused slots point at page 0; they must not clear or set page 0
    sel = torch.tensor([[[0, 3, 5, 0], [2, 0, 0, 0]]], dtype=torch.int32)
    nsel = torch.tensor([[3, 1]], dtype=torch.int32)
    m = AB._membership(sel, nsel, 7)
    assert m.shape == (1, 2, 7)
    assert m[0, 0].tolist() == [True, False, False, True, False, True, False]
    assert m[0, 1].tolist() == [False, False, True, False, False, False, False]
    nsel0 = torch.tensor([[0, 0]], dtype=torch.int32)
    assert not AB._membership(sel, nsel0, 7).any()


def test_membership_matches_python_sets():
    rng = np.random.default_rng(0)
    B, H, K, P = 3, 2, 9, 40
    sel = np.zeros((B, H, K), np.int32)
    nsel = rng.integers(0, K + 1, (B, H)).astype(np.int32)
    for b in range(B):
        for h in range(H):
            sel[b, h, :nsel[b, h]] = np.sort(rng.choice(P, nsel[b, h], replace=False))
    m = AB._membership(torch.from_numpy(sel), torch.from_numpy(nsel), P).numpy()
    for b in range(B):
        for h in range(H):
            assert set(np.flatnonzero(m[b, h])) == set(sel[b, h, :nsel[b, h]].tolist())


def test_carrier_mask():
    carriers = [[np.array([1, 4]), np.array([], np.int64)], [np.array([0]), np.array([2, 3])]]
    m = AB.carrier_mask(carriers, (2, 2, 5), "cpu")
    assert m.sum().item() == 5
    assert m[0, 0, 1] and m[0, 0, 4] and m[1, 0, 0] and m[1, 1, 2] and m[1, 1, 3]


def test_selection_metrics_hand_worked():
    """One (request, kv head) of 4 pages, 2 query heads: every metric by hand."""
    import math
    share = torch.tensor([[[0.4, 0.3, 0.2, 0.1]]], dtype=torch.float64)
    exact_sel = torch.tensor([[[True, True, False, False]]])
    chosen = torch.tensor([[[True, False, True, False]]])
    carriers = torch.tensor([[[False, True, True, False]]])
    exact_scores = torch.zeros((1, 2, 4))
    scores = torch.tensor([[[0.0, 0.5, -0.25, 0.0], [0.1, 0.0, 0.0, 9.0]]])
    live = torch.tensor([[[True, True, True, False]]])        # page 3 is past the sequence
    m = AB.selection_metrics(chosen, exact_sel, share, carriers, scores, exact_scores, live)
    assert m["recall"] == 0.5                                 # {0} of {0, 1}
    assert m["mass"] == 0.6                                   # 0.4 + 0.2
    assert m["mass_vs_exact"] == round(0.6 / 0.7, 4)
    assert m["carriers_kept"] == 0.5                          # page 2 of {1, 2}
    assert m["eta"] == 0.5                                    # page 3's 9.0 is not live
    assert m["mean_score_err"] == round((0.5 + 0.25 + 0.1) / 6, 5)
    assert m["theorem1_bound"] == round(math.exp(-2.0), 4)
