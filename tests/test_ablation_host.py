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
