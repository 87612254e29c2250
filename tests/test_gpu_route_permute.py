"""Routing, counts/offsets and permute vs the oracle (bit-exact indices,
counts, offsets, slots and permuted rows; weights within 1e-6)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import gpu_ops, to_np
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [  # T, E, k, score, normalize, zipf
    (256, 8, 2, "softmax", True, None),
    (1000, 8, 2, "softmax", False, None),
    (333, 64, 6, "sigmoid", False, None),
    (8192, 8, 2, "softmax", True, None),
    (24576, 256, 8, "sigmoid", True, None),
    (24576, 256, 8, "sigmoid", True, 1.2),
    (7, 4, 4, "softmax", True, None),
    (129, 1024, 32, "softmax", True, None),
]


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _score(ops, s):
    return ops.MOE_SCORE_SOFTMAX if s == "softmax" else ops.MOE_SCORE_SIGMOID


@pytest.mark.parametrize("T,E,k,score,norm,zipf", CASES)
def test_route_topk(ops, T, E, k, score, norm, zipf):
    logits = synth.make_logits(T, E, 0, "cuda", zipf)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w, counts, offsets = ops.moe_route_topk(logits, k, _score(ops, score), norm, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ridx, rw = O.route_topk(logits.cpu().numpy(), k, score, norm)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy() - rw)) <= 1e-6
    rc = O.group_counts(ridx, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), O.group_offsets(rc))
    if zipf:
        # skewed load: many empty experts, the largest group above 20% of tokens
        assert (rc == 0).sum() >= 30 and rc.max() > 0.2 * T


def test_route_ties_go_to_lower_index(ops):
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    logits = torch.randint(-2, 3, (4096, 16), generator=g, device="cuda").float()
    idx, w, _, _ = ops.moe_route_topk(logits, 5, ops.MOE_SCORE_SOFTMAX, True)
    torch.cuda.synchronize()
    ridx, rw = O.route_topk(logits.cpu().numpy(), 5, "softmax", True)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy() - rw)) <= 1e-6


def test_route_empty_batch(ops):
    logits = torch.zeros((0, 8), device="cuda")
    idx, w, counts, offsets = ops.moe_route_topk(logits, 2)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and offsets.cpu().tolist() == [0] * 9


@pytest.mark.parametrize("T,E,k,d", [(256, 8, 2, 512), (1000, 64, 6, 256), (24576, 256, 8, 7168), (3, 8, 2, 128),
                                     (500, 1024, 32, 128)])       # the largest E and k
def test_permute(ops, T, E, k, d):
    logits = synth.make_logits(T, E, 0, "cuda")
    x = synth.make_normal_bf16((T, d), 1, "cuda")
    idx, _, counts, _ = ops.moe_route_topk(logits, k)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gofs, slot_of, row_id, x_perm = ops.moe_permute(x, idx, E, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    idx_n = idx.cpu().numpy()
    r_slot, r_row = O.permute_slots(idx_n, E, align=128)
    r_gofs = O.aligned_group_offsets(O.group_counts(idx_n, E), 128)
    assert np.array_equal(gofs.cpu().numpy(), r_gofs)
    assert np.array_equal(slot_of.cpu().numpy(), r_slot)
    Rp = int(r_gofs[-1])
    assert np.array_equal(row_id[:Rp].cpu().numpy(), r_row)
    rows = np.arange(Rp) if Rp <= 8192 else np.sort(np.random.default_rng(0).choice(Rp, 4096, replace=False))
    want = O.permute(to_np(x), r_row[rows], k)
    got = to_np(x_perm[torch.from_numpy(rows).cuda()])
    assert np.array_equal(got, want)


def test_permute_rejects_bad_expert_index(ops):
    idx = torch.tensor([[0, 1], [2, 9], [3, 3]], dtype=torch.int32, device="cuda")
    x = torch.ones((3, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_permute(x, idx, 8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ops.MOE_ERR_BAD_EXPERT


def test_permute_duplicate_choice_gets_no_slot(ops):
    """A token that names one expert twice: the error word says so, the
    repeated choice (and an out-of-range one) gets slot -1, and the valid
    choices keep distinct slots whose row_id entries point back at them."""
    idx = torch.tensor([[0, 1], [2, 9], [3, 3], [1, 3]], dtype=torch.int32, device="cuda")
    x = torch.ones((4, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gofs, slot_of, row_id, _ = ops.moe_permute(x, idx, 8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ops.MOE_ERR_BAD_EXPERT
    s = slot_of.cpu().numpy()
    assert s[1, 1] == -1 and s[2, 1] == -1              # out of range; repeated expert 3
    valid = [(t, j) for t in range(4) for j in range(2) if s[t, j] >= 0]
    assert len(valid) == 6 and len({s[t, j] for t, j in valid}) == 6
    rid = row_id.cpu().numpy()
    for t, j in valid:
        assert rid[s[t, j]] == t * 2 + j
    # counts (and so the group offsets) see each valid choice once
    g = gofs.cpu().numpy()
    assert g[-1] == 128 * 4            # experts 0, 1, 2, 3 hold rows
