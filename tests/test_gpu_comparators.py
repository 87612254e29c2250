"""The prior-art comparators (per-expert GEMM loop, capacity-based MoE)
against the grouped dropless layer and the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_bf16_close, gpu_ops, to_np
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu

OUTS = ("out", "dx", "dlogits", "dW1", "dW2")


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _inputs(L, T, d, E, f, zipf=None):
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", zipf_s=zipf)
    L.set_weights(inp["W1"], inp["W2"])
    L.logits.copy_(inp["logits"])
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    return inp


@pytest.mark.parametrize("T,d,E,k,f,zipf", [
    (256, 512, 8, 2, 256, None),
    (2048, 1024, 32, 4, 512, 1.5),      # skewed: large, small and empty experts
])
def test_loop_of_gemms_matches_grouped_bit_for_bit(ops, T, d, E, k, f, zipf):
    """One GEMM per expert (single-group launches on per-expert MXFP8
    layouts, counts read on the host) gives exactly the grouped step's
    outputs and weight gradients."""
    from grouped_gemm_top_gb300.comparators import LoopMoE
    from grouped_gemm_top_gb300.layer import MoELayer
    L = MoELayer(T, d, E, k, f, "softmax", True)
    inp = _inputs(L, T, d, E, f, zipf)
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    ref = {n: getattr(L, n).clone() for n in OUTS}
    counts = L.counts.cpu().numpy()
    for n in OUTS:
        getattr(L, n).fill_(7)
    loop = LoopMoE(L)
    loop.set_weights(inp["W1"], inp["W2"])
    loop.step_()
    torch.cuda.synchronize()
    L.check_err()
    for n in OUTS:
        assert torch.equal(getattr(L, n), ref[n]), n
    assert loop.launches == 9 + 9 * int(np.count_nonzero(counts)) + 2 * int(np.count_nonzero(counts == 0))
    if zipf:
        assert np.count_nonzero(counts == 0) >= 1 or counts.max() > 4 * counts.mean()


def test_capacity_without_drops_matches_dropless(ops):
    """With a budget above every expert's load nothing is dropped, and the
    capacity-based layer (static padded groups) computes exactly what the
    dropless one does: each row's results depend only on its own operands
    and its expert, and the extra padding rows are zeros."""
    from grouped_gemm_top_gb300.comparators import CapacityMoE
    from grouped_gemm_top_gb300.layer import MoELayer
    T, d, E, k, f = 512, 512, 8, 2, 256
    L = MoELayer(T, d, E, k, f, "sigmoid", True)
    inp = _inputs(L, T, d, E, f)
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    C = CapacityMoE(T, d, E, k, f, "sigmoid", True, capacity_factor=2.0)
    C.set_weights(inp["W1"], inp["W2"])
    for n in ("logits", "x", "dout"):
        getattr(C, n).copy_(getattr(L, n))
    C.step_()
    torch.cuda.synchronize()
    C.check_err()
    assert int(L.counts.max()) <= C.C
    assert C.dropped_fraction() == 0.0
    for n in OUTS:
        assert torch.equal(getattr(C, n), getattr(L, n)), n


@pytest.mark.parametrize("cf", [0.5, 1.0])
def test_capacity_drops_the_choices_beyond_the_budget(ops, cf):
    """Capacity factor below the load: the choices kept are the first C of
    each expert in token order (exact), dropped choices contribute nothing,
    and the kept rows' outputs are the dropless layer's rows."""
    from grouped_gemm_top_gb300.comparators import CapacityMoE, capacity_rows
    from grouped_gemm_top_gb300.layer import MoELayer
    T, d, E, k, f = 1024, 512, 8, 2, 256
    L = MoELayer(T, d, E, k, f, "softmax", True)
    inp = _inputs(L, T, d, E, f, zipf=1.0)
    L.step_()
    torch.cuda.synchronize()
    C = CapacityMoE(T, d, E, k, f, "softmax", True, capacity_factor=cf)
    assert C.C == capacity_rows(T, E, k, cf)
    C.set_weights(inp["W1"], inp["W2"])
    for n in ("logits", "x", "dout"):
        getattr(C, n).copy_(getattr(L, n))
    C.step_()
    torch.cuda.synchronize()
    C.check_err()
    idx, _ = O.route_topk(inp["logits"].cpu().numpy(), k, "softmax", True)
    slot_dl, _ = O.permute_slots(idx, E, 1)          # unpadded: slot - start of expert = rank
    starts = np.concatenate([[0], np.cumsum(O.group_counts(idx, E))])
    rank = slot_dl - starts[idx]
    keep = rank < C.C
    want_slot = np.where(keep, idx * C.C + rank, E * C.C)
    assert np.array_equal(C.slot_of.cpu().numpy(), want_slot)
    assert C.dropped_fraction() == pytest.approx(1.0 - keep.mean())
    assert keep.mean() < 1.0
    # out = sum over kept choices of w * (the dropless layer's row)
    y0 = to_np(L.y_perm)
    w = L.topk_w.cpu().numpy().astype(np.float64)
    slot0 = L.slot_of.cpu().numpy()
    want = np.zeros((T, d))
    for j in range(k):
        want += np.where(keep[:, j:j + 1], w[:, j:j + 1] * y0[slot0[:, j]], 0.0)
    assert_bf16_close(C.out, want, what="capacity out")
    yc = to_np(C.y_perm)
    kept_rows = want_slot[keep]
    assert np.array_equal(yc[kept_rows], y0[slot0[keep]])
