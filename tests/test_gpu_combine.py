"""Combine (weighted and plain), combine backward and router backward vs
the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_bf16_close, assert_fp32_close, gpu_ops, to_np
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _routed(ops, T, E, k, d, score="softmax", norm=True):
    logits = synth.make_logits(T, E, 0, "cuda")
    idx, w, _, _ = ops.moe_route_topk(logits, k, ops.MOE_SCORE_SOFTMAX if score == "softmax" else
                                      ops.MOE_SCORE_SIGMOID, norm)
    gofs, slot_of, row_id, _ = ops.moe_permute(None, idx, E, want_x_perm=False)
    M = row_id.shape[0]
    y = synth.make_normal_bf16((M, d), 5, "cuda")
    return logits, idx, w, gofs, slot_of, row_id, y


@pytest.mark.parametrize("T,E,k,d", [(256, 8, 2, 512), (500, 64, 8, 1024), (24576, 256, 8, 7168)])
def test_combine(ops, T, E, k, d):
    logits, idx, w, gofs, slot_of, row_id, y = _routed(ops, T, E, k, d)
    out = ops.moe_unpermute_combine(y, slot_of, w)
    plain = ops.moe_unpermute_combine(y, slot_of, None)
    torch.cuda.synchronize()
    sl, wn = slot_of.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    tok = np.arange(T) if T <= 4096 else np.random.default_rng(1).choice(T, 2048, replace=False)
    yn = to_np(y)
    assert_bf16_close(to_np(out)[tok], O.combine(yn, sl[tok], wn[tok]), what="combine")
    assert_bf16_close(to_np(plain)[tok], O.combine(yn, sl[tok], None), what="unpermute-sum")


def test_combine_k1_unit_weight_is_exact_unpermute(ops):
    T, E, k, d = 300, 8, 1, 256
    logits = synth.make_logits(T, E, 0, "cuda")
    x = synth.make_normal_bf16((T, d), 1, "cuda")
    idx, _, _, _ = ops.moe_route_topk(logits, k)
    gofs, slot_of, row_id, x_perm = ops.moe_permute(x, idx, E)
    back = ops.moe_unpermute_combine(x_perm, slot_of, None)
    torch.cuda.synchronize()
    assert torch.equal(back, x)


@pytest.mark.parametrize("T,E,k,d", [(256, 8, 2, 512), (700, 32, 4, 1024)])
def test_combine_bwd(ops, T, E, k, d):
    logits, idx, w, gofs, slot_of, row_id, y = _routed(ops, T, E, k, d)
    dout = synth.make_normal_bf16((T, d), 6, "cuda")
    M = row_id.shape[0]
    dy = torch.full((M, d), 9.0, dtype=torch.bfloat16, device="cuda")
    dy, dw = ops.moe_combine_bwd(dout, y, slot_of, w, row_id, gofs, E, dy_perm=dy)
    torch.cuda.synchronize()
    Rp = int(gofs[-1].item())
    rdy, rdw = O.combine_bwd(to_np(dout), to_np(y), slot_of.cpu().numpy(), w.cpu().numpy(), Rp)
    assert_bf16_close(dy[:Rp], rdy, what="dy_perm")
    pad = (row_id[:Rp] < 0)
    assert torch.all(dy[:Rp][pad] == 0)
    assert torch.all(dy[Rp:] == 9.0)
    assert_fp32_close(dw, rdw, what="dw")


@pytest.mark.parametrize("score,norm", [("softmax", True), ("softmax", False), ("sigmoid", True), ("sigmoid", False)])
@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (1000, 256, 8), (64, 1024, 32)])
def test_route_bwd(ops, score, norm, T, E, k):
    sc = ops.MOE_SCORE_SOFTMAX if score == "softmax" else ops.MOE_SCORE_SIGMOID
    logits = synth.make_logits(T, E, 0, "cuda")
    idx, w, _, _ = ops.moe_route_topk(logits, k, sc, norm)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    dw = torch.randn((T, k), generator=g, device="cuda")
    dl = ops.moe_route_bwd(logits, idx, dw, sc, norm)
    torch.cuda.synchronize()
    ref = O.route_bwd(logits.cpu().numpy(), idx.cpu().numpy(), dw.cpu().numpy(), score, norm)
    got = dl.double().cpu().numpy()
    scale = np.abs(ref).max() + 1e-30
    assert np.max(np.abs(got - ref)) <= 1e-5 * scale + 1e-7
