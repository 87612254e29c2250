"""The whole layer (MoELayer: fwd + bwd) stage by stage against the oracle,
CUDA-graph replay, and the larger workloads on sampled rows."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_bf16_close, assert_fp32_close, atoms_to_rowmajor, batched_weight_operand,
                     colwise_scales_rowmajor, glu_perm, gpu_ops, to_np)
from layer_checks import sampled_checks
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def _layer(ops, T, d, E, k, f, score, norm, zipf=None, seed_offset=0, n_shared=0):
    from grouped_gemm_top_gb300.layer import MoELayer
    L = MoELayer(T, d, E, k, f, score, norm, store_intermediates=True, n_shared=n_shared)
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", zipf_s=zipf, seed_offset=seed_offset, n_shared=n_shared)
    L.set_weights(inp["W1"], inp["W2"])
    L.logits.copy_(inp["logits"])
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    return L, inp


def _w_fwd(L, which):
    """Oracle B [G, K, N] from the fwd weight operand (columnwise codes)."""
    E, d, f = L.G, L.d, L.f
    if which == 1:
        q, s, K, N = L.W1f, L.W1f_s, d, 2 * f
    else:
        q, s, K, N = L.W2f, L.W2f_s, f, d
    # per-expert operands [E][N][K] (W1: gate/up interleaved rows)
    return batched_weight_operand(q.cpu().numpy(), s.cpu().numpy(), E, N, K, glu=(which == 1))


def _w_dgrad(L, which):
    """Oracle B [G, K, N] for dgrad from the rowwise weight copy."""
    E, d, f = L.G, L.d, L.f
    if which == 1:     # dXp = dA W1^T: B_g = W1_g^T, [2f, d]
        q, s, R, C = L.W1d, L.W1d_s, E * d, 2 * f
        W = O.mxfp8_dequantize_rows(q.cpu().numpy(), atoms_to_rowmajor(s.cpu().numpy(), R, C)).reshape(E, d, 2 * f)
    else:              # dH = dY W2^T: B_g = W2_g^T, [d, f]
        q, s, R, C = L.W2d, L.W2d_s, E * f, d
        W = O.mxfp8_dequantize_rows(q.cpu().numpy(), atoms_to_rowmajor(s.cpu().numpy(), R, C)).reshape(E, f, d)
    return np.transpose(W, (0, 2, 1))


def _deq_act(q, s, M, C):
    return O.mxfp8_dequantize_rows(q.cpu().numpy(), atoms_to_rowmajor(s.cpu().numpy(), M, C))


def _deq_actT(q, s, C, M, Rp, tile224=False):
    sc = colwise_scales_rowmajor(s.cpu().numpy(), C, M, tile224)
    return O.mxfp8_dequantize_cols(q.cpu().numpy()[:, :Rp], sc[:, :Rp // 32])


@pytest.mark.parametrize("score,norm,S,T,E0,k0", [("softmax", True, 0, 256, 8, 2), ("sigmoid", True, 0, 256, 8, 2),
                                                 ("softmax", True, 1, 256, 8, 2), ("sigmoid", True, 2, 256, 8, 2),
                                                 ("softmax", False, 0, 1000, 5, 3), ("sigmoid", True, 1, 77, 6, 4),
                                                 ("softmax", True, 0, 256, 4, 4), ("sigmoid", False, 0, 300, 1, 1)])
def test_tiny_layer_stagewise(ops, score, norm, S, T, E0, k0):
    """Small dropless layers (d=512, f=256; T tokens, E0 routed experts,
    top-k0, S shared experts; T=1000 and T=77 give ragged groups and a
    token count that is not a multiple of any tile; k = E sends every token
    to every expert; E = k = 1 is a dense FFN): every stage of fwd and bwd
    against the oracle applied to the GPU's own stage inputs."""
    d, f = 512, 256
    L, inp = _layer(ops, T, d, E0, k0, f, score, norm, n_shared=S)
    E, k = E0 + S, k0 + S          # expert groups and choices per token
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    M = L.row_cap
    logits = inp["logits"].cpu().numpy()
    idx0, w0 = O.route_topk(logits, k0, score, norm)
    assert np.array_equal(L.route_idx.cpu().numpy(), idx0)
    assert np.max(np.abs(L.route_w.cpu().numpy() - w0)) <= 1e-6
    idx, w = O.append_shared(idx0, L.route_w.cpu().numpy(), E0, S)
    assert np.array_equal(L.topk_idx.cpu().numpy(), idx)
    assert np.array_equal(L.topk_w.cpu().numpy(), w)
    slot_of, row_id = O.permute_slots(idx, E, 128)
    gofs = O.aligned_group_offsets(O.group_counts(idx, E), 128)
    Rp = int(gofs[-1])
    assert np.array_equal(L.gofs.cpu().numpy(), gofs)
    assert np.array_equal(L.slot_of.cpu().numpy(), slot_of)
    assert np.array_equal(L.row_id.cpu().numpy()[:Rp], row_id)
    # x_perm (never stored) quantized along both axes straight from x
    xp = O.permute(to_np(inp["x"]), row_id, k)
    rq, rs = O.mxfp8_quantize_rows(xp)
    assert np.array_equal(L.xq.cpu().numpy()[:Rp], rq)
    assert np.array_equal(atoms_to_rowmajor(L.xs.cpu().numpy(), M, d)[:Rp], rs)
    xcq, xcs, _ = O.mxfp8_quantize_cols_grouped(xp, gofs)
    assert np.array_equal(L.xqT.cpu().numpy()[:, :Rp], xcq)
    assert np.array_equal(atoms_to_rowmajor(L.xsT.cpu().numpy(), d, M)[:, :Rp // 32], xcs)
    # up/gate GEMM + SwiGLU
    A = O.grouped_gemm(O.mxfp8_dequantize_rows(rq, rs), _w_fwd(L, 1), gofs)
    assert_bf16_close(L.a_pre[:Rp], A, what="a_pre")
    assert_bf16_close(L.h[:Rp], O.swiglu(A), what="h")
    # h quantized from the GPU's bf16 h
    hq, hs = O.mxfp8_quantize_rows(to_np(L.h)[:Rp])
    assert np.array_equal(L.hq.cpu().numpy()[:Rp], hq)
    Y = O.grouped_gemm(O.mxfp8_dequantize_rows(hq, hs), _w_fwd(L, 2), gofs)
    assert_bf16_close(L.y_perm[:Rp], Y, what="y_perm")
    wg = L.topk_w.cpu().numpy().astype(np.float64)
    assert_bf16_close(L.out, O.combine(to_np(L.y_perm)[:Rp], slot_of, wg), what="out")
    # ---- backward
    dy, dw = O.combine_bwd(to_np(inp["dout"]), to_np(L.y_perm)[:Rp], slot_of, wg, Rp)
    if S:
        assert_fp32_close(L.dw_all, dw, what="dw (every choice)")
        dw = dw[:, :k0]
    assert_fp32_close(L.dw, dw, what="dw")
    # dy_perm (never stored) = bf16(fp32(w * dout)), quantized both ways
    dyg = O.permute_scaled_bf16(to_np(inp["dout"]), row_id, k, wg)
    assert_bf16_close(dyg, dy, what="dy_perm")
    dq, ds = O.mxfp8_quantize_rows(dyg)
    assert np.array_equal(L.dyq.cpu().numpy()[:Rp], dq)
    dcq, dcs, _ = O.mxfp8_quantize_cols_grouped(dyg, gofs)
    assert np.array_equal(L.dyqT.cpu().numpy()[:, :Rp], dcq)
    assert np.array_equal(colwise_scales_rowmajor(L.dysT.cpu().numpy(), d, M, L.wgrad_t224)[:, :Rp // 32], dcs)
    dH = O.grouped_gemm(O.mxfp8_dequantize_rows(dq, ds), _w_dgrad(L, 2), gofs)
    assert_fp32_close(L.dH[:Rp], dH[:Rp], what="dH")
    dA = O.swiglu_bwd(to_np(L.a_pre)[:Rp], dH)
    assert_bf16_close(L.dA[:Rp], dA, what="dA")
    # wgrad dW2 = h^T dy per group (columnwise operands)
    Hh = _deq_actT(L.hqT, L.hsT, f, M, Rp)
    DYh = _deq_actT(L.dyqT, L.dysT, d, M, Rp, L.wgrad_t224)
    rq2, rs2, _ = O.mxfp8_quantize_cols_grouped(to_np(L.h)[:Rp], gofs)
    assert np.array_equal(L.hqT.cpu().numpy()[:, :Rp], rq2)
    dW2 = O.grouped_gemm_wgrad(Hh, DYh, gofs)
    for g in range(E):
        assert_bf16_close(L.dW2[g], dW2[g], what=f"dW2[{g}]")
    daq, das = O.mxfp8_quantize_rows(to_np(L.dA)[:Rp])
    assert np.array_equal(L.dAq.cpu().numpy()[:Rp], daq)
    dacq, dacs, _ = O.mxfp8_quantize_cols_grouped(to_np(L.dA)[:Rp], gofs)
    assert np.array_equal(L.dAqT.cpu().numpy()[:, :Rp], dacq)
    assert np.array_equal(colwise_scales_rowmajor(L.dAsT.cpu().numpy(), 2 * f, M, L.wgrad_t224)[:, :Rp // 32], dacs)
    dXp = O.grouped_gemm(O.mxfp8_dequantize_rows(daq, das), _w_dgrad(L, 1), gofs)
    assert_bf16_close(L.dx_perm[:Rp], dXp, what="dx_perm")
    Xh = _deq_actT(L.xqT, L.xsT, d, M, Rp)
    DAh = _deq_actT(L.dAqT, L.dAsT, 2 * f, M, Rp, L.wgrad_t224)
    dW1 = O.grouped_gemm_wgrad(Xh, DAh, gofs)
    for g in range(E):
        assert_bf16_close(L.dW1[g], dW1[g], what=f"dW1[{g}]")
    assert_bf16_close(L.dx, O.combine(to_np(L.dx_perm)[:Rp], slot_of, None), what="dx")
    dl = O.route_bwd(logits, idx0, L.dw.double().cpu().numpy(), score, norm)
    got = L.dlogits.double().cpu().numpy()
    assert np.max(np.abs(got - dl)) <= 1e-5 * (np.abs(dl).max() + 1e-30) + 1e-7


def test_graph_replay_matches_eager(ops):
    T, d, E, k, f = 256, 512, 8, 2, 256
    L, inp = _layer(ops, T, d, E, k, f, "softmax", True)
    L.step_()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (L.out, L.dx, L.dlogits, L.dW1, L.dW2)]
    L.capture()
    # new inputs through the captured buffers, then back to the first ones
    L.logits.copy_(synth.make_logits(T, E, 5, "cuda"))
    L.replay()
    torch.cuda.synchronize()
    assert not torch.equal(L.out, ref[0])
    L.logits.copy_(inp["logits"])
    L.replay()
    torch.cuda.synchronize()
    L.check_err()
    for a, b in zip((L.out, L.dx, L.dlogits, L.dW1, L.dW2), ref):
        assert torch.equal(a, b)


def test_pipelined_steps_match_single_steps(ops):
    """run_pipelined (three sets of inputs/outputs, copies overlapping the
    other steps' kernels, every set reused) returns for every step exactly
    what step() returns for that batch alone."""
    T, d, E, k, f = 256, 512, 8, 2, 256
    L, inp = _layer(ops, T, d, E, k, f, "softmax", True)
    batches, refs = [], []
    for i in range(5):          # more steps than buffer sets: every set is reused
        x = synth.make_normal_bf16((T, d), 100 + i, "cuda").cpu().pin_memory()
        logits = synth.make_logits(T, E, 200 + i, "cuda").cpu().pin_memory()
        dout = synth.make_normal_bf16((T, d), 300 + i, "cuda").cpu().pin_memory()
        refs.append(tuple(t.clone() for t in L.step(x, logits, dout)))
        outs = (torch.empty((T, d), dtype=torch.bfloat16).pin_memory(),
                torch.empty((T, d), dtype=torch.bfloat16).pin_memory(),
                torch.empty((T, E), dtype=torch.float32).pin_memory())
        batches.append((x, logits, dout) + outs)
    L.run_pipelined(batches)
    torch.cuda.synchronize()
    L.check_err()
    for b, ref in zip(batches, refs):
        for got, want in zip(b[3:], ref):
            assert torch.equal(got, want)


@pytest.mark.parametrize("name,T,d,E,k,f,score,zipf,S", [
    ("mixtral-shaped", 8192, 4096, 8, 2, 14336, "softmax", None, 0),
    ("deepseek-v3-shaped", 24576, 7168, 256, 8, 2048, "sigmoid", None, 0),
    ("deepseek-v3-zipf", 24576, 7168, 256, 8, 2048, "sigmoid", 1.2, 0),
    ("deepseek-v3-shared-expert", 24576, 7168, 256, 8, 2048, "sigmoid", None, 1),
])
def test_large_layer_sampled(ops, name, T, d, E, k, f, score, zipf, S):
    L, inp = _layer(ops, T, d, E, k, f, score, True, zipf=zipf, n_shared=S)
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    sampled_checks(L, inp, score, True)
    del L, inp
    torch.cuda.empty_cache()


def test_wgrad_split_matches_single_launch(ops):
    """Skewed routing over 8 experts (T = 4096, top-2: groups of 256 to 3328
    padded rows): with the weight gradients split (224-wide tiles for the
    groups in the layer's WGRAD224_ROWS band, 256-wide tiles for the rest),
    the band's groups equal the single 224-wide launch's bit for bit and the
    rest within bf16 rounding; all of them against the oracle on sampled
    entries (the largest group always)."""
    from grouped_gemm_top_gb300.layer import MoELayer, WGRAD224_ROWS
    T, d, E, k, f = 4096, 512, 8, 2, 256
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", zipf_s=1.2)
    layers = []
    for band in (None, (0, 0)):
        L = MoELayer(T, d, E, k, f, "softmax", True, store_intermediates=True, wgrad224_rows=band)
        L.set_weights(inp["W1"], inp["W2"])
        L.logits.copy_(inp["logits"])
        L.x.copy_(inp["x"])
        L.dout.copy_(inp["dout"])
        L.step_()
        torch.cuda.synchronize()
        L.check_err()
        layers.append(L)
    Ls, Lu = layers
    assert Ls.wgrad_t224 and Ls.wgrad_split and Ls.wgrad224_rows == WGRAD224_ROWS and not Lu.wgrad_split
    rows = np.diff(Ls.gofs.cpu().numpy())
    assert np.array_equal(rows, np.diff(Lu.gofs.cpu().numpy()))
    lo, hi = WGRAD224_ROWS
    band = (rows >= lo) & ((rows < hi) if hi else True)
    assert band.sum() >= 2 and (~band).sum() >= 2          # both launches have work
    for a, b, name in ((Ls.dW1, Lu.dW1, "dW1"), (Ls.dW2, Lu.dW2, "dW2")):
        for g in range(E):
            if band[g]:
                assert torch.equal(a[g], b[g]), f"{name} g={g}"
            else:
                assert_bf16_close(a[g], to_np(b[g]), what=f"{name} g={g} (256-wide vs 224-wide)")
    sampled_checks(Ls, inp, "softmax", True)
