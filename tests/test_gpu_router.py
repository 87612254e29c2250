"""Router path on the GPU vs the oracle: the bf16 tcgen05 GEMM (logits,
router backward), the bf16 transpose, the combine with an fp32 addend, and
the tiny layer with its router stage by stage."""
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


@pytest.mark.parametrize("M,N,K", [(128, 8, 512), (256, 256, 7168), (384, 520, 200), (1024, 4096, 256),
                                   (128, 64, 8)])
def test_gemm_bf16_nt(ops, M, N, K):
    """D = A B^T in fp32 from bf16 operands: any N % 8 (columns past N not
    stored), K % 8 (the last 64-element step zero-filled)."""
    a = synth.make_normal_bf16((M, K), 11, "cuda")
    b = synth.make_normal_bf16((N, K), 12, "cuda")
    d = ops.gemm_bf16_nt(a, b)
    torch.cuda.synchronize()
    assert_fp32_close(d, to_np(a) @ to_np(b).T, what="gemm_bf16_nt")


def test_gemm_bf16_nt_leaves_neighbours(ops):
    """Rows of D are N wide: nothing past column N of a row is written."""
    M, N, K = 128, 16, 64
    a = synth.make_normal_bf16((M, K), 13, "cuda")
    b = synth.make_normal_bf16((N, K), 14, "cuda")
    buf = torch.full((M * N + 64,), -7.0, dtype=torch.float32, device="cuda")
    ops.gemm_bf16_nt(a, b, buf[:M * N].view(M, N))
    torch.cuda.synchronize()
    assert torch.all(buf[M * N:] == -7.0)
    assert_fp32_close(buf[:M * N].view(M, N), to_np(a) @ to_np(b).T, what="gemm")


@pytest.mark.parametrize("rows,cols", [(256, 7168), (100, 37), (24576, 8)])
def test_transpose_exact(ops, rows, cols):
    xb = synth.make_normal_bf16((rows, cols), 15, "cuda")
    assert torch.equal(ops.moe_transpose_bf16(xb), xb.t().contiguous())
    xf = torch.randn((rows, cols), device="cuda") * 100
    assert torch.equal(ops.moe_transpose_bf16(xf), xf.t().contiguous().to(torch.bfloat16))


def test_combine_add(ops):
    T, E, k, d = 512, 8, 2, 256
    logits = synth.make_logits(T, E, 0, "cuda")
    idx, w, _, _ = ops.moe_route_topk(logits, k)
    gofs, slot_of, row_id, _ = ops.moe_permute(None, idx, E, want_x_perm=False)
    y = synth.make_normal_bf16((row_id.shape[0], d), 16, "cuda")
    add = torch.randn((T, d), device="cuda") * 4
    out = ops.moe_unpermute_combine_add(y, slot_of, w, add)
    torch.cuda.synchronize()
    ref = O.combine(to_np(y), slot_of.cpu().numpy(), w.double().cpu().numpy()) + add.double().cpu().numpy()
    assert_bf16_close(out, ref, what="combine + addend")


@pytest.mark.parametrize("score,S", [("softmax", 0), ("sigmoid", 0), ("sigmoid", 1)])
def test_tiny_layer_with_router_stagewise(ops, score, S):
    """logits = x W_r on the GPU (fp32, against the oracle on the same bf16
    operands), routing from the GPU's logits bit-exact (with S shared
    experts appended), the router backward from the GPU's dlogits, and
    dx = dx_moe + dx_r."""
    from grouped_gemm_top_gb300.layer import MoELayer
    T, d, E, k, f = 256, 512, 8, 2, 256
    L = MoELayer(T, d, E, k, f, score, True, router=True, n_shared=S)
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", n_shared=S)
    L.set_weights(inp["W1"], inp["W2"])
    Wr = synth.make_normal_bf16((d, E), 21, "cuda", std=0.05)
    L.set_router_weights(Wr)
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    x, Wn = to_np(inp["x"]), to_np(Wr)
    assert_fp32_close(L.logits, O.router_logits(x, Wn), what="logits")
    logits = L.logits.cpu().numpy()
    idx, w = O.route_topk(logits, k, score, True)
    assert np.array_equal(L.route_idx.cpu().numpy(), idx)
    idx_all, _ = O.append_shared(idx, w, E, S)
    assert np.array_equal(L.topk_idx.cpu().numpy(), idx_all)
    dl = L.dlogits.double().cpu().numpy()
    dx_r, dWr = O.router_backward(x, Wn, dl)
    assert_fp32_close(L.dx_r, dx_r, what="dx_r")
    assert_fp32_close(L.dWr, dWr, what="dW_r")
    slot_of = L.slot_of.cpu().numpy()
    Rp = int(L.gofs[-1].item())
    ref_dx = O.combine(to_np(L.dx_perm)[:Rp], slot_of, None) + L.dx_r.double().cpu().numpy()
    assert_bf16_close(L.dx, ref_dx, what="dx = dx_moe + dx_r")


def test_pipelined_steps_with_router_and_shared_expert_match_single_steps(ops):
    """run_pipelined (three graphs per buffer set: forward, backward to dx and
    dlogits, dW1) on the layer with its router and a shared expert returns
    for every step what step() returns for that batch alone."""
    from grouped_gemm_top_gb300.layer import MoELayer
    T, d, E, k, f, S = 256, 512, 8, 2, 256, 1
    L = MoELayer(T, d, E, k, f, "sigmoid", True, router=True, n_shared=S)
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", n_shared=S)
    L.set_weights(inp["W1"], inp["W2"])
    L.set_router_weights(synth.make_normal_bf16((d, E), 21, "cuda", std=0.05))
    batches, refs = [], []
    for i in range(4):
        x = synth.make_normal_bf16((T, d), 400 + i, "cuda").cpu().pin_memory()
        logits = torch.zeros((T, E), dtype=torch.float32).pin_memory()      # the router computes them
        dout = synth.make_normal_bf16((T, d), 500 + i, "cuda").cpu().pin_memory()
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
