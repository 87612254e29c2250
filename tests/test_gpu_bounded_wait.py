"""The kernels' bounded waits end with an error status instead of hanging:
a wait on an mbarrier that nothing arrives at gives up after its limit,
reports MOE_ERR_DEVICE_TIMEOUT in the error word, and the context stays
usable for the next launches."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from helpers import gpu_ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


@pytest.mark.parametrize("timeout_ms", [5, 50])
def test_wait_on_a_barrier_nothing_arrives_at_times_out(ops, timeout_ms):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ops.moe_selftest_bounded_wait(timeout_ms * 1_000_000, err, done)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert done.item() == 0
    assert err.item() == ops.MOE_ERR_DEVICE_TIMEOUT
    assert timeout_ms * 1e-3 * 0.9 <= dt < timeout_ms * 1e-3 + 2.0


def test_context_usable_after_a_timeout(ops):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_selftest_bounded_wait(1_000_000, err, done)
    torch.cuda.synchronize()
    assert err.item() == ops.MOE_ERR_DEVICE_TIMEOUT
    # a routing launch and a grouped GEMM on the same context afterwards
    logits = torch.randn((256, 8), device="cuda")
    idx, w, counts, offsets = ops.moe_route_topk(logits, 2)
    torch.cuda.synchronize()
    ref_idx, _ = O.route_topk(logits.cpu().numpy(), 2, "softmax", True)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    x = torch.randn((256, 256), device="cuda").bfloat16()
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE)
    gofs = torch.tensor([0, 128, 256], dtype=torch.int32, device="cuda")
    W = torch.randn((2 * 256, 256), device="cuda").bfloat16()
    bq, bs = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, q, s, bq, bs, ops.MOE_B_GNK, gofs, 2, 256, 256, 256, err=err2)
    torch.cuda.synchronize()
    assert err2.item() == 0 and torch.isfinite(d.float()).all()
