"""Library utilities on the GPU: the scale-layout conversion (against the
test-side reading of the atom layout and the oracle's canonical scales),
the workspace dispatcher driving a routing + permute, and the write-only
fill used to measure the write ceiling."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import atoms_to_rowmajor, gpu_ops, to_np
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 640), (1024, 7168)])
def test_scale_layout_round_trip(ops, rows, cols):
    x = synth.make_normal_bf16((rows, cols), 3, "cuda")
    q, s = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE)
    canon = ops.mxfp8_scale_layout(s, rows, cols, to_canonical=True)
    torch.cuda.synchronize()
    got = canon.cpu().numpy().reshape(rows, cols // 32)
    assert np.array_equal(got, atoms_to_rowmajor(s.cpu().numpy(), rows, cols))
    # the canonical scales are the oracle's own scale bytes
    _, rs = O.mxfp8_quantize_rows(to_np(x))
    assert np.array_equal(got, rs)
    back = ops.mxfp8_scale_layout(canon, rows, cols, to_canonical=False)
    torch.cuda.synchronize()
    assert torch.equal(back, s)


def test_workspace_size_drives_route_and_permute(ops):
    T, d, E, k, f = 1000, 256, 64, 6, 128
    ws_r = torch.empty(ops.moe_workspace_size(ops.MOE_OP_ROUTE_TOPK, T, d, E, k, f), dtype=torch.uint8, device="cuda")
    ws_p = torch.empty(ops.moe_workspace_size(ops.MOE_OP_PERMUTE, T, d, E, k, f), dtype=torch.uint8, device="cuda")
    for op in (ops.MOE_OP_GROUP_QUANTIZE, ops.MOE_OP_GATHER_QUANTIZE, ops.MOE_OP_GROUPED_GEMM,
               ops.MOE_OP_UNPERMUTE_COMBINE, ops.MOE_OP_COMBINE_BWD, ops.MOE_OP_ROUTE_BWD):
        assert ops.moe_workspace_size(op, T, d, E, k, f) == 0
    logits = synth.make_logits(T, E, 0, "cuda")
    x = synth.make_normal_bf16((T, d), 1, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, _, _, _ = ops.moe_route_topk(logits, k, ws=ws_r, err=err)
    gofs, slot_of, _, _ = ops.moe_permute(x, idx, E, ws=ws_p, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ridx, _ = O.route_topk(logits.cpu().numpy(), k, "softmax", True)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    r_slot, _ = O.permute_slots(ridx, E, align=128)
    assert np.array_equal(slot_of.cpu().numpy(), r_slot)


@pytest.mark.parametrize("method", [0, 1])
@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (32 << 20) + 32768 + 16])
def test_hbm_fill(ops, method, nbytes):
    buf = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    ops.moe_hbm_fill(buf[:nbytes], 0xA5C3E1F0, method)
    torch.cuda.synchronize()
    words = buf[:nbytes].view(torch.int32).cpu().numpy().view(np.uint32)
    assert np.all(words == 0xA5C3E1F0)
    assert torch.all(buf[nbytes:] == 0)            # nothing past the buffer
