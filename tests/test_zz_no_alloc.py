"""moe_route_topk_noalloc: the routing entry point for callers that cannot
hand the library any device memory (plugin-style interfaces that pass only
input/output pointers, fixed memory pools, code that must not call
cudaMalloc).  It must give the same results as moe_route_topk, whose
scratch comes from a caller workspace, on consecutive calls that share the
library's fixed scratch array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from helpers import gpu_ops
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("T,E,k,score,norm", [(24576, 256, 8, 1, 1), (1000, 64, 6, 0, 0), (300, 8, 2, 0, 1)])
def test_noalloc_matches_workspace_entry_point(T, E, k, score, norm):
    ops = gpu_ops()
    lib = ops.lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):      # two calls in a row on the shared scratch array
        logits = synth.make_logits(T, E, 11 + call, "cuda")
        ridx, rw, rc, ro = ops.moe_route_topk(logits, k, score, norm)
        idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
        counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = lib.moe_route_topk_noalloc(_p(logits), T, E, k, score, norm, _p(idx), _p(w), _p(counts), _p(offsets),
                                        _p(err), stream)
        assert st == ops.MOE_OK, ops.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(idx, ridx)
        assert torch.equal(counts, rc) and torch.equal(offsets, ro)
        assert int(offsets[-1].item()) == T * k
        assert np.max(np.abs(w.cpu().numpy() - rw.cpu().numpy())) <= 1e-6


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ops = gpu_ops()
    T, E, k = 131073, 256, 8                     # ceil(T/128) * E = 262400 > 262144
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = ops.lib.moe_route_topk_noalloc(_p(dummy), T, E, k, 0, 1, _p(dummy), _p(dummy), _p(dummy), _p(dummy), None,
                                        None)
    assert st == ops.MOE_ERR_WORKSPACE
