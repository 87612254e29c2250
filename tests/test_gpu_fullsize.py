"""Full-size parity of the configurations the path is measured on.

* Mixtral-shaped layer (T = 8192, d = 4096, E = 8, top-2, f = 14336): every
  rowwise and group-aware columnwise MXFP8 code and scale byte of the four
  quantized activations of the step (x_perm, h, dy_perm, dA), against the
  oracle, over the whole tensors.
* DeepSeek-V3-shaped layer (T = 24576, d = 7168, E = 256, top-8 sigmoid,
  f = 2048), uniform and Zipf(1.2)-skewed routing: the same, on 16 whole
  groups (the largest, the smallest non-empty and 14 seeded others), all
  their rows and columns.
* The Zipf-skewed step captured once in a CUDA graph and replayed over five
  routing seeds: routing, offsets and permutation exact per seed, plus
  sampled GEMM rows, tokens and weight-gradient entries.
* Three points of the grouped-GEMM sweep (Dirichlet(0.3) group sizes, N(0,1)
  operands): sampled rows of sampled groups against the oracle's grouped
  GEMM on the GPU's own quantized operands.

The oracle's quantization of the whole tensors runs in a process pool over
the host's cores (parity_pool.py)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_bf16_close, atoms_block_range, atoms_rows_subset, atoms_to_rowmajor, bf16_bits_of,
                     colwise_scales_rowmajor, gpu_ops, tile224_block_range, to_np)
from layer_checks import sampled_checks
from parity_pool import OraclePool, bf16_bits
from grouped_gemm_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


@pytest.fixture(scope="module")
def pool():
    p = OraclePool()
    yield p
    p.close()


def _layer(ops, T, d, E, k, f, score, zipf=None):
    from grouped_gemm_top_gb300.layer import MoELayer
    L = MoELayer(T, d, E, k, f, score, True, store_intermediates=True)
    inp = synth.make_layer_inputs(T, d, E, f, "cuda", zipf_s=zipf)
    L.set_weights(inp["W1"], inp["W2"])
    del inp["W1"], inp["W2"]
    L.logits.copy_(inp["logits"])
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    return L, inp


def _routing(L, inp, score):
    """Oracle routing and permutation, checked exactly against the GPU's."""
    idx, w = O.route_topk(inp["logits"].cpu().numpy(), L.k, score, True)
    assert np.array_equal(L.topk_idx.cpu().numpy(), idx)
    assert np.max(np.abs(L.topk_w.cpu().numpy() - w)) <= 1e-6
    counts = O.group_counts(idx, L.G)
    gofs = O.aligned_group_offsets(counts, 128)
    slot_of, row_id = O.permute_slots(idx, L.G, 128)
    assert np.array_equal(L.gofs.cpu().numpy(), gofs)
    assert np.array_equal(L.slot_of.cpu().numpy(), slot_of)
    assert np.array_equal(L.row_id[:int(gofs[-1])].cpu().numpy(), row_id)
    return counts, gofs, row_id


def _quantized(L):
    """name -> (rowwise codes, rowwise scale atoms, columnwise codes, columnwise
    scales, columns, columnwise scales in the tile-224 layout) of the step's
    four quantized activations (dy_perm and dA, the weight gradients' right
    operands, carry the layer's tile-224 scales)."""
    d, f, t = L.d, L.f, L.wgrad_t224
    return {"x_perm": (L.xq, L.xs, L.xqT, L.xsT, d, False), "h": (L.hq, L.hs, L.hqT, L.hsT, f, False),
            "dy_perm": (L.dyq, L.dys, L.dyqT, L.dysT, d, t), "dA": (L.dAq, L.dAs, L.dAqT, L.dAsT, 2 * f, t)}


def test_mixtral_every_code_and_scale_both_axes(ops, pool):
    T, d, E, k, f = 8192, 4096, 8, 2, 14336
    L, inp = _layer(ops, T, d, E, k, f, "softmax")
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    counts, gofs, row_id = _routing(L, inp, "softmax")
    assert counts.sum() == T * k
    Rp, M = int(gofs[-1]), L.row_cap
    wg = L.topk_w.cpu().numpy().astype(np.float64)
    sources = {
        "x_perm": lambda: bf16_bits(O.permute(to_np(inp["x"]), row_id, k)),
        "h": lambda: bf16_bits_of(L.h[:Rp]),
        "dy_perm": lambda: bf16_bits(O.permute_scaled_bf16(to_np(inp["dout"]), row_id, k, wg)),
        "dA": lambda: bf16_bits_of(L.dA[:Rp]),
    }
    bad = []
    for name, (q, s, qT, sT, C, t224) in _quantized(L).items():
        src = sources[name]()
        assert src.shape == (Rp, C)
        bad += pool.check_both_axes(name, src, gofs, q[:Rp].cpu().numpy(),
                                    atoms_to_rowmajor(s.cpu().numpy(), M, C)[:Rp], qT[:, :Rp].cpu().numpy(),
                                    colwise_scales_rowmajor(sT.cpu().numpy(), C, M, t224)[:, :Rp // 32])
    assert not bad, bad[:8]


@pytest.mark.parametrize("zipf", [None, 1.2])
def test_deepseek_whole_groups_both_axes(ops, pool, zipf):
    T, d, E, k, f = 24576, 7168, 256, 8, 2048
    L, inp = _layer(ops, T, d, E, k, f, "sigmoid", zipf=zipf)
    L.step_()
    torch.cuda.synchronize()
    L.check_err()
    counts, gofs, row_id = _routing(L, inp, "sigmoid")
    if zipf:       # the skewed workload's shape: a dominant expert and many idle ones
        assert counts.max() > 0.2 * T and int((counts == 0).sum()) >= 30
    M = L.row_cap
    nonempty = np.nonzero(counts)[0]
    big = int(nonempty[np.argmax(counts[nonempty])])
    small = int(nonempty[np.argmin(counts[nonempty])])
    rest = np.setdiff1d(nonempty, [big, small])
    groups = [big, small] + [int(g) for g in np.random.default_rng(7).choice(rest, 14, replace=False)]
    xn, dn = to_np(inp["x"]), to_np(inp["dout"])
    wg = L.topk_w.cpu().numpy().astype(np.float64)
    quant = _quantized(L)
    atoms = {name: (s.cpu().numpy(), sT.cpu().numpy()) for name, (_, s, _, sT, _, _) in quant.items()}
    bad = []
    for g in groups:
        lo, hi = int(gofs[g]), int(gofs[g + 1])
        rid, rows = row_id[lo:hi], np.arange(lo, hi)
        sources = {
            "x_perm": lambda: bf16_bits(O.permute(xn, rid, k)),
            "h": lambda: bf16_bits_of(L.h[lo:hi]),
            "dy_perm": lambda: bf16_bits(O.permute_scaled_bf16(dn, rid, k, wg)),
            "dA": lambda: bf16_bits_of(L.dA[lo:hi]),
        }
        for name, (q, _, qT, _, C, t224) in quant.items():
            s_at, sT_at = atoms[name]
            col_sc = (tile224_block_range(sT_at, C, M, lo // 32, hi // 32) if t224
                      else atoms_block_range(sT_at, C, M, lo // 32, hi // 32))
            if t224 and L.col_sf == ops.MOE_SF_TILE224_AND_ATOMS:
                # the atom copy after the tile-224 bytes (the split weight
                # gradients' 256-wide launch reads it): the same scales
                n224 = ops.sf_bytes_tile224(C, M)
                at = atoms_block_range(sT_at[n224:], C, M, lo // 32, hi // 32)
                if not np.array_equal(at, col_sc):
                    bad.append(f"{name} group {g}: atom copy of the columnwise scales differs")
            bad += pool.check_both_axes(f"{name} group {g} ({counts[g]} rows)", sources[name](),
                                        np.array([0, hi - lo]), q[lo:hi].cpu().numpy(),
                                        atoms_rows_subset(s_at, M, C, rows), qT[:, lo:hi].cpu().numpy(), col_sc)
    assert not bad, bad[:8]


def test_zipf_step_graph_replayed_over_seeds(ops):
    """One captured graph, five routing draws: only the logits buffer
    changes, so group sizes (a dominant expert, >= 30 idle ones) change on
    the device only."""
    T, d, E, k, f = 24576, 7168, 256, 8, 2048
    L, inp = _layer(ops, T, d, E, k, f, "sigmoid", zipf=1.2)
    L.step_()
    torch.cuda.synchronize()
    L.capture()
    for seed in range(1, 6):
        logits = synth.make_logits(T, E, synth.SEED_LOGITS + seed, "cuda", 1.2)
        L.logits.copy_(logits)
        L.replay()
        torch.cuda.synchronize()
        L.check_err()
        counts = L.counts.cpu().numpy()
        assert counts.sum() == T * k and counts.max() > 0.2 * T and int((counts == 0).sum()) >= 30
        sampled_checks(L, dict(inp, logits=logits), "sigmoid", True, n_rows=48, n_groups=4, seed=seed)


@pytest.mark.parametrize("G,M_total,NK", [(256, 16384, 7168), (8, 262144, 2048), (64, 65536, 7168)])
def test_sweep_point_sampled_rows(ops, G, M_total, NK):
    """Grouped GEMM (FWD, the library's kernel choice, as the sweep times it)
    on Dirichlet(0.3) groups; for the largest, the smallest non-empty and
    four seeded other groups, 4 sampled rows each over their full
    contraction."""
    N = K = NK
    sizes = synth.dirichlet_group_sizes(G, M_total, 0.3, 0)
    gofs = np.concatenate([[0], np.cumsum((sizes + 127) // 128 * 128)])
    M = int(gofs[-1])
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    src = synth.make_normal_bf16((M_total, K), 100, "cuda")
    r = 0
    for g, m in enumerate(sizes):
        x[int(gofs[g]):int(gofs[g]) + int(m)] = src[r:r + int(m)]
        r += int(m)
    del src
    gofs_t = torch.tensor(gofs, dtype=torch.int32, device="cuda")
    xq, xs = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE, gofs_t, G)
    W = synth.make_normal_bf16((G * N, K), 200, "cuda")
    bq, bs = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
    del W
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, ops.MOE_B_GNK, gofs_t, G, M, N, K, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    nonempty = np.nonzero(sizes)[0]
    rng = np.random.default_rng(1)
    big, small = int(nonempty[np.argmax(sizes[nonempty])]), int(nonempty[np.argmin(sizes[nonempty])])
    rest = np.setdiff1d(nonempty, [big, small])
    groups = [big, small] + [int(g) for g in rng.choice(rest, min(4, len(rest)), replace=False)]
    xs_at, bs_at = xs.cpu().numpy(), bs.cpu().numpy()
    for g in groups:
        lo = int(gofs[g])
        rows = np.sort(rng.choice(np.arange(lo, lo + int(sizes[g])), min(4, int(sizes[g])), replace=False))
        rt = torch.from_numpy(rows).cuda()
        # A's codes of those rows are the oracle's, then the oracle's GEMM on them
        aq, asc = O.mxfp8_quantize_rows(to_np(x[rt]))
        assert np.array_equal(xq[rt].cpu().numpy(), aq)
        assert np.array_equal(atoms_rows_subset(xs_at, M, K, rows), asc)
        wr = np.arange(g * N, (g + 1) * N)
        Bg = O.mxfp8_dequantize_rows(bq[g * N:(g + 1) * N].cpu().numpy(), atoms_rows_subset(bs_at, G * N, K, wr))
        ref = O.mxfp8_dequantize_rows(aq, asc) @ Bg.T
        assert_bf16_close(d[rt], ref, what=f"G={G} M={M_total} N=K={NK} group {g} ({sizes[g]} rows)")
