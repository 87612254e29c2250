"""Checks of a whole MoELayer step at large sizes against the oracle: exact
routing and permutation, and sampled rows, tokens and weight-gradient
entries, each over its full contraction (the layer ran on the GPU; the
oracle works on the GPU's own stage inputs)."""
import numpy as np
import torch

import oracle as O
from helpers import assert_bf16_close, assert_fp32_close, glu_perm, to_np


def sampled_checks(L, inp, score, norm, n_rows=256, n_groups=None, seed=0):
    """Large workloads: exact routing/permute, sampled GEMM rows and
    sampled wgrad entries (each over its full contraction).  n_groups
    limits the sampled rows to that many (seeded) groups, which bounds the
    weight blocks the oracle dequantizes."""
    T, d, E, k, f, M = L.T, L.d, L.G, L.kk, L.f, L.row_cap
    rng = np.random.default_rng(seed)
    logits = inp["logits"].cpu().numpy()
    idx, w = O.route_topk(logits, L.k, score, norm)
    assert np.array_equal(L.route_idx.cpu().numpy(), idx)
    assert np.max(np.abs(L.route_w.cpu().numpy() - w)) <= 1e-6
    if L.S:
        idx, w = O.append_shared(idx, L.route_w.cpu().numpy(), L.E, L.S)
        assert np.array_equal(L.topk_idx.cpu().numpy(), idx)
    counts = O.group_counts(idx, E)
    gofs = O.aligned_group_offsets(counts, 128)
    assert np.array_equal(L.gofs.cpu().numpy(), gofs)
    slot_of, row_id = O.permute_slots(idx, E, 128)
    assert np.array_equal(L.slot_of.cpu().numpy(), slot_of)
    Rp = int(gofs[-1])
    gl = L.row_id[:Rp].cpu().numpy()
    assert np.array_equal(gl, row_id)
    valid = np.nonzero(row_id >= 0)[0]
    if n_groups is not None:
        vg = np.searchsorted(gofs, valid, side="right") - 1
        ne = np.unique(vg)
        keep = rng.choice(ne, size=min(n_groups, len(ne)), replace=False)
        valid = valid[np.isin(vg, keep)]
    rows = np.sort(rng.choice(valid, size=min(n_rows, len(valid)), replace=False))
    grp = np.searchsorted(gofs, rows, side="right") - 1
    rt = torch.from_numpy(rows).cuda()
    # permute + quantize of the sampled rows
    xp = O.permute(to_np(inp["x"]), row_id[rows], k)
    rq, rs = O.mxfp8_quantize_rows(xp)
    assert np.array_equal(L.xq[rt].cpu().numpy(), rq)
    # per sampled row: the row's group weights, fetched group by group

    def take_sf(atoms_t, rows_total, r_idx, b_lo, b_hi, tile224=False):
        r = np.asarray(r_idx)[:, None]
        b = np.arange(b_lo, b_hi)[None, :]
        if tile224:           # the tile-224 layout of the weight gradients' right operands
            T, rp = (rows_total + 223) // 224, r % 224
            off = ((b // 4) * T + r // 224) * 1024 + (rp // 128) * 512 + (rp % 32) * 16 + ((rp // 32) % 4) * 4 \
                + (b % 4)
        else:
            off = ((b // 4) * (rows_total // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
        return atoms_t[torch.from_numpy(off.reshape(-1)).cuda()].cpu().numpy().reshape(off.shape)

    def b_fwd(q, s, g, K, N, glu):   # per-expert codes [E][N][K] -> logical [K, N] of group g
        codes = q[g].cpu().numpy()
        sc = take_sf(s, E * N, np.arange(g * N, (g + 1) * N), 0, K // 32)
        deq = np.empty((N, K))
        perm = glu_perm(N) if glu else np.arange(N)
        deq[perm] = O.mxfp8_dequantize_rows(codes, sc)
        return deq.T

    def b_dgrad(q, s, g, Rw, C):  # rowwise [E*Rw, C] -> B = W_g^T [C, Rw]
        r = np.arange(g * Rw, (g + 1) * Rw)
        codes = q[g * Rw:(g + 1) * Rw].cpu().numpy()
        return O.mxfp8_dequantize_rows(codes, take_sf(s, E * Rw, r, 0, C // 32)).T

    A_rows = O.mxfp8_dequantize_rows(rq, rs)
    a_pre = np.zeros((len(rows), 2 * f))
    y = np.zeros((len(rows), d))
    hq_rows = L.hq[rt].cpu().numpy()
    h_rows = to_np(L.h[rt])
    hq_ref, hs_ref = O.mxfp8_quantize_rows(h_rows)
    assert np.array_equal(hq_rows, hq_ref)
    Hd = O.mxfp8_dequantize_rows(hq_ref, hs_ref)
    wall = L.topk_w.cpu().numpy().astype(np.float64)
    dq_ref, ds_ref = O.mxfp8_quantize_rows(O.permute_scaled_bf16(to_np(inp["dout"]), row_id[rows], k, wall))
    assert np.array_equal(L.dyq[rt].cpu().numpy(), dq_ref)
    DYd = O.mxfp8_dequantize_rows(dq_ref, ds_ref)
    daq_ref, das_ref = O.mxfp8_quantize_rows(to_np(L.dA[rt]))
    assert np.array_equal(L.dAq[rt].cpu().numpy(), daq_ref)
    DAd = O.mxfp8_dequantize_rows(daq_ref, das_ref)
    dH = np.zeros((len(rows), f))
    dxp = np.zeros((len(rows), d))
    for g in np.unique(grp):
        sel = grp == g
        a_pre[sel] = A_rows[sel] @ b_fwd(L.W1f, L.W1f_s, g, d, 2 * f, True)
        y[sel] = Hd[sel] @ b_fwd(L.W2f, L.W2f_s, g, f, d, False)
        dH[sel] = DYd[sel] @ b_dgrad(L.W2d, L.W2d_s, g, f, d)
        dxp[sel] = DAd[sel] @ b_dgrad(L.W1d, L.W1d_s, g, d, 2 * f)
    assert_bf16_close(L.a_pre[rt], a_pre, what="a_pre rows")
    assert_bf16_close(L.h[rt], O.swiglu(a_pre), what="h rows")
    assert_bf16_close(L.y_perm[rt], y, what="y_perm rows")
    assert_fp32_close(L.dH[rt], dH, what="dH rows")
    assert_bf16_close(L.dA[rt], O.swiglu_bwd(to_np(L.a_pre[rt]), dH), what="dA rows")
    assert_bf16_close(L.dx_perm[rt], dxp, what="dx_perm rows")
    # combine + combine bwd on sampled tokens
    tok = np.sort(rng.choice(T, size=min(256, T), replace=False))
    need = np.unique(slot_of[tok].reshape(-1))          # rows those tokens read
    sl = np.searchsorted(need, slot_of[tok])            # slots into the compact row set
    need_t = torch.from_numpy(need).cuda()
    tok_t = torch.from_numpy(tok).cuda()
    ysub = to_np(L.y_perm[need_t])
    wg = L.topk_w.cpu().numpy().astype(np.float64)[tok]
    assert_bf16_close(to_np(L.out[tok_t]), O.combine(ysub, sl, wg), what="out tokens")
    _, rdw = O.combine_bwd(to_np(L.dout[tok_t]), ysub, sl, wg, len(need))
    assert_fp32_close(L.dw.double().cpu().numpy()[tok], rdw[:, :L.k], what="dw tokens")
    assert_bf16_close(to_np(L.dx[tok_t]), O.combine(to_np(L.dx_perm[need_t]), sl, None), what="dx tokens")
    # wgrad: sampled (g, m, n) entries over the full group contraction
    nonempty = np.nonzero(counts)[0]
    for which in (2, 1):
        if which == 2:
            aT, asT, bT, bsT, Mo, No, dW = L.hqT, L.hsT, L.dyqT, L.dysT, f, d, L.dW2
        else:
            aT, asT, bT, bsT, Mo, No, dW = L.xqT, L.xsT, L.dAqT, L.dAsT, d, 2 * f, L.dW1
        # the largest group always (under skew it runs on the 256-wide tiles
        # of a split weight gradient), and random others
        big = int(nonempty[np.argmax(counts[nonempty])])
        gs = np.unique(np.concatenate([[big], rng.choice(nonempty, size=min(4, len(nonempty)), replace=False)]))
        for g in gs:
            lo, hi = int(gofs[g]), int(gofs[g + 1])
            ms = rng.choice(Mo, size=8, replace=False)
            ns = rng.choice(No, size=8, replace=False)
            aq = aT[torch.from_numpy(ms).cuda(), lo:hi].cpu().numpy()
            bq = bT[torch.from_numpy(ns).cuda(), lo:hi].cpu().numpy()
            asc = take_sf(asT, Mo, ms, lo // 32, hi // 32)
            bsc = take_sf(bsT, No, ns, lo // 32, hi // 32, L.wgrad_t224)
            Ah = O.mxfp8_dequantize_rows(aq, asc)      # [8, rows of g]
            Bh = O.mxfp8_dequantize_rows(bq, bsc)
            ref = Ah @ Bh.T
            got = to_np(dW[g][torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()])
            rms = np.sqrt(np.mean(ref ** 2)) + 1e-30
            assert np.all(np.abs(got - ref) <= 1e-2 * (np.abs(ref) + rms)), (which, g)
            assert np.linalg.norm(got - O.bf16_round(ref)) <= 1e-3 * np.linalg.norm(ref) + 1e-30
        empty = np.nonzero(counts == 0)[0]
        for g in empty[:3]:
            assert torch.all(dW[g] == 0)
