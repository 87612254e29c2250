"""The prior-art ways of running the same MoE layer, as measured comparators
for the grouped path ([TE-JAX] "How is dropless MoE different from
capacity-based MoE?" and "Optimization 1: Grouped GEMM").

LoopMoE -- one GEMM per expert with that expert's own token count.  The host
has to know the counts before it can issue the launches, so every step copies
the group offsets to the host and synchronises ([TE-JAX] "Optimization 1":
that copy is what keeps the loop out of a CUDA graph).  Each expert's
operands are quantized by their own launches (per-expert MXFP8 layouts) and
its GEMMs are single-group launches of the same kernels, so the loop gives
the grouped step's results bit for bit; what differs is the number of
launches, the host round trip and how well a GEMM of one expert's rows fills
the GPU.

CapacityMoE -- capacity-based MoE: every expert gets the same static budget
of C rows (C = capacity_factor x T k / E, rounded up to the 128-row tile),
choices beyond an expert's budget are dropped (their combine weight meets a
zero row) and unused budget rows are computed as zero padding.  Shapes are
static, so the step is graph-capturable, at the price of padded FLOPs and
dropped tokens ([TE-JAX] "How is dropless MoE different…").

Both reuse MoELayer's buffers and kernels; neither is part of the dropless
path.  Layout remapping in CapacityMoE uses plain torch index operations.
"""
from __future__ import annotations

import math

import torch

from . import ops
from .layer import MoELayer


class LoopMoE:
    """Per-expert loop over a MoELayer's buffers (no shared experts, no router
    GEMM).  set_weights() quantizes each expert's weights on its own."""

    def __init__(self, layer: MoELayer):
        assert layer.S == 0 and not layer.router, "loop comparator: routed experts only"
        self.L = layer
        dev = layer.device
        G, d, f = layer.G, layer.d, layer.f
        # single-group offsets [0, 128 j] for every possible padded count
        n = layer.row_cap // 128
        tab = torch.zeros((n + 1, 2), dtype=torch.int32)
        tab[:, 1] = 128 * torch.arange(n + 1, dtype=torch.int32)
        self.tab = tab.to(dev)
        self.gofs_host = torch.empty((G + 1,), dtype=torch.int32).pin_memory()
        u8 = torch.uint8

        def z(shape):
            return torch.zeros(shape, dtype=u8, device=dev)

        self.W1f, self.W1f_s = z((G, 2 * f, d)), z((G, ops.sf_bytes(2 * f, d)))
        self.W2f, self.W2f_s = z((G, d, f)), z((G, ops.sf_bytes(d, f)))
        self.W1d, self.W1d_s = z((G, d, 2 * f)), z((G, ops.sf_bytes(d, 2 * f)))
        self.W2d, self.W2d_s = z((G, f, d)), z((G, ops.sf_bytes(f, d)))
        self.launches = 0

    def set_weights(self, W1, W2):
        L = self.L
        for g in range(L.G):
            ops.mxfp8_group_quantize(W1[g], ops.MOE_QUANT_COLWISE_BATCHED_GLU, None, 1, self.W1f[g], self.W1f_s[g],
                                     err=L.err)
            ops.mxfp8_group_quantize(W2[g], ops.MOE_QUANT_COLWISE_BATCHED, None, 1, self.W2f[g], self.W2f_s[g],
                                     err=L.err)
            ops.mxfp8_group_quantize(W1[g], ops.MOE_QUANT_ROWWISE, None, 0, self.W1d[g], self.W1d_s[g], err=L.err)
            ops.mxfp8_group_quantize(W2[g], ops.MOE_QUANT_ROWWISE, None, 0, self.W2d[g], self.W2d_s[g], err=L.err)

    @staticmethod
    def _cols(t, s, e, c):
        """Per-expert block [c, e - s] of a flat column-major buffer."""
        return t.view(-1)[s * c:e * c].view(c, e - s)

    @staticmethod
    def _sf(t, s, e, c):
        return t[s * c // 32:e * c // 32]

    def _sfc(self, t, s, e, c):
        """Per-expert slice of a columnwise scale buffer of the layer's layout
        (tile-224: whole k-blocks of ceil(c / 224) 1024-byte tiles)."""
        if not self.L.wgrad_t224:
            return self._sf(t, s, e, c)
        tb = (c + 223) // 224 * 1024
        return t[s // 128 * tb:e // 128 * tb]

    def step_(self):
        """One fwd+bwd step: route and permute once, read the group offsets
        on the host, then per expert its quantizations and GEMMs."""
        L = self.L
        G, k, d, f, err = L.G, L.kk, L.d, L.f, L.err
        B = ops.MOE_B_GNK
        L.route_permute_()
        self.gofs_host.copy_(L.gofs, non_blocking=True)
        torch.cuda.current_stream(L.device).synchronize()
        go = self.gofs_host.tolist()
        cols, sf = self._cols, self._sf
        live = [(g, go[g], go[g + 1]) for g in range(G) if go[g + 1] > go[g]]
        for g, s, e in live:
            m, gt = e - s, self.tab[(e - s) // 128]
            ops.mxfp8_gather_quantize(L.x, gt, 1, m, L.row_id[s:e], k, None, True, True, L.xq[s:e],
                                      sf(L.xs, s, e, d), cols(L.xqT, s, e, d), sf(L.xsT, s, e, d), err)
            ops.grouped_gemm_mxfp8_swiglu_quant(L.xq[s:e], sf(L.xs, s, e, d), self.W1f[g], self.W1f_s[g], B, gt, 1,
                                                m, 2 * f, d, L.a_pre[s:e], None if L.h is None else L.h[s:e], False,
                                                L.hq[s:e], sf(L.hs, s, e, f), cols(L.hqT, s, e, f),
                                                sf(L.hsT, s, e, f), err)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, L.hq[s:e], sf(L.hs, s, e, f), self.W2f[g], self.W2f_s[g], B,
                                   gt, 1, m, d, f, ops.MOE_EPI_NONE, None, L.y_perm[s:e], None, err)
        ops.moe_unpermute_combine(L.y_perm, L.slot_of, L.topk_w, L.out, err)
        ops.moe_combine_bwd(L.dout, L.y_perm, L.slot_of, L.topk_w, None, None, G, None, L.dw, err, want_dy=False)
        for g, s, e in live:
            m, gt = e - s, self.tab[(e - s) // 128]
            dyqT, dysT = cols(L.dyqT, s, e, d), self._sfc(L.dysT, s, e, d)
            ops.mxfp8_gather_quantize(L.dout, gt, 1, m, L.row_id[s:e], k, L.topk_w, True, True, L.dyq[s:e],
                                      sf(L.dys, s, e, d), dyqT, dysT, err, col_sf_layout=L.col_sf)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_DGRAD, L.dyq[s:e], sf(L.dys, s, e, d), self.W2d[g], self.W2d_s[g],
                                   B, gt, 1, m, f, d, ops.MOE_EPI_NONE_F32, None, L.dH[s:e], None, err)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, cols(L.hqT, s, e, f), sf(L.hsT, s, e, f), dyqT, dysT, L.wgrad_b,
                                   gt, 1, f, d, m, ops.MOE_EPI_NONE, None, L.dW2[g:g + 1], None, err)
            dAqT, dAsT = cols(L.dAqT, s, e, 2 * f), self._sfc(L.dAsT, s, e, 2 * f)
            ops.mxfp8_swiglu_bwd_quantize(L.dH[s:e], L.a_pre[s:e], gt, 1, None if L.dA is None else L.dA[s:e],
                                          False, L.dAq[s:e], sf(L.dAs, s, e, 2 * f), dAqT, dAsT, err,
                                          col_sf_layout=L.col_sf)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_DGRAD, L.dAq[s:e], sf(L.dAs, s, e, 2 * f), self.W1d[g],
                                   self.W1d_s[g], B, gt, 1, m, d, 2 * f, ops.MOE_EPI_NONE, None, L.dx_perm[s:e], None,
                                   err)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, cols(L.xqT, s, e, d), sf(L.xsT, s, e, d), dAqT, dAsT,
                                   L.wgrad_b, gt, 1, d, 2 * f, m, ops.MOE_EPI_NONE, None, L.dW1[g:g + 1], None, err)
        for g in range(G):           # an expert without tokens has zero weight gradients
            if go[g + 1] == go[g]:
                L.dW1[g].zero_()
                L.dW2[g].zero_()
        ops.moe_route_bwd(L.logits, L.route_idx, L.dw, L.score, L.normalize, L.dlogits, err)
        ops.moe_unpermute_combine(L.dx_perm, L.slot_of, None, L.dx, err)
        # route (2), permute (3), combine, combine bwd, route bwd, combine
        # (dx), 3 + 6 per expert with tokens, 2 memsets per expert without
        self.launches = 9 + 9 * len(live) + 2 * (G - len(live))


def capacity_rows(T, E, k, capacity_factor):
    """Per-expert budget: capacity_factor * T k / E rows, rounded up to 128."""
    return int(math.ceil(capacity_factor * T * k / E / 128.0)) * 128


class CapacityMoE(MoELayer):
    """Capacity-based MoE on the same kernels: static groups of C rows.
    Choices beyond their expert's C rows are dropped; a zero row after the
    E C budget rows stands in for them in the combine."""

    def __init__(self, T, d, E, k, f, score="softmax", normalize=True, device="cuda:0", capacity_factor=1.25,
                 store_intermediates=False):
        self.C = capacity_rows(T, E, k, capacity_factor)
        self.capacity_factor = capacity_factor
        super().__init__(T, d, E, k, f, score, normalize, device, store_intermediates=store_intermediates,
                         row_cap=E * self.C + 128)
        dev = self.device
        cap = ops.moe_row_capacity(T, E, k)
        # the dropless layout the permute kernel produces, remapped each step
        self.gofs_dl = torch.zeros((E + 1,), dtype=torch.int32, device=dev)
        self.slot_dl = torch.zeros((T, k), dtype=torch.int32, device=dev)
        self.row_id_dl = torch.zeros((cap,), dtype=torch.int32, device=dev)
        self.gofs.copy_(self.C * torch.arange(E + 1, dtype=torch.int32, device=dev))
        self.choice = torch.arange(T * k, dtype=torch.int32, device=dev).view(T, k)
        self.dl_cap = cap

    def route_permute_(self):
        err, E, k = self.err, self.E, self.k
        ops.moe_route_topk(self.logits, k, self.score, self.normalize, self.route_idx, self.route_w,
                           self.counts, self.offsets, self.ws_route, err)
        ops.moe_permute(self.x, self.topk_idx, E, self.dl_cap, self.gofs_dl, self.slot_dl, self.row_id_dl, None,
                        False, self.ws_perm, err)
        # rank of each choice inside its expert, then its budget row (or the
        # zero row E*C when the budget is full)
        e = self.topk_idx.long()
        rank = self.slot_dl - self.gofs_dl[e]
        keep = rank < self.C
        slot = torch.where(keep, e.int() * self.C + rank, torch.full_like(rank, E * self.C))
        self.slot_of.copy_(slot)
        # row_id of every budget row: its choice, -1 for padding (dropped
        # choices all write -1 to the zero row; no host sync, capturable)
        self.row_id.fill_(-1)
        self.row_id.index_put_((slot.view(-1).long(),), torch.where(keep, self.choice, -1).view(-1))

    def dropped_fraction(self):
        """Fraction of the T k routed choices the last step dropped."""
        return float((self.slot_of == self.E * self.C).sum().item()) / (self.T * self.k)
