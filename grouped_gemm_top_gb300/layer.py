"""MoELayer: the dropless-MoE fwd+bwd step as a fixed sequence of libmoe calls.

Every buffer is allocated once, sized from (T, d, E, k, f) and the static row
capacity, so the step allocates nothing, never reads counts on the host and
can be captured in one CUDA graph ([TE-JAX] "What specialized optimizations
are required for dropless MoE?": shapes must work while invisible to the CPU,
to enable CUDA graphs).  The step follows [TE-JAX] Figure 3 (route, dispatch,
two grouped GEMMs, combine) plus its backward.
"""
from __future__ import annotations

import torch

from . import ops

_SCORES = {"softmax": ops.MOE_SCORE_SOFTMAX, "sigmoid": ops.MOE_SCORE_SIGMOID}

# When the weight gradients use 224-wide tiles, only the groups with
# lo <= rows < hi (padded rows; hi = 0: no upper bound) do; the others take
# 256 x 256 tiles in a second launch (MoELayer wgrad224_rows).  Measured on
# the DeepSeek-V3 step: balanced routing (every group 640-896 rows) runs as
# with 224-wide tiles throughout; Zipf(1.2)-skewed routing, whose few large
# groups want the full-width MMA and whose many small ones the fewer, wider
# tiles, 28.25-28.28 ms against 29.10-29.16 ms (all 224) and 28.15-28.34 ms
# (all 256).
WGRAD224_ROWS = (512, 4096)


def wgrad_band_filters(lo, hi):
    """The weight-gradient group filters (moe_gemm_opts_t wgrad_rows_lo,
    wgrad_rows_hi) of the 224-wide launch over the groups of lo <= rows < hi
    (hi = 0: no upper bound) and of the 256-wide launch over all the others."""
    return (lo, hi), ((hi, lo) if hi else (0, lo))


class MoELayer:
    def __init__(self, T, d, E, k, f, score="softmax", normalize=True, device="cuda:0", store_intermediates=False,
                 router=False, n_shared=0, row_cap=None, wgrad_tiles=None, wgrad224_rows=None):
        """store_intermediates: also write h and dA in bf16 (the step itself
        only needs their MXFP8 codes, which the up/gate GEMM's epilogue and
        the fused SwiGLU-backward quantization produce).
        router: the step starts from x alone: logits = x W_r with a bf16
        router weight W_r [d, E] (set_router_weights), and the backward adds
        the router's input gradient to dx and computes dW_r [d, E] (fp32).
        n_shared: S shared experts that every token uses with weight 1
        ([CH1] §2.3.2, DeepSeek-V3's shared expert).  They are expert groups
        E .. E+S-1 of the same grouped GEMMs (weights [E+S, ...]), entered as
        S extra choices per token, so the layer runs G = E+S groups over
        T (k+S) rows; the router and its logits cover the E routed experts.
        wgrad_tiles: 224 or 256 forces the weight-gradient GEMMs' pair-tile
        width; None chooses (see below).
        wgrad224_rows: (lo, hi) with 224-wide weight-gradient tiles, only
        the groups of lo <= rows < hi (hi = 0: no upper bound) use them, the
        others 256-wide tiles in a second launch per weight gradient (the
        device picks the groups from the step's offsets); (0, 0) = every
        group on the 224-wide tiles; None = WGRAD224_ROWS."""
        self.T, self.d, self.E, self.k, self.f = T, d, E, k, f
        self.S = int(n_shared)
        self.G, self.kk = E + self.S, k + self.S      # expert groups, choices per token
        self.score = _SCORES[score]
        self.normalize = bool(normalize)
        self.device = torch.device(device)
        ops.moe_init(self.device.index or 0)
        self.R = T * self.kk
        self.row_cap = ops.moe_row_capacity(T, self.G, self.kk) if row_cap is None else int(row_cap)
        G, kk = self.G, self.kk
        M, dev = self.row_cap, self.device

        def z(shape, dtype):
            return torch.zeros(shape, dtype=dtype, device=dev)

        # inputs (resident)
        self.logits = z((T, E), torch.float32)
        self.x = z((T, d), torch.bfloat16)
        self.dout = z((T, d), torch.bfloat16)
        # routing / layout
        self.err = z((1,), torch.int32)
        # route_idx / route_w: the router's top-k; topk_idx / topk_w: every
        # choice the layer computes (the top-k, then the shared experts)
        self.route_idx = z((T, k), torch.int32)
        self.route_w = z((T, k), torch.float32)
        if self.S:
            self.topk_idx = z((T, kk), torch.int32)
            self.topk_w = z((T, kk), torch.float32)
        else:
            self.topk_idx, self.topk_w = self.route_idx, self.route_w
        self.counts = z((E,), torch.int32)
        self.offsets = z((E + 1,), torch.int32)
        self.gofs = z((G + 1,), torch.int32)
        self.slot_of = z((T, kk), torch.int32)
        self.row_id = z((M,), torch.int32)
        self.ws_route = z((ops.moe_route_workspace_size(T, E),), torch.uint8)
        self.ws_perm = z((ops.moe_permute_workspace_size(T, G),), torch.uint8)
        # forward activations (x_perm and dy_perm never exist in bf16: both
        # are quantized, along both axes, straight from x and dout)
        self.xq, self.xs = z((M, d), torch.uint8), z((ops.sf_bytes(M, d),), torch.uint8)
        self.a_pre = z((M, 2 * f), torch.bfloat16)
        self.h = z((M, f), torch.bfloat16) if store_intermediates else None
        self.hq, self.hs = z((M, f), torch.uint8), z((ops.sf_bytes(M, f),), torch.uint8)
        self.y_perm = z((M, d), torch.bfloat16)
        self.out = z((T, d), torch.bfloat16)
        # backward activations
        self.dw_all = z((T, kk), torch.float32) if self.S else None
        self.dw = z((T, k), torch.float32)
        # the weight gradients' right operands (dy_perm^T, dA^T) carry their
        # scales in the tile-224 layout when both weight-gradient GEMMs can run
        # 256 x 224 pair tiles (their M = f and d multiples of 256) and the
        # groups are short on average (at most 1024 rows: eight 128-deep
        # k-steps a tile).  Two TMEM accumulators hide each short tile's
        # drain; a long contraction loses more to the narrower MMA (1/8 of
        # the tensor rate) than its single drain costs.
        can224 = d % 256 == 0 and f % 256 == 0
        if wgrad_tiles is None:
            self.wgrad_t224 = can224 and self.R <= 1024 * self.G
        elif wgrad_tiles in (224, 256):
            if wgrad_tiles == 224 and not can224:
                raise ValueError("224-wide weight-gradient tiles need d and f multiples of 256")
            self.wgrad_t224 = wgrad_tiles == 224
        else:
            raise ValueError("wgrad_tiles: None, 224 or 256")
        # Under skewed routing a few groups hold thousands of rows; their
        # long contractions run faster on the full-width 256 x 256 tiles, so
        # each weight gradient is split in two launches by group size, the
        # right operands' scales written in both layouts.
        lo, hi = WGRAD224_ROWS if wgrad224_rows is None else (int(wgrad224_rows[0]), int(wgrad224_rows[1]))
        if lo < 0 or hi < 0 or (hi and hi <= lo):
            raise ValueError("wgrad224_rows: 0 <= lo, and hi == 0 or hi > lo")
        self.wgrad_split = self.wgrad_t224 and (lo > 0 or hi > 0)
        self.wgrad224_rows = (lo, hi) if self.wgrad_split else (0, 0)
        if self.wgrad_split:
            self.col_sf = ops.MOE_SF_TILE224_AND_ATOMS
            f224, f256 = wgrad_band_filters(lo, hi)
            self.wg_224 = ops.gemm_opts(wgrad_rows=f224)
            self.wg_256 = ops.gemm_opts(wgrad_rows=f256)
        else:
            self.col_sf = ops.MOE_SF_TILE224 if self.wgrad_t224 else ops.MOE_SF_ATOMS
        self.wgrad_b = ops.MOE_B_SF_TILE224 if self.wgrad_t224 else ops.MOE_B_GNK

        def sfc(C):              # bytes of the columnwise scales of a [M, C] matrix
            return ops.col_sf_bytes(self.col_sf, M, C)

        self.dyq, self.dys = z((M, d), torch.uint8), z((ops.sf_bytes(M, d),), torch.uint8)
        self.dyqT, self.dysT = z((d, M), torch.uint8), z((sfc(d),), torch.uint8)
        self.hqT, self.hsT = z((f, M), torch.uint8), z((ops.sf_bytes(M, f),), torch.uint8)
        self.dH = z((M, f), torch.float32)
        self.dA = z((M, 2 * f), torch.bfloat16) if store_intermediates else None
        self.dAq, self.dAs = z((M, 2 * f), torch.uint8), z((ops.sf_bytes(M, 2 * f),), torch.uint8)
        self.dAqT, self.dAsT = z((2 * f, M), torch.uint8), z((sfc(2 * f),), torch.uint8)
        self.xqT, self.xsT = z((d, M), torch.uint8), z((ops.sf_bytes(M, d),), torch.uint8)
        self.dx_perm = z((M, d), torch.bfloat16)
        self.dx = z((T, d), torch.bfloat16)
        self.dlogits = z((T, E), torch.float32)
        self.dW1 = z((G, d, 2 * f), torch.bfloat16)
        self.dW2 = z((G, f, d), torch.bfloat16)
        self.router = bool(router)
        if self.router:
            assert T % 128 == 0 and d % 8 == 0 and E % 8 == 0, "router GEMMs: T % 128, d % 8, E % 8"
            self.Wr = z((d, E), torch.bfloat16)            # logits = x @ Wr
            self.WrT = z((E, d), torch.bfloat16)
            self.xT = z((d, T), torch.bfloat16)
            self.dlogitsT = z((E, T), torch.bfloat16)
            self.dlogits_bf = z((T, E), torch.bfloat16)
            self.dx_r = z((T, d), torch.float32)
            self.dWr = z((d, E), torch.float32)
        self.graph = None
        self.weights_ready = False
        # when a list, every grouped-GEMM launch of a step appends a pair of
        # CUDA events recorded around it on the current stream
        self.gemm_events = None
        self.router_events = None      # the same for the router's GEMMs
        # when a dict, the memory-bound launches of a step (quantizations,
        # combines) append their event pairs under their names
        self.mem_events = None

    # ------------------------------------------------------------ weights --
    def set_weights(self, W1, W2):
        """Quantize bf16 W1 [G, d, 2f] and W2 [G, f, d] along both axes (done
        once per weight update, outside the step; G = E + n_shared, the
        shared experts last)."""
        E, d, f = self.G, self.d, self.f
        dev = self.device
        W1v = W1.reshape(E * d, 2 * f)
        W2v = W2.reshape(E * f, d)
        # fwd operands: blocks along the contraction axis (d for W1, f for W2),
        # stored per expert as [E][N][K] (W1's gate/up halves interleaved in
        # 64-row chunks for the SwiGLU epilogue)
        self.W1f, self.W1f_s = ops.mxfp8_group_quantize(W1v, ops.MOE_QUANT_COLWISE_BATCHED_GLU, None, E,
                                                        err=self.err)
        self.W2f, self.W2f_s = ops.mxfp8_group_quantize(W2v, ops.MOE_QUANT_COLWISE_BATCHED, None, E, err=self.err)
        # dgrad operands: blocks along the other axis (2f for W1, d for W2)
        self.W1d, self.W1d_s = ops.mxfp8_group_quantize(W1v, ops.MOE_QUANT_ROWWISE, err=self.err)
        self.W2d, self.W2d_s = ops.mxfp8_group_quantize(W2v, ops.MOE_QUANT_ROWWISE, err=self.err)
        self.weights_ready = True

    def set_router_weights(self, Wr):
        """bf16 router weight W_r [d, E] (and its transposed copy)."""
        assert self.router
        self.Wr.copy_(Wr)
        ops.moe_transpose_bf16(self.Wr, self.WrT)

    def _timed(self, fn, *args):
        if self.gemm_events is None:
            return fn(*args)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        r = fn(*args)
        e.record()
        self.gemm_events.append((s, e))
        return r

    def _mem(self, name, fn, *args, **kw):
        if self.mem_events is None:
            return fn(*args, **kw)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        r = fn(*args, **kw)
        e.record()
        self.mem_events.setdefault(name, []).append((s, e))
        return r

    def _gemm(self, *args):
        return self._timed(ops.grouped_gemm_mxfp8, *args)

    def _router_gemm(self, *args):
        if self.router_events is None:
            return ops.gemm_bf16_nt(*args)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        r = ops.gemm_bf16_nt(*args)
        e.record()
        self.router_events.append((s, e))
        return r

    def _gemm_swiglu_quant(self, *args):
        return self._timed(ops.grouped_gemm_mxfp8_swiglu_quant, *args)

    def _wgrad(self, a, a_sf, b, b_sf, Mo, No, d_out):
        """d_out[g] = A_g B_g^T over each group's rows (one timed launch, or
        the 224-wide launch over the groups in the wgrad224_rows band and the
        256-wide one over the rest, under a single pair of events)."""
        E, K, err = self.G, self.row_cap, self.err
        if not self.wgrad_split:
            return self._gemm(ops.MOE_GEMM_WGRAD, a, a_sf, b, b_sf, self.wgrad_b, self.gofs, E, Mo, No, K,
                              ops.MOE_EPI_NONE, None, d_out, None, err)
        n224 = ops.sf_bytes_tile224(No, K)

        def both():
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, a, a_sf, b, b_sf[:n224], ops.MOE_B_SF_TILE224, self.gofs, E,
                                   Mo, No, K, ops.MOE_EPI_NONE, None, d_out, None, err, opts=self.wg_224)
            ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, a, a_sf, b, b_sf[n224:], ops.MOE_B_GNK, self.gofs, E,
                                   Mo, No, K, ops.MOE_EPI_NONE, None, d_out, None, err, opts=self.wg_256)
        return self._timed(both)

    # ------------------------------------------------------------- step ----
    def route_permute_(self):
        """Router GEMM (if any), top-k routing, shared choices (if any) and
        the permutation: gofs, slot_of and row_id of the step."""
        err = self.err
        if self.router:      # logits = x W_r (bf16 operands, fp32 logits)
            self._router_gemm(self.x, self.WrT, self.logits, err)
        ops.moe_route_topk(self.logits, self.k, self.score, self.normalize, self.route_idx, self.route_w,
                           self.counts, self.offsets, self.ws_route, err)
        if self.S:
            ops.moe_route_append_shared(self.route_idx, self.route_w, self.E, self.S, self.topk_idx, self.topk_w)
        ops.moe_permute(self.x, self.topk_idx, self.G, self.row_cap, self.gofs, self.slot_of, self.row_id, None,
                        False, self.ws_perm, err)

    def forward_(self):
        E, k, d, f, M = self.G, self.kk, self.d, self.f, self.row_cap
        err = self.err
        self.route_permute_()
        # x_perm = x[row_id // k], both axes: rowwise for the up GEMM, the
        # columnwise copy for the dW1 wgrad of the backward
        self._mem("quant_x", ops.mxfp8_gather_quantize, self.x, self.gofs, E, M, self.row_id, k, None, True, True,
                  self.xq, self.xs, self.xqT, self.xsT, err)
        # up/gate GEMM; its SwiGLU epilogue writes a_pre and h's MXFP8 codes
        # on both axes (h itself only if store_h)
        self._gemm_swiglu_quant(self.xq, self.xs, self.W1f, self.W1f_s, ops.MOE_B_GNK, self.gofs, E, M, 2 * f, d,
                                self.a_pre, self.h, False, self.hq, self.hs, self.hqT, self.hsT, err)
        self._gemm(ops.MOE_GEMM_FWD, self.hq, self.hs, self.W2f, self.W2f_s, ops.MOE_B_GNK, self.gofs,
                   E, M, d, f, ops.MOE_EPI_NONE, None, self.y_perm, None, err)
        self._mem("combine_out", ops.moe_unpermute_combine, self.y_perm, self.slot_of, self.topk_w, self.out, err)

    def backward_(self):
        self.backward_outputs_()
        self.backward_dw1_()

    def backward_outputs_(self):
        """The backward up to the step's outputs dx and dlogits (and dW2):
        everything but the last weight gradient, so that dx and dlogits can
        leave the GPU while dW1 is computed."""
        E, k, d, f, M = self.G, self.kk, self.d, self.f, self.row_cap
        err = self.err
        # dw = <dout, y_perm> per (token, choice); dy_perm = w * dout is only
        # ever materialised as its MXFP8 codes (both axes)
        dw = self.dw_all if self.S else self.dw
        self._mem("combine_bwd_dw", ops.moe_combine_bwd, self.dout, self.y_perm, self.slot_of, self.topk_w, None,
                  None, E, None, dw, err, want_dy=False)
        if self.S:       # the shared choices' weights are constants
            ops.moe_route_drop_shared(self.dw_all, self.k, self.dw)
        self._mem("quant_dy", ops.mxfp8_gather_quantize, self.dout, self.gofs, E, M, self.row_id, k, self.topk_w,
                  True, True, self.dyq, self.dys, self.dyqT, self.dysT, err, col_sf_layout=self.col_sf)
        # dH = dY W2^T (fp32)
        self._gemm(ops.MOE_GEMM_DGRAD, self.dyq, self.dys, self.W2d, self.W2d_s, ops.MOE_B_GNK,
                   self.gofs, E, M, f, d, ops.MOE_EPI_NONE_F32, None, self.dH, None, err)
        # dW2_g = H_g^T dY_g
        self._wgrad(self.hqT, self.hsT, self.dyqT, self.dysT, f, d, self.dW2)
        # dA = [dgate | dup] = SwiGLU backward of (a_pre, dH), quantized on
        # both axes in the same pass
        self._mem("swiglu_bwd_quant_dA", ops.mxfp8_swiglu_bwd_quantize, self.dH, self.a_pre, self.gofs, E, self.dA,
                  False, self.dAq, self.dAs, self.dAqT, self.dAsT, err, col_sf_layout=self.col_sf)
        # dX_perm = dA W1^T
        self._gemm(ops.MOE_GEMM_DGRAD, self.dAq, self.dAs, self.W1d, self.W1d_s, ops.MOE_B_GNK,
                   self.gofs, E, M, d, 2 * f, ops.MOE_EPI_NONE, None, self.dx_perm, None, err)
        ops.moe_route_bwd(self.logits, self.route_idx, self.dw, self.score, self.normalize, self.dlogits, err)
        if self.router:
            # dx_r = bf16(dlogits) W_r^T, dW_r = x^T bf16(dlogits); dx = dx_r + sum_j dX_perm[slot]
            ops.moe_transpose_bf16(self.dlogits, self.dlogitsT)
            ops.moe_transpose_bf16(self.dlogitsT, self.dlogits_bf)
            ops.moe_transpose_bf16(self.x, self.xT)
            self._router_gemm(self.dlogits_bf, self.Wr, self.dx_r, err)
            self._router_gemm(self.xT, self.dlogitsT, self.dWr, err)
            ops.moe_unpermute_combine_add(self.dx_perm, self.slot_of, None, self.dx_r, self.dx, err)
        else:
            self._mem("combine_dx", ops.moe_unpermute_combine, self.dx_perm, self.slot_of, None, self.dx, err)

    def backward_dw1_(self):
        """The last weight gradient, dW1_g = X_g^T dA_g."""
        self._wgrad(self.xqT, self.xsT, self.dAqT, self.dAsT, self.d, 2 * self.f, self.dW1)

    def step_(self):
        """One fwd+bwd pass over the resident inputs (no allocation, no sync)."""
        assert self.weights_ready, "set_weights() first"
        self.forward_()
        self.backward_()

    # ------------------------------------------------------ CUDA graphs ----
    def capture(self, warmup=1):
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            for _ in range(warmup):
                self.step_()
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step_()
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            self.step_()
        else:
            self.graph.replay()

    # ------------------------------------------------------- public API ----
    def step(self, x, logits, dout, out_host=None, dx_host=None, dlogits_host=None):
        """End-to-end step from host (or device) tensors: copy the inputs in,
        run fwd+bwd, copy out, dx and dlogits back.  Returns those three.
        Outputs for which a host tensor is given are copied asynchronously
        into it (pinned memory): synchronize the current stream before
        reading them; the others are returned as new CPU tensors (a
        synchronous copy)."""
        self.x.copy_(x, non_blocking=True)
        self.logits.copy_(logits, non_blocking=True)
        self.dout.copy_(dout, non_blocking=True)
        self.replay()
        outs = []
        for dev_t, host_t in ((self.out, out_host), (self.dx, dx_host), (self.dlogits, dlogits_host)):
            if host_t is None:
                outs.append(dev_t.to("cpu"))
            else:
                host_t.copy_(dev_t, non_blocking=True)
                outs.append(host_t)
        return tuple(outs)

    # ------------------------------------------- pipelined host stepping ----
    _IO = ("x", "logits", "dout", "out", "dx", "dlogits")

    def enable_pipelining(self, warmup=1, nsets=3):
        """nsets buffer sets of the step's inputs and outputs, and per set
        three CUDA graphs (forward; backward up to dx and dlogits; dW1), so
        that run_pipelined() can copy later steps' inputs in and earlier
        steps' outputs out while a step computes.  With three sets, step i's
        inputs wait for step i-3's outputs to leave, so the copies have two
        steps' compute time to finish (with two, a slow host link would have
        to move one step's outputs and the next inputs within a single
        step)."""
        if getattr(self, "_sets", None) is not None:
            return
        first = {n: getattr(self, n) for n in self._IO}
        sets = [first] + [{n: torch.zeros_like(t) for n, t in first.items()} for _ in range(nsets - 1)]
        parts = (self.forward_, self.backward_outputs_, self.backward_dw1_)
        graphs, whole = [], []
        for bufs in sets:
            for n, t in bufs.items():
                setattr(self, n, t)
            self.graph = None
            whole.append(self.capture(warmup))      # also the warm-up of this set
            gs = []
            for fn in parts:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn()
                gs.append(g)
            graphs.append(tuple(gs))
        for n, t in first.items():
            setattr(self, n, t)
        self.graph = whole[0]
        self._sets = tuple(sets)
        self._graphs = graphs
        self._h2d_stream = torch.cuda.Stream(device=self.device)
        self._d2h_stream = torch.cuda.Stream(device=self.device)

    def run_pipelined(self, batches):
        """Run one fwd+bwd step per element of `batches`, each a tuple
        (x, logits, dout, out_host, dx_host, dlogits_host) of host tensors
        (pinned, for asynchronous copies).  Step i uses buffer set i % nsets:
        its inputs are copied in on an input-copy stream (once the outputs of
        the last step that used the set have been copied out), its graphs
        run on the current stream, and its outputs are copied out on an
        output-copy stream while later work computes (the GPU's copy engines
        run both directions beside the kernels).  Within a step the forward
        waits only for x and logits (dout arrives meanwhile), out leaves
        while the backward runs, and dx and dlogits leave while dW1 is
        computed.  Returns with the current stream ordered after the last
        copy.  The weight gradients and the error word are those of the last
        step."""
        self.enable_pipelining()
        comp = torch.cuda.current_stream(self.device)
        h2d, d2h = self._h2d_stream, self._d2h_stream
        nsets = len(self._sets)
        free = [None] * nsets        # events: the set's outputs have been copied out

        def mark(stream):
            e = torch.cuda.Event()
            e.record(stream)
            return e

        for i, (x, logits, dout, out_h, dx_h, dl_h) in enumerate(batches):
            b = i % nsets
            bufs = self._sets[b]
            g_fwd, g_bwd, g_dw1 = self._graphs[b]
            with torch.cuda.stream(h2d):
                if free[b] is not None:
                    h2d.wait_event(free[b])
                bufs["logits"].copy_(logits, non_blocking=True)
                bufs["x"].copy_(x, non_blocking=True)
                fwd_in = mark(h2d)
                bufs["dout"].copy_(dout, non_blocking=True)
                bwd_in = mark(h2d)
            comp.wait_event(fwd_in)
            g_fwd.replay()
            fwd_done = mark(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(fwd_done)
                out_h.copy_(bufs["out"], non_blocking=True)
            comp.wait_event(bwd_in)
            g_bwd.replay()
            bwd_done = mark(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(bwd_done)
                dx_h.copy_(bufs["dx"], non_blocking=True)
                dl_h.copy_(bufs["dlogits"], non_blocking=True)
                free[b] = mark(d2h)
            g_dw1.replay()
        comp.wait_stream(h2d)
        comp.wait_stream(d2h)

    def check_err(self):
        v = int(self.err.item())
        if v != 0:
            raise ops.MoEError("device", v)

    def flops_per_step(self):
        return 18.0 * self.R * self.d * self.f
