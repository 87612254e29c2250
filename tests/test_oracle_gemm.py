"""Pins for the oracle's grouped GEMM (fwd / dgrad / wgrad), SwiGLU and the
whole-layer backward (CPU)."""
import numpy as np
import pytest

import oracle as O


def _triple_loop(A, B):
    M, K = A.shape
    N = B.shape[1]
    D = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = 0.0
            for kk in range(K):
                s += A[i, kk] * B[kk, j]
            D[i, j] = s
    return D


def test_grouped_gemm_brute_force_with_empty_groups():
    rng = np.random.default_rng(20)
    sizes = [3, 0, 1, 5, 0]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    A = rng.standard_normal((offs[-1] + 2, 6))        # 2 rows belong to no group
    B = rng.standard_normal((len(sizes), 6, 4))
    D = O.grouped_gemm(A, B, offs)
    for g, m in enumerate(sizes):
        lo, hi = offs[g], offs[g + 1]
        if m:
            assert np.allclose(D[lo:hi], _triple_loop(A[lo:hi], B[g]), rtol=1e-13)
    assert np.all(D[offs[-1]:] == 0)                  # no output rows outside groups


def test_all_tokens_to_one_expert_is_dense_gemm():
    rng = np.random.default_rng(21)
    A = rng.standard_normal((9, 5))
    B = rng.standard_normal((4, 5, 3))
    offs = np.array([0, 0, 0, 9, 9])                  # every row in group 2
    assert np.allclose(O.grouped_gemm(A, B, offs), _triple_loop(A, B[2]), rtol=1e-13)


def test_identity_and_permutation_weights_are_exact():
    rng = np.random.default_rng(22)
    A = np.round(rng.standard_normal((10, 8)) * 16) / 16
    P = np.eye(8)[rng.permutation(8)]
    B = np.stack([np.eye(8), P, 2.0 * np.eye(8)])
    offs = np.array([0, 4, 7, 10])
    D = O.grouped_gemm(A, B, offs)
    assert np.array_equal(D[:4], A[:4])
    assert np.array_equal(D[4:7], A[4:7] @ P)
    assert np.array_equal(D[7:], 2 * A[7:])


def test_wgrad_brute_force_and_empty_group_zero():
    rng = np.random.default_rng(23)
    sizes = [4, 0, 7]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    A = rng.standard_normal((offs[-1], 3))
    G = rng.standard_normal((offs[-1], 5))
    dB = O.grouped_gemm_wgrad(A, G, offs)
    assert dB.shape == (3, 3, 5)
    assert np.all(dB[1] == 0)
    for g in (0, 2):
        lo, hi = offs[g], offs[g + 1]
        assert np.allclose(dB[g], _triple_loop(A[lo:hi].T.copy(), G[lo:hi]), rtol=1e-13)
    one = O.grouped_gemm_wgrad(A, G, np.array([0, offs[-1]]))
    assert np.allclose(one[0], _triple_loop(A.T.copy(), G), rtol=1e-13)


def test_swiglu_special_values():
    a = np.array([[0.0, 3.0, 5.0, 0.0], [40.0, -40.0, 2.0, 3.0]])   # f = 2: [g | u]
    h = O.swiglu(a)
    assert h[0, 0] == 0.0 and h[0, 1] == 0.0          # g = 0 or u = 0
    assert np.isclose(h[1, 0], 40.0 * 2.0, rtol=1e-15)  # silu(40) ~ 40
    assert abs(h[1, 1]) < 1e-15                        # silu(-40) ~ 0
    g = 1.3
    assert np.isclose(O.swiglu(np.array([[g, 2.0]]))[0, 0], g / (1 + np.exp(-g)) * 2.0, rtol=1e-15)


def test_swiglu_bwd_finite_differences():
    rng = np.random.default_rng(24)
    a = rng.standard_normal((5, 8)) * 2
    dh = rng.standard_normal((5, 4))
    da = O.swiglu_bwd(a, dh)
    eps = 1e-6
    for i in range(5):
        for j in range(8):
            ap, am = a.copy(), a.copy()
            ap[i, j] += eps
            am[i, j] -= eps
            fd = np.sum((O.swiglu(ap) - O.swiglu(am)) * dh) / (2 * eps)
            assert np.isclose(fd, da[i, j], rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_layer_backward_finite_differences(score):
    """The whole unquantized layer: gradients of L = <out, dout> with respect
    to x, logits, W1 and W2 against central differences."""
    rng = np.random.default_rng(25)
    T, d, E, k, f = 12, 6, 4, 2, 5
    x = rng.standard_normal((T, d))
    # well separated logits so the top-k choice cannot flip under eps
    logits = np.stack([rng.permutation(E) * 1.0 for _ in range(T)]) + 0.1 * rng.standard_normal((T, E))
    W1 = rng.standard_normal((E, d, 2 * f)) * 0.5
    W2 = rng.standard_normal((E, f, d)) * 0.5
    dout = rng.standard_normal((T, d))
    out, saved = O.layer_forward(x, logits, W1, W2, k, score, True, align=1)
    g = O.layer_backward(dout, logits, W1, W2, k, saved, score, True)

    def loss(x_, l_, W1_, W2_):
        o, _ = O.layer_forward(x_, l_, W1_, W2_, k, score, True, align=1)
        return np.sum(o * dout)

    eps = 1e-6
    args = [x, logits, W1, W2]
    grads = [g["dx"], g["dlogits"], g["dW1"], g["dW2"]]
    for which in range(4):
        flat = args[which].reshape(-1)
        for pos in rng.choice(flat.size, size=min(12, flat.size), replace=False):
            p = [a.copy() for a in args]
            m = [a.copy() for a in args]
            p[which].reshape(-1)[pos] += eps
            m[which].reshape(-1)[pos] -= eps
            fd = (loss(*p) - loss(*m)) / (2 * eps)
            an = grads[which].reshape(-1)[pos]
            assert np.isclose(fd, an, rtol=1e-5, atol=1e-7), (which, pos, fd, an)


def test_layer_padding_does_not_change_results():
    rng = np.random.default_rng(26)
    T, d, E, k, f = 30, 8, 4, 2, 4
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W1 = rng.standard_normal((E, d, 2 * f))
    W2 = rng.standard_normal((E, f, d))
    dout = rng.standard_normal((T, d))
    o1, s1 = O.layer_forward(x, logits, W1, W2, k, align=1)
    o2, s2 = O.layer_forward(x, logits, W1, W2, k, align=128)
    assert np.allclose(o1, o2, rtol=1e-13)
    g1 = O.layer_backward(dout, logits, W1, W2, k, s1)
    g2 = O.layer_backward(dout, logits, W1, W2, k, s2)
    for key in ("dx", "dlogits", "dW1", "dW2"):
        assert np.allclose(g1[key], g2[key], rtol=1e-12, atol=1e-12)


def test_router_logits_by_hand_and_one_hot():
    x = np.array([[1.0, 2.0, -3.0], [0.5, 0.0, 4.0]])
    Wr = np.array([[1.0, 0.0], [0.0, 2.0], [1.0, -1.0]])
    assert np.array_equal(O.router_logits(x, Wr), np.array([[1 - 3, 4 + 3], [0.5 + 4, -4.0]]))
    # one-hot columns pick input features exactly
    rng = np.random.default_rng(3)
    xb = O.bf16_round(rng.standard_normal((16, 8)))
    pick = np.array([5, 0, 7, 2])
    oh = np.zeros((8, 4))
    oh[pick, np.arange(4)] = 1.0
    assert np.array_equal(O.router_logits(xb, oh), xb[:, pick])


def test_router_backward_adjoint_and_bf16_rounding():
    rng = np.random.default_rng(4)
    T, d, E = 12, 10, 6
    x = O.bf16_round(rng.standard_normal((T, d)))
    Wr = O.bf16_round(rng.standard_normal((d, E)))
    G = O.bf16_round(rng.standard_normal((T, E)))        # already bf16: no rounding
    dx, dW = O.router_backward(x, Wr, G)
    # <router_logits(x, W), G> = <x, dx> = <W, dW>
    v = np.sum(O.router_logits(x, Wr) * G)
    assert np.isclose(v, np.sum(x * dx), rtol=1e-12) and np.isclose(v, np.sum(Wr * dW), rtol=1e-12)
    # dlogits are rounded to bf16 before the GEMMs: 1 + 2^-9 becomes 1
    g = np.zeros((T, E))
    g[0, 0] = 1.0 + 2.0 ** -9
    dx1, _ = O.router_backward(x, Wr, g)
    assert np.array_equal(dx1[0], Wr[:, 0])


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_layer_with_router_finite_differences(score):
    """The router's gradients close the layer's chain: L(x, W_r) =
    <layer(x, router_logits(x, W_r)), dout>; dL/dx = dx_moe + dx_r and
    dL/dW_r = dW_r, checked by central differences on the unquantized fp64
    layer.  router_backward rounds dlogits to bf16 once, so the comparison
    allows that rounding (rtol 1e-2)."""
    rng = np.random.default_rng(5)
    T, d, E, k, f = 6, 8, 5, 2, 4
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((d, E)) * 0.5
    W1 = rng.standard_normal((E, d, 2 * f)) * 0.4
    W2 = rng.standard_normal((E, f, d)) * 0.4
    dout = rng.standard_normal((T, d))

    def loss(x_, Wr_):
        o, _ = O.layer_forward(x_, O.router_logits(x_, Wr_), W1, W2, k, score, True, align=1)
        return float(np.sum(o * dout))

    logits = O.router_logits(x, Wr)
    out, saved = O.layer_forward(x, logits, W1, W2, k, score, True, align=1)
    g = O.layer_backward(dout, logits, W1, W2, k, saved, score, True)
    dx_r, dWr = O.router_backward(x, Wr, g["dlogits"])
    gx, gW = g["dx"] + dx_r, dWr
    eps = 1e-6
    for (t, j) in [(0, 0), (3, 5), (5, 7)]:
        xp, xm = x.copy(), x.copy()
        xp[t, j] += eps
        xm[t, j] -= eps
        fd = (loss(xp, Wr) - loss(xm, Wr)) / (2 * eps)
        assert np.isclose(fd, gx[t, j], rtol=1e-2, atol=1e-3 * (np.abs(gx).max() + 1e-12))
    for (j, e) in [(0, 0), (4, 2), (7, 4)]:
        Wp, Wm = Wr.copy(), Wr.copy()
        Wp[j, e] += eps
        Wm[j, e] -= eps
        fd = (loss(x, Wp) - loss(x, Wm)) / (2 * eps)
        assert np.isclose(fd, gW[j, e], rtol=1e-2, atol=1e-3 * (np.abs(gW).max() + 1e-12))


def test_append_shared_by_hand():
    idx = np.array([[2, 0], [1, 3]])
    w = np.array([[0.7, 0.3], [0.6, 0.4]])
    i2, w2 = O.append_shared(idx, w, 4, 2)
    assert np.array_equal(i2, np.array([[2, 0, 4, 5], [1, 3, 4, 5]]))
    assert np.array_equal(w2, np.array([[0.7, 0.3, 1.0, 1.0], [0.6, 0.4, 1.0, 1.0]]))


def test_shared_expert_is_a_dense_ffn_added_to_the_routed_layer():
    """With S shared experts the layer's output is the routed layer's plus,
    for each shared expert, swiglu(x W1_s) W2_s on every token (computed
    here densely, with no routing or permutation)."""
    rng = np.random.default_rng(6)
    T, d, E, k, f, S = 9, 8, 5, 2, 4, 2
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E))
    W1 = rng.standard_normal((E + S, d, 2 * f)) * 0.5
    W2 = rng.standard_normal((E + S, f, d)) * 0.5
    routed, _ = O.layer_forward(x, logits, W1[:E], W2[:E], k, align=4)
    both, saved = O.layer_forward(x, logits, W1, W2, k, align=4, n_shared=S)
    dense = sum(O.swiglu(x @ W1[E + s]) @ W2[E + s] for s in range(S))
    assert np.allclose(both, routed + dense, rtol=1e-12, atol=1e-12)
    # every token is in each shared expert's group
    gofs = saved["gofs"]
    assert all(gofs[E + s + 1] - gofs[E + s] >= T for s in range(S))


def test_shared_expert_finite_differences():
    rng = np.random.default_rng(7)
    T, d, E, k, f, S = 6, 8, 4, 2, 4, 1
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E))
    W1 = rng.standard_normal((E + S, d, 2 * f)) * 0.4
    W2 = rng.standard_normal((E + S, f, d)) * 0.4
    dout = rng.standard_normal((T, d))
    out, saved = O.layer_forward(x, logits, W1, W2, k, "sigmoid", True, align=1, n_shared=S)
    g = O.layer_backward(dout, logits, W1, W2, k, saved, "sigmoid", True)

    def loss(x_, l_, W1_):
        o, _ = O.layer_forward(x_, l_, W1_, W2, k, "sigmoid", True, align=1, n_shared=S)
        return float(np.sum(o * dout))

    eps = 1e-6
    for t, j in [(0, 1), (5, 7)]:
        xp, xm = x.copy(), x.copy()
        xp[t, j] += eps
        xm[t, j] -= eps
        assert np.isclose((loss(xp, logits, W1) - loss(xm, logits, W1)) / (2 * eps), g["dx"][t, j], rtol=1e-5,
                          atol=1e-8)
    for t, e in [(0, 0), (3, 2)]:
        lp, lm = logits.copy(), logits.copy()
        lp[t, e] += eps
        lm[t, e] -= eps
        assert np.isclose((loss(x, lp, W1) - loss(x, lm, W1)) / (2 * eps), g["dlogits"][t, e], rtol=1e-5,
                          atol=1e-8)
    # the shared expert's weights get gradients from every token
    Wp, Wm = W1.copy(), W1.copy()
    Wp[E, 3, 5] += eps
    Wm[E, 3, 5] -= eps
    assert np.isclose((loss(x, logits, Wp) - loss(x, logits, Wm)) / (2 * eps), g["dW1"][E, 3, 5], rtol=1e-5,
                      atol=1e-8)

