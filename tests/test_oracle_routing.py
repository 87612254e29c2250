"""Pins for the oracle's routing, counts/offsets, permute and combine (CPU)."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_softmax_worked_example():
    g = _golden("softmax_worked_example.json")
    scores = np.array([g["scores"]], dtype=np.float32)
    idx, w = O.route_topk(scores, k=4, score="softmax", normalize=False)
    p = np.zeros(4)
    p[idx[0]] = w[0]
    assert np.array_equal(np.round(p, g["decimals"]), np.array(g["softmax"]))
    assert list(idx[0]) == [1, 3, 0, 2]             # descending score
    # with all experts chosen, renormalising changes nothing
    _, wn = O.route_topk(scores, k=4, score="softmax", normalize=True)
    assert np.allclose(wn, w, rtol=0, atol=1e-15)


def test_top2_renormalised_equals_online_softmax_rescale():
    g = _golden("online_softmax_rescale.json")
    scores = np.array([g["scores"]], dtype=np.float32)
    idx, w = O.route_topk(scores, k=g["k"], score="softmax", normalize=True)
    assert list(idx[0]) == g["top_idx"]
    assert round(w[0, 0], g["decimals"]) == g["ratio"] == round(g["l1"] / g["l2"], g["decimals"])
    assert round(w[0, 1], g["decimals"]) == round(1 - g["ratio"], g["decimals"])


def _check_selection(l, idx):
    """Independent characterisation of top-k: every chosen expert beats every
    unchosen one (higher logit, or equal logit and lower index), and the
    chosen list is in that same order."""
    T, E = l.shape
    for t in range(T):
        S = list(idx[t])
        assert len(set(S)) == len(S)
        beats = lambda a, b: l[t, a] > l[t, b] or (l[t, a] == l[t, b] and a < b)
        for a in S:
            for b in range(E):
                if b not in S:
                    assert beats(a, b)
        for a, b in zip(S, S[1:]):
            assert beats(a, b)


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3), (5, 5)])
def test_topk_brute_force_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    l = rng.integers(-2, 3, size=(40, E)).astype(np.float32)      # many ties
    idx, w = O.route_topk(l, k, "softmax", True)
    _check_selection(l, idx)
    # brute force over all k-subsets: the chosen set is the best subset in
    # the (logit desc, index asc) order
    for t in range(l.shape[0]):
        key = lambda S: sorted(((-l[t, e], e) for e in S))
        best = min(itertools.combinations(range(E), k), key=key)
        assert set(best) == set(idx[t])


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_weights_sum_to_one_and_raw_scores(score):
    rng = np.random.default_rng(7)
    l = rng.standard_normal((64, 16)).astype(np.float32)
    idx, w = O.route_topk(l, 4, score, True)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-14)
    _, raw = O.route_topk(l, 4, score, False)
    chosen = np.take_along_axis(l.astype(np.float64), idx.astype(np.int64), 1)
    if score == "sigmoid":
        ref = 1 / (1 + np.exp(-chosen))
    else:
        ref = np.exp(chosen) / np.exp(l.astype(np.float64)).sum(axis=1, keepdims=True)
    assert np.allclose(raw, ref, rtol=1e-13)
    assert np.allclose(w, raw / raw.sum(axis=1, keepdims=True), rtol=1e-13)


def test_counts_offsets_dropless():
    rng = np.random.default_rng(8)
    l = rng.standard_normal((100, 8)).astype(np.float32)
    idx, _ = O.route_topk(l, 2)
    c = O.group_counts(idx, 8)
    assert c.sum() == 200 and np.all(c >= 0)
    for e in range(8):
        assert c[e] == int(np.sum(idx == e))
    off = O.group_offsets(c)
    assert off[0] == 0 and off[-1] == 200 and np.all(np.diff(off) == c)
    gofs = O.aligned_group_offsets(c, 128)
    assert np.all(gofs % 128 == 0) and np.all(np.diff(gofs) >= c) and np.all(np.diff(gofs) - c < 128)
    assert np.array_equal(O.aligned_group_offsets(c, 1), off)


@pytest.mark.parametrize("align", [1, 32, 128])
def test_permute_is_stable_bijection(align):
    rng = np.random.default_rng(9)
    T, E, k = 77, 6, 3
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, 5] -= 10                                    # expert 5 gets no token
    idx, _ = O.route_topk(l, k)
    slot_of, row_id = O.permute_slots(idx, E, align)
    c = O.group_counts(idx, E)
    gofs = O.aligned_group_offsets(c, align)
    assert c[5] == 0 and gofs[5] == gofs[6]          # empty group has no rows
    flat = slot_of.reshape(-1)
    assert len(np.unique(flat)) == T * k             # unique slots
    assert np.array_equal(np.sort(flat[row_id[flat] >= 0]), np.sort(flat))
    for s in range(len(row_id)):
        if row_id[s] >= 0:
            t, j = divmod(row_id[s], k)
            assert slot_of[t, j] == s
    for e in range(E):
        ids = row_id[gofs[e]:gofs[e] + c[e]]
        assert np.all(ids >= 0) and np.all(idx.reshape(-1)[ids] == e)
        assert np.all(np.diff(ids // k) > 0)        # token order inside the group
        assert np.all(row_id[gofs[e] + c[e]:gofs[e + 1]] == -1)
    if align == 1:
        assert np.array_equal(np.sort(flat), np.arange(T * k))


def test_unpermute_of_permute_is_identity():
    rng = np.random.default_rng(10)
    T, E, d = 50, 8, 16
    x = np.round(rng.standard_normal((T, d)) * 64) / 64    # few significant bits: sums are exact
    for k in (1, 2, 4, 8):
        idx, _ = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
        slot_of, row_id = O.permute_slots(idx, E, 128)
        xp = O.permute(x, row_id, k)
        assert np.all(xp[row_id < 0] == 0)
        out = O.combine(xp, slot_of, np.full((T, k), 1.0 / k))
        assert np.array_equal(out, x)
        assert np.array_equal(O.combine(xp, slot_of, None), k * x)


def test_combine_weighted_sum_by_hand():
    y = np.arange(12, dtype=np.float64).reshape(6, 2)
    slot_of = np.array([[4, 0], [1, 5]])
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    out = O.combine(y, slot_of, w)
    assert np.array_equal(out, np.array([[0.25 * 8 + 0.75 * 0, 0.25 * 9 + 0.75 * 1],
                                         [0.5 * 2 + 0.5 * 10, 0.5 * 3 + 0.5 * 11]]))


def test_combine_bwd_is_adjoint_and_fd():
    rng = np.random.default_rng(11)
    T, E, k, d = 20, 5, 2, 8
    idx, w = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    slot_of, row_id = O.permute_slots(idx, E, 32)
    R = len(row_id)
    y = rng.standard_normal((R, d))
    y[row_id < 0] = 0
    dout = rng.standard_normal((T, d))
    dy, dw = O.combine_bwd(dout, y, slot_of, w, R)
    # <combine(y), dout> == <y, dy>  (linear in y)
    assert np.isclose(np.sum(O.combine(y, slot_of, w) * dout), np.sum(y * dy), rtol=1e-12)
    assert np.all(dy[row_id < 0] == 0)
    # dw by central differences of L(w) = <combine(y, w), dout>
    eps = 1e-6
    for t, j in [(0, 0), (3, 1), (19, 0)]:
        wp, wm = w.copy(), w.copy()
        wp[t, j] += eps
        wm[t, j] -= eps
        fd = (np.sum(O.combine(y, slot_of, wp) * dout) - np.sum(O.combine(y, slot_of, wm) * dout)) / (2 * eps)
        assert np.isclose(fd, dw[t, j], rtol=1e-6, atol=1e-9)


def test_fp32_round_ties_and_spacing():
    one = 1.0
    assert O.fp32_round(one + 2.0 ** -24) == one                 # tie -> even
    assert O.fp32_round(one + 3 * 2.0 ** -24) == one + 2.0 ** -22  # tie -> even (up)
    assert O.fp32_round(one + 2.0 ** -24 + 2.0 ** -40) == one + 2.0 ** -23
    assert O.fp32_round(2.0 ** -149) == 2.0 ** -149              # smallest subnormal
    assert O.fp32_round(2.0 ** -151) == 0.0
    assert np.isinf(O.fp32_round(3.5e38))


def test_permute_scaled_bf16_special_cases():
    rng = np.random.default_rng(13)
    T, E, k, d = 40, 6, 3, 16
    idx, w = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    slot_of, row_id = O.permute_slots(idx, E, 32)
    src = O.bf16_round(rng.standard_normal((T, d)))
    # unit weights: exactly the permute; powers of two: exactly w * src
    assert np.array_equal(O.permute_scaled_bf16(src, row_id, k, np.ones((T, k))), O.permute(src, row_id, k))
    p2 = 2.0 ** rng.integers(-6, 3, size=(T, k)).astype(np.float64)
    dy_exact, _ = O.combine_bwd(src, np.zeros((len(row_id), d)), slot_of, p2, len(row_id))
    assert np.array_equal(O.permute_scaled_bf16(src, row_id, k, p2), dy_exact)
    # general weights: within one bf16 rounding of the fp64 combine_bwd rows
    dy_ref, _ = O.combine_bwd(src, np.zeros((len(row_id), d)), slot_of, w, len(row_id))
    got = O.permute_scaled_bf16(src, row_id, k, w)
    assert np.all(got[row_id < 0] == 0)
    assert np.all(np.abs(got - dy_ref) <= 2.0 ** -8 * np.abs(dy_ref) * (1 + 1e-6))


def test_permute_scaled_bf16_double_rounding_by_hand():
    # src = 0x1.02p1 (bf16), w = 0x1.4e633ap-1 (fp32).  The exact product
    # 0x1.51000074p0 lies just above the bf16 tie 0x1.51p0 (fraction bits
    # 0101 0001); its fp32 rounding drops the tail (fraction bit 24 is 0)
    # and lands exactly on the tie, which bf16 rounds to even: 0x1.50p0 =
    # 1.3125.  A single rounding of the exact product gives 0x1.52p0.
    src = np.array([[float.fromhex("0x1.02p1"), 512.0] + [0.0] * 30])
    w = np.array([[float.fromhex("0x1.4e633ap-1")]])
    got = O.permute_scaled_bf16(src, np.array([0]), 1, w)
    assert got[0, 0] == 1.3125
    assert O.bf16_round(src[0, 0] * w[0, 0]) == float.fromhex("0x1.52p0")
    # the rounding reaches the MXFP8 code: the block max 512 w ~ 334.4 gives
    # scale 2^0, and 1.3125 is the E4M3 tie between 1.25 (0x3A, even) and
    # 1.375 (0x3B); 0x1.52p0 = 1.328125 would round up to 0x3B.
    codes, scales = O.mxfp8_quantize_rows(got)
    assert scales[0, 0] == 127 and codes[0, 0] == 0x3A
    alt = got.copy()
    alt[0, 0] = float.fromhex("0x1.52p0")
    assert O.mxfp8_quantize_rows(alt)[0][0, 0] == 0x3B


@pytest.mark.parametrize("score,normalize", [("softmax", True), ("softmax", False),
                                             ("sigmoid", True), ("sigmoid", False)])
def test_route_bwd_finite_differences(score, normalize):
    rng = np.random.default_rng(12)
    T, E, k = 6, 7, 3
    l = rng.standard_normal((T, E))
    idx, w = O.route_topk(l, k, score, normalize)
    dw = rng.standard_normal((T, k))
    dl = O.route_bwd(l, idx, dw, score, normalize)
    eps = 1e-6
    for t in range(T):
        for e in range(E):
            lp, lm = l.copy(), l.copy()
            lp[t, e] += eps
            lm[t, e] -= eps
            ip, wp = O.route_topk(lp, k, score, normalize)
            im, wm = O.route_topk(lm, k, score, normalize)
            assert np.array_equal(ip, idx) and np.array_equal(im, idx)   # selection is stable
            fd = np.sum((wp - wm) * dw) / (2 * eps)
            assert np.isclose(fd, dl[t, e], rtol=1e-5, atol=1e-8), (t, e, fd, dl[t, e])
