"""Pins for the CPU oracle: each check ties it to something other than itself.

Kinds of pin used (no check re-types the oracle's own formula):
* library routines: numpy matmul, torch's bf16 cast, scipy softmax, Python's
  stable sort;
* closed forms: one-hot expert weights with a known output, softmax of
  [0, ln 3], sigmoid(0);
* invariants stated by the pages: sum of tokens_per_expert = T*k, permute
  then unpermute is the identity ("Expert Parallelism (EP)" section 5), H
  shards summing to the full output ("NCCL course 32", tensor-parallel
  matrix split; "Expert Tensor Parallel design" section 4.3);
* the worked example of "NCCL course 32", section "Expert Parallel / MoE
  data flow" (7:1 skewed top-1 routing gives expert loads 112 / 16).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- rounding

def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(1000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    one = 1.0
    assert oracle.round_bf16(one + 2.0 ** -8) == 1.0                        # tie, even below
    assert oracle.round_bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6       # tie, even above
    assert oracle.round_bf16(one + 2.0 ** -8 + 2.0 ** -20) == one + 2.0 ** -7
    assert oracle.round_bf16(-(one + 2.0 ** -8)) == -1.0
    assert oracle.round_bf16(0.0) == 0.0
    assert math.isinf(oracle.round_bf16(3.4e38))


# ---------------------------------------------------------------- SiLU

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert oracle.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    v = oracle.silu(-800.0)
    assert v == 0.0 and not math.isnan(v)


# ---------------------------------------------------------------- router

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_router_logits_match_numpy_matmul(dt):
    rng = np.random.default_rng(2)
    T, D, E = 37, 96, 11
    x = rng.standard_normal((T, D)).astype(np.float32)
    wg = (rng.standard_normal((E, D)) * 0.05).astype(np.float32)
    b = rng.standard_normal(E)
    if dt == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        wt = torch.from_numpy(wg).to(torch.bfloat16)
        xa, wa = (xt.view(torch.int16).numpy().view(np.uint16), wt.view(torch.int16).numpy().view(np.uint16))
        xv, wv = xt.to(torch.float64).numpy(), wt.to(torch.float64).numpy()
    else:
        xa, wa, xv, wv = x, wg, x.astype(np.float64), wg.astype(np.float64)
    got = oracle.router_logits(xa, wa, b)
    ref = xv @ wv.T + b[None, :]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _brute_topk(l, k):
    # full stable sort of all experts by (NaN last, value desc, index asc)
    order = sorted(range(len(l)), key=lambda e: (math.isnan(l[e]), -l[e] if not math.isnan(l[e]) else 0.0, e))
    return order[:k]


def test_topk_matches_full_sort_with_ties():
    rng = np.random.default_rng(3)
    T, E = 200, 16
    l = rng.integers(-3, 4, size=(T, E)).astype(np.float32)   # many exact ties
    for k in (1, 2, 5, 16):
        idx, st = oracle.topk(l, k)
        assert st == oracle.OK
        for t in range(T):
            assert list(idx[t]) == _brute_topk(list(map(float, l[t])), k)


def test_topk_tie_goes_to_lower_index_from_duplicated_router_rows():
    rng = np.random.default_rng(4)
    T, D, E = 50, 32, 8
    x = rng.standard_normal((T, D)).astype(np.float32)
    wg = rng.standard_normal((E, D)).astype(np.float32)
    wg[5] = wg[2]            # experts 2 and 5 always tie exactly
    keys = oracle.router_logits(x, wg).astype(np.float32)
    idx, _ = oracle.topk(keys, E)
    for t in range(T):
        pos = {int(e): j for j, e in enumerate(idx[t])}
        assert pos[2] < pos[5]


def test_topk_nan_and_signed_zero():
    l = np.array([[0.0, np.nan, -np.inf, -0.0, 1.0]], np.float32)
    idx, st = oracle.topk(l, 5)
    assert st == oracle.BAD_ROUTING
    assert list(idx[0]) == [4, 0, 3, 2, 1]       # +0 and -0 tie -> lower index first


# ---------------------------------------------------------------- group-limited top-k
# Reading of the "Expert Parallelism (EP)" page, section 3 (DeepSeek-V3 style
# group-limited routing): n_group equal groups of consecutive experts; a group
# scores the fp32 sum of its m = k / topk_group best keys; the topk_group best
# groups (ties to the lower group) are the only ones a token may use.

def test_group_limited_topk_hand_example():
    # keys of 8 experts, groups {0,1} {2,3} {4,5} {6,7}, k = 4, topk_group = 2,
    # so m = 2: group scores 9+0=9, 5+5=10, 8+1=9, 7+7=14 -> groups 3 and 1;
    # the top-4 of experts {2,3,6,7} by (key desc, index asc) is 6, 7, 2, 3.
    # Plain top-4 would be 0, 4, 6, 7.
    keys = np.array([[9, 0, 5, 5, 8, 1, 7, 7]], np.float32)
    idx, st = oracle.topk(keys, 4, n_group=4, topk_group=2)
    assert st == oracle.OK and idx.tolist() == [[6, 7, 2, 3]]
    assert oracle.topk(keys, 4)[0].tolist() == [[0, 4, 6, 7]]
    # tied group scores go to the lower group: m = 1 gives 9, 5, 9, 7; with
    # topk_group = 1 group 0 wins the tie with group 2
    idx, _ = oracle.topk(keys, 1, n_group=4, topk_group=1)
    assert idx.tolist() == [[0]]
    keys2 = np.array([[0, 9, 5, 5, 9, 1, 7, 7]], np.float32)
    idx, _ = oracle.topk(keys2, 2, n_group=4, topk_group=2)   # m = 1: 9, 5, 9, 7 -> groups 0, 2
    assert idx.tolist() == [[1, 4]]


def _grouped_topk_by_sorting(keys, k, G, tg):
    """Independent statement of the reading with Python sorts."""
    T, E = keys.shape
    gs, m = E // G, k // tg
    out = np.empty((T, k), np.int32)
    for t in range(T):
        sc = []
        for g in range(G):
            best = sorted(range(g * gs, (g + 1) * gs), key=lambda e: (-keys[t, e], e))[:m]
            s32 = np.float32(0)
            for e in best:
                s32 = np.float32(s32 + keys[t, e])
            sc.append((-float(s32), g))
        chosen = {g for _, g in sorted(sc)[:tg]}
        allowed = [e for e in range(E) if e // gs in chosen]
        out[t] = sorted(allowed, key=lambda e: (-keys[t, e], e))[:k]
    return out


@pytest.mark.parametrize("E,G,tg,k", [(8, 4, 2, 4), (16, 4, 2, 2), (32, 8, 4, 8), (24, 3, 1, 5),
                                      (64, 8, 3, 7)])
def test_group_limited_topk_matches_sorting(E, G, tg, k):
    rng = np.random.default_rng(E * 100 + k)
    keys = rng.integers(-4, 5, size=(300, E)).astype(np.float32)   # many ties
    keys[:100] = rng.standard_normal((100, E)).astype(np.float32)
    idx, st = oracle.topk(keys, k, n_group=G, topk_group=tg)
    assert st == oracle.OK
    assert np.array_equal(idx, _grouped_topk_by_sorting(keys, k, G, tg))


def test_group_limited_topk_reduces_to_plain():
    rng = np.random.default_rng(7)
    keys = rng.integers(-3, 4, size=(200, 32)).astype(np.float32)
    plain, _ = oracle.topk(keys, 6)
    assert np.array_equal(oracle.topk(keys, 6, n_group=1, topk_group=1)[0], plain)
    assert np.array_equal(oracle.topk(keys, 6, n_group=4, topk_group=4)[0], plain)   # every group allowed


def test_group_limited_topk_rejects_bad_groupings():
    keys = np.zeros((2, 12), np.float32)
    assert oracle.topk(keys, 2, n_group=5, topk_group=2)[1] == oracle.BAD_ARG    # 12 % 5
    assert oracle.topk(keys, 1, n_group=4, topk_group=2)[1] == oracle.BAD_ARG    # k < topk_group
    assert oracle.topk(keys, 7, n_group=4, topk_group=2)[1] == oracle.BAD_ARG    # 7 > 2 groups x 3
    nan = keys.copy()
    nan[1, 3] = np.nan
    assert oracle.topk(nan, 2, n_group=4, topk_group=2)[1] == oracle.BAD_ROUTING


def test_scores_closed_forms():
    l = np.array([[0.0, math.log(3.0)]], np.float32)
    idx, _ = oracle.topk(l, 2)
    w = oracle.topk_weights(l, idx, oracle.SOFTMAX, False)
    np.testing.assert_allclose(w[0], [0.75, 0.25], rtol=1e-7)   # ln3 rounded to fp32
    s = oracle.topk_weights(np.zeros((1, 4), np.float32), np.array([[0, 1]], np.int32),
                            oracle.SIGMOID, False)
    assert s[0, 0] == 0.5 and s[0, 1] == 0.5
    sr = oracle.topk_weights(np.zeros((1, 4), np.float32), np.array([[0, 1]], np.int32),
                             oracle.SIGMOID, True)
    assert sr[0, 0] == 0.5 and sr[0, 1] == 0.5


def test_scores_against_scipy_softmax_and_sums():
    from scipy.special import softmax, expit
    rng = np.random.default_rng(5)
    T, E = 64, 12
    l = (rng.standard_normal((T, E)) * 3).astype(np.float32)
    idx, _ = oracle.topk(l, E)
    w = oracle.topk_weights(l, idx, oracle.SOFTMAX, False)
    ref = softmax(l.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, idx, 1), rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)
    # k = E with renormalisation is the plain softmax again
    wr = oracle.topk_weights(l, idx, oracle.SOFTMAX, True)
    np.testing.assert_allclose(wr, w, rtol=1e-13)
    # renormalised top-k weights sum to one, for both score functions
    idx4, _ = oracle.topk(l, 4)
    for sc in (oracle.SOFTMAX, oracle.SIGMOID):
        np.testing.assert_allclose(oracle.topk_weights(l, idx4, sc, True).sum(1), 1.0, rtol=1e-13)
    sg = oracle.topk_weights(l, idx4, oracle.SIGMOID, False)
    np.testing.assert_allclose(sg, np.take_along_axis(expit(l.astype(np.float64)), idx4, 1),
                               rtol=1e-13)


# ---------------------------------------------------------------- layout

def test_ep_toy_skewed_counts_golden():
    g = json.load(open(os.path.join(GOLDEN, "ep_toy_skewed_counts.json")))
    n = g["tokens_per_source"]
    for case in ("skewed", "balanced"):
        s0, s1 = g[case]["input_splits"]
        # x[t] = +1 routes to expert 0, -1 to expert 1 through a 1-dim router
        xs = []
        for _src in range(g["sources"]):
            xs += [1.0] * s0 + [-1.0] * s1
        x = np.array(xs, np.float32)[:, None]
        wg = np.array([[1.0], [-1.0]], np.float32)
        _, _, idx, _, st = oracle.route(x, wg, None, 1, oracle.SOFTMAX, False)
        assert st == oracle.OK
        lay = oracle.layout(idx, 2, align_m=1)
        assert list(lay["tokens_per_expert"]) == g[case]["tokens_per_expert"]
        recv = [[int((idx[src * n:(src + 1) * n, 0] == e).sum()) for src in range(2)] for e in range(2)]
        assert recv == g[case]["receive"]


def _check_layout_properties(idx, lay, E, e_first, E_local, align_m, masked=False, cap=0):
    T, k = idx.shape
    cnt, seg, row_of, tor = (lay["tokens_per_expert"], lay["seg_offsets"], lay["row_of"],
                             lay["token_of_row"])
    assert cnt.sum() == T * k                                          # sum = T*k
    assert np.array_equal(cnt, np.bincount(idx.ravel(), minlength=E))
    for i in range(E_local):
        e = e_first + i
        if masked:
            assert seg[i] == i * cap
        else:
            assert seg[i] % align_m == 0
            assert seg[i + 1] - seg[i] == -(-cnt[e] // align_m) * align_m
        toks = np.nonzero((idx == e).any(1))[0]                        # ascending tokens
        rows = seg[i] + np.arange(len(toks))
        assert np.array_equal(tor[rows], toks)
        pad_end = seg[i + 1] if not masked else seg[i] + cap
        assert (tor[seg[i] + len(toks):pad_end] == -1).all()
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            if e_first <= e < e_first + E_local:
                assert tor[row_of[t, j]] == t
            else:
                assert row_of[t, j] == -1


@pytest.mark.parametrize("align_m", [1, 8, 128])
def test_layout_properties_and_sort_reference(align_m):
    from moe_inputs import random_topk_idx
    T, E, k = 300, 12, 3
    idx = random_topk_idx(T, E, k, seed=6, skew=1.5)
    lay = oracle.layout(idx, E, align_m=align_m)
    assert lay["status"] == oracle.OK
    _check_layout_properties(idx, lay, E, 0, E, align_m)
    # reference by a library stable sort of (expert, token) pairs
    flat_e = idx.ravel()
    flat_t = np.repeat(np.arange(T), k)
    order = np.lexsort((flat_t, flat_e))
    seg = lay["seg_offsets"]
    pos = 0
    for e in range(E):
        n = int(lay["tokens_per_expert"][e])
        sel = order[pos:pos + n]
        assert np.array_equal(lay["row_of"].ravel()[sel], seg[e] + np.arange(n))
        pos += n


def test_layout_expert_range_and_masked():
    from moe_inputs import random_topk_idx
    T, E, k = 90, 16, 4
    idx = random_topk_idx(T, E, k, seed=7, skew=0.5)
    lay = oracle.layout(idx, E, e_first=4, E_local=8, align_m=16)
    assert lay["status"] == oracle.OK
    _check_layout_properties(idx, lay, E, 4, 8, 16)
    cap = int(np.bincount(idx.ravel(), minlength=E).max())
    lm = oracle.layout(idx, E, e_first=0, E_local=E, layout_kind=oracle.MASKED, capacity=cap)
    assert lm["status"] == oracle.OK and lm["rows_alloc"] == E * cap
    _check_layout_properties(idx, lm, E, 0, E, 1, masked=True, cap=cap)
    over = oracle.layout(idx, E, layout_kind=oracle.MASKED, capacity=cap - 1)
    assert over["status"] == oracle.CAPACITY


# A routing table with one out-of-range id (t3 slot 0), one negative id (t4
# slot 1) and one id repeated within a token (t2 slot 1).  Every expected
# array below was worked out by hand from the layout's definition: valid
# slots counted per expert, segments in expert order, tokens ascending inside
# a segment.
_BAD_IDX = np.array([[0, 1], [1, 0], [2, 2], [5, 1], [0, -1], [3, 0]], np.int32)


def test_layout_bad_ids_hand_example():
    """Reading R15: an invalid slot is neither counted nor placed."""
    lay = oracle.layout(_BAD_IDX, 4, align_m=1)
    assert lay["status"] == oracle.BAD_ROUTING
    assert list(lay["tokens_per_expert"]) == [4, 3, 1, 1]          # 9 = 12 - 3 slots
    assert list(lay["seg_offsets"]) == [0, 4, 7, 8, 9]
    assert lay["row_of"].tolist() == [[0, 4], [5, 1], [7, -1], [-1, 6], [2, -1], [8, 3]]
    assert list(lay["token_of_row"][:9]) == [0, 1, 4, 5, 0, 1, 3, 2, 5]
    assert (lay["token_of_row"][9:] == -1).all()
    # an expert range [1, 3) padded to 2 rows
    lr = oracle.layout(_BAD_IDX, 4, e_first=1, E_local=2, align_m=2)
    assert lr["status"] == oracle.BAD_ROUTING
    assert list(lr["tokens_per_expert"]) == [4, 3, 1, 1]
    assert list(lr["seg_offsets"]) == [0, 4, 6]
    assert lr["row_of"].tolist() == [[-1, 0], [1, -1], [4, -1], [-1, 2], [-1, -1], [-1, -1]]
    assert list(lr["token_of_row"][:6]) == [0, 1, 3, -1, 2, -1]
    assert (lr["token_of_row"][6:] == -1).all()


def test_layout_capacity_overflow_hand_example():
    """Reading R7: a masked expert over capacity keeps its first `capacity`
    tokens in token order; the count still covers every routed token."""
    idx = np.array([[0, 1], [1, 0], [2, 0], [0, 3]], np.int32)
    lay = oracle.layout(idx, 4, layout_kind=oracle.MASKED, capacity=2)
    assert lay["status"] == oracle.CAPACITY
    assert lay["rows_alloc"] == 8
    assert list(lay["tokens_per_expert"]) == [4, 2, 1, 1]
    assert list(lay["seg_offsets"]) == [0, 2, 4, 6, 8]
    assert lay["row_of"].tolist() == [[0, 2], [3, 1], [4, -1], [-1, 6]]
    assert list(lay["token_of_row"]) == [0, 1, 0, 1, 2, -1, 3, -1]
    # with invalid slots as well: both rules apply, capacity is reported first
    lb = oracle.layout(_BAD_IDX, 4, layout_kind=oracle.MASKED, capacity=2)
    assert lb["status"] == oracle.CAPACITY
    assert list(lb["tokens_per_expert"]) == [4, 3, 1, 1]
    assert lb["row_of"].tolist() == [[0, 2], [3, 1], [4, -1], [-1, -1], [-1, -1], [6, -1]]
    assert list(lb["token_of_row"]) == [0, 1, 0, 1, 2, -1, 5, -1]
    # capacity 0: nothing is placed
    l0 = oracle.layout(idx, 4, layout_kind=oracle.MASKED, capacity=0)
    assert l0["status"] == oracle.CAPACITY and l0["rows_alloc"] == 0
    assert (l0["row_of"] == -1).all()


def test_layout_rejected_arguments_leave_sentinels():
    """A rejected argument writes nothing; the wrapper's arrays then hold a
    sentinel that no layout contains, so they cannot match a result."""
    lay = oracle.layout(_BAD_IDX, 4, e_first=3, E_local=2)        # range beyond E
    assert lay["status"] == oracle.BAD_ARG
    assert (lay["row_of"] < -1).all()


def test_permute_then_unpermute_is_identity():
    from moe_inputs import random_topk_idx
    rng = np.random.default_rng(8)
    T, E, k, D = 120, 10, 3, 24
    idx = random_topk_idx(T, E, k, seed=8)
    x = rng.standard_normal((T, D)).astype(np.float32)
    lay = oracle.layout(idx, E, align_m=8)
    xp = oracle.permute_rows(x, lay["token_of_row"])
    for t in range(T):
        for j in range(k):
            assert np.array_equal(xp[lay["row_of"][t, j]], x[t])          # bitwise copy
    # unpermute with dyadic weights summing to one returns x exactly
    w = np.tile(np.array([0.5, 0.25, 0.25]), (T, 1))
    out = oracle.unpermute_combine(xp, lay["row_of"], w)
    assert np.array_equal(out, x.astype(np.float64))
    # k = 1 with unit weights: combine(permute(x)) == x
    idx1 = idx[:, :1].copy()
    l1 = oracle.layout(idx1, E, align_m=4)
    out1 = oracle.unpermute_combine(oracle.permute_rows(x, l1["token_of_row"]), l1["row_of"],
                                    np.ones((T, 1)))
    assert np.array_equal(out1, x.astype(np.float64))


# ---------------------------------------------------------------- experts

def test_expert_ffn_one_hot_closed_form():
    D, H = 7, 5            # D != H so a transposed index cannot pass
    d0, h0, d1 = 3, 4, 6
    a, b, c, s = 1.5, -2.0, 0.75, 0.5
    v = np.zeros(D); v[d0] = s
    w1 = np.zeros((H, D)); w1[h0, d0] = a
    w3 = np.zeros((H, D)); w3[h0, d0] = b
    w2 = np.zeros((D, H)); w2[d1, h0] = c
    y = oracle.expert_ffn(v, w1, w3, w2)
    ref = np.zeros(D); ref[d1] = c * (a * s / (1.0 + math.exp(-a * s))) * (b * s)
    np.testing.assert_allclose(y, ref, rtol=1e-15, atol=0)
    # gate and up on different hidden units never meet: output is zero
    w3b = np.zeros((H, D)); w3b[1, d0] = b
    assert not oracle.expert_ffn(v, w1, w3b, w2).any()


def _numpy_moe(x, w1, w3, w2, idx, w, e_first=0, E_local=None, round_fn=None, round_y=True):
    """Layer output written with numpy matmuls (F.linear: X @ W^T)."""
    T, D = x.shape
    E_local = w1.shape[0] if E_local is None else E_local
    out = np.zeros((T, D))
    for i in range(E_local):
        e = e_first + i
        tok, slot = np.nonzero(idx == e)
        if len(tok) == 0:
            continue
        X = x[tok]
        g = X @ w1[i].T
        u = X @ w3[i].T
        hh = g / (1.0 + np.exp(-g)) * u
        if round_fn:
            hh = round_fn(hh)
        y = hh @ w2[i].T
        if round_fn and round_y:
            y = round_fn(y)
        np.add.at(out, tok, w[tok, slot][:, None] * y)
    return out


def _small_problem(seed, T=64, D=40, H=24, E=6, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, D))
    wg = rng.standard_normal((E, D)) * 0.1
    w1 = rng.standard_normal((E, H, D)) * 0.1
    w3 = rng.standard_normal((E, H, D)) * 0.1
    w2 = rng.standard_normal((E, D, H)) * 0.1
    _, _, idx, w, _ = oracle.route(x, wg, None, k, oracle.SOFTMAX, True)
    return x, w1, w3, w2, idx, w


def test_moe_tokens_matches_numpy_and_grouped_layout():
    x, w1, w3, w2, idx, w = _small_problem(9)
    T, D = x.shape
    E = w1.shape[0]
    brute = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w)
    np.testing.assert_allclose(brute, _numpy_moe(x, w1, w3, w2, idx, w), rtol=1e-11, atol=1e-13)
    # grouped form over the permuted layout gives the same output
    lay = oracle.layout(idx, E, align_m=8)
    xp = oracle.permute_rows(x, lay["token_of_row"])
    cnt = lay["tokens_per_expert"]
    h = oracle.grouped_gemm1_swiglu(xp, lay["seg_offsets"], cnt, list(w1), list(w3))
    y = oracle.grouped_gemm2(h, lay["seg_offsets"], cnt, list(w2))
    out = oracle.unpermute_combine(np.nan_to_num(y), lay["row_of"], w)
    np.testing.assert_allclose(out, brute, rtol=1e-12, atol=1e-14)


def test_bf16_rounding_points_match_torch():
    x, w1, w3, w2, idx, w = _small_problem(10)
    T = x.shape[0]

    def tround(a):
        return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w, round_h=True,
                            round_y=True)
    # numpy evaluation rounding h and y through torch's bf16 cast; an fp64 ->
    # fp32 -> bf16 double rounding may differ by one bf16 step in rare cases
    ref = _numpy_moe(x, w1, w3, w2, idx, w, round_fn=tround)
    err = np.abs(got - ref).max() / np.sqrt((ref ** 2).mean())
    assert err < 1e-2
    unrounded = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w)
    assert np.abs(got - unrounded).max() > 0     # the rounding points are real
    # h alone: numpy evaluation rounding only h
    got_h = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w, round_h=True)
    ref_h = _numpy_moe(x, w1, w3, w2, idx, w, round_fn=tround, round_y=False)
    assert np.abs(got_h - ref_h).max() / np.sqrt((ref_h ** 2).mean()) < 1e-2
    assert np.abs(got_h - got).max() > 0 and np.abs(got_h - unrounded).max() > 0


def test_h_shards_sum_to_full_output():
    x, w1, w3, w2, idx, w = _small_problem(11, H=24)
    T = x.shape[0]
    full = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w)
    for tp in (2, 3, 4):
        Hl = w1.shape[1] // tp
        acc = np.zeros_like(full)
        for r in range(tp):
            sl = slice(r * Hl, (r + 1) * Hl)
            acc += oracle.moe_tokens(np.arange(T), x, list(w1[:, sl, :]), list(w3[:, sl, :]),
                                     list(w2[:, :, sl]), idx, w)
        np.testing.assert_allclose(acc, full, rtol=1e-11, atol=1e-13)


def test_expert_ranges_sum_to_full_output():
    x, w1, w3, w2, idx, w = _small_problem(12, E=8, k=3)
    T = x.shape[0]
    full = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w)
    acc = np.zeros_like(full)
    for r in range(4):
        e0 = 2 * r
        acc += oracle.moe_tokens(np.arange(T), x, list(w1[e0:e0 + 2]), list(w3[e0:e0 + 2]),
                                 list(w2[e0:e0 + 2]), idx, w, e_first=e0)
    np.testing.assert_allclose(acc, full, rtol=1e-11, atol=1e-13)


def test_missing_expert_weights_is_an_error():
    x, w1, w3, w2, idx, w = _small_problem(13)
    w1s = list(w1)
    w1s[int(idx[0, 0])] = None
    with pytest.raises(ValueError):
        oracle.moe_tokens([0], x, w1s, list(w3), list(w2), idx, w)
