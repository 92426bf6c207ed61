"""GPU parity of each step of the path against the CPU oracle, via the C ABI.

Integer work (routing indices, counts, offsets, permutation, x_perm bytes)
is compared bit for bit; floats against the oracle with the tolerances of
tests/helpers.py (max |gpu - oracle| / rms(oracle): 1e-4 fp32, 2e-2 bf16).
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import (assert_grouped_parity as _assert_grouped_parity, check_layout_properties,
                     rel_err, to_f64, within_bf16_rounding)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("score,renorm", [("softmax", False), ("softmax", True), ("sigmoid", True),
                                          ("sigmoid", False)])
@pytest.mark.parametrize("n_group,topk_group", [(0, 0), (8, 3), (4, 1)])
def test_route_exact_logits_bitexact(moe, dt, score, renorm, n_group, topk_group):
    """Integer-valued inputs make every logit exact in fp32, ties included;
    also with group-limited routing (groups of 9 or 18 experts)."""
    T, D, E, k = 300, 264, 72, 6
    x, wg = moe_inputs.exact_router_inputs(T, D, E, seed=11)
    bias = (np.arange(E) % 5 - 2).astype(np.float32) / 8.0
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k,
                     dtype=moe.MOE_F32 if dt == "f32" else moe.MOE_BF16,
                     score=moe.MOE_SCORE_SOFTMAX if score == "softmax" else moe.MOE_SCORE_SIGMOID,
                     renorm=int(renorm), n_group=n_group, topk_group=topk_group)
    ws = moe.alloc_workspace(cfg)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    gidx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(cfg, _dev(x, tdt), _dev(wg, tdt), _dev(bias), logits, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    ref = oracle.router_logits(x, wg, bias.astype(np.float64))
    assert np.array_equal(logits.cpu().numpy(), ref.astype(np.float32))      # exact
    keys = ref.astype(np.float32)
    oidx, st = oracle.topk(keys, k, n_group, topk_group)
    assert st == oracle.OK
    n_ties = sum(len(set(keys[t])) < E for t in range(T))
    assert n_ties > T // 2                                   # the case exercises ties
    if n_group:
        assert (oidx != oracle.topk(keys, k)[0]).any()       # the grouping changes choices
    assert np.array_equal(gidx.cpu().numpy(), oidx)
    ow = oracle.topk_weights(keys, oidx, oracle.SOFTMAX if score == "softmax" else oracle.SIGMOID,
                             renorm)
    np.testing.assert_allclose(gw.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,D,E,k,score", [
    (4096, 2048, 64, 6, "softmax"),    # 32 m-tiles: the D reduction split 4 ways per cluster
    (4096, 1024, 256, 8, "sigmoid"),
    (8192, 1024, 64, 6, "softmax"),    # 64 m-tiles: 2 splits
    (8192, 1024, 256, 8, "sigmoid"),
    (16384, 512, 64, 8, "softmax"),    # 128 m-tiles: 1 split
    (16384, 512, 256, 8, "sigmoid"),
])
@pytest.mark.parametrize("mode", ["cluster", "split"])
def test_route_exact_logits_full_batch_sizes(moe, T, D, E, k, score, mode, monkeypatch):
    """The batch sizes of the bf16 workloads, where the router splits the D
    reduction 4, 2 or 1 ways: on exact-integer inputs the fp32 logits, the
    whole batch's top-k and the weights equal the oracle's (one cluster launch
    and the two-kernel form)."""
    if mode == "split":
        monkeypatch.setenv("MOE_ROUTER_KERNEL", "split")
    x, wg = moe_inputs.exact_router_inputs(T, D, E, seed=T + E)
    bias = ((np.arange(E) * 7) % 9 - 4).astype(np.float32) / 4.0
    renorm = True
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                     score=moe.MOE_SCORE_SOFTMAX if score == "softmax" else moe.MOE_SCORE_SIGMOID,
                     renorm=int(renorm))
    ws = moe.alloc_workspace(cfg)
    logits = torch.full((T, E), float("nan"), device="cuda")
    gidx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    gw = torch.full((T, k), float("nan"), device="cuda")
    moe.moe_route_topk(cfg, _dev(x, torch.bfloat16), _dev(wg, torch.bfloat16), _dev(bias),
                       logits, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    ref = oracle.router_logits(x, wg, bias.astype(np.float64))
    keys = ref.astype(np.float32)
    assert np.array_equal(logits.cpu().numpy(), keys)                    # exact
    oidx, st = oracle.topk(keys, k)
    assert st == oracle.OK
    assert sum(len(set(keys[t])) < E for t in range(0, T, 16)) > T // 64   # ties occur
    assert np.array_equal(gidx.cpu().numpy(), oidx)                       # whole batch
    ow = oracle.topk_weights(keys, oidx, oracle.SOFTMAX if score == "softmax" else oracle.SIGMOID,
                             renorm)
    np.testing.assert_allclose(gw.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name", moe_inputs.WORKLOAD_ORDER)
def test_route_workload_shapes(moe, name):
    """Config-shaped random inputs: logits within tolerance, selection valid."""
    w = moe_inputs.WORKLOADS[name].scaled(T=min(moe_inputs.WORKLOADS[name].T, 1024))
    inp = moe_inputs.make_inputs(w, device="cuda", seed=5, weights=False)
    from helpers import cfg_for, oracle_route, routing_agreement
    cfg = cfg_for(moe, w)
    ws = moe.alloc_workspace(cfg)
    logits = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    gidx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, logits, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    l64, keys, oidx, ow, st = oracle_route(inp, w, inp.bias)
    gl = logits.cpu().numpy()
    lerr = np.abs(gl - l64).max()
    assert lerr < 1e-4 * max(1.0, np.abs(l64).max())
    g = gidx.cpu().numpy()
    same_set, same_order = routing_agreement(g, oidx, keys, key_tol=4 * lerr + 1e-6)
    assert same_order.mean() > 0.99
    # the GPU's choice is exact for its own logits: sorted by (key desc, index asc)
    for t in range(w.T):
        order = sorted(range(w.E), key=lambda e: (-gl[t, e], e))[:w.k]
        assert list(g[t]) == order
    np.testing.assert_allclose(gw.cpu().numpy()[same_order], ow[same_order], rtol=1e-4, atol=1e-6)


def test_route_group_limited_workload(moe):
    """DeepSeek-V3-shaped router with 8 groups, top-4 groups: the GPU's
    choice is exactly the grouped selection on its own fp32 logits, agrees
    with the oracle's routing on > 99% of tokens and uses at most 4 groups."""
    w = moe_inputs.WORKLOADS["deepseek-v3-shaped"].scaled(T=1024, n_group=8, topk_group=4)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=5, weights=False)
    from helpers import cfg_for, oracle_route, routing_agreement
    cfg = cfg_for(moe, w)
    ws = moe.alloc_workspace(cfg)
    logits = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    gidx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, logits, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    gl = logits.cpu().numpy()
    g = gidx.cpu().numpy()
    own, _ = oracle.topk(gl, w.k, w.n_group, w.topk_group)
    assert np.array_equal(g, own)
    assert max(len(set(row // (w.E // w.n_group))) for row in g) <= w.topk_group
    l64, keys, oidx, ow, st = oracle_route(inp, w, inp.bias)
    lerr = np.abs(gl - l64).max()
    same_set = np.array([set(a) == set(b) for a, b in zip(g, oidx)])
    assert same_set.mean() > 0.99, f"{same_set.mean():.4f} (logit error {lerr:.2e})"
    assert (oidx != oracle.topk(keys, w.k)[0]).any()
    np.testing.assert_allclose(gw.cpu().numpy()[same_set], ow[same_set], rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("T,D,E,k,score", [(1000, 2048, 64, 6, "softmax"), (300, 7168, 256, 8, "sigmoid"),
                                           (77, 512, 8, 2, "softmax"), (4096, 2048, 64, 6, "softmax")])
def test_route_one_kernel_equals_two(moe, T, D, E, k, score, monkeypatch):
    """bf16 router: one cluster launch (split-D partials summed through
    distributed shared memory) and the two-kernel form (partials through the
    workspace) add the same partials in the same order: bitwise equal."""
    g = torch.Generator(device="cuda").manual_seed(T + E)
    x = torch.randn((T, D), generator=g, device="cuda").to(torch.bfloat16)
    wg = (torch.randn((E, D), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    bias = torch.randn((E,), generator=g, device="cuda") * 0.1
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                     score=moe.MOE_SCORE_SOFTMAX if score == "softmax" else moe.MOE_SCORE_SIGMOID)
    ws = moe.alloc_workspace(cfg)
    outs = {}
    for mode in ("cluster", "split"):
        if mode == "split":
            monkeypatch.setenv("MOE_ROUTER_KERNEL", "split")
        logits = torch.full((T, E), float("nan"), device="cuda")
        gidx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        gw = torch.full((T, k), float("nan"), device="cuda")
        n0 = moe.kernel_launches()
        moe.moe_route_topk(cfg, x, wg, bias, logits, gidx, gw, ws)
        n = moe.kernel_launches() - n0
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        outs[mode] = (logits, gidx, gw, n)
    assert outs["cluster"][3] == 1 and outs["split"][3] == 2
    for a, b in zip(outs["cluster"][:3], outs["split"][:3]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_route_largest_E_and_k_bitexact(moe, dt):
    """E = 1024 and k = 32, the largest the ABI accepts (the bf16 router runs
    the SIMT form above 256 experts); with and without 32 groups."""
    T, D, E, k = 160, 96, 1024, 32
    x, wg = moe_inputs.exact_router_inputs(T, D, E, seed=3)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    ref = oracle.router_logits(x, wg, None)
    keys = ref.astype(np.float32)
    for n_group, topk_group in ((0, 0), (32, 8)):
        cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k,
                         dtype=moe.MOE_F32 if dt == "f32" else moe.MOE_BF16,
                         score=moe.MOE_SCORE_SIGMOID, renorm=1, n_group=n_group,
                         topk_group=topk_group)
        ws = moe.alloc_workspace(cfg)
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        gidx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        moe.moe_route_topk(cfg, _dev(x, tdt), _dev(wg, tdt), None, logits, gidx, gw, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        assert np.array_equal(logits.cpu().numpy(), keys)
        oidx, st = oracle.topk(keys, k, n_group, topk_group)
        assert st == oracle.OK
        assert np.array_equal(gidx.cpu().numpy(), oidx)
        ow = oracle.topk_weights(keys, oidx, oracle.SIGMOID, True)
        np.testing.assert_allclose(gw.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n_group,topk_group", [(0, 0), (4, 2)])
def test_route_special_keys_order(moe, dt, n_group, topk_group):
    """+inf, -inf and NaN keys in one token: the selection takes +inf first,
    -inf after every finite key and NaN last, equal keys by lower index --
    the same as the oracle's top-k on the GPU's own logits."""
    T, D, E, k = 96, 64, 32, 10
    rng = np.random.default_rng(5)
    x = rng.integers(-3, 4, size=(T, D)).astype(np.float32)
    wg = rng.integers(-2, 3, size=(E, D)).astype(np.float32)
    # where x[t, 0] = inf: per 8 experts one +inf, one -inf and six NaN keys,
    # so the 10 slots take 4 x +inf, 4 x -inf and the 2 lowest NaN experts
    wg[:, 0] = np.tile([1.0, 0.0, -1.0, 0.0, 0.0, 0.0, 0.0, 0.0], E // 8)
    x[::3, 0] = np.inf                                    # a third of the tokens
    x[1::6, 0] = -np.inf                                  # and a sixth with -inf
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k,
                     dtype=moe.MOE_F32 if dt == "f32" else moe.MOE_BF16,
                     score=moe.MOE_SCORE_SIGMOID, renorm=1, n_group=n_group,
                     topk_group=topk_group)
    ws = moe.alloc_workspace(cfg)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    gidx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(cfg, _dev(x, tdt), _dev(wg, tdt), None, logits, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BAD_ROUTING
    keys = logits.cpu().numpy()
    assert np.isnan(keys).any() and np.isposinf(keys).any() and np.isneginf(keys).any()
    oidx, st = oracle.topk(keys, k, n_group, topk_group)
    assert st == oracle.BAD_ROUTING
    assert np.array_equal(gidx.cpu().numpy(), oidx)


def test_route_nan_logit_sets_status(moe):
    T, D, E, k = 64, 64, 16, 4
    x = torch.randn(T, D, device="cuda")
    x[7, 3] = float("nan")
    wg = torch.randn(E, D, device="cuda")
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_F32)
    ws = moe.alloc_workspace(cfg)
    gidx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(cfg, x, wg, None, None, gidx, gw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BAD_ROUTING
    assert moe.moe_get_device_status(ws) == moe.MOE_OK          # read clears
    g = gidx.cpu().numpy()
    assert ((g >= 0) & (g < E)).all()
    assert all(len(set(r)) == k for r in g)


# ------------------------------------------------------------------ permute

def _run_permute(moe, cfg, x, idx, ws=None):
    ra = moe.rows_alloc(cfg)
    el = cfg.e_local
    ws = moe.alloc_workspace(cfg) if ws is None else ws
    tpe = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    seg = torch.empty(el + 1, dtype=torch.int32, device="cuda")
    row_of = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    tor = torch.full((ra,), 7777, dtype=torch.int32, device="cuda")
    xp = torch.zeros((ra, cfg.D), dtype=x.dtype, device="cuda")
    moe.moe_permute(cfg, x, _dev(idx), tpe, seg, row_of, tor, xp, ws)
    st = moe.moe_get_device_status(ws)
    return st, tpe.cpu().numpy(), seg.cpu().numpy(), row_of.cpu().numpy(), tor.cpu().numpy(), xp


@pytest.mark.parametrize("T,E,k,align,e_first,E_local,skew", [
    (1000, 16, 4, 128, 0, 16, 1.3),      # ragged tail block, empty experts
    (257, 64, 6, 128, 0, 64, 0.0),
    (31, 8, 2, 1, 0, 8, 0.0),            # fewer tokens than a warp, no padding
    (40, 256, 8, 128, 0, 256, 0.5),      # fewer tokens than experts: a warp pads several segments
    (2000, 32, 8, 8, 8, 12, 0.8),        # expert range, small alignment
    (513, 256, 8, 128, 0, 256, 0.3),
    (700, 5, 1, 16, 2, 2, 0.0),          # k = 1
    (32768, 64, 8, 128, 0, 64, 0.5),     # 128 x 64 counts: the largest two-launch case
    (20000, 256, 8, 128, 0, 256, 0.3),   # count matrix above the fused-scan limit
    (3000, 1024, 32, 128, 0, 1024, 0.5),  # the largest E and k the ABI accepts
    (70000, 64, 8, 128, 0, 64, 1.0),     # T above 2^16, R = 560000 rows
])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_permute_bitexact(moe, T, E, k, align, e_first, E_local, skew, dt):
    D = 136
    idx = moe_inputs.random_topk_idx(T, E, k, seed=T + E, skew=skew)
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, e_first=e_first, E_local=E_local,
                     dtype=moe.MOE_BF16 if dt == torch.bfloat16 else moe.MOE_F32, align_m=align)
    x = torch.randn(T, D, device="cuda").to(dt)
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx)
    assert st == moe.MOE_OK
    lay = oracle.layout(idx, E, e_first, E_local, oracle.CONTIGUOUS, align)
    assert lay["status"] == oracle.OK
    assert np.array_equal(tpe, lay["tokens_per_expert"])
    assert np.array_equal(seg, lay["seg_offsets"])
    assert np.array_equal(row_of, lay["row_of"])
    assert np.array_equal(tor, lay["token_of_row"])
    filled = lay["token_of_row"] >= 0
    xh = moe_inputs.host_array(x)
    ref = oracle.permute_rows(xh, lay["token_of_row"])
    assert np.array_equal(moe_inputs.host_array(xp)[filled], ref[filled])   # bit for bit


def test_permute_workspace_reuse(moe):
    """Back-to-back permutes on one workspace: the count kernel's completion
    ticket returns to zero after every call, so each call's layout is exact."""
    T, E, k, D = 3000, 64, 6, 64
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(cfg)
    x = torch.randn(T, D, device="cuda").to(torch.bfloat16)
    for seed, skew in ((1, 0.0), (2, 1.2), (3, 0.4)):
        idx = moe_inputs.random_topk_idx(T, E, k, seed=seed, skew=skew)
        st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx, ws)
        assert st == moe.MOE_OK
        lay = oracle.layout(idx, E, 0, E, oracle.CONTIGUOUS, 128)
        assert np.array_equal(seg, lay["seg_offsets"])
        assert np.array_equal(row_of, lay["row_of"])
        assert np.array_equal(tor, lay["token_of_row"])


def test_permute_masked_and_capacity(moe):
    T, E, k, D = 400, 12, 3, 64
    idx = moe_inputs.random_topk_idx(T, E, k, seed=3, skew=1.0)
    cnt = np.bincount(idx.ravel(), minlength=E)
    cap = int(cnt.max())
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                     layout=moe.MOE_LAYOUT_MASKED, capacity=cap)
    x = torch.randn(T, D, device="cuda").to(torch.bfloat16)
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx)
    assert st == moe.MOE_OK
    lay = oracle.layout(idx, E, 0, E, oracle.MASKED, 1, cap)
    for a, b in ((tpe, "tokens_per_expert"), (seg, "seg_offsets"), (row_of, "row_of"),
                 (tor, "token_of_row")):
        assert np.array_equal(a, lay[b])
    check_layout_properties(idx, (tpe, seg, row_of, tor), E, 0, E, masked_cap=cap)
    # capacity exceeded (reading R7): the first `cap2` tokens of each expert
    # kept, the rest dropped and flagged -- the oracle's layout bit for bit
    cap2 = int(np.median(cnt))
    cfg2 = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                      layout=moe.MOE_LAYOUT_MASKED, capacity=cap2)
    st2, tpe2, seg2, row2, tor2, xp2 = _run_permute(moe, cfg2, x, idx)
    lay2 = oracle.layout(idx, E, 0, E, oracle.MASKED, 1, cap2)
    assert lay2["status"] == oracle.CAPACITY
    assert st2 == moe.MOE_ERR_CAPACITY
    for a, b in ((tpe2, "tokens_per_expert"), (seg2, "seg_offsets"), (row2, "row_of"),
                 (tor2, "token_of_row")):
        assert np.array_equal(a, lay2[b])
    filled = lay2["token_of_row"] >= 0
    ref = oracle.permute_rows(moe_inputs.host_array(x), lay2["token_of_row"])
    assert np.array_equal(moe_inputs.host_array(xp2)[filled], ref[filled])


@pytest.mark.parametrize("cap", [5, 1, 0])
def test_permute_masked_few_tokens(moe, cap):
    """Masked layout with fewer tokens than local experts, an expert range,
    and capacities that do (1, 0) and may not (5) overflow: every array equals
    the oracle's layout, whatever the status; unused capacity rows are -1."""
    T, E, k, D = 20, 48, 4, 64
    idx = moe_inputs.random_topk_idx(T, E, k, seed=12, skew=0.7)
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                     layout=moe.MOE_LAYOUT_MASKED, capacity=cap, e_first=4, E_local=40)
    x = torch.randn(T, D, device="cuda").to(torch.bfloat16)
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx)
    lay = oracle.layout(idx, E, 4, 40, oracle.MASKED, 1, cap)
    assert lay["status"] in (oracle.OK, oracle.CAPACITY)
    if cap < 2:
        assert lay["status"] == oracle.CAPACITY               # the case overflows
    assert st == (moe.MOE_OK if lay["status"] == oracle.OK else moe.MOE_ERR_CAPACITY)
    for a, b in ((tpe, "tokens_per_expert"), (seg, "seg_offsets"), (row_of, "row_of"),
                 (tor, "token_of_row")):
        assert np.array_equal(a, lay[b])


@pytest.mark.parametrize("layout", ["contiguous", "masked"])
def test_permute_bad_ids_flagged_and_skipped(moe, layout):
    """Reading R15: out-of-range, negative and repeated ids are skipped and
    flagged; the rest of the layout equals the oracle's bit for bit."""
    T, E, k, D = 100, 8, 2, 32
    idx = moe_inputs.random_topk_idx(T, E, k, seed=9)
    idx[5, 1] = E          # out of range
    idx[9, 0] = -3         # negative
    idx[11, 1] = idx[11, 0]  # duplicate expert within a token
    masked = layout == "masked"
    cap = T if masked else 0
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, dtype=moe.MOE_F32, align_m=4,
                     layout=moe.MOE_LAYOUT_MASKED if masked else moe.MOE_LAYOUT_CONTIGUOUS,
                     capacity=cap)
    x = torch.randn(T, D, device="cuda")
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx)
    assert st == moe.MOE_ERR_BAD_ROUTING
    lay = oracle.layout(idx, E, 0, E, oracle.MASKED if masked else oracle.CONTIGUOUS,
                        1 if masked else 4, cap)
    assert lay["status"] == oracle.BAD_ROUTING
    assert row_of[5, 1] == -1 and row_of[9, 0] == -1 and row_of[11, 1] == -1
    assert tpe.sum() == T * k - 3
    for a, b in ((tpe, "tokens_per_expert"), (seg, "seg_offsets"), (row_of, "row_of"),
                 (tor, "token_of_row")):
        assert np.array_equal(a, lay[b])
    filled = lay["token_of_row"] >= 0
    ref = oracle.permute_rows(moe_inputs.host_array(x), lay["token_of_row"])
    assert np.array_equal(moe_inputs.host_array(xp)[filled], ref[filled])


def test_permute_empty_batch(moe):
    cfg = moe.Config(T=0, D=64, H_local=8, E=8, k=2, dtype=moe.MOE_BF16)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, np.zeros((0, 2), np.int32))
    assert st == moe.MOE_OK
    assert (tpe == 0).all() and (seg == 0).all()
    assert (tor == -1).all()


# ------------------------------------------------------------------ grouped GEMMs

def _grouped_case(moe, dt, T, E_local, k, D, H, align, seed, skew=1.0):
    idx = moe_inputs.random_topk_idx(T, E_local, k, seed=seed, skew=skew)
    lay = oracle.layout(idx, E_local, 0, E_local, oracle.CONTIGUOUS, align)
    ra = lay["rows_alloc"]
    g = torch.Generator(device="cuda").manual_seed(seed)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    xp = torch.randn((ra, D), generator=g, device="cuda").to(tdt)
    w1 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(tdt)
    w3 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(tdt)
    w2 = (torch.randn((E_local, D, H), generator=g, device="cuda") * 0.05).to(tdt)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=k, align_m=align,
                     dtype=moe.MOE_BF16 if dt == "bf16" else moe.MOE_F32)
    assert moe.rows_alloc(cfg) == ra
    ws = moe.alloc_workspace(cfg)
    h = torch.full((ra, H), float("nan"), device="cuda").to(tdt)
    y = torch.full((ra, D), float("nan"), device="cuda").to(cfg.y_dtype)
    moe.moe_grouped_swiglu(cfg, xp, _dev(lay["seg_offsets"]), _dev(lay["tokens_per_expert"]),
                           w1, w3, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    return lay, xp, w1, w3, w2, h, y


@pytest.mark.parametrize("dt,T,E_local,k,D,H,align", [
    ("bf16", 700, 6, 2, 640, 200, 128),   # N tails (640 = 2.5 x 256, 200 = 1.56 x 128), K tail
    ("bf16", 1500, 9, 3, 512, 384, 128),  # several m-tiles per expert, empty experts
    ("bf16", 333, 5, 2, 256, 128, 1),     # unpadded segments: tiles start mid-buffer
    ("bf16", 900, 4, 1, 1024, 256, 64),   # k = 1, segments aligned to half a tile
    ("f32", 600, 6, 2, 128, 256, 128),
    ("f32", 301, 7, 3, 136, 72, 8),
])
@pytest.mark.parametrize("kernel", ["pair", "pair2", "single"])
def test_grouped_swiglu_parity(moe, dt, T, E_local, k, D, H, align, kernel, monkeypatch):
    # bf16: the CTA-pair (cta_group::2) kernel in one launch (GEMM1 and GEMM2
    # tiles interleaved) and in two, and the one-CTA-per-tile kernel
    if dt == "f32" and kernel != "pair":
        pytest.skip("one fp32 implementation")
    monkeypatch.setenv("MOE_GROUPED_KERNEL", kernel)
    lay, xp, w1, w3, w2, h, y = _grouped_case(moe, dt, T, E_local, k, D, H, align, seed=T + H)
    _assert_grouped_parity(lay, xp, w1, w3, w2, h, y, dt == "bf16")


@pytest.mark.parametrize("kernel", ["pair", "pair2", "single"])
def test_grouped_tile_shapes(moe, kernel, monkeypatch):
    """Every tile shape the grouped kernels choose from, by exact expert
    counts: transposed tail tiles (1..128 valid rows, N = 32..128), full
    tiles with partial rows (129..255), several tiles per expert, empty
    experts; H and D with N tails."""
    counts = [1, 31, 32, 33, 0, 64, 96, 127, 128, 129, 200, 255, 256, 257, 384, 0, 500, 17]
    E_local, D, H = len(counts), 320, 192
    idx = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]
    idx = idx[np.random.default_rng(3).permutation(len(idx))]
    T = len(idx)
    lay = oracle.layout(idx, E_local, 0, E_local, oracle.CONTIGUOUS, 128)
    assert lay["tokens_per_expert"].tolist() == counts
    monkeypatch.setenv("MOE_GROUPED_KERNEL", kernel)
    ra = lay["rows_alloc"]
    g = torch.Generator(device="cuda").manual_seed(11)
    xp = torch.randn((ra, D), generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w3 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E_local, D, H), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=1, align_m=128, dtype=moe.MOE_BF16)
    assert moe.rows_alloc(cfg) == ra
    ws = moe.alloc_workspace(cfg)
    h = torch.full((ra, H), float("nan"), device="cuda").to(torch.bfloat16)
    y = torch.full((ra, D), float("nan"), device="cuda").to(cfg.y_dtype)
    moe.moe_grouped_swiglu(cfg, xp, _dev(lay["seg_offsets"]), _dev(lay["tokens_per_expert"]),
                           w1, w3, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    _assert_grouped_parity(lay, xp, w1, w3, w2, h, y, True)


def _grouped_run(moe, cfg, lay, xp, w1, w3, w2, ws):
    ra, H, D = lay["rows_alloc"], cfg.H_local, cfg.D
    h = torch.full((ra, H), float("nan"), device="cuda").to(torch.bfloat16)
    y = torch.full((ra, D), float("nan"), device="cuda").to(cfg.y_dtype)
    before = moe.kernel_launches()
    moe.moe_grouped_swiglu(cfg, xp, _dev(lay["seg_offsets"]), _dev(lay["tokens_per_expert"]),
                           w1, w3, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    return h, y, moe.kernel_launches() - before


@pytest.mark.parametrize("T,E_local,k,D,H,skew", [
    (1500, 9, 3, 512, 384, 1.0),
    (4096, 64, 6, 2048, 1408, 1.0),    # the fine-grained layer's shapes
    (3000, 16, 4, 768, 640, 1.5),      # skewed: a few long segments, several empty
])
def test_grouped_one_launch_equals_two(moe, T, E_local, k, D, H, skew, monkeypatch):
    """The one-launch schedule (GEMM2 tiles wait on per-block GEMM1 counters)
    gives bit-identical h and y to GEMM1 and GEMM2 run as two launches, also
    when the workspace (and its counters) was used by a different problem
    just before."""
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=k, align_m=128, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(cfg)
    cases = []
    for seed in (5, 6):
        idx = moe_inputs.random_topk_idx(T, E_local, k, seed=seed, skew=skew)
        lay = oracle.layout(idx, E_local, 0, E_local, oracle.CONTIGUOUS, 128)
        g = torch.Generator(device="cuda").manual_seed(seed)
        xp = torch.randn((lay["rows_alloc"], D), generator=g, device="cuda").to(torch.bfloat16)
        ws_ = [(torch.randn(s, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
               for s in ((E_local, H, D), (E_local, H, D), (E_local, D, H))]
        cases.append((lay, xp, ws_))
    monkeypatch.setenv("MOE_GROUPED_KERNEL", "pair")
    for lay, xp, (w1, w3, w2) in cases:
        h1, y1, n1 = _grouped_run(moe, cfg, lay, xp, w1, w3, w2, ws)
    assert n1 == 1
    monkeypatch.setenv("MOE_GROUPED_KERNEL", "pair2")
    h2, y2, n2 = _grouped_run(moe, cfg, lay, xp, w1, w3, w2, ws)
    assert n2 == 2
    filled = torch.from_numpy(lay["token_of_row"] >= 0).cuda()
    assert torch.equal(h1[filled], h2[filled])
    assert torch.equal(y1[filled], y2[filled])
    assert torch.isnan(y1[~filled]).all()


def test_grouped_overlapping_segments_flagged(moe):
    """Segments that overlap cover more 256-row blocks than the buffer has;
    the one-launch schedule then computes nothing and flags the routing."""
    E_local, D, H, T = 3, 128, 128, 1024
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=1, dtype=moe.MOE_BF16)
    ra = moe.rows_alloc(cfg)
    ws = moe.alloc_workspace(cfg)
    seg = _dev(np.array([0, ra, 0, ra], np.int32))   # experts 0 and 2 both claim every row
    cnt = _dev(np.array([ra, 0, ra], np.int32))
    xp = torch.zeros((ra, D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((E_local, H, D), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((E_local, D, H), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((ra, H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((ra, D), dtype=cfg.y_dtype, device="cuda")
    moe.moe_grouped_swiglu(cfg, xp, seg, cnt, w, w, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BAD_ROUTING


def test_grouped_swiglu_bad_offsets_flagged(moe):
    E_local, D, H = 3, 128, 128
    cfg = moe.Config(T=64, D=D, H_local=H, E=E_local, k=1, dtype=moe.MOE_BF16)
    ra = moe.rows_alloc(cfg)
    ws = moe.alloc_workspace(cfg)
    seg = _dev(np.array([0, 128, 64, ra + 500], np.int32))     # decreasing, then out of range
    cnt = _dev(np.array([10, 10, 10], np.int32))
    xp = torch.zeros((ra, D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((E_local, H, D), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((E_local, D, H), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((ra, H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((ra, D), dtype=cfg.y_dtype, device="cuda")
    moe.moe_grouped_swiglu(cfg, xp, seg, cnt, w, w, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BAD_ROUTING


@pytest.mark.parametrize("kernel", ["pair", "pair2", "single"])
def test_grouped_fp16_range_flagged(moe, kernel, monkeypatch):
    """A bf16 layer stores y_perm in fp16.  An expert whose outputs exceed
    fp16's range (|y| >= 65520 rounds to infinity) must be reported
    (MOE_ERR_UNSUPPORTED), whether its tile is a transposed tail (20 rows),
    a full tile or an M=128 tail (300 rows); the flag is cleared by the read
    and the next in-range call reports MOE_OK."""
    counts = [20, 64, 300, 130]
    E_local, D, H = len(counts), 320, 192
    idx = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]
    idx = idx[np.random.default_rng(5).permutation(len(idx))]
    T = len(idx)
    lay = oracle.layout(idx, E_local, 0, E_local, oracle.CONTIGUOUS, 128)
    monkeypatch.setenv("MOE_GROUPED_KERNEL", kernel)
    ra = lay["rows_alloc"]
    g = torch.Generator(device="cuda").manual_seed(12)
    xp = torch.randn((ra, D), generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w3 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E_local, D, H), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=1, align_m=128, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(cfg)
    seg, cnt = _dev(lay["seg_offsets"]), _dev(lay["tokens_per_expert"])
    h = torch.empty((ra, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((ra, D), dtype=cfg.y_dtype, device="cuda")
    assert y.dtype == torch.float16
    for big in ([0], [2], [0, 2]):
        w2b = w2.clone()
        for e in big:
            w2b[e] = (w2b[e].float() * 4.0e5).to(torch.bfloat16)
        moe.moe_grouped_swiglu(cfg, xp, seg, cnt, w1, w3, w2b, h, y, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_ERR_UNSUPPORTED, big
        for e in big:
            rows = slice(int(lay["seg_offsets"][e]), int(lay["seg_offsets"][e]) + counts[e])
            assert torch.isinf(y[rows]).any()
        # the status word was cleared by the read; an in-range call is clean
        moe.moe_grouped_swiglu(cfg, xp, seg, cnt, w1, w3, w2, h, y, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        assert torch.isfinite(y[torch.from_numpy(lay["token_of_row"] >= 0).cuda()]).all()


# ------------------------------------------------------------------ combine

@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("T,E,k,D,e_first,E_local", [(513, 16, 4, 264, 0, 16), (200, 64, 8, 2048, 16, 32),
                                                     (77, 4, 1, 8, 0, 4), (300, 32, 12, 136, 0, 32),
                                                     (41, 8, 3, 3080, 0, 8)])
def test_combine_parity(moe, dt, T, E, k, D, e_first, E_local):
    idx = moe_inputs.random_topk_idx(T, E, k, seed=T)
    lay = oracle.layout(idx, E, e_first, E_local, oracle.CONTIGUOUS, 128)
    ra = lay["rows_alloc"]
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    w = moe_inputs.random_weights(T, k, seed=T)
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, e_first=e_first, E_local=E_local,
                     dtype=moe.MOE_BF16 if dt == "bf16" else moe.MOE_F32)
    y = torch.randn((ra, D), device="cuda").to(cfg.y_dtype)     # fp16 (bf16 layers) or fp32
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((T, D), dtype=tdt, device="cuda")
    moe.moe_unpermute_combine(cfg, y, _dev(lay["row_of"]), _dev(w), out, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    yh = y.double().cpu().numpy()                                # exact
    ref = oracle.unpermute_combine(yh, lay["row_of"], w.astype(np.float64))
    # bound: fp32 accumulation error (k terms) plus one final rounding (one ulp)
    yabs = np.abs(to_f64(y))
    mag = oracle.unpermute_combine(yabs, lay["row_of"], np.abs(w).astype(np.float64))
    got = to_f64(out)
    ulp = 2.0 ** -7 if dt == "bf16" else 2.0 ** -23
    assert (np.abs(got - ref) <= ulp * np.abs(ref) + 2 * k * 2.0 ** -24 * mag).all()
    none_local = (lay["row_of"] < 0).all(1)
    assert (got[none_local] == 0).all()


def test_permute_then_combine_is_identity(moe):
    T, E, D = 999, 24, 520
    idx = moe_inputs.random_topk_idx(T, E, 1, seed=1)
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=1, dtype=moe.MOE_BF16)
    # multiples of 1/8 up to 16: exact in bf16, in the fp16 of y_perm and in fp32
    x = (torch.randint(-128, 129, (T, D), device="cuda").float() / 8).to(torch.bfloat16)
    st, tpe, seg, row_of, tor, xp = _run_permute(moe, cfg, x, idx)
    assert st == moe.MOE_OK
    out = torch.empty_like(x)
    ws = moe.alloc_workspace(cfg)
    moe.moe_unpermute_combine(cfg, xp.to(cfg.y_dtype), _dev(row_of), torch.ones((T, 1), device="cuda"),
                              out, ws)
    assert torch.equal(out, x)
