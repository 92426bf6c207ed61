"""GPU parity of the FP8 e4m3 dispatch and GEMM1 against the CPU oracle.

The quantisation is integer work decided in binary32 on both sides (one
scale amax / 448 per row, codes of the correctly rounded quotients), so the
codes and scales are compared bit for bit.  The FP8 grouped GEMM then runs
on exactly the values value(code) * scale that the oracle evaluates in fp64:
h (bf16) is compared per element within one bf16 rounding, y through the
bound the bf16 path uses, and the layer output within the bf16 layer's
tolerance (max error <= 2e-2 of the RMS).
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import (cfg_for, oracle_route, rel_err, routing_agreement, to_f64,
                     within_bf16_rounding)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _dev(a, dtype=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def _np(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 2048), (300, 336)])
def test_quantize_rows_bitexact(moe, rows, cols):
    g = torch.Generator(device="cuda").manual_seed(rows)
    x = torch.randn((rows, cols), generator=g, device="cuda")
    x = x * torch.exp(torch.empty((rows, 1), device="cuda").uniform_(-8, 8, generator=g))
    if rows > 3:
        x[1] = 0.0                                    # all-zero row: scale 1, codes 0
        x[2, : cols // 2] = 1e-30                     # far below the row's largest value
    x = x.to(torch.bfloat16)
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows,), dtype=torch.float32, device="cuda")
    moe.moe_quantize_rows_fp8(x, q, s)
    torch.cuda.synchronize()
    oq, osc = oracle.quantize_rows_e4m3(moe_inputs.host_array(x))
    assert np.array_equal(_np(s), osc)
    assert np.array_equal(_np(q), oq)


def _weights_fp8(moe, w):
    q, s = moe.quantize_weights_fp8(w)
    E, H, D = w.shape
    oq, osc = oracle.quantize_rows_e4m3(moe_inputs.host_array(w).reshape(E * H, D))
    assert np.array_equal(_np(q).reshape(E * H, D), oq)
    assert np.array_equal(_np(s).reshape(E * H), osc)
    return q, s


@pytest.mark.parametrize("T,E,k,D,align", [(700, 16, 4, 512, 128), (333, 5, 2, 336, 1)])
def test_permute_fp8_bitexact(moe, T, E, k, D, align):
    idx = moe_inputs.random_topk_idx(T, E, k, seed=T)
    g = torch.Generator(device="cuda").manual_seed(T)
    x = torch.randn((T, D), generator=g, device="cuda").to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=64, E=E, k=k, align_m=align, dtype=moe.MOE_BF16)
    ra = moe.rows_alloc(cfg)
    ws = moe.alloc_workspace(cfg)
    outs = {}
    for fp8 in (False, True):
        tpe = torch.empty(E, dtype=torch.int32, device="cuda")
        seg = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        row_of = torch.empty((T, k), dtype=torch.int32, device="cuda")
        tor = torch.empty(ra, dtype=torch.int32, device="cuda")
        if fp8:
            xq = torch.zeros((ra, D), dtype=torch.uint8, device="cuda")
            xs = torch.full((ra,), -1.0, device="cuda")
            moe.moe_permute_fp8(cfg, x, _dev(idx), tpe, seg, row_of, tor, xq, xs, ws)
        else:
            xp = torch.empty((ra, D), dtype=torch.bfloat16, device="cuda")
            moe.moe_permute(cfg, x, _dev(idx), tpe, seg, row_of, tor, xp, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        outs[fp8] = [_np(t) for t in (tpe, seg, row_of, tor)]
    # the layout is the bf16 permute's, bit for bit
    for a, b in zip(outs[False], outs[True]):
        assert np.array_equal(a, b)
    tor = outs[True][3]
    filled = tor >= 0
    oq, osc = oracle.quantize_rows_e4m3(moe_inputs.host_array(x))
    assert np.array_equal(_np(xq)[filled], oq[tor[filled]])
    assert np.array_equal(_np(xs)[filled], osc[tor[filled]])
    assert (_np(xs)[~filled] == -1.0).all()            # rows without a token untouched


def _fp8_grouped_parity(lay, xq, xs, w1q, w1s, w3q, w3s, w2, h, y):
    H_ = moe_inputs.host_array
    seg, cnt = lay["seg_offsets"], lay["tokens_per_expert"]
    E_local = len(cnt)
    filled = lay["token_of_row"] >= 0
    xd = np.zeros(xq.shape, np.float64)
    xd[filled] = oracle.dequantize_rows_e4m3(_np(xq)[filled], _np(xs)[filled])
    w1d = [oracle.dequantize_rows_e4m3(_np(w1q[i]), _np(w1s[i])) for i in range(E_local)]
    w3d = [oracle.dequantize_rows_e4m3(_np(w3q[i]), _np(w3s[i])) for i in range(E_local)]
    oh = oracle.grouped_gemm1_swiglu(xd, seg, cnt, w1d, w3d, round_h=True)
    gh = to_f64(h)
    assert within_bf16_rounding(gh[filled], oh[filled]) <= 1.0
    # GEMM2 (bf16) from the oracle's own h
    oy = oracle.grouped_gemm2(oh.astype(np.float32), seg, cnt, list(H_(w2)))
    gy = to_f64(y)
    w2h = to_f64(w2)
    dh = np.abs(np.nan_to_num(gh) - np.nan_to_num(oh))
    for i in range(E_local):
        rows = np.arange(seg[i], seg[i] + cnt[i])
        if len(rows) == 0:
            continue
        aw2 = np.abs(w2h[i])
        bound = dh[rows] @ aw2.T + 2.0 ** -20 * (np.abs(oh[rows]) @ aw2.T) + 1e-30
        # plus y's one rounding to fp16 (2^-11 relative, 2^-25 absolute below 2^-14)
        bound = bound + 2.0 ** -11 * (np.abs(oy[rows]) + bound) + 2.0 ** -25
        assert (np.abs(gy[rows] - oy[rows]) <= bound).all(), f"expert {i}"
    tail = ~filled
    if tail.any():
        tt = torch.from_numpy(tail).cuda()
        assert torch.isnan(h.float()[tt]).all() and torch.isnan(y[tt]).all()


@pytest.mark.parametrize("kernel", ["pair", "pair2"])
def test_grouped_fp8_tile_shapes(moe, kernel, monkeypatch):
    """Every tile shape of the pair kernel (transposed tails of 1..32 rows,
    M=128 tiles, full and partial 256-row tiles, several per expert, empty
    experts) with e4m3 GEMM1, a K tail (D = 2.5 K blocks of 128) and N tails."""
    counts = [1, 31, 32, 33, 0, 64, 96, 127, 128, 129, 200, 255, 256, 257, 384, 0, 500, 17]
    E_local, D, H = len(counts), 320, 192
    idx = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]
    idx = idx[np.random.default_rng(3).permutation(len(idx))]
    T = len(idx)
    lay = oracle.layout(idx, E_local, 0, E_local, oracle.CONTIGUOUS, 128)
    monkeypatch.setenv("MOE_GROUPED_KERNEL", kernel)
    ra = lay["rows_alloc"]
    g = torch.Generator(device="cuda").manual_seed(12)
    xsrc = torch.randn((ra, D), generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w3 = (torch.randn((E_local, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E_local, D, H), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    xq = torch.empty((ra, D), dtype=torch.uint8, device="cuda")
    xs = torch.empty((ra,), dtype=torch.float32, device="cuda")
    moe.moe_quantize_rows_fp8(xsrc, xq, xs)
    w1q, w1s = _weights_fp8(moe, w1)
    w3q, w3s = _weights_fp8(moe, w3)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E_local, k=1, align_m=128, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(cfg)
    h = torch.full((ra, H), float("nan"), device="cuda").to(torch.bfloat16)
    y = torch.full((ra, D), float("nan"), device="cuda").to(cfg.y_dtype)
    moe.moe_grouped_swiglu_fp8(cfg, xq, xs, _dev(lay["seg_offsets"]), _dev(lay["tokens_per_expert"]),
                               w1q, w1s, w3q, w3s, w2, h, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    _fp8_grouped_parity(lay, xq, xs, w1q, w1s, w3q, w3s, w2, h, y)


@pytest.mark.parametrize("name,over,n_sample", [
    ("fine-grained-bf16", dict(T=640), 96),
    ("fine-grained-bf16", dict(), 24),      # the benchmark's FP8 step at full size, sampled
    ("deepseek-v3-shaped", dict(T=300), 12),
    ("decode-masked", dict(), 16),           # masked layout, capacity = T
])
def test_layer_fp8_matches_oracle(moe, name, over, n_sample):
    w = moe_inputs.WORKLOADS[name].scaled(**over)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=2)
    cfg = cfg_for(moe, w)
    w1q, w1s = _weights_fp8(moe, inp.w1)
    w3q, w3s = _weights_fp8(moe, inp.w3)
    ws = moe.alloc_workspace(cfg, layer=True)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward_fp8(cfg, inp.x, inp.wg, inp.bias, w1q, w1s, w3q, w3s, inp.w2, out, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    views = moe.layer_views(cfg, ws)
    # routing: the bf16 router on the bf16 x
    l64, keys, oidx, owts, st = oracle_route(inp, w, inp.bias)
    gidx = views["topk_idx"].cpu().numpy()
    same_set, _ = routing_agreement(gidx, oidx, keys, key_tol=1e-3)
    assert same_set.mean() > 0.99
    rng = np.random.default_rng(0)
    cand = np.nonzero(same_set)[0]
    toks = np.sort(rng.choice(cand, size=min(n_sample, len(cand)), replace=False))
    # the experts evaluated on value(code) * scale: tokens' rows of x and the used experts' rows
    xq, xs = oracle.quantize_rows_e4m3(moe_inputs.host_array(inp.x))
    xd = oracle.dequantize_rows_e4m3(xq, xs)
    used = set(int(e) for e in np.unique(oidx[toks]))
    w1d, w3d, w2h = [], [], []
    for e in range(w.E):
        if e in used:
            w1d.append(oracle.dequantize_rows_e4m3(_np(w1q[e]), _np(w1s[e])))
            w3d.append(oracle.dequantize_rows_e4m3(_np(w3q[e]), _np(w3s[e])))
            w2h.append(to_f64(inp.w2[e]))
        else:
            w1d.append(None); w3d.append(None); w2h.append(None)
    ref = oracle.moe_tokens(toks, xd, w1d, w3d, w2h, oidx, owts, round_h=True)
    got = to_f64(out)[toks]
    err = rel_err(got, ref)
    assert err < 2e-2, f"{name}: max err / rms = {err:.3e}"
    # the layer's codes and scales are the oracle's (bit for bit)
    tor = views["token_of_row"].cpu().numpy()
    filled = tor >= 0
    assert np.array_equal(views["x_perm_q"].cpu().numpy()[filled], xq[tor[filled]])
    assert np.array_equal(views["x_scale"].cpu().numpy()[filled], xs[tor[filled]])
    # and the FP8 output stays close to the bf16 layer's (quantisation error only)
    out16 = torch.empty_like(out)
    ws16 = moe.alloc_workspace(cfg, layer=True)
    moe.moe_layer_forward(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out16, ws16)
    a, b = to_f64(out), to_f64(out16)
    assert np.sqrt(np.mean((a - b) ** 2)) / np.sqrt(np.mean(b ** 2)) < 0.1


def test_fp8_rejects_unsupported(moe):
    cfg = moe.Config(T=8, D=24, H_local=64, E=4, k=2, dtype=moe.MOE_BF16)   # D % 16 != 0
    ws = moe.alloc_workspace(cfg, layer=True)
    x = torch.zeros((8, 24), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((4, 64, 24), dtype=torch.uint8, device="cuda")
    s = torch.ones((4, 64), device="cuda")
    w2 = torch.zeros((4, 24, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    with pytest.raises(moe.MoeError):
        moe.moe_layer_forward_fp8(cfg, x, wg, None, q, s, q, s, w2, out, ws)


def test_layer_fp8_expert_ranges_sum_to_layer(moe):
    """Expert-range shards of the FP8 layer add up to the whole FP8 layer."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=512, D=512, H=256, E=16)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=6)
    w1q, w1s = _weights_fp8(moe, inp.w1)
    w3q, w3s = _weights_fp8(moe, inp.w3)

    def run(cfg, e0, el):
        ws = moe.alloc_workspace(cfg, layer=True)
        out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device="cuda")
        moe.moe_layer_forward_fp8(cfg, inp.x, inp.wg, inp.bias, w1q[e0:e0 + el], w1s[e0:e0 + el],
                                  w3q[e0:e0 + el], w3s[e0:e0 + el], inp.w2[e0:e0 + el], out, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        return out.double()

    full = run(cfg_for(moe, w), 0, w.E)
    total = sum(run(cfg_for(moe, w, e_first=e0, E_local=8), e0, 8) for e0 in (0, 8))
    rms = full.pow(2).mean().sqrt().item()
    assert (total - full).abs().max().item() <= 2e-2 * rms
