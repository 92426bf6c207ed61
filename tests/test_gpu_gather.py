"""The dispatch fused into GEMM1's operand load: no x_perm.

moe_permute_index writes the layout without copying rows, and
moe_grouped_swiglu_gather reads row r of the layout as x[token_of_row[r]]
(gather warps of the CTA-pair kernel copy the rows into the swizzled stages
TMA would have filled).  Every output must equal the copy path's bit for
bit -- the A operand bytes are the same -- and the oracle's within the
grouped GEMM's bounds.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import assert_grouped_parity, cfg_for, check_layout_properties

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _layouts(moe, cfg, x, idx, ws):
    """The layout by moe_permute (with x_perm) and by moe_permute_index."""
    ra = moe.rows_alloc(cfg)
    out = []
    for copy in (True, False):
        tpe = torch.full((cfg.E,), -9, dtype=torch.int32, device="cuda")
        seg = torch.full((cfg.e_local + 1,), -9, dtype=torch.int32, device="cuda")
        row_of = torch.full((cfg.T, cfg.k), -9, dtype=torch.int32, device="cuda")
        tor = torch.full((ra,), -9, dtype=torch.int32, device="cuda")
        if copy:
            xp = torch.full((ra, cfg.D), float("nan"), device="cuda").to(x.dtype)
            moe.moe_permute(cfg, x, idx, tpe, seg, row_of, tor, xp, ws)
        else:
            xp = None
            moe.moe_permute_index(cfg, idx, tpe, seg, row_of, tor, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        out.append((tpe, seg, row_of, tor, xp))
    return out


def _grouped_both(moe, cfg, x, lay_copy, lay_idx, w1, w3, w2, ws):
    ra = moe.rows_alloc(cfg)
    res = []
    for gather in (False, True):
        tpe, seg, row_of, tor, xp = lay_idx if gather else lay_copy
        h = torch.full((ra, cfg.H_local), float("nan"), device="cuda").to(torch.bfloat16)
        y = torch.full((ra, cfg.D), float("nan"), device="cuda").to(cfg.y_dtype)
        if gather:
            moe.moe_grouped_swiglu_gather(cfg, x, tor, seg, tpe, w1, w3, w2, h, y, ws)
        else:
            moe.moe_grouped_swiglu(cfg, xp, seg, tpe, w1, w3, w2, h, y, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        res.append((h, y))
    return res


def _check_case(moe, cfg, x, idx, w1, w3, w2, align):
    ws = moe.alloc_workspace(cfg)
    lay_copy, lay_idx = _layouts(moe, cfg, x, _dev(idx), ws)
    # the layout without the copy is the layout with it, and the oracle's
    for a, b in zip(lay_copy[:4], lay_idx[:4]):
        assert torch.equal(a, b)
    lay = oracle.layout(idx, cfg.E, cfg.e_first, cfg.e_local, oracle.CONTIGUOUS, align)
    assert lay["status"] == oracle.OK
    for a, key in zip(lay_idx[:4], ("tokens_per_expert", "seg_offsets", "row_of", "token_of_row")):
        assert np.array_equal(a.cpu().numpy(), lay[key]), key
    (h0, y0), (h1, y1) = _grouped_both(moe, cfg, x, lay_copy, lay_idx, w1, w3, w2, ws)
    filled = torch.from_numpy(lay["token_of_row"] >= 0).cuda()
    assert torch.equal(h1[filled], h0[filled])                 # bit for bit
    assert torch.equal(y1[filled], y0[filled])
    assert torch.isnan(y1[~filled]).all()                     # no row without a token is written
    # and against the oracle, on the rows the layout names (a copy made by the oracle)
    xp_o = oracle.permute_rows(moe_inputs.host_array(x), lay["token_of_row"])
    xp_t = torch.from_numpy(xp_o.view(np.int16)).view(torch.bfloat16).cuda()
    lay_local = dict(lay)
    lay_local["tokens_per_expert"] = lay["tokens_per_expert"][cfg.e_first:cfg.e_first + cfg.e_local]
    assert_grouped_parity(lay_local, xp_t, w1, w3, w2, h1, y1, True)


def _weights(E_local, H, D, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return [(torch.randn(s, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
            for s in ((E_local, H, D), (E_local, H, D), (E_local, D, H))]


@pytest.mark.parametrize("kernel", ["pair", "pair2"])
def test_gather_tile_shapes(moe, kernel, monkeypatch):
    """Every tile shape of the pair kernel by exact expert counts: transposed
    tails (1..32 rows, token rows in the B slot), M=128 tails (33..128),
    partial and several full tiles, empty experts; D = 328 leaves a K tail
    of 8 columns that the gather zero-fills; one launch and two."""
    monkeypatch.setenv("MOE_GROUPED_KERNEL", kernel)
    counts = [1, 31, 32, 33, 0, 64, 96, 127, 128, 129, 200, 255, 256, 257, 384, 0, 500, 17]
    E, D, H = len(counts), 328, 192
    idx = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]
    idx = idx[np.random.default_rng(3).permutation(len(idx))]
    T = len(idx)
    g = torch.Generator(device="cuda").manual_seed(4)
    x = torch.randn((T, D), generator=g, device="cuda").to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E, k=1, align_m=128, dtype=moe.MOE_BF16)
    _check_case(moe, cfg, x, idx, *_weights(E, H, D, 5), 128)


@pytest.mark.parametrize("T,E,k,D,H,align,skew,e_first,E_local", [
    (700, 6, 2, 640, 200, 128, 1.0, 0, 6),      # N tails, K tail
    (333, 5, 2, 256, 128, 1, 1.0, 0, 5),        # unpadded segments: tiles start mid-buffer
    (900, 4, 1, 1024, 256, 64, 1.0, 0, 4),      # k = 1, half-tile alignment
    (2000, 32, 8, 512, 256, 128, 0.8, 8, 12),   # an expert range
    (4096, 64, 6, 2048, 1408, 128, 0.0, 0, 64),  # the fine-grained layer's shapes
])
def test_gather_random_routing(moe, T, E, k, D, H, align, skew, e_first, E_local):
    idx = moe_inputs.random_topk_idx(T, E, k, seed=T + E, skew=skew)
    g = torch.Generator(device="cuda").manual_seed(T)
    x = torch.randn((T, D), generator=g, device="cuda").to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E, k=k, e_first=e_first, E_local=E_local,
                     align_m=align, dtype=moe.MOE_BF16)
    _check_case(moe, cfg, x, idx, *_weights(E_local, H, D, T + 1), align)


def test_permute_index_chain_and_masked(moe):
    """moe_permute_index on the four-launch chain (above 16384 count cells)
    and on the masked layout with capacity overflow: the layout and status
    of moe_permute, without touching x_perm."""
    for T, E, k, layout, cap in ((20000, 256, 8, "contiguous", 0), (400, 12, 3, "masked", 90)):
        idx = moe_inputs.random_topk_idx(T, E, k, seed=7, skew=1.0)
        cfg = moe.Config(T=T, D=64, H_local=8, E=E, k=k, dtype=moe.MOE_BF16,
                         layout=moe.MOE_LAYOUT_MASKED if layout == "masked" else moe.MOE_LAYOUT_CONTIGUOUS,
                         capacity=cap)
        ws = moe.alloc_workspace(cfg)
        ra = moe.rows_alloc(cfg)
        tpe = torch.empty(E, dtype=torch.int32, device="cuda")
        seg = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        row_of = torch.empty((T, k), dtype=torch.int32, device="cuda")
        tor = torch.empty(ra, dtype=torch.int32, device="cuda")
        moe.moe_permute_index(cfg, _dev(idx), tpe, seg, row_of, tor, ws)
        st = moe.moe_get_device_status(ws)
        lay = oracle.layout(idx, E, 0, E, oracle.MASKED if layout == "masked" else oracle.CONTIGUOUS,
                            1 if layout == "masked" else 128, cap)
        assert st == (moe.MOE_ERR_CAPACITY if lay["status"] == oracle.CAPACITY else moe.MOE_OK)
        for a, key in ((tpe, "tokens_per_expert"), (seg, "seg_offsets"), (row_of, "row_of"),
                       (tor, "token_of_row")):
            assert np.array_equal(a.cpu().numpy(), lay[key]), key


LAYER_CASES = [
    ("fine-grained-bf16", dict(T=1024)),
    ("deepseek-v3-shaped", dict(T=512, E=64, D=1024, H=512)),
    ("zipf-skewed", dict(T=2048, D=1024, H=512)),
    ("decode-masked", dict()),
    ("fine-grained-bf16", dict(T=700, n_group=8, topk_group=3)),
]


@pytest.mark.parametrize("name,over", LAYER_CASES)
def test_layer_forward_gather_equals_forward(moe, name, over):
    """moe_layer_forward_gather gives moe_layer_forward's output bit for bit
    (the decode layout included: the gather always runs the pair kernel, so
    the copy path is forced onto it too for the comparison)."""
    w = moe_inputs.WORKLOADS[name].scaled(**over)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=21)
    cfg = cfg_for(moe, w)
    outs = []
    for fn in (moe.moe_layer_forward, moe.moe_layer_forward_gather):
        ws = moe.alloc_workspace(cfg, layer=True)
        out = torch.full((w.T, w.D), float("nan"), device="cuda").to(torch.bfloat16)
        fn(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        outs.append((out, moe.layer_views(cfg, ws)))
    (o0, v0), (o1, v1) = outs
    for key in ("topk_idx", "tokens_per_expert", "seg_offsets", "row_of", "token_of_row"):
        assert torch.equal(v0[key], v1[key]), key
    if w.layout == "masked":
        # the copy path ran the one-CTA-per-tile kernel: compare within h's rounding
        d = (o1.float() - o0.float()).abs().max().item()
        rms = o0.float().pow(2).mean().sqrt().item()
        assert d <= 2e-2 * rms
    else:
        assert torch.equal(o1, o0)
    idx = v1["topk_idx"].cpu().numpy()
    lay = (v1["tokens_per_expert"].cpu().numpy(), v1["seg_offsets"].cpu().numpy(),
           v1["row_of"].cpu().numpy(), v1["token_of_row"].cpu().numpy())
    if w.layout == "masked":
        check_layout_properties(idx, lay, w.E, 0, w.E, masked_cap=cfg.capacity)
    else:
        check_layout_properties(idx, lay, w.E, 0, w.E, align_m=cfg.align_m)


def test_layer_forward_gather_decode_on_pair_kernel_bitwise(moe, monkeypatch):
    """With the copy path forced onto the pair kernel too, the masked decode
    layout's outputs are bitwise equal as well."""
    monkeypatch.setenv("MOE_GROUPED_KERNEL", "pair")
    w = moe_inputs.WORKLOADS["decode-masked"].scaled(E=64, D=1024, H=512)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=22)
    cfg = cfg_for(moe, w)
    outs = []
    for fn in (moe.moe_layer_forward, moe.moe_layer_forward_gather):
        ws = moe.alloc_workspace(cfg, layer=True)
        out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device="cuda")
        fn(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_gather_rejects_fp32(moe):
    w = moe_inputs.WORKLOADS["tiny-fp32"]
    inp = moe_inputs.make_inputs(w, device="cuda", seed=1)
    cfg = cfg_for(moe, w)
    ws = moe.alloc_workspace(cfg, layer=True)
    out = torch.empty((w.T, w.D), device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_layer_forward_gather(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, ws)
