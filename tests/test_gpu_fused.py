"""GPU parity of moe_layer_forward_fused (the combine fused into GEMM2's
epilogue with fp32 atomic adds) against the CPU oracle and the unfused layer.

The fused layer computes the same sums as moe_layer_forward, but the slots of
a token are added in the order their tiles finish: it is held to the same
oracle tolerance as the bf16 layer, and against the unfused output to one
bf16 rounding per element (the fp32 sums differ by reassociation only).
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_inputs
from helpers import cfg_for, to_f64
from test_gpu_layer import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def run_fused(moe, cfg, inp, w1=None, w3=None, w2=None):
    ws = moe.alloc_workspace(cfg, layer=True)
    out = torch.full((cfg.T, cfg.D), float("nan"), device="cuda").to(torch.bfloat16)
    moe.moe_layer_forward_fused(cfg, inp.x, inp.wg, inp.bias, inp.w1 if w1 is None else w1,
                                inp.w3 if w3 is None else w3, inp.w2 if w2 is None else w2, out, ws)
    st = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK, moe.status_string(st)
    return out, moe.layer_views(cfg, ws)


def _within_one_rounding(a, b, ysum=None):
    """Elements of two bf16 results differ by at most one bf16 step of the
    larger magnitude (2^-7 relative), plus what reassociating the fp32 slot
    sum can move a result that nearly cancels: a few fp32 roundings of the
    slot terms, bounded here by 2^-16 of the largest output.  ysum, when
    given, is sum_j w_j |y_j| of b's slots, whose y_j b read after one
    rounding to fp16 (at most 2^-11 relative each) while a used the fp32
    accumulators themselves."""
    a, b = to_f64(a), to_f64(b)
    m = np.maximum(np.abs(a), np.abs(b))
    slack = 2.0 ** -16 * np.abs(b).max()
    bound = m * 2.0 ** -7 + slack
    if ysum is not None:
        bound = bound + 2.0 ** -11 * ysum
    return bool((np.abs(a - b) <= bound).all())


def _weighted_abs_slot_sum(views, D):
    """sum_j topk_w[t, j] |y_perm[row_of[t, j]]| per element, from a layer
    workspace (rows < 0 contribute nothing)."""
    row_of = views["row_of"].long()
    y = views["y_perm"].double()
    wts = views["topk_w"].double()
    acc = torch.zeros((row_of.shape[0], D), dtype=torch.float64, device=y.device)
    for j in range(row_of.shape[1]):
        r = row_of[:, j]
        ok = r >= 0
        acc[ok] += wts[ok, j, None].abs() * y[r[ok]].abs()
    return acc.cpu().numpy()


@pytest.mark.parametrize("name,over,n_sample", [
    ("fine-grained-bf16", dict(T=640), 96),
    ("deepseek-v3-shaped", dict(T=300), 12),
    ("zipf-skewed", dict(T=1500), 48),
    ("decode-masked", dict(), 16),
])
def test_fused_layer_matches_oracle_and_unfused(moe, name, over, n_sample, monkeypatch):
    w = moe_inputs.WORKLOADS[name].scaled(**over)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=3)
    cfg = cfg_for(moe, w)
    out, views = run_fused(moe, cfg, inp)
    assert not torch.isnan(out.float()).any()
    check_against_oracle(moe, w, inp, out, views, n_sample)
    # the unfused reference on the same GEMM kernel as the fused path (the
    # one-CTA kernel, chosen for small segments, can round h differently)
    monkeypatch.setenv("MOE_GROUPED_KERNEL", "pair")
    ref = torch.empty_like(out)
    ws = moe.alloc_workspace(cfg, layer=True)
    moe.moe_layer_forward(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, ref, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    ysum = _weighted_abs_slot_sum(moe.layer_views(cfg, ws), cfg.D)
    assert _within_one_rounding(out, ref, ysum)


def test_fused_expert_ranges_sum_to_layer(moe):
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=512, D=512, H=256, E=16)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=4)
    full, _ = run_fused(moe, cfg_for(moe, w), inp)
    total = torch.zeros((w.T, w.D), dtype=torch.float64, device="cuda")
    for e0 in (0, 8):
        cfg = cfg_for(moe, w, e_first=e0, E_local=8)
        part, _ = run_fused(moe, cfg, inp, inp.w1[e0:e0 + 8], inp.w3[e0:e0 + 8], inp.w2[e0:e0 + 8])
        total += part.double()
    err = (total - full.double()).abs().max().item()
    rms = full.double().pow(2).mean().sqrt().item()
    assert err <= 2e-2 * rms


def test_fused_tokens_without_local_rows_are_zero(moe):
    # every token routes to experts 0..3; the shard holding 4..7 outputs zeros
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=256, D=256, H=128, E=8, k=2)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=5)
    bias = torch.zeros(w.E, device="cuda")
    bias[4:] = -30.0
    inp = dataclasses.replace(inp, bias=bias)
    cfg = cfg_for(moe, w, e_first=4, E_local=4)
    out, _ = run_fused(moe, cfg, inp, inp.w1[4:], inp.w3[4:], inp.w2[4:])
    assert (out.float() == 0).all()
