"""End-to-end GPU parity of moe_layer_forward against the CPU oracle.

Reduced-T versions of every workload are checked token by token on a
sample; the full-size workloads (the launch configuration the benchmark
times) are checked on sampled tokens plus properties of the whole layout.
Shards (expert ranges and H shards) are summed on the host and compared
with the unsharded output.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import (cfg_for, check_layout_properties, oracle_out_tokens, oracle_route, oscore,
                     rel_err, routing_agreement, to_f64, tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def run_layer(moe, cfg, inp, w1=None, w3=None, w2=None):
    ws = moe.alloc_workspace(cfg, layer=True)
    out = torch.empty((cfg.T, cfg.D), dtype=cfg.torch_dtype, device="cuda")
    moe.moe_layer_forward(cfg, inp.x, inp.wg, inp.bias, inp.w1 if w1 is None else w1,
                          inp.w3 if w3 is None else w3, inp.w2 if w2 is None else w2, out, ws)
    st = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK, moe.status_string(st)
    return out, moe.layer_views(cfg, ws), ws


def check_against_oracle(moe, w, inp, out, views, n_sample, seed=0):
    l64, keys, oidx, owts, st = oracle_route(inp, w, inp.bias)
    gidx = views["topk_idx"].cpu().numpy()
    gl_err = 1e-3  # generous key tolerance for near ties (logits are O(1))
    same_set, _ = routing_agreement(gidx, oidx, keys, key_tol=gl_err)
    assert same_set.mean() > 0.99
    rng = np.random.default_rng(seed)
    cand = np.nonzero(same_set)[0]
    toks = np.sort(rng.choice(cand, size=min(n_sample, len(cand)), replace=False))
    ref = oracle_out_tokens(inp, w, toks, oidx, owts)
    got = to_f64(out)[toks]
    err = rel_err(got, ref)
    assert err < tol(w), f"{w.name}: max err / rms = {err:.3e}"
    return err


SMALL = [
    ("tiny-fp32", dict(), 256),
    ("fine-grained-bf16", dict(T=640), 96),
    ("deepseek-v3-shaped", dict(T=300), 12),
    ("zipf-skewed", dict(T=1500), 48),
    ("decode-masked", dict(), 16),
]


@pytest.mark.parametrize("name,over,n_sample", SMALL)
def test_layer_reduced_workloads(moe, name, over, n_sample):
    w = moe_inputs.WORKLOADS[name].scaled(**over)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=1)
    cfg = cfg_for(moe, w)
    out, views, _ = run_layer(moe, cfg, inp)
    check_against_oracle(moe, w, inp, out, views, n_sample)
    # layout of the whole batch, by properties that fix it uniquely
    idx = views["topk_idx"].cpu().numpy()
    lay = (views["tokens_per_expert"].cpu().numpy(), views["seg_offsets"].cpu().numpy(),
           views["row_of"].cpu().numpy(), views["token_of_row"].cpu().numpy())
    if w.layout == "masked":
        check_layout_properties(idx, lay, w.E, 0, w.E, masked_cap=cfg.capacity)
    else:
        check_layout_properties(idx, lay, w.E, 0, w.E, align_m=cfg.align_m)


def test_tiny_fp32_whole_batch_and_tp2_shards(moe):
    w = moe_inputs.WORKLOADS["tiny-fp32"]
    inp = moe_inputs.make_inputs(w, device="cuda", seed=0)
    cfg = cfg_for(moe, w)
    out, views, _ = run_layer(moe, cfg, inp)
    l64, keys, oidx, owts, _ = oracle_route(inp, w)
    assert np.array_equal(views["topk_idx"].cpu().numpy(), oidx)
    ref = oracle_out_tokens(inp, w, np.arange(w.T), oidx, owts)
    assert rel_err(to_f64(out), ref) < 1e-4
    # H shards: w1/w3 split on dim 1, w2 on dim 2; partial outputs sum to the layer
    Hl = w.H // w.tp
    acc = np.zeros((w.T, w.D))
    for r in range(w.tp):
        sl = slice(r * Hl, (r + 1) * Hl)
        c = cfg_for(moe, w, H_local=Hl)
        part, _, _ = run_layer(moe, c, inp, inp.w1[:, sl].contiguous(), inp.w3[:, sl].contiguous(),
                               inp.w2[:, :, sl].contiguous())
        acc += to_f64(part)
        pref = oracle_out_tokens(inp, w, np.arange(w.T), oidx, owts, h0=r * Hl, Hl=Hl)
        assert rel_err(to_f64(part), pref) < 1e-4
    assert rel_err(acc, ref) < 1e-4


def test_decode_masked_expert_ranges_times_h_shards(moe):
    """8 expert ranges x 4 H shards; the 32 partials sum to the whole layer."""
    w = moe_inputs.WORKLOADS["decode-masked"]
    inp = moe_inputs.make_inputs(w, device="cuda", seed=2)
    cfg = cfg_for(moe, w)
    full, views, _ = run_layer(moe, cfg, inp)
    El, Hl = w.E // w.ep, w.H // w.tp
    acc = torch.zeros((w.T, w.D), dtype=torch.float64, device="cuda")
    for er in range(w.ep):
        es = slice(er * El, (er + 1) * El)
        for r in range(w.tp):
            hs = slice(r * Hl, (r + 1) * Hl)
            c = cfg_for(moe, w, e_first=er * El, E_local=El, H_local=Hl)
            part, pv, _ = run_layer(moe, c, inp, inp.w1[es, hs].contiguous(),
                                    inp.w3[es, hs].contiguous(), inp.w2[es, :, hs].contiguous())
            acc += part.double()
            if er == 0 and r == 0:
                # counts cover every expert; segments only the local range
                assert int(pv["tokens_per_expert"].sum()) == w.T * w.k
                assert pv["seg_offsets"].cpu().numpy().tolist() == [i * w.T for i in range(El + 1)]
    accn = acc.cpu().numpy()
    fulln = to_f64(full)
    assert rel_err(accn, fulln) < 2e-2
    l64, keys, oidx, owts, _ = oracle_route(inp, w)
    toks = np.arange(0, w.T, 8)
    assert np.array_equal(views["topk_idx"].cpu().numpy()[toks], oidx[toks])
    ref = oracle_out_tokens(inp, w, toks, oidx, owts)
    assert rel_err(accn[toks], ref) < 2e-2


def test_layer_without_local_experts_gives_zeros(moe):
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=100, E=16, D=256, H=128)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=4)
    cfg = cfg_for(moe, w, e_first=16, E_local=0)
    e0 = inp.w1[:0]
    out, views, _ = run_layer(moe, cfg, inp, e0, e0, inp.w2[:0])
    assert (out.float() == 0).all()
    assert int(views["tokens_per_expert"].sum()) == w.T * w.k


def test_layer_single_token_and_k1(moe):
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=1, E=8, k=1, D=512, H=256)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=6)
    out, views, _ = run_layer(moe, cfg_for(moe, w), inp)
    check_against_oracle(moe, w, inp, out, views, 1)


@pytest.mark.parametrize("T,E,k,D,H,renorm", [
    (300, 1, 1, 256, 128, True),    # one expert: every token in one segment, weight 1
    (200, 4, 4, 128, 64, False),    # k = E: every token to every expert (softmax weights)
    (100, 8, 2, 8, 8, True),        # the smallest widths: D = H = 8 (one 16-byte row)
    (1, 64, 6, 2048, 1408, True),   # one token at full widths: six one-row expert segments
])
def test_layer_degenerate_shapes(moe, T, E, k, D, H, renorm):
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=T, E=E, k=k, D=D, H=H, renorm=renorm)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=T + E)
    cfg = cfg_for(moe, w)
    out, views, _ = run_layer(moe, cfg, inp)
    check_against_oracle(moe, w, inp, out, views, min(T, 32))
    idx = views["topk_idx"].cpu().numpy()
    lay = (views["tokens_per_expert"].cpu().numpy(), views["seg_offsets"].cpu().numpy(),
           views["row_of"].cpu().numpy(), views["token_of_row"].cpu().numpy())
    check_layout_properties(idx, lay, w.E, 0, w.E, align_m=cfg.align_m)
    if k == E:
        assert (np.sort(idx, axis=1) == np.arange(E)).all()
    if E == 1:
        assert np.allclose(views["topk_w"].cpu().numpy(), 1.0)


def test_layer_is_deterministic(moe):
    w = moe_inputs.WORKLOADS["zipf-skewed"].scaled(T=3000)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=8)
    cfg = cfg_for(moe, w)
    a, _, _ = run_layer(moe, cfg, inp)
    b, _, _ = run_layer(moe, cfg, inp)
    assert torch.equal(a, b)


def test_layer_group_limited_routing(moe):
    w = moe_inputs.WORKLOADS["deepseek-v3-shaped"].scaled(T=300, n_group=8, topk_group=4)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=12)
    out, views, _ = run_layer(moe, cfg_for(moe, w), inp)
    check_against_oracle(moe, w, inp, out, views, 12)
    idx = views["topk_idx"].cpu().numpy()
    assert max(len(set(row // (w.E // w.n_group))) for row in idx) <= w.topk_group


@pytest.mark.parametrize("pinned_out", [True, False])
def test_layer_forward_host_buffers(moe, pinned_out):
    """The host-buffer entry point around the same layer: bit-identical to
    moe_layer_forward, also on a second call that reuses the workspace with
    another input -- with a page-locked out_host (the combine writes it
    directly) and a pageable one (staged and copied back)."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=700, D=512, H=384)
    cfg = cfg_for(moe, w)
    hws = moe.alloc_workspace(cfg, host=True)
    for seed in (13, 14):
        inp = moe_inputs.make_inputs(w, device="cuda", seed=seed)
        ref, _, _ = run_layer(moe, cfg, inp)
        x_host = inp.x.cpu().pin_memory()
        out_host = torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16)
        if pinned_out:
            out_host = out_host.pin_memory()
        moe.moe_layer_forward_host(cfg, x_host, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out_host,
                                   hws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(hws) == moe.MOE_OK
        assert torch.equal(out_host, ref.cpu())


@pytest.mark.parametrize("pinned", [True, False])
def test_host_pipeline_matches_layer_forward(moe, pinned):
    """Five calls queued back to back on the host pipeline, each with its own
    input and output buffer (the two device slots are each reused twice or
    more), then a sixth after a sync: every output is bit-identical to
    moe_layer_forward on the same input, with page-locked and with pageable
    host buffers."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=700, D=512, H=384)
    cfg = cfg_for(moe, w)
    base = moe_inputs.make_inputs(w, device="cuda", seed=21)
    xs = [moe_inputs.make_inputs(w, device="cuda", seed=30 + i, weights=False).x for i in range(6)]
    refs = []
    lws = moe.alloc_workspace(cfg, layer=True)
    for x in xs:
        out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device="cuda")
        moe.moe_layer_forward(cfg, x, base.wg, base.bias, base.w1, base.w3, base.w2, out, lws)
        refs.append(out.cpu())
    assert moe.moe_get_device_status(lws) == moe.MOE_OK

    def host(t):
        return t.pin_memory() if pinned else t

    pipe = moe.HostPipeline(cfg)
    try:
        x_hosts = [host(x.cpu()) for x in xs]
        outs = [host(torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16)) for _ in xs]
        for i in range(5):
            pipe.submit(x_hosts[i], base.wg, base.bias, base.w1, base.w3, base.w2, outs[i])
        pipe.sync()
        pipe.submit(x_hosts[5], base.wg, base.bias, base.w1, base.w3, base.w2, outs[5])
        other = torch.cuda.Stream()
        with pytest.raises(moe.MoeError):     # another stream while a call is pending
            pipe.submit(x_hosts[0], base.wg, base.bias, base.w1, base.w3, base.w2, outs[0],
                        stream=other)
        pipe.sync()
    finally:
        pipe.close()
    for i in range(6):
        assert torch.equal(outs[i], refs[i]), i


def test_host_pipeline_shard_and_masked_layout(moe):
    """The host pipeline on an expert-range x H shard of the masked (decode)
    layout: three queued calls, each bit-identical to moe_layer_forward on
    the same shard."""
    w = moe_inputs.WORKLOADS["decode-masked"].scaled(D=1024, H=512)
    El, Hl = w.E // w.ep, w.H // w.tp
    es, hs = slice(2 * El, 3 * El), slice(Hl, 2 * Hl)
    cfg = cfg_for(moe, w, e_first=2 * El, E_local=El, H_local=Hl)
    base = moe_inputs.make_inputs(w, device="cuda", seed=51)
    w1, w3 = base.w1[es, hs].contiguous(), base.w3[es, hs].contiguous()
    w2 = base.w2[es, :, hs].contiguous()
    xs = [moe_inputs.make_inputs(w, device="cuda", seed=52 + i, weights=False).x for i in range(3)]
    lws = moe.alloc_workspace(cfg, layer=True)
    refs = []
    for x in xs:
        out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device="cuda")
        moe.moe_layer_forward(cfg, x, base.wg, base.bias, w1, w3, w2, out, lws)
        refs.append(out.cpu())
    assert moe.moe_get_device_status(lws) == moe.MOE_OK
    pipe = moe.HostPipeline(cfg)
    try:
        x_hosts = [x.cpu().pin_memory() for x in xs]
        outs = [torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16).pin_memory()
                for _ in xs]
        for xh, oh in zip(x_hosts, outs):
            pipe.submit(xh, base.wg, base.bias, w1, w3, w2, oh)
        pipe.sync()
    finally:
        pipe.close()
    for i in range(3):
        assert torch.equal(outs[i], refs[i]), i


def test_fp8_layer_in_cuda_graph(moe):
    """moe_layer_forward_fp8 (quantising dispatch, e4m3 GEMM1) captured into a
    CUDA graph after a warm-up call and replayed on new inputs: bit-identical
    to direct calls."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=600, D=512, H=384)
    cfg = cfg_for(moe, w)
    base = moe_inputs.make_inputs(w, device="cuda", seed=61)
    w1q, w1s = moe.quantize_weights_fp8(base.w1)
    w3q, w3s = moe.quantize_weights_fp8(base.w3)
    x = base.x.clone()
    out = torch.empty_like(x)
    ws = moe.alloc_workspace(cfg, layer=True)

    def call(xx, oo, wws, stream=None):
        moe.moe_layer_forward_fp8(cfg, xx, base.wg, base.bias, w1q, w1s, w3q, w3s, base.w2, oo,
                                  wws, stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(x, out, ws, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(x, out, ws, s)
    ref_ws = moe.alloc_workspace(cfg, layer=True)
    for seed in (62, 63):
        xi = moe_inputs.make_inputs(w, device="cuda", seed=seed, weights=False).x
        x.copy_(xi)
        g.replay()
        torch.cuda.synchronize()
        ref = torch.empty_like(x)
        call(xi, ref, ref_ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), seed
    assert moe.moe_get_device_status(ws) == moe.MOE_OK


@pytest.mark.parametrize("name,over", [
    ("fine-grained-bf16", dict(T=700, D=512, H=384)),
    ("tiny-fp32", dict()),
])
def test_layer_forward_in_cuda_graph(moe, name, over):
    """moe_layer_forward captured once into a CUDA graph (after a warm-up call
    outside the capture) and replayed on new inputs written into the same
    buffers: every replay is bit-identical to a direct call."""
    w = moe_inputs.WORKLOADS[name].scaled(**over)
    cfg = cfg_for(moe, w)
    base = moe_inputs.make_inputs(w, device="cuda", seed=41)
    x = base.x.clone()
    out = torch.empty_like(x)
    ws = moe.alloc_workspace(cfg, layer=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_layer_forward(cfg, x, base.wg, base.bias, base.w1, base.w3, base.w2, out, ws, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward(cfg, x, base.wg, base.bias, base.w1, base.w3, base.w2, out, ws, s)
    ref_ws = moe.alloc_workspace(cfg, layer=True)
    for seed in (42, 43, 44):
        xi = moe_inputs.make_inputs(w, device="cuda", seed=seed, weights=False).x
        x.copy_(xi)
        g.replay()
        torch.cuda.synchronize()
        ref = torch.empty_like(x)
        moe.moe_layer_forward(cfg, xi, base.wg, base.bias, base.w1, base.w3, base.w2, ref, ref_ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), seed
    assert moe.moe_get_device_status(ws) == moe.MOE_OK


def test_layer_k32_many_experts(moe):
    """k = 32 of E = 256 (the largest k the ABI accepts), bf16."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=96, E=256, k=32, D=256, H=128)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=15)
    out, views, _ = run_layer(moe, cfg_for(moe, w), inp)
    check_against_oracle(moe, w, inp, out, views, 24)


@pytest.mark.parametrize("kernel", ["auto", "pair"])
def test_layer_max_experts(moe, kernel, monkeypatch):
    """E = 1024, the most experts the ABI accepts: the SIMT router above 256
    experts, a count matrix of 6 x 1024 cells, about 12 rows per expert (the
    one-CTA grouped kernel is chosen; "pair" forces the CTA-pair kernel and
    its 1024-expert tile table)."""
    if kernel == "pair":
        monkeypatch.setenv("MOE_GROUPED_KERNEL", "pair")
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=1500, D=256, H=128, E=1024, k=8)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=17)
    cfg = cfg_for(moe, w)
    out, views, _ = run_layer(moe, cfg, inp)
    check_against_oracle(moe, w, inp, out, views, 48)
    idx = views["topk_idx"].cpu().numpy()
    lay = (views["tokens_per_expert"].cpu().numpy(), views["seg_offsets"].cpu().numpy(),
           views["row_of"].cpu().numpy(), views["token_of_row"].cpu().numpy())
    check_layout_properties(idx, lay, w.E, 0, w.E, align_m=cfg.align_m)


def test_layer_launch_count(moe):
    # bf16, E <= 256: router logits on the tensor cores with the top-k in the
    # same cluster launch (1), count with the scan in its last block (1;
    # 4 blocks x 64 experts fit it), ranks with the row copy (1), GEMM1 and
    # GEMM2 in one pair-kernel launch (1), combine (1)
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=1024, D=512, H=256)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=9)
    cfg = cfg_for(moe, w)
    run_layer(moe, cfg, inp)
    before = moe.kernel_launches()
    run_layer(moe, cfg, inp)
    assert moe.kernel_launches() - before == 5


# ------------------------------------------------------------------ full sizes

FULL = [
    ("fine-grained-bf16", 48),
    ("deepseek-v3-shaped", 4),
    ("zipf-skewed", 24),
    ("decode-masked", 16),
]


@pytest.mark.parametrize("name,n_sample", FULL)
def test_layer_full_size_sampled(moe, name, n_sample):
    w = moe_inputs.WORKLOADS[name]
    inp = moe_inputs.make_inputs(w, device="cuda", seed=0)
    cfg = cfg_for(moe, w)
    out, views, ws = run_layer(moe, cfg, inp)
    check_against_oracle(moe, w, inp, out, views, n_sample, seed=1)
    idx = views["topk_idx"].cpu().numpy()
    # whole-batch routing: the router call on the same inputs returns the
    # layer's top-k and its fp32 logits; the oracle's selection on those
    # logits is the same for every token, and so are the weights
    logits = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    gidx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    rws = moe.alloc_workspace(cfg)
    moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, logits, gidx, gw, rws)
    assert moe.moe_get_device_status(rws) == moe.MOE_OK
    assert np.array_equal(gidx.cpu().numpy(), idx)
    assert torch.equal(gw, views["topk_w"])
    keys = logits.cpu().numpy()
    oidx, st = oracle.topk(keys, w.k, w.n_group, w.topk_group)
    assert st == oracle.OK
    assert np.array_equal(idx, oidx)
    ow = oracle.topk_weights(keys, oidx, oscore(w), w.renorm)
    np.testing.assert_allclose(gw.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)
    cnt = views["tokens_per_expert"].cpu().numpy()
    assert int(cnt.sum()) == w.T * w.k
    lay = (cnt, views["seg_offsets"].cpu().numpy(), views["row_of"].cpu().numpy(),
           views["token_of_row"].cpu().numpy())
    if w.layout == "masked":
        check_layout_properties(idx, lay, w.E, 0, w.E, masked_cap=cfg.capacity)
    else:
        check_layout_properties(idx, lay, w.E, 0, w.E, align_m=cfg.align_m)
    # x_perm rows are the tokens' rows, bit for bit
    row_of = views["row_of"]
    sel = row_of[:, 0].long()
    assert torch.equal(views["x_perm"][sel], inp.x)
    if w.zipf_s:
        assert (cnt == 0).sum() >= w.zipf_empty
    del inp, out, views, ws
    torch.cuda.empty_cache()


def test_layer_empty_batch(moe):
    """T = 0: the layer call launches nothing and returns MOE_OK; the training
    backward has no dx rows to write and sets every parameter gradient to
    zero (in fp32 and in bf16)."""
    w = moe_inputs.WORKLOADS["fine-grained-bf16"].scaled(T=64, E=8, D=256, H=128)
    inp = moe_inputs.make_inputs(w, device="cuda", seed=2)
    cfg = cfg_for(moe, w, T=0)
    x = torch.empty((0, w.D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, w.D), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg, layer=True)
    n0 = moe.kernel_launches()
    moe.moe_layer_forward(cfg, x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, ws)
    assert moe.kernel_launches() == n0
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    tws = moe.alloc_workspace(cfg, train=True)
    moe.moe_layer_forward_train(cfg, x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, tws)
    for wdt in (torch.float32, torch.bfloat16):
        dwg = torch.full((w.E, w.D), float("nan"), device="cuda")
        dbias = torch.full((w.E,), float("nan"), device="cuda")
        dws = [torch.full(s, float("nan"), dtype=wdt, device="cuda")
               for s in ((w.E, w.H, w.D), (w.E, w.H, w.D), (w.E, w.D, w.H))]
        moe.moe_layer_backward(cfg, x, inp.wg, inp.w1, inp.w3, inp.w2, out, out, dwg, dbias,
                               *dws, tws)
        assert moe.moe_get_device_status(tws) == moe.MOE_OK
        for t in (dwg, dbias, *dws):
            assert (t.float() == 0).all()
