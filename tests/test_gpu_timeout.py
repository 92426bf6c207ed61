"""A bounded device wait that runs out (failure detection without a fault).

The one-launch grouped SwiGLU runs GEMM1 and GEMM2 in one cooperative
launch; a GEMM2 producer waits (acquire, bounded at one second of
%globaltimer) until every GEMM1 tile of its 256-row block has stored h.
The test plants GEMM1 block counts in the workspace that can never reach
their target -- a flag that nothing sets -- so every such wait runs out.
The kernel must then stop its roles, meet its peer, free its tensor memory
and return; the call reports MOE_ERR_TIMEOUT through the workspace status;
the last CTA still leaves the counters at zero, so the next call on the same
workspace is correct again.  Nothing faults or waits forever.
"""
import time

import numpy as np
import pytest
import torch

import moe_inputs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import routing_grouped_gemm_gb300 as m
    assert torch.cuda.is_available()
    return m


def _grouped_counters(moe, cfg, ws):
    """int32 view of the grouped kernel's counters at the end of the step
    workspace: [0] CTAs finished, [32 ..] GEMM1 epilogue signals per block
    (the library's workspace layout: 32 + ceil(rows/256) + E_local ints,
    rounded up to 256 bytes, after the permute and router scratch)."""
    ra = moe.rows_alloc(cfg)
    n_ints = 32 + -(-ra // 256) + cfg.e_local
    nbytes = -(-4 * n_ints // 256) * 256
    off = moe.workspace_size(cfg) - nbytes
    return ws[off:off + 4 * n_ints].view(torch.int32)


def test_grouped_wait_runs_out_and_the_next_call_recovers(moe, monkeypatch):
    monkeypatch.delenv("MOE_GROUPED_KERNEL", raising=False)
    T, E, k, D, H = 600, 4, 2, 256, 256
    idx = moe_inputs.random_topk_idx(T, E, k, seed=31, skew=0.3)
    lay = oracle.layout(idx, E, 0, E, oracle.CONTIGUOUS, 128)
    ra = lay["rows_alloc"]
    g = torch.Generator(device="cuda").manual_seed(31)
    xp = torch.randn((ra, D), generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn((E, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w3 = (torch.randn((E, H, D), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E, D, H), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    cfg = moe.Config(T=T, D=D, H_local=H, E=E, k=k, dtype=moe.MOE_BF16)
    assert moe.rows_alloc(cfg) == ra
    seg = torch.from_numpy(lay["seg_offsets"]).cuda()
    tpe = torch.from_numpy(lay["tokens_per_expert"]).cuda()
    ws = moe.alloc_workspace(cfg)
    valid = torch.from_numpy(lay["token_of_row"] >= 0).cuda()

    def call():
        h = torch.zeros((ra, H), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros((ra, D), dtype=cfg.y_dtype, device="cuda")
        n0 = moe.kernel_launches()
        moe.moe_grouped_swiglu(cfg, xp, seg, tpe, w1, w3, w2, h, y, ws)
        n = moe.kernel_launches() - n0
        return h, y, n

    h0, y0, n = call()
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert n == 1                                   # the one-launch cooperative form
    ctr = _grouped_counters(moe, cfg, ws)
    assert int(ctr.abs().sum()) == 0                # every call leaves them at zero

    # GEMM1 block counts that can never reach their target (one per 256-row
    # block of the pair kernel's tile table)
    n_blocks = int(sum(-(-int(c) // 256) for c in lay["tokens_per_expert"]))
    assert 0 < n_blocks <= ctr.numel() - 32
    ctr[32:32 + n_blocks] = -(1 << 30)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    call()
    st = moe.moe_get_device_status(ws)              # synchronises
    elapsed = time.perf_counter() - t0
    assert st == moe.MOE_ERR_TIMEOUT, moe.status_string(st)
    assert 0.9 < elapsed < 30.0                     # the waits ran their full second, then ended
    assert moe.moe_get_device_status(ws) == moe.MOE_OK   # the read cleared the status
    assert int(ctr.abs().sum()) == 0                # the last CTA reset the counters

    # the context and the workspace are usable: the same call is correct again
    h1, y1, _ = call()
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(h1[valid], h0[valid])
    assert torch.equal(y1[valid], y0[valid])
    # and agrees with the oracle on a few rows (the GEMM itself is checked elsewhere)
    rows = np.nonzero(lay["token_of_row"] >= 0)[0][::97]
    xh = xp.float().cpu().numpy().astype(np.float64)
    for r in rows:
        e = int(np.searchsorted(lay["seg_offsets"], r, side="right") - 1)
        ref = oracle.expert_ffn(xh[r], moe_inputs.host_array(w1[e]), moe_inputs.host_array(w3[e]),
                                moe_inputs.host_array(w2[e]), round_h=True)
        got = y1[r].double().cpu().numpy()
        assert np.abs(got - ref).max() <= 2e-2 * np.sqrt((ref ** 2).mean())
