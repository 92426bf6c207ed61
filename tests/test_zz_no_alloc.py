"""moe_permute_noalloc: the permute for callers that cannot allocate.

Some callers cannot call cudaMalloc where they dispatch tokens (they run in
a memory pool they do not own, or are handed only their input and output
tensors), so they cannot provide moe_permute's workspace.  The no-alloc
entry point keeps that scratch in a fixed array inside the library.  These
checks call it through the C ABI twice in a row -- the second call on a
different problem, so it starts from the first call's leftovers -- and
compare every output with moe_permute on the same inputs, bit for bit (the
tolerance of all integer and byte work in these tests), and the layout with
the CPU oracle's.  The cases take each form of the counting sort: up to 8192
count cells (ceil(T / 256) * E), 8192 to 16384, and above that up to the
fixed array's limit.  This file is collected last on purpose.
"""
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


def _outputs(moe, cfg):
    ra = moe.rows_alloc(cfg)
    return dict(
        tpe=torch.full((cfg.E,), -5, dtype=torch.int32, device="cuda"),
        seg=torch.full((cfg.e_local + 1,), -5, dtype=torch.int32, device="cuda"),
        row_of=torch.full((cfg.T, cfg.k), -5, dtype=torch.int32, device="cuda"),
        tor=torch.full((ra,), -5, dtype=torch.int32, device="cuda"),
        xp=torch.zeros((ra, cfg.D), dtype=cfg.torch_dtype, device="cuda"))


def _case(moe, T, E, k, D, align, skew, seed, e_first=0, E_local=-1):
    cfg = moe.Config(T=T, D=D, H_local=8, E=E, k=k, e_first=e_first, E_local=E_local,
                     dtype=moe.MOE_BF16, align_m=align)
    idx = torch.from_numpy(moe_inputs.random_topk_idx(T, E, k, seed=seed, skew=skew)).cuda()
    x = torch.randn((T, D), generator=torch.Generator(device="cuda").manual_seed(seed),
                    device="cuda").to(torch.bfloat16)
    return cfg, idx, x


def _compare(moe, cfg, idx, x):
    ref = _outputs(moe, cfg)
    ws = moe.alloc_workspace(cfg)
    moe.moe_permute(cfg, x, idx, ref["tpe"], ref["seg"], ref["row_of"], ref["tor"], ref["xp"], ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    del ws
    got = _outputs(moe, cfg)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute_noalloc(cfg, x, idx, got["tpe"], got["seg"], got["row_of"], got["tor"],
                            got["xp"], flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    for name in ("tpe", "seg", "row_of", "tor"):
        assert torch.equal(got[name], ref[name]), name
    filled = ref["tor"] >= 0
    assert torch.equal(got["xp"][filled], ref["xp"][filled])
    assert int(got["tpe"].sum()) == cfg.T * cfg.k
    lay = oracle.layout(idx.cpu().numpy(), cfg.E, cfg.e_first, cfg.e_local, oracle.CONTIGUOUS,
                        cfg.align_m)
    assert lay["status"] == oracle.OK
    for name, key in (("tpe", "tokens_per_expert"), ("seg", "seg_offsets"),
                      ("row_of", "row_of"), ("tor", "token_of_row")):
        assert np.array_equal(got[name].cpu().numpy(), lay[key]), name
    return got


def test_noalloc_matches_permute_on_two_calls_in_a_row(moe):
    # first call: a large skewed batch (4096 count cells: the two-launch form)
    cfg1, idx1, x1 = _case(moe, T=16384, E=64, k=8, D=512, align=128, skew=1.2, seed=21)
    _compare(moe, cfg1, idx1, x1)
    # second call: a different, smaller problem over an expert range; the
    # scratch still holds the first call's counts
    cfg2, idx2, x2 = _case(moe, T=777, E=48, k=6, D=264, align=8, skew=0.4, seed=22,
                           e_first=8, E_local=30)
    _compare(moe, cfg2, idx2, x2)


@pytest.mark.parametrize("T,E,k", [
    (16384, 256, 8),    # 16384 count cells: the index kernel re-derives the scan
    (131072, 256, 8),   # 131072 cells: count, scan, index, copy; exactly the array's limit
])
def test_noalloc_large_count_matrices(moe, T, E, k):
    cfg, idx, x = _case(moe, T=T, E=E, k=k, D=64, align=128, skew=0.6, seed=T + E)
    cells = -(-T // 256) * E
    assert cells > 8192
    got = _compare(moe, cfg, idx, x)
    del got
    # and a small call right after it, on what the large one left in the array
    cfg2, idx2, x2 = _case(moe, T=300, E=16, k=4, D=128, align=16, skew=0.9, seed=5)
    _compare(moe, cfg2, idx2, x2)

