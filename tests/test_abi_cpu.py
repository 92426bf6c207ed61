"""Host-side checks of the C ABI library (no GPU needed, no compute calls).

The library must build for sm_103a, load, export every function that
include/moe.h declares, and reject bad arguments on the host before anything
is launched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import routing_grouped_gemm_gb300 as m
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(moe):
    declared = header_functions()
    assert declared, "no declarations found in include/moe.h"
    assert sorted(moe.ABI_SYMBOLS) == declared
    lib = ctypes.CDLL(moe.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_library_is_built_for_sm103a():
    import __graft_entry__
    assert "arch=compute_103a,code=sm_103a" in __graft_entry__._build_module().ARCH


def _cfg(moe, **kw):
    base = dict(T=64, D=128, H_local=64, E=8, k=2, dtype=moe.MOE_BF16)
    base.update(kw)
    return moe.Config(**base)


@pytest.mark.parametrize("bad", [
    dict(D=12), dict(D=0), dict(H_local=4), dict(E=0), dict(E=2000), dict(k=0), dict(k=9),
    dict(T=-1), dict(e_first=6, E_local=4), dict(dtype=7), dict(score=3), dict(align_m=0),
    dict(layout=1, capacity=-1), dict(layout=5),
])
def test_invalid_configs_rejected(moe, bad):
    assert moe.validate_config(_cfg(moe, **bad)) == moe.MOE_ERR_INVALID_ARG
    assert moe.rows_alloc(_cfg(moe, **bad)) == -1
    assert moe.workspace_size(_cfg(moe, **bad)) == -1


def test_rows_alloc_formula_matches_oracle(moe):
    import oracle
    for kw in (dict(), dict(align_m=1), dict(e_first=2, E_local=3), dict(E_local=1, k=2),
               dict(layout=1, capacity=40), dict(T=0)):
        cfg = _cfg(moe, **kw)
        el = cfg.e_local
        ref = oracle.rows_alloc(cfg.T, cfg.k, el, cfg.layout, cfg.align_m, cfg.capacity)
        assert moe.rows_alloc(cfg) == ref


def test_workspace_sizes_are_positive_and_ordered(moe):
    cfg = _cfg(moe)
    assert 256 <= moe.workspace_size(cfg) <= moe.layer_workspace_size(cfg)
    assert moe.layer_workspace_size(cfg) % 256 == 0


def test_host_errors_before_any_launch(moe):
    lib = moe._lib
    c = _cfg(moe).c()
    # NULL workspace
    st = lib.moe_route_topk(ctypes.byref(c), 16, 16, None, None, 16, 16, None, 0, None)
    assert st == moe.MOE_ERR_WORKSPACE
    # misaligned workspace
    st = lib.moe_permute(ctypes.byref(c), 16, 16, 16, 16, 16, 16, 16, 1024 + 8, 1 << 20, None)
    assert st == moe.MOE_ERR_WORKSPACE
    # workspace too small
    st = lib.moe_unpermute_combine(ctypes.byref(c), 16, 16, 16, 16, 256 * 64, 256, None)
    assert st == moe.MOE_ERR_WORKSPACE
    # NULL tensor with a large enough fake workspace
    big = moe.layer_workspace_size(_cfg(moe))
    st = lib.moe_grouped_swiglu(ctypes.byref(c), None, 16, 16, 16, 16, 16, 16, 16, 1 << 20, big,
                                None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # misaligned expert weights
    st = lib.moe_layer_forward(ctypes.byref(c), 256, 256, None, 8, 256, 256, 256, 1 << 20, big, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert "misaligned" in moe.last_error_string()
    # invalid config wins over everything else
    bad = _cfg(moe, k=99).c()
    assert lib.moe_layer_forward(ctypes.byref(bad), 0, 0, None, 0, 0, 0, 0, 0, 0, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(None, 0, None) == moe.MOE_ERR_WORKSPACE


@pytest.mark.parametrize("n_group,topk_group,k,ok", [
    (0, 0, 6, True), (1, 0, 6, True), (8, 4, 8, True), (8, 8, 8, True), (32, 4, 8, True),
    (7, 2, 6, False),    # 7 does not divide 64
    (64, 2, 6, False),   # more than 32 groups
    (8, 0, 6, False), (8, 9, 9, False),   # topk_group out of 1..n_group
    (8, 4, 3, False),    # k < topk_group
    (16, 1, 5, False),   # k > topk_group * E / n_group = 4
])
def test_group_limited_config_validation(moe, n_group, topk_group, k, ok):
    cfg = moe.Config(T=16, D=64, H_local=64, E=64, k=k, n_group=n_group, topk_group=topk_group)
    st = moe.validate_config(cfg)
    assert (st == moe.MOE_OK) == ok, moe.last_error_string()


def test_layer_host_workspace_size(moe):
    cfg = moe.Config(T=1000, D=264, H_local=64, E=16, k=4)
    extra = 2 * ((1000 * 264 * 2 + 255) // 256 * 256)
    assert moe.layer_host_workspace_size(cfg) == moe.layer_workspace_size(cfg) + extra


@pytest.mark.parametrize("over", [dict(dtype=1), dict(e_first=2, E_local=6), dict(D=96),
                                  dict(H_local=80), dict(align_m=32)])
def test_training_path_rejects_unsupported_configs(moe, over):
    kw = dict(T=64, D=128, H_local=128, E=8, k=2)
    kw.update(over)
    if "dtype" in over:
        kw["dtype"] = moe.MOE_F32
    cfg = moe.Config(**kw)
    assert moe.validate_config(cfg) == moe.MOE_OK
    assert moe.layer_train_workspace_size(cfg) == -1
    c = cfg.c()
    assert moe._lib.moe_layer_forward_train(ctypes.byref(c), 0, 0, None, 0, 0, 0, 0, 0, 0, None) == \
        moe.MOE_ERR_UNSUPPORTED


def test_host_rejections_launch_nothing(moe):
    lib = moe._lib
    before = moe.kernel_launches()
    bad = moe.Config(T=10, D=12, H_local=8, E=4, k=5).c()
    assert lib.moe_layer_forward(ctypes.byref(bad), 0, 0, None, 0, 0, 0, 0, 0, 0, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(ctypes.byref(bad), 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert moe.kernel_launches() == before


def test_host_pipeline_host_checks(moe):
    """The host pipeline checks its config, workspace and handle on the host,
    before it creates a stream or queues anything."""
    lib = moe._lib
    cfg = _cfg(moe)
    n = moe.host_pipeline_workspace_size(cfg)
    assert n >= moe.layer_host_workspace_size(cfg) > 0
    assert moe.host_pipeline_workspace_size(_cfg(moe, D=12)) == -1
    h = ctypes.c_void_p(123)
    c = cfg.c()
    assert lib.moe_host_pipeline_create(ctypes.byref(c), None, n, ctypes.byref(h)) == \
        moe.MOE_ERR_WORKSPACE
    assert not h.value                                   # NULL on failure
    bad = _cfg(moe, k=0).c()
    assert lib.moe_host_pipeline_create(ctypes.byref(bad), 256, n, ctypes.byref(h)) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_host_pipeline_create(ctypes.byref(c), 256, n, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_host_pipeline_create(ctypes.byref(c), 256, n - 1, ctypes.byref(h)) == \
        moe.MOE_ERR_WORKSPACE
    assert lib.moe_host_pipeline_submit(None, 0, 0, None, 0, 0, 0, 0, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_host_pipeline_sync(None) == moe.MOE_ERR_INVALID_ARG
    lib.moe_host_pipeline_destroy(None)                  # a no-op


def test_status_strings(moe):
    assert moe.status_string(moe.MOE_OK) == "MOE_OK"
    assert moe.status_string(moe.MOE_ERR_CAPACITY) == "MOE_ERR_CAPACITY"
    assert moe.status_string(1234) == "MOE_ERR_UNKNOWN"
    assert moe.abi_version() >= 20000  # y_perm of bf16 layers is fp16 from 2.0.0


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "routing_grouped_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "moe_oracle" not in txt and "liboracle" not in txt, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            txt = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+(routing_grouped_gemm_gb300|moe_inputs)", txt,
                                 flags=re.M), f
            assert "libmoe" not in txt, f


def test_permute_noalloc_rejects_problems_beyond_its_scratch_on_the_host(moe):
    """The size check of moe_permute_noalloc runs before any CUDA call."""
    lib = moe._lib
    # 2 * ceil(T/256) * E = 2 * 1024 * 256 = 524288 int32 > the 262144 of its fixed scratch
    c = _cfg(moe, T=262144, E=256, k=8).c()
    st = lib.moe_permute_noalloc(ctypes.byref(c), 256, 256, 256, 256, 256, 256, 256, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert "fixed scratch" in moe.last_error_string()
    bad = _cfg(moe, k=0).c()
    assert lib.moe_permute_noalloc(ctypes.byref(bad), 0, 0, 0, 0, 0, 0, 0, None, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_noalloc_permute_limit_checked_on_the_host(moe):
    """moe_permute_noalloc refuses, before any launch or pointer check, a
    problem one 256-token count block past its fixed array; the largest
    problem that fits gets past the limit (and then fails on the NULL
    tensors, still on the host)."""
    lib = moe._lib
    over = _cfg(moe, T=131072 + 256, D=64, E=256, k=1).c()
    st = lib.moe_permute_noalloc(ctypes.byref(over), None, None, None, None, None, None, None,
                                 None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert "fixed scratch" in moe.last_error_string()
    fits = _cfg(moe, T=131072, D=64, E=256, k=1).c()
    st = lib.moe_permute_noalloc(ctypes.byref(fits), None, None, None, None, None, None, None,
                                 None, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_empty_batch_backward_checks_gradients_on_the_host(moe):
    """With T = 0 the backward zeroes the parameter gradients; a NULL or
    misaligned gradient pointer is rejected on the host before that."""
    cfg = moe.Config(T=0, D=128, H_local=128, E=8, k=2, dtype=moe.MOE_BF16)
    n = moe.layer_train_workspace_size(cfg)
    assert n > 0
    c = cfg.c()
    lib = moe._lib
    n0 = moe.kernel_launches()
    # dwg NULL, then dw1 misaligned; the workspace pointer is only checked for alignment
    assert lib.moe_layer_backward_ex(ctypes.byref(c), 0, 0, 0, 0, 0, 0, 0, None, None, 256, 256,
                                     256, moe.MOE_F32, 256, n, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_backward_ex(ctypes.byref(c), 0, 0, 0, 0, 0, 0, 0, 256, None, 264, 256,
                                     256, moe.MOE_F32, 256, n, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.kernel_launches() == n0
