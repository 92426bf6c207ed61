"""Pins of the oracle's backward of the layer (CPU only).

The backward ("Expert Parallelism (EP)" page, section 5: the backward runs
the forward's steps in mirror -- combine-bwd is a dispatch, dispatch-bwd a
combine -- with m-grouped dgrad and k-grouped wgrad for the expert weights)
is checked against central finite differences of the oracle's own fp64
forward, for every parameter kind and every score mode, and the fp64
forward is checked against the fp32-keyed forward the parity tests use.
"""
import numpy as np
import pytest

import oracle


def _problem(seed, T=3, D=5, H=4, E=6):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((T, D)), wg=rng.standard_normal((E, D)),
                bias=rng.standard_normal(E) * 0.1,
                w1=rng.standard_normal((E, H, D)) * 0.5, w3=rng.standard_normal((E, H, D)) * 0.5,
                w2=rng.standard_normal((E, D, H)) * 0.5,
                dout=rng.standard_normal((T, D)))


def _loss(p, k, score, renorm, n_group, topk_group):
    out, idx = oracle.moe_forward64(p["x"], p["wg"], p["bias"], p["w1"], p["w3"], p["w2"], k, score,
                                    renorm, n_group, topk_group)
    return float((p["dout"] * out).sum()), idx


MODES = [(oracle.SOFTMAX, False), (oracle.SOFTMAX, True), (oracle.SIGMOID, False),
         (oracle.SIGMOID, True)]


@pytest.mark.parametrize("score,renorm", MODES)
@pytest.mark.parametrize("k,n_group,topk_group", [(2, 0, 0), (3, 3, 2)])
def test_backward_matches_finite_differences(score, renorm, k, n_group, topk_group):
    p = _problem(seed=11 + 7 * score + int(renorm) + k)
    g = oracle.moe_backward(p["x"], p["wg"], p["bias"], p["w1"], p["w3"], p["w2"], p["dout"], k,
                            score, renorm, n_group, topk_group)
    _, idx0 = _loss(p, k, score, renorm, n_group, topk_group)
    assert np.array_equal(g["topk_idx"], idx0)
    grads = dict(x=g["dx"], wg=g["dwg"], bias=g["dbias"], w1=g["dw1"], w3=g["dw3"], w2=g["dw2"])
    rng = np.random.default_rng(5)
    eps = 1e-6
    checked = 0
    for name, grad in grads.items():
        flat = p[name].reshape(-1)
        picks = rng.choice(flat.size, size=min(12, flat.size), replace=False)
        for i in picks:
            keep = flat[i]
            flat[i] = keep + eps
            lp, ip = _loss(p, k, score, renorm, n_group, topk_group)
            flat[i] = keep - eps
            lm, im = _loss(p, k, score, renorm, n_group, topk_group)
            flat[i] = keep
            if not (np.array_equal(ip, idx0) and np.array_equal(im, idx0)):
                continue   # the selection moved: no derivative there
            fd = (lp - lm) / (2 * eps)
            an = grad.reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, i, fd, an)
            checked += 1
    assert checked >= 60


def test_backward_zero_routes_give_zero_expert_grads():
    """Experts no token selects get no weight gradient; with dout = 0 every
    gradient is zero."""
    p = _problem(seed=3, T=2, E=8)
    g = oracle.moe_backward(p["x"], p["wg"], p["bias"], p["w1"], p["w3"], p["w2"], p["dout"], 2,
                            oracle.SOFTMAX, True)
    used = set(g["topk_idx"].reshape(-1).tolist())
    for e in range(8):
        if e not in used:
            assert not g["dw1"][e].any() and not g["dw3"][e].any() and not g["dw2"][e].any()
    z = oracle.moe_backward(p["x"], p["wg"], p["bias"], p["w1"], p["w3"], p["w2"],
                            np.zeros_like(p["dout"]), 2, oracle.SIGMOID, False)
    for key in ("dx", "dwg", "dbias", "dw1", "dw3", "dw2"):
        assert not z[key].any()


def test_forward64_matches_fp32_keyed_forward():
    """The fp64 layer equals the forward used by the parity tests (which
    selects and weighs on fp32 keys) up to the fp32 rounding of the keys."""
    rng = np.random.default_rng(9)
    T, D, H, E, k = 40, 24, 16, 8, 2
    x = rng.standard_normal((T, D))
    wg = rng.standard_normal((E, D)) * 0.3
    w1 = rng.standard_normal((E, H, D)) * 0.2
    w3 = rng.standard_normal((E, H, D)) * 0.2
    w2 = rng.standard_normal((E, D, H)) * 0.2
    out64, idx64 = oracle.moe_forward64(x, wg, None, w1, w3, w2, k, oracle.SOFTMAX, True)
    l64, keys, idx, w, st = oracle.route(x, wg, None, k, oracle.SOFTMAX, True)
    assert np.array_equal(idx, idx64)
    ref = oracle.moe_tokens(np.arange(T), x, list(w1), list(w3), list(w2), idx, w)
    assert np.abs(out64 - ref).max() <= 1e-6 * np.abs(ref).max()
