"""Shared helpers of the GPU parity tests (marshalling and comparisons only)."""
import numpy as np
import torch

import moe_inputs
import oracle

TOL_F32 = 1e-4   # max |gpu - oracle| / rms(oracle), fp32 workloads
TOL_BF16 = 2e-2  # same measure, bf16 workloads


def tol(w):
    return TOL_F32 if w.dtype == "f32" else TOL_BF16


def cfg_for(moe, w, **over):
    kw = dict(T=w.T, D=w.D, H_local=w.H, E=w.E, k=w.k,
              dtype=moe.MOE_F32 if w.dtype == "f32" else moe.MOE_BF16,
              score=moe.MOE_SCORE_SOFTMAX if w.score == "softmax" else moe.MOE_SCORE_SIGMOID,
              renorm=int(w.renorm),
              layout=moe.MOE_LAYOUT_MASKED if w.layout == "masked" else moe.MOE_LAYOUT_CONTIGUOUS,
              align_m=128, capacity=w.T if w.layout == "masked" else 0,
              n_group=w.n_group, topk_group=w.topk_group)
    kw.update(over)
    return moe.Config(**kw)


def oscore(w):
    return oracle.SOFTMAX if w.score == "softmax" else oracle.SIGMOID


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt((ref ** 2).mean())
    return float(np.abs(got - ref).max() / max(rms, 1e-30))


def within_bf16_rounding(got, ref):
    """Element-wise bound for a bf16 intermediate that both sides round once.

    The two sides round values that differ only by accumulation-order error,
    so they can land on neighbouring bf16 values: at most one unit in the
    last place (2^-7 relative) at the element's own magnitude, or at the
    tensor's RMS for elements near zero.  Returns the worst ratio of the
    observed difference to that bound (<= 1 passes).
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt((ref ** 2).mean())
    bound = 2.0 ** -7 * np.maximum(np.abs(ref), rms)
    return float((np.abs(got - ref) / bound).max())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_route(inp, w, bias=None):
    H = moe_inputs.host_array
    b = None if bias is None else bias.detach().cpu().numpy().astype(np.float64)
    return oracle.route(H(inp.x), H(inp.wg), b, w.k, oscore(w), w.renorm, n_group=w.n_group,
                        topk_group=w.topk_group)


def routing_agreement(gidx: np.ndarray, oidx: np.ndarray, keys: np.ndarray, key_tol: float):
    """Tokens where GPU and oracle choose the same expert set.

    A token whose sets differ is accepted only as a near tie: every expert
    chosen by one side and not the other has an oracle key within key_tol of
    the oracle's k-th key.  Returns (same_set mask, same_order mask).
    """
    T, k = oidx.shape
    same_order = (gidx == oidx).all(1)
    same_set = np.array([set(gidx[t]) == set(oidx[t]) for t in range(T)])
    for t in np.nonzero(~same_set)[0]:
        kth = keys[t, oidx[t, -1]]
        diff = set(gidx[t]) ^ set(oidx[t])
        for e in diff:
            assert 0 <= e < keys.shape[1], f"token {t}: expert id {e} out of range"
            assert abs(float(keys[t, e]) - float(kth)) <= key_tol, \
                f"token {t}: routing differs beyond a near tie ({gidx[t]} vs {oidx[t]})"
    return same_set, same_order


def oracle_out_tokens(inp, w, toks, idx, wts, e_first=0, E_local=None, h0=0, Hl=None,
                      needed_only=True):
    """Oracle layer output on listed tokens; copies only the experts they use."""
    E_local = w.E - e_first if E_local is None else E_local
    Hl = w.H if Hl is None else Hl
    used = set(int(e) for e in np.unique(idx[toks])) if needed_only else set(range(w.E))
    H = moe_inputs.host_array
    w1s, w3s, w2s = [], [], []
    for i in range(E_local):
        e = e_first + i
        if e in used:
            w1s.append(H(inp.w1[e, h0:h0 + Hl]))
            w3s.append(H(inp.w3[e, h0:h0 + Hl]))
            w2s.append(H(inp.w2[e, :, h0:h0 + Hl]))
        else:
            w1s.append(None); w3s.append(None); w2s.append(None)
    if all(a is None for a in w1s):
        return np.zeros((len(toks), w.D))
    return oracle.moe_tokens(np.asarray(toks), H(inp.x), w1s, w3s, w2s, idx, wts,
                             e_first=e_first, round_h=(w.dtype == "bf16"))


def check_layout_properties(idx, lay, E, e_first, E_local, align_m=None, masked_cap=None):
    """Properties that fix the layout uniquely (hold at any size)."""
    T, k = idx.shape
    cnt, seg, row_of, tor = lay
    assert int(cnt.sum()) == T * k
    assert np.array_equal(cnt, np.bincount(idx.ravel(), minlength=E))
    for i in range(E_local):
        e = e_first + i
        size = seg[i + 1] - seg[i]
        if masked_cap is not None:
            assert seg[i] == i * masked_cap
        else:
            assert seg[i] % align_m == 0 and size == -(-cnt[e] // align_m) * align_m
        toks = np.nonzero((idx == e).any(1))[0]
        assert np.array_equal(tor[seg[i]:seg[i] + len(toks)], toks)
        assert (tor[seg[i] + len(toks):seg[i + 1]] == -1).all()
    local = (idx >= e_first) & (idx < e_first + E_local)
    assert (row_of[~local] == -1).all()
    tt = np.broadcast_to(np.arange(T)[:, None], idx.shape)
    assert np.array_equal(tor[row_of[local]], tt[local])


def assert_grouped_parity(lay, xp, w1, w3, w2, h, y, rb):
    """Grouped SwiGLU outputs h and y (CUDA tensors) against the oracle's
    grouped form over the layout `lay`, on the A rows xp (CUDA tensor
    [rows, D]); rb: bf16 (element-wise bounds) or fp32 (1e-4)."""
    H_ = moe_inputs.host_array
    seg, cnt = lay["seg_offsets"], lay["tokens_per_expert"]
    E_local = len(cnt)
    oh = oracle.grouped_gemm1_swiglu(H_(xp), seg, cnt, list(H_(w1)), list(H_(w3)), round_h=rb)
    filled = lay["token_of_row"] >= 0
    gh = to_f64(h)
    # second GEMM from the oracle's own h (no GPU value feeds the oracle)
    ohb = oh.astype(np.float32)
    oy = oracle.grouped_gemm2(ohb, seg, cnt, list(H_(w2)))
    gy = to_f64(y)
    if rb:
        # h is a bf16 intermediate rounded once on each side: compared per element
        assert within_bf16_rounding(gh[filled], oh[filled]) <= 1.0
        # y differs by what those h differences carry through w2, plus fp32
        # accumulation error, |dh| |w2|^T + 2^-20 |h| |w2|^T, plus the one
        # rounding of the accumulator to y's storage type: fp16 (11
        # significant bits: 2^-11 relative, 2^-25 absolute below 2^-14)
        w2h = to_f64(w2)
        dh = np.abs(np.nan_to_num(gh) - np.nan_to_num(oh))
        half = y.dtype == torch.float16
        for i in range(E_local):
            rows = np.arange(seg[i], seg[i] + cnt[i])
            if len(rows) == 0:
                continue
            aw2 = np.abs(w2h[i])
            bound = dh[rows] @ aw2.T + 2.0 ** -20 * (np.abs(oh[rows]) @ aw2.T) + 1e-30
            if half:
                bound = bound + 2.0 ** -11 * (np.abs(oy[rows]) + bound) + 2.0 ** -25
            assert (np.abs(gy[rows] - oy[rows]) <= bound).all(), f"expert {i}"
        assert rel_err(gy[filled], oy[filled]) < 1e-2
    else:
        assert rel_err(gh[filled], oh[filled]) < 1e-4
        assert rel_err(gy[filled], oy[filled]) < 1e-4
    # rows that hold no token (padding and past the last segment) are never written
    tail = ~filled
    if tail.any():
        tt = torch.from_numpy(tail).cuda()
        assert torch.isnan(h.float()[tt]).all() and torch.isnan(y[tt]).all()
