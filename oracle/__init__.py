"""Plain CPU oracle for the MoE layer's local data path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product library
(``routing_grouped_gemm_gb300``) never imports, links or calls it, and this
package imports nothing from the product.  The two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64 accumulation);
this module only compiles it with gcc on first use and marshals numpy arrays.

Array conventions
-----------------
* ``np.float32`` / ``np.float64`` arrays are read as those types.
* ``np.uint16`` arrays are bf16 bit patterns (the upper half of a binary32).
* Integer outputs are ``np.int32``; float outputs are ``np.float64``.

What each function follows (page title, section):
* ``router_logits``       "Expert Parallelism (EP)" section 1, gating logits
* ``topk``/``topk_weights`` same section, "top-k + score_func"
* ``layout``/``permute_rows`` same section (tokens_per_expert, permute) and
                          section 2 (expert-contiguous, M-tile aligned layout)
* ``expert_ffn``/``moe_tokens``/``grouped_*`` same section, grouped
                          fc1 -> act -> fc2, with the SwiGLU expert of the
                          "Expert Tensor Parallel design" page, section 4.3
* ``unpermute_combine``   "Expert Parallelism (EP)" section 1, combine
                          post-process (top-k weighted reduce back to order)
* ``e4m3_*``/``quantize_rows_e4m3`` the FP8 step of the same page's next
                          steps (e4m3 dispatched activations with scales);
                          the scale granularity is a reading (one binary32
                          scale per row: amax / 448)

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force and the worked example of the
"NCCL course 32" page, section "Expert Parallel / MoE data flow").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
SOFTMAX, SIGMOID = 0, 1
CONTIGUOUS, MASKED = 0, 1
OK, BAD_ARG, CAPACITY, BAD_ROUTING = 0, 1, 3, 6
ROUND_H, ROUND_Y = 1, 2   # rounding points: h (bf16 tensor) and y

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``_lib/liboracle.so`` (gcc, -O2)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            lib.oracle_round_bf16.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16_array.argtypes = [L, P, P]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_router_logits.argtypes = [I, I, I, P, I, P, I, P, P, I]
            lib.oracle_topk.restype = I
            lib.oracle_topk.argtypes = [I, I, I, P, P]
            lib.oracle_topk_grouped.restype = I
            lib.oracle_topk_grouped.argtypes = [I, I, I, I, I, P, P]
            lib.oracle_moe_forward64.restype = I
            lib.oracle_moe_forward64.argtypes = [I, I, I, I, I, P, P, P, P, P, P, I, I, I, I, P, P]
            lib.oracle_moe_backward.restype = I
            lib.oracle_moe_backward.argtypes = [I, I, I, I, I, P, P, P, P, P, P, I, I, I, I, P,
                                                P, P, P, P, P, P, P]
            lib.oracle_topk_weights.argtypes = [I, I, I, P, P, I, I, P]
            lib.oracle_rows_alloc.restype = L
            lib.oracle_rows_alloc.argtypes = [I, I, I, I, I, I]
            lib.oracle_layout.restype = I
            lib.oracle_layout.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, L]
            lib.oracle_permute_rows.argtypes = [L, I, I, P, P, P]
            lib.oracle_expert_ffn.argtypes = [I, I, P, P, P, I, P, I, P]
            lib.oracle_moe_tokens.restype = I
            lib.oracle_moe_tokens.argtypes = [I, P, I, I, I, I, I, P, I, P, P, P, I,
                                              P, P, I, P, I]
            lib.oracle_grouped_gemm1_swiglu.argtypes = [I, I, I, P, P, P, I, P, P, I, I, P, I]
            lib.oracle_grouped_gemm2.argtypes = [I, I, I, P, P, P, I, P, I, I, P, I]
            lib.oracle_unpermute_combine.argtypes = [I, I, I, P, I, P, P, P]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [I]
            lib.oracle_e4m3_encode.restype = I
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_quantize_rows_e4m3.argtypes = [L, I, P, P, P]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle: unsupported element type {a.dtype}")


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def _p(a) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if a is None else a.ctypes.data)


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def round_bf16(a) -> np.ndarray:
    """Nearest bf16 value (ties to even) of each element, as float64."""
    a = np.asarray(a, dtype=np.float64)
    src = _c(a)
    out = np.empty_like(src)
    _load().oracle_round_bf16_array(src.size, _p(src), _p(out))
    return out.reshape(a.shape)


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, wg: np.ndarray, bias=None, nthreads=None) -> np.ndarray:
    """fp64 logits[t, e] = sum_d x[t,d] wg[e,d] (+ bias[e])."""
    x = _c(x)
    wg = _c(wg)
    T, D = x.shape
    E = wg.shape[0]
    assert wg.shape[1] == D
    b = None if bias is None else _c(bias, np.float64)
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits(T, D, E, _p(x), _dt(x), _p(wg), _dt(wg), _p(b),
                                 _p(out), nthreads or default_threads())
    return out


def topk(logits_f32: np.ndarray, k: int, n_group: int = 0, topk_group: int = 0):
    """(topk_idx int32 [T,k], status) from fp32 keys; ties -> lower index.

    With n_group > 1: group-limited selection (only experts of the
    topk_group best groups; a group scores the fp32 sum of its k/topk_group
    best keys).
    """
    l = _c(logits_f32, np.float32)
    T, E = l.shape
    idx = np.empty((T, k), np.int32)
    if n_group and n_group > 1:
        st = _load().oracle_topk_grouped(T, E, k, n_group, topk_group, _p(l), _p(idx))
    else:
        st = _load().oracle_topk(T, E, k, _p(l), _p(idx))
    return idx, st


def topk_weights(logits_f32: np.ndarray, idx: np.ndarray, score: int, renorm: bool) -> np.ndarray:
    l = _c(logits_f32, np.float32)
    idx = _c(idx, np.int32)
    T, E = l.shape
    k = idx.shape[1]
    w = np.empty((T, k), np.float64)
    _load().oracle_topk_weights(T, E, k, _p(l), _p(idx), int(score), int(bool(renorm)), _p(w))
    return w


def route(x, wg, bias, k: int, score: int, renorm: bool, nthreads=None, n_group: int = 0,
          topk_group: int = 0):
    """Whole router on the oracle's own logits.

    Returns (logits_f64, keys_f32, topk_idx, topk_w, status); the selection
    key is the fp32 rounding of the fp64 logit.
    """
    l64 = router_logits(x, wg, bias, nthreads)
    keys = l64.astype(np.float32)
    idx, st = topk(keys, k, n_group, topk_group)
    w = topk_weights(keys, idx, score, renorm)
    return l64, keys, idx, w, st


# --------------------------------------------------------------------------
# layout
# --------------------------------------------------------------------------

def rows_alloc(T, k, E_local, layout=CONTIGUOUS, align_m=128, capacity=0) -> int:
    return int(_load().oracle_rows_alloc(T, k, E_local, layout, align_m, capacity))


def layout(idx: np.ndarray, E: int, e_first: int = 0, E_local=None,
           layout_kind: int = CONTIGUOUS, align_m: int = 128, capacity: int = 0):
    """tokens_per_expert, segment offsets and the permutation (dict).

    The layout is complete for every status but BAD_ARG: a masked expert over
    ``capacity`` keeps its first ``capacity`` tokens (status CAPACITY), and a
    slot with an id outside [0, E) or an id repeated within its token is left
    out (status BAD_ROUTING; CAPACITY is reported first when both happen).
    """
    idx = _c(idx, np.int32)
    T, k = idx.shape
    if E_local is None:
        E_local = E - e_first
    ra = rows_alloc(T, k, E_local, layout_kind, align_m, capacity)
    # outputs start as a sentinel no layout contains, so an array the C code
    # did not write (a rejected argument) cannot pass for a result
    unset = np.iinfo(np.int32).min
    cnt = np.full(E, unset, np.int32)
    seg = np.full(E_local + 1, unset, np.int32)
    row_of = np.full((T, k), unset, np.int32)
    tor = np.full(max(ra, 1), unset, np.int32)
    st = _load().oracle_layout(T, k, E, e_first, E_local, layout_kind, align_m, capacity,
                               _p(idx), _p(cnt), _p(seg), _p(row_of), _p(tor), ra)
    return dict(status=st, tokens_per_expert=cnt, seg_offsets=seg, row_of=row_of,
                token_of_row=tor[:ra], rows_alloc=ra)


def permute_rows(x: np.ndarray, token_of_row: np.ndarray, fill=0) -> np.ndarray:
    """x_perm[r] = x[token_of_row[r]] (exact copy); unfilled rows = ``fill``."""
    x = _c(x)
    tor = _c(token_of_row, np.int32)
    out = np.full((tor.shape[0], x.shape[1]), fill, dtype=x.dtype)
    _load().oracle_permute_rows(tor.shape[0], x.shape[1], x.itemsize, _p(x), _p(tor), _p(out))
    return out


# --------------------------------------------------------------------------
# experts
# --------------------------------------------------------------------------

def _rounding(round_h: bool, round_y: bool) -> int:
    return (ROUND_H if round_h else 0) | (ROUND_Y if round_y else 0)


def expert_ffn(v: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray,
               round_h: bool = False, round_y: bool = False) -> np.ndarray:
    """FFN(v) = w2 . (SiLU(w1 . v) * (w3 . v)) for one expert (fp64 result).

    ``round_h`` / ``round_y`` round the hidden activation / the expert output
    to bf16 (nearest, ties to even) where a bf16 pipeline stores them.
    """
    v = _c(v, np.float64)
    w1, w3, w2 = _c(w1), _c(w3), _c(w2)
    Hl, D = w1.shape
    assert w3.shape == (Hl, D) and w2.shape == (D, Hl) and v.shape == (D,)
    assert w1.dtype == w3.dtype == w2.dtype
    y = np.empty(D, np.float64)
    _load().oracle_expert_ffn(D, Hl, _p(w1), _p(w3), _p(w2), _dt(w1), _p(v),
                              _rounding(round_h, round_y), _p(y))
    return y


def _ptr_table(ws, n):
    arr = (ctypes.c_void_p * n)()
    keep = []
    for i in range(n):
        w = ws[i] if i < len(ws) else None
        if w is None:
            arr[i] = None
        else:
            w = _c(w)
            keep.append(w)
            arr[i] = w.ctypes.data
    return arr, keep


def moe_tokens(tokens, x, w1s, w3s, w2s, topk_idx, topk_w, e_first: int = 0,
               round_h: bool = False, round_y: bool = False, nthreads=None) -> np.ndarray:
    """Brute-force per-token layer output (no permutation) for listed tokens.

    ``w1s[i]``, ``w3s[i]`` ([Hl, D]) and ``w2s[i]`` ([D, Hl]) are the weights
    of local expert ``e_first + i``; entries may be ``None`` for experts no
    listed token uses.  Returns fp64 [len(tokens), D].
    """
    tokens = _c(np.asarray(tokens), np.int32)
    x = _c(x)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float64)
    E_local = len(w1s)
    first = next(a for a in w1s if a is not None)
    Hl, D = first.shape
    wdt = _dt(first)
    t1, k1 = _ptr_table(w1s, E_local)
    t3, k3 = _ptr_table(w3s, E_local)
    t2, k2 = _ptr_table(w2s, E_local)
    out = np.empty((tokens.shape[0], D), np.float64)
    st = _load().oracle_moe_tokens(tokens.shape[0], _p(tokens), D, Hl, idx.shape[1], e_first,
                                   E_local, _p(x), _dt(x), t1, t3, t2, wdt, _p(idx), _p(w),
                                   _rounding(round_h, round_y), _p(out),
                                   nthreads or default_threads())
    if st != OK:
        raise ValueError("oracle.moe_tokens: a listed token uses an expert whose weights are missing")
    del k1, k3, k2
    return out


def grouped_gemm1_swiglu(x_perm, seg_offsets, cnt_local, w1s, w3s, round_h=False,
                         nthreads=None) -> np.ndarray:
    """h over the permuted layout (fp64 [rows, Hl]; unfilled rows are NaN)."""
    x_perm = _c(x_perm)
    seg = _c(seg_offsets, np.int32)
    cnt = _c(cnt_local, np.int32)
    E_local = len(w1s)
    first = next(a for a in w1s if a is not None)
    Hl, D = first.shape
    t1, k1 = _ptr_table(w1s, E_local)
    t3, k3 = _ptr_table(w3s, E_local)
    h = np.full((x_perm.shape[0], Hl), np.nan)
    _load().oracle_grouped_gemm1_swiglu(D, Hl, E_local, _p(seg), _p(cnt), _p(x_perm), _dt(x_perm),
                                        t1, t3, _dt(first), _rounding(round_h, False), _p(h),
                                        nthreads or default_threads())
    del k1, k3
    return h


def grouped_gemm2(h, seg_offsets, cnt_local, w2s, round_y=False, nthreads=None) -> np.ndarray:
    """y_perm over the permuted layout (fp64 [rows, D]; unfilled rows NaN)."""
    h = _c(h)
    seg = _c(seg_offsets, np.int32)
    cnt = _c(cnt_local, np.int32)
    E_local = len(w2s)
    first = next(a for a in w2s if a is not None)
    D, Hl = first.shape
    t2, k2 = _ptr_table(w2s, E_local)
    y = np.full((h.shape[0], D), np.nan)
    _load().oracle_grouped_gemm2(D, Hl, E_local, _p(seg), _p(cnt), _p(h), _dt(h), t2, _dt(first),
                                 _rounding(False, round_y), _p(y), nthreads or default_threads())
    del k2
    return y


def unpermute_combine(y_perm, row_of, topk_w) -> np.ndarray:
    """out[t] = sum_j w[t,j] y_perm[row_of[t,j]] (fp64 [T, D])."""
    y = _c(y_perm)
    ro = _c(row_of, np.int32)
    w = _c(topk_w, np.float64)
    T, k = ro.shape
    D = y.shape[1]
    out = np.empty((T, D), np.float64)
    _load().oracle_unpermute_combine(T, k, D, _p(y), _dt(y), _p(ro), _p(w), _p(out))
    return out


# --------------------------------------------------------------------------
# backward (fp64 throughout)
# --------------------------------------------------------------------------

def _f64(a):
    return None if a is None else _c(np.asarray(a, dtype=np.float64), np.float64)


def moe_forward64(x, wg, bias, w1, w3, w2, k: int, score: int, renorm: bool, n_group: int = 0,
                  topk_group: int = 0):
    """The whole layer in fp64 (selection on the fp64 logits), the function
    moe_backward differentiates.  x [T,D], wg [E,D], bias [E] or None,
    w1/w3 [E,H,D], w2 [E,D,H].  Returns (out [T,D], topk_idx [T,k])."""
    x, wg, b, w1, w3, w2 = (_f64(a) for a in (x, wg, bias, w1, w3, w2))
    T, D = x.shape
    E, H = w1.shape[0], w1.shape[1]
    out = np.empty((T, D), np.float64)
    idx = np.empty((T, k), np.int32)
    st = _load().oracle_moe_forward64(T, D, H, E, k, _p(x), _p(wg), _p(b) if b is not None else None,
                                      _p(w1), _p(w3), _p(w2), int(score), int(bool(renorm)),
                                      int(n_group), int(topk_group), _p(out), _p(idx))
    if st != OK:
        raise ValueError("oracle.moe_forward64: bad arguments")
    return out, idx


def moe_backward(x, wg, bias, w1, w3, w2, dout, k: int, score: int, renorm: bool,
                 n_group: int = 0, topk_group: int = 0) -> dict:
    """Gradients of sum(dout * out) for the fp64 layer of moe_forward64:
    keys dx, dwg, dbias, dw1, dw3, dw2 (and topk_idx, the selection used)."""
    x, wg, b, w1, w3, w2, go = (_f64(a) for a in (x, wg, bias, w1, w3, w2, dout))
    T, D = x.shape
    E, H = w1.shape[0], w1.shape[1]
    r = dict(dx=np.empty((T, D)), dwg=np.empty((E, D)), dbias=np.empty(E),
             dw1=np.empty((E, H, D)), dw3=np.empty((E, H, D)), dw2=np.empty((E, D, H)),
             topk_idx=np.empty((T, k), np.int32))
    st = _load().oracle_moe_backward(T, D, H, E, k, _p(x), _p(wg), _p(b) if b is not None else None,
                                     _p(w1), _p(w3), _p(w2), int(score), int(bool(renorm)),
                                     int(n_group), int(topk_group), _p(go), _p(r["dx"]),
                                     _p(r["dwg"]), _p(r["dbias"]), _p(r["dw1"]), _p(r["dw3"]),
                                     _p(r["dw2"]), _p(r["topk_idx"]))
    if st != OK:
        raise ValueError("oracle.moe_backward: bad arguments")
    return r


# --------------------------------------------------------------------------
# FP8 e4m3
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of an e4m3 ("fn": no infinities, max 448) code."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_encode(v: float) -> int:
    """Nearest e4m3 code of the binary32 value v (ties to even, saturating)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(v))))


def e4m3_table() -> np.ndarray:
    """float64 [256]: the value of every code (NaN for the two NaN codes)."""
    return np.array([e4m3_value(c) for c in range(256)], np.float64)


def quantize_rows_e4m3(src) -> tuple:
    """Row-wise e4m3 quantisation of a [rows, cols] array of binary32 values
    (bf16 bit patterns are widened exactly): (codes uint8, scales float32)."""
    a = np.asarray(src)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    a = _c(a, np.float32)
    rows, cols = a.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty(rows, np.float32)
    _load().oracle_quantize_rows_e4m3(rows, cols, _p(a), _p(q), _p(sc))
    return q, sc


def dequantize_rows_e4m3(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 scale[r] * value(codes[r, c]) (exact in fp64)."""
    tab = e4m3_table()
    return tab[np.asarray(codes, np.uint8)] * np.asarray(scales, np.float64)[:, None]
