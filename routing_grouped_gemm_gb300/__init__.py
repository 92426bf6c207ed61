"""Python binding of the GB300 MoE local data path (``include/moe.h``).

Argument marshalling only: every function below checks shapes and dtypes,
passes raw device pointers and the current CUDA stream to the C ABI of
``_lib/libmoe.so`` and turns a non-OK status into ``MoeError``.  All compute
runs in the library's sm_103a kernels; there is no fallback of any kind --
importing this package fails if the library has not been built.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CAPACITY = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_BAD_ROUTING, MOE_ERR_WORKSPACE = 4, 5, 6, 7
MOE_F32, MOE_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_LAYOUT_CONTIGUOUS, MOE_LAYOUT_MASKED = 0, 1

# every symbol include/moe.h declares
ABI_SYMBOLS = (
    "moe_status_string", "moe_last_error_string", "moe_abi_version", "moe_validate_config",
    "moe_rows_alloc", "moe_workspace_size", "moe_layer_workspace_size", "moe_route_topk",
    "moe_permute", "moe_grouped_swiglu", "moe_unpermute_combine", "moe_layer_forward",
    "moe_get_device_status", "moe_permute_noalloc", "moe_kernel_launches",
    "moe_layer_host_workspace_size", "moe_layer_forward_host",
    "moe_layer_train_workspace_size", "moe_layer_forward_train", "moe_layer_backward",
    "moe_quantize_rows_fp8", "moe_permute_fp8", "moe_grouped_swiglu_fp8", "moe_layer_forward_fp8",
    "moe_layer_forward_fused", "moe_layer_backward_ex",
    "moe_host_pipeline_workspace_size", "moe_host_pipeline_create", "moe_host_pipeline_submit",
    "moe_host_pipeline_sync", "moe_host_pipeline_destroy",
    "moe_permute_index", "moe_grouped_swiglu_gather", "moe_layer_forward_gather",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({last_error_string()})")


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "D", "H_local", "E", "k", "e_first", "E_local", "dtype", "score", "renorm",
        "layout", "align_m", "capacity", "n_group", "topk_group")]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with routing_grouped_gemm_gb300.build.build() "
            "(nvcc, sm_103a). There is no CPU or eager fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    C = ctypes.POINTER(moe_config)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_last_error_string": (ctypes.c_char_p, []),
        "moe_abi_version": (I32, []),
        "moe_validate_config": (I32, [C]),
        "moe_rows_alloc": (I64, [C]),
        "moe_workspace_size": (I64, [C]),
        "moe_layer_workspace_size": (I64, [C]),
        "moe_route_topk": (I32, [C, P, P, P, P, P, P, P, SZ, P]),
        "moe_permute": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_grouped_swiglu": (I32, [C, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_unpermute_combine": (I32, [C, P, P, P, P, P, SZ, P]),
        "moe_layer_forward": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_get_device_status": (I32, [P, SZ, P]),
        "moe_permute_noalloc": (I32, [C, P, P, P, P, P, P, P, P, P]),
        "moe_kernel_launches": (ctypes.c_uint64, []),
        "moe_layer_host_workspace_size": (I64, [C]),
        "moe_layer_forward_host": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_train_workspace_size": (I64, [C]),
        "moe_layer_forward_train": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_backward": (I32, [C, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_quantize_rows_fp8": (I32, [P, I64, I32, P, P, P]),
        "moe_permute_fp8": (I32, [C, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_grouped_swiglu_fp8": (I32, [C, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_forward_fp8": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_forward_fused": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_backward_ex": (I32, [C, P, P, P, P, P, P, P, P, P, P, P, P, I32, P, SZ, P]),
        "moe_host_pipeline_workspace_size": (I64, [C]),
        "moe_host_pipeline_create": (I32, [C, P, SZ, ctypes.POINTER(P)]),
        "moe_host_pipeline_submit": (I32, [P, P, P, P, P, P, P, P, P]),
        "moe_host_pipeline_sync": (I32, [P]),
        "moe_host_pipeline_destroy": (None, [P]),
        "moe_permute_index": (I32, [C, P, P, P, P, P, P, SZ, P]),
        "moe_grouped_swiglu_gather": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_layer_forward_gather": (I32, [C, P, P, P, P, P, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


# --------------------------------------------------------------------------
# configuration
# --------------------------------------------------------------------------

@dataclass
class Config:
    T: int
    D: int
    H_local: int
    E: int
    k: int
    e_first: int = 0
    E_local: int = -1          # -1: every expert from e_first on
    dtype: int = MOE_BF16
    score: int = MOE_SCORE_SOFTMAX
    renorm: int = 0
    layout: int = MOE_LAYOUT_CONTIGUOUS
    align_m: int = 128
    capacity: int = 0
    n_group: int = 0           # > 1: group-limited routing over n_group expert groups
    topk_group: int = 0

    def c(self) -> moe_config:
        el = self.E - self.e_first if self.E_local < 0 else self.E_local
        return moe_config(self.T, self.D, self.H_local, self.E, self.k, self.e_first, el,
                          self.dtype, self.score, int(bool(self.renorm)), self.layout,
                          self.align_m, self.capacity, self.n_group, self.topk_group)

    @property
    def e_local(self) -> int:
        return self.E - self.e_first if self.E_local < 0 else self.E_local

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == MOE_BF16 else torch.float32

    @property
    def y_dtype(self) -> torch.dtype:
        """Element type of y_perm: fp16 for bf16 layers, fp32 for fp32 ones."""
        return torch.float16 if self.dtype == MOE_BF16 else torch.float32


def status_string(st: int) -> str:
    return _lib.moe_status_string(int(st)).decode()


def last_error_string() -> str:
    return _lib.moe_last_error_string().decode()


def abi_version() -> int:
    return int(_lib.moe_abi_version())


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(_lib.moe_kernel_launches())


def validate_config(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_validate_config(ctypes.byref(c)))


def rows_alloc(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_rows_alloc(ctypes.byref(c)))


def workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_workspace_size(ctypes.byref(c)))


def layer_workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_layer_workspace_size(ctypes.byref(c)))


def layer_host_workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_layer_host_workspace_size(ctypes.byref(c)))


def layer_train_workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_layer_train_workspace_size(ctypes.byref(c)))


def alloc_workspace(cfg: Config, layer: bool = False, device="cuda", host: bool = False,
                    train: bool = False) -> torch.Tensor:
    """Zero-filled workspace of the size the library asks for (torch-owned).

    layer: for moe_layer_forward; host: for moe_layer_forward_host; train: for
    moe_layer_forward_train / moe_layer_backward."""
    n = (layer_train_workspace_size(cfg) if train else
         layer_host_workspace_size(cfg) if host else
         layer_workspace_size(cfg) if layer else workspace_size(cfg))
    if n < 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "workspace size")
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(t) -> int:
    if t is None:
        return 0
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoeError(st, what)


def _expect(t, shape, dtype, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


# --------------------------------------------------------------------------
# the ABI calls (same names as include/moe.h)
# --------------------------------------------------------------------------

def moe_route_topk(cfg: Config, x, wg, bias, logits_out, topk_idx, topk_w, ws, stream=None):
    dt = cfg.torch_dtype
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    if logits_out is not None:
        _expect(logits_out, (cfg.T, cfg.E), torch.float32, "logits_out")
    _expect(topk_idx, (cfg.T, cfg.k), torch.int32, "topk_idx")
    _expect(topk_w, (cfg.T, cfg.k), torch.float32, "topk_w")
    c = cfg.c()
    _check(_lib.moe_route_topk(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(logits_out),
                               _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_topk")


def moe_permute(cfg: Config, x, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                x_perm, ws, stream=None):
    ra = rows_alloc(cfg)
    _expect(x, (cfg.T, cfg.D), cfg.torch_dtype, "x")
    _expect(topk_idx, (cfg.T, cfg.k), torch.int32, "topk_idx")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(seg_offsets, (cfg.e_local + 1,), torch.int32, "seg_offsets")
    _expect(row_of, (cfg.T, cfg.k), torch.int32, "row_of")
    _expect(token_of_row, (ra,), torch.int32, "token_of_row")
    _expect(x_perm, (ra, cfg.D), cfg.torch_dtype, "x_perm")
    c = cfg.c()
    _check(_lib.moe_permute(ctypes.byref(c), _ptr(x), _ptr(topk_idx), _ptr(tokens_per_expert),
                            _ptr(seg_offsets), _ptr(row_of), _ptr(token_of_row), _ptr(x_perm),
                            _ptr(ws), ws.numel(), _stream(stream)), "moe_permute")


def moe_permute_index(cfg: Config, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                      ws, stream=None):
    """moe_permute without the row copy: the layout arrays only."""
    ra = rows_alloc(cfg)
    _expect(topk_idx, (cfg.T, cfg.k), torch.int32, "topk_idx")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(seg_offsets, (cfg.e_local + 1,), torch.int32, "seg_offsets")
    _expect(row_of, (cfg.T, cfg.k), torch.int32, "row_of")
    _expect(token_of_row, (ra,), torch.int32, "token_of_row")
    c = cfg.c()
    _check(_lib.moe_permute_index(ctypes.byref(c), _ptr(topk_idx), _ptr(tokens_per_expert),
                                  _ptr(seg_offsets), _ptr(row_of), _ptr(token_of_row), _ptr(ws),
                                  ws.numel(), _stream(stream)), "moe_permute_index")


def moe_permute_noalloc(cfg: Config, x, topk_idx, tokens_per_expert, seg_offsets, row_of,
                        token_of_row, x_perm, device_flags=None, stream=None):
    """moe_permute for callers that cannot allocate: no workspace argument.

    The library keeps the counting-sort scratch in a fixed device array of
    its own (limit 2 * ceil(T/256) * E <= 262144 int32), shared by every
    call -- calls must not overlap on the GPU.  ``device_flags`` is an
    optional int32 CUDA tensor of one element that receives the status flags.
    """
    ra = rows_alloc(cfg)
    _expect(x, (cfg.T, cfg.D), cfg.torch_dtype, "x")
    _expect(topk_idx, (cfg.T, cfg.k), torch.int32, "topk_idx")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(seg_offsets, (cfg.e_local + 1,), torch.int32, "seg_offsets")
    _expect(row_of, (cfg.T, cfg.k), torch.int32, "row_of")
    _expect(token_of_row, (ra,), torch.int32, "token_of_row")
    _expect(x_perm, (ra, cfg.D), cfg.torch_dtype, "x_perm")
    if device_flags is not None:
        _expect(device_flags, (1,), torch.int32, "device_flags")
    c = cfg.c()
    _check(_lib.moe_permute_noalloc(ctypes.byref(c), _ptr(x), _ptr(topk_idx),
                                    _ptr(tokens_per_expert), _ptr(seg_offsets), _ptr(row_of),
                                    _ptr(token_of_row), _ptr(x_perm), _ptr(device_flags),
                                    _stream(stream)), "moe_permute_noalloc")


def moe_grouped_swiglu(cfg: Config, x_perm, seg_offsets, tokens_per_expert, w1, w3, w2, h, y_perm,
                       ws, stream=None):
    ra = rows_alloc(cfg)
    dt = cfg.torch_dtype
    el = cfg.e_local
    _expect(x_perm, (ra, cfg.D), dt, "x_perm")
    _expect(seg_offsets, (el + 1,), torch.int32, "seg_offsets")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(h, (ra, cfg.H_local), dt, "h")
    _expect(y_perm, (ra, cfg.D), cfg.y_dtype, "y_perm")
    c = cfg.c()
    _check(_lib.moe_grouped_swiglu(ctypes.byref(c), _ptr(x_perm), _ptr(seg_offsets),
                                   _ptr(tokens_per_expert), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(h),
                                   _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_swiglu")


def moe_unpermute_combine(cfg: Config, y_perm, row_of, topk_w, out, ws, stream=None):
    ra = rows_alloc(cfg)
    dt = cfg.torch_dtype
    _expect(y_perm, (ra, cfg.D), cfg.y_dtype, "y_perm")
    _expect(row_of, (cfg.T, cfg.k), torch.int32, "row_of")
    _expect(topk_w, (cfg.T, cfg.k), torch.float32, "topk_w")
    _expect(out, (cfg.T, cfg.D), dt, "out")
    c = cfg.c()
    _check(_lib.moe_unpermute_combine(ctypes.byref(c), _ptr(y_perm), _ptr(row_of), _ptr(topk_w),
                                      _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_unpermute_combine")


def moe_layer_forward(cfg: Config, x, wg, bias, w1, w3, w2, out, ws, stream=None):
    dt = cfg.torch_dtype
    el = cfg.e_local
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(out, (cfg.T, cfg.D), dt, "out")
    c = cfg.c()
    _check(_lib.moe_layer_forward(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w1),
                                  _ptr(w3), _ptr(w2), _ptr(out), _ptr(ws), ws.numel(),
                                  _stream(stream)), "moe_layer_forward")


def moe_layer_forward_host(cfg: Config, x_host, wg, bias, w1, w3, w2, out_host, ws, stream=None):
    """moe_layer_forward with x and out in host memory (page-locked for
    asynchronous copies); the weights are CUDA tensors."""
    dt = cfg.torch_dtype
    el = cfg.e_local
    for t, shape, name in ((x_host, (cfg.T, cfg.D), "x_host"), (out_host, (cfg.T, cfg.D), "out_host")):
        if tuple(t.shape) != shape or t.dtype != dt or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous host tensor {shape} {dt}")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    c = cfg.c()
    _check(_lib.moe_layer_forward_host(ctypes.byref(c), x_host.data_ptr(), _ptr(wg), _ptr(bias),
                                       _ptr(w1), _ptr(w3), _ptr(w2), out_host.data_ptr(), _ptr(ws),
                                       ws.numel(), _stream(stream)), "moe_layer_forward_host")


def host_pipeline_workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(_lib.moe_host_pipeline_workspace_size(ctypes.byref(c)))


class HostPipeline:
    """moe_host_pipeline: moe_layer_forward calls on host activations whose
    input and output copies overlap the neighbouring calls' compute.

    submit() queues one call (x_host, out_host: contiguous host tensors,
    page-locked for overlap; every call on the same compute stream); sync()
    waits for all of them, output copies included, and raises on a flagged
    device status.  Host buffers must stay valid, and x_host unchanged,
    until sync() returns."""

    def __init__(self, cfg: Config, device="cuda"):
        n = host_pipeline_workspace_size(cfg)
        if n < 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "host pipeline workspace size")
        self.cfg = cfg
        self.ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
        self._c = cfg.c()
        h = ctypes.c_void_p()
        _check(_lib.moe_host_pipeline_create(ctypes.byref(self._c), _ptr(self.ws), self.ws.numel(),
                                             ctypes.byref(h)), "moe_host_pipeline_create")
        self._h = h
        self._keep = []

    def submit(self, x_host, wg, bias, w1, w3, w2, out_host, stream=None):
        cfg = self.cfg
        dt = cfg.torch_dtype
        el = cfg.e_local
        for t, shape, name in ((x_host, (cfg.T, cfg.D), "x_host"),
                               (out_host, (cfg.T, cfg.D), "out_host")):
            if tuple(t.shape) != shape or t.dtype != dt or t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name}: expected a contiguous host tensor {shape} {dt}")
        _expect(wg, (cfg.E, cfg.D), dt, "wg")
        if bias is not None:
            _expect(bias, (cfg.E,), torch.float32, "bias")
        _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
        _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
        _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
        self._keep.append((x_host, out_host))  # alive until sync()
        _check(_lib.moe_host_pipeline_submit(self._h, x_host.data_ptr(), _ptr(wg), _ptr(bias),
                                             _ptr(w1), _ptr(w3), _ptr(w2), out_host.data_ptr(),
                                             _stream(stream)), "moe_host_pipeline_submit")

    def sync(self):
        st = int(_lib.moe_host_pipeline_sync(self._h))
        self._keep.clear()
        if st != MOE_OK:
            raise MoeError(st, "moe_host_pipeline_sync")

    def close(self):
        if self._h:
            _lib.moe_host_pipeline_destroy(self._h)
            self._h = None
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_layer_forward_train(cfg: Config, x, wg, bias, w1, w3, w2, out, ws, stream=None):
    dt = cfg.torch_dtype
    el = cfg.e_local
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(out, (cfg.T, cfg.D), dt, "out")
    c = cfg.c()
    _check(_lib.moe_layer_forward_train(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w1),
                                        _ptr(w3), _ptr(w2), _ptr(out), _ptr(ws), ws.numel(),
                                        _stream(stream)), "moe_layer_forward_train")


def moe_layer_backward(cfg: Config, x, wg, w1, w3, w2, dout, dx, dwg, dbias, dw1, dw3, dw2, ws,
                       stream=None):
    """Gradients for the forward last run by moe_layer_forward_train on ws.

    dw1, dw3 and dw2 may be fp32 or bf16 (all three the same); dwg and dbias
    are fp32.
    """
    dt = cfg.torch_dtype
    el = cfg.e_local
    f32 = torch.float32
    wdt = dw1.dtype if dw1 is not None else f32
    if wdt not in (torch.float32, torch.bfloat16):
        raise ValueError("dw1, dw3, dw2: float32 or bfloat16")
    _expect(dout, (cfg.T, cfg.D), dt, "dout")
    _expect(dx, (cfg.T, cfg.D), dt, "dx")
    _expect(dwg, (cfg.E, cfg.D), f32, "dwg")
    if dbias is not None:
        _expect(dbias, (cfg.E,), f32, "dbias")
    _expect(dw1, (el, cfg.H_local, cfg.D), wdt, "dw1")
    _expect(dw3, (el, cfg.H_local, cfg.D), wdt, "dw3")
    _expect(dw2, (el, cfg.D, cfg.H_local), wdt, "dw2")
    c = cfg.c()
    _check(_lib.moe_layer_backward_ex(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(w1), _ptr(w3),
                                      _ptr(w2), _ptr(dout), _ptr(dx), _ptr(dwg), _ptr(dbias),
                                      _ptr(dw1), _ptr(dw3), _ptr(dw2),
                                      MOE_BF16 if wdt == torch.bfloat16 else MOE_F32, _ptr(ws),
                                      ws.numel(), _stream(stream)), "moe_layer_backward")


# --------------------------------------------------------------------------
# FP8 e4m3 dispatch and GEMM1 (codes are torch.uint8 tensors)
# --------------------------------------------------------------------------

def moe_quantize_rows_fp8(src, dst, scale, stream=None):
    """Row-wise e4m3 codes and fp32 scales of a bf16 tensor viewed as [rows, cols]."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src: a contiguous bf16 CUDA tensor")
    cols = src.shape[-1]
    rows = src.numel() // cols if cols else 0
    _expect(dst, tuple(src.shape), torch.uint8, "dst")
    _expect(scale, tuple(src.shape[:-1]), torch.float32, "scale")
    _check(_lib.moe_quantize_rows_fp8(_ptr(src), rows, cols, _ptr(dst), _ptr(scale),
                                      _stream(stream)), "moe_quantize_rows_fp8")


def quantize_weights_fp8(w, stream=None):
    """(codes uint8, scales fp32 [..., rows]) of a bf16 weight [E, H, D] (one scale per row)."""
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    moe_quantize_rows_fp8(w, q, sc, stream)
    return q, sc


def moe_permute_fp8(cfg: Config, x, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                    x_perm_q, x_scale, ws, stream=None):
    ra = rows_alloc(cfg)
    _expect(x, (cfg.T, cfg.D), torch.bfloat16, "x")
    _expect(topk_idx, (cfg.T, cfg.k), torch.int32, "topk_idx")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(seg_offsets, (cfg.e_local + 1,), torch.int32, "seg_offsets")
    _expect(row_of, (cfg.T, cfg.k), torch.int32, "row_of")
    _expect(token_of_row, (ra,), torch.int32, "token_of_row")
    _expect(x_perm_q, (ra, cfg.D), torch.uint8, "x_perm_q")
    _expect(x_scale, (ra,), torch.float32, "x_scale")
    c = cfg.c()
    _check(_lib.moe_permute_fp8(ctypes.byref(c), _ptr(x), _ptr(topk_idx), _ptr(tokens_per_expert),
                                _ptr(seg_offsets), _ptr(row_of), _ptr(token_of_row),
                                _ptr(x_perm_q), _ptr(x_scale), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_permute_fp8")


def moe_grouped_swiglu_fp8(cfg: Config, x_perm_q, x_scale, seg_offsets, tokens_per_expert, w1_q,
                           w1_scale, w3_q, w3_scale, w2, h, y_perm, ws, stream=None):
    ra = rows_alloc(cfg)
    el = cfg.e_local
    _expect(x_perm_q, (ra, cfg.D), torch.uint8, "x_perm_q")
    _expect(x_scale, (ra,), torch.float32, "x_scale")
    _expect(seg_offsets, (el + 1,), torch.int32, "seg_offsets")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(w1_q, (el, cfg.H_local, cfg.D), torch.uint8, "w1_q")
    _expect(w3_q, (el, cfg.H_local, cfg.D), torch.uint8, "w3_q")
    _expect(w1_scale, (el, cfg.H_local), torch.float32, "w1_scale")
    _expect(w3_scale, (el, cfg.H_local), torch.float32, "w3_scale")
    _expect(w2, (el, cfg.D, cfg.H_local), torch.bfloat16, "w2")
    _expect(h, (ra, cfg.H_local), torch.bfloat16, "h")
    _expect(y_perm, (ra, cfg.D), cfg.y_dtype, "y_perm")
    c = cfg.c()
    _check(_lib.moe_grouped_swiglu_fp8(ctypes.byref(c), _ptr(x_perm_q), _ptr(x_scale),
                                       _ptr(seg_offsets), _ptr(tokens_per_expert), _ptr(w1_q),
                                       _ptr(w1_scale), _ptr(w3_q), _ptr(w3_scale), _ptr(w2),
                                       _ptr(h), _ptr(y_perm), _ptr(ws), ws.numel(),
                                       _stream(stream)), "moe_grouped_swiglu_fp8")


def moe_layer_forward_fp8(cfg: Config, x, wg, bias, w1_q, w1_scale, w3_q, w3_scale, w2, out, ws,
                          stream=None):
    el = cfg.e_local
    _expect(x, (cfg.T, cfg.D), torch.bfloat16, "x")
    _expect(wg, (cfg.E, cfg.D), torch.bfloat16, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1_q, (el, cfg.H_local, cfg.D), torch.uint8, "w1_q")
    _expect(w3_q, (el, cfg.H_local, cfg.D), torch.uint8, "w3_q")
    _expect(w1_scale, (el, cfg.H_local), torch.float32, "w1_scale")
    _expect(w3_scale, (el, cfg.H_local), torch.float32, "w3_scale")
    _expect(w2, (el, cfg.D, cfg.H_local), torch.bfloat16, "w2")
    _expect(out, (cfg.T, cfg.D), torch.bfloat16, "out")
    c = cfg.c()
    _check(_lib.moe_layer_forward_fp8(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w1_q),
                                      _ptr(w1_scale), _ptr(w3_q), _ptr(w3_scale), _ptr(w2),
                                      _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_layer_forward_fp8")


def moe_grouped_swiglu_gather(cfg: Config, x, token_of_row, seg_offsets, tokens_per_expert, w1,
                              w3, w2, h, y_perm, ws, stream=None):
    """moe_grouped_swiglu with GEMM1's rows read from x by token_of_row."""
    ra = rows_alloc(cfg)
    dt = cfg.torch_dtype
    el = cfg.e_local
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(token_of_row, (ra,), torch.int32, "token_of_row")
    _expect(seg_offsets, (el + 1,), torch.int32, "seg_offsets")
    _expect(tokens_per_expert, (cfg.E,), torch.int32, "tokens_per_expert")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(h, (ra, cfg.H_local), dt, "h")
    _expect(y_perm, (ra, cfg.D), cfg.y_dtype, "y_perm")
    c = cfg.c()
    _check(_lib.moe_grouped_swiglu_gather(ctypes.byref(c), _ptr(x), _ptr(token_of_row),
                                          _ptr(seg_offsets), _ptr(tokens_per_expert), _ptr(w1),
                                          _ptr(w3), _ptr(w2), _ptr(h), _ptr(y_perm), _ptr(ws),
                                          ws.numel(), _stream(stream)), "moe_grouped_swiglu_gather")


def moe_layer_forward_gather(cfg: Config, x, wg, bias, w1, w3, w2, out, ws, stream=None):
    """moe_layer_forward with the dispatch fused into GEMM1's operand load
    (no x_perm); bitwise the same output."""
    el = cfg.e_local
    dt = cfg.torch_dtype
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(out, (cfg.T, cfg.D), dt, "out")
    c = cfg.c()
    _check(_lib.moe_layer_forward_gather(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w1),
                                         _ptr(w3), _ptr(w2), _ptr(out), _ptr(ws), ws.numel(),
                                         _stream(stream)), "moe_layer_forward_gather")


def moe_layer_forward_fused(cfg: Config, x, wg, bias, w1, w3, w2, out, ws, stream=None):
    """moe_layer_forward with the combine fused into GEMM2's epilogue (fp32
    atomics; not bitwise reproducible run to run)."""
    el = cfg.e_local
    dt = cfg.torch_dtype
    _expect(x, (cfg.T, cfg.D), dt, "x")
    _expect(wg, (cfg.E, cfg.D), dt, "wg")
    if bias is not None:
        _expect(bias, (cfg.E,), torch.float32, "bias")
    _expect(w1, (el, cfg.H_local, cfg.D), dt, "w1")
    _expect(w3, (el, cfg.H_local, cfg.D), dt, "w3")
    _expect(w2, (el, cfg.D, cfg.H_local), dt, "w2")
    _expect(out, (cfg.T, cfg.D), dt, "out")
    c = cfg.c()
    _check(_lib.moe_layer_forward_fused(ctypes.byref(c), _ptr(x), _ptr(wg), _ptr(bias), _ptr(w1),
                                        _ptr(w3), _ptr(w2), _ptr(out), _ptr(ws), ws.numel(),
                                        _stream(stream)), "moe_layer_forward_fused")


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace status word (returns a code)."""
    return int(_lib.moe_get_device_status(_ptr(ws), ws.numel(), _stream(stream)))


def layer_views(cfg: Config, ws: torch.Tensor) -> dict:
    """Views of the intermediates moe_layer_forward keeps in its workspace.

    Mirrors the carving order of the library (256-byte aligned regions after
    the step workspace): topk_idx, topk_w, tokens_per_expert, seg_offsets,
    row_of, token_of_row, x_perm (x_perm_q: the FP8 layer's codes in the same
    bytes), h, y_perm, x_scale (the FP8 layer's row scales).
    """
    def up(n):
        return (n + 255) // 256 * 256
    off = workspace_size(cfg)
    R = cfg.T * cfg.k
    ra = rows_alloc(cfg)
    el = cfg.e_local
    dt = cfg.torch_dtype
    out = {}
    for name, n, tdt, shape in (
            ("topk_idx", R, torch.int32, (cfg.T, cfg.k)),
            ("topk_w", R, torch.float32, (cfg.T, cfg.k)),
            ("tokens_per_expert", cfg.E, torch.int32, (cfg.E,)),
            ("seg_offsets", el + 1, torch.int32, (el + 1,)),
            ("row_of", R, torch.int32, (cfg.T, cfg.k)),
            ("token_of_row", ra, torch.int32, (ra,)),
            ("x_perm", ra * cfg.D, dt, (ra, cfg.D)),
            ("h", ra * cfg.H_local, dt, (ra, cfg.H_local)),
            ("y_perm", ra * cfg.D, cfg.y_dtype, (ra, cfg.D)),
            ("x_scale", ra, torch.float32, (ra,))):
        nbytes = n * (4 if tdt in (torch.int32, torch.float32) else 2)
        region = nbytes
        if name == "y_perm" and cfg.dtype == MOE_BF16:
            region = max(nbytes, cfg.T * cfg.D * 4)   # also holds the fused combine's fp32 sums
        out[name] = ws[off:off + nbytes].view(tdt).view(shape)
        if name == "x_perm":
            # moe_layer_forward_fp8 keeps the e4m3 codes at the start of this buffer
            out["x_perm_q"] = ws[off:off + ra * cfg.D].view(ra, cfg.D)
        off += up(region)
    return out
