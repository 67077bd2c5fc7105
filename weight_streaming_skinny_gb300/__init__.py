"""GB300 (sm_103a) decode-linear weight streaming: Python binding.

y[M, N] = x[M, K] . W[N, K]^T (+ bias) for M = 1..16 decode tokens, with bf16
weights or weight-only FP8 (e4m3, one fp32 scale per 128x128 block).  Every
step runs in the CUDA kernels of ``libdecode_linear.so`` behind the C ABI in
``include/dl_linear.h``; this module only checks torch tensors and passes raw
device pointers, sizes and the current stream through ctypes.  There is no CPU
fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass

import torch

__all__ = [
    "BF16", "FP8_B128", "KERNEL_AUTO", "KERNEL_SIMT", "KERNEL_MMA", "DLError", "Layer",
    "library_path", "load", "version", "workspace_bytes", "Workspace", "linear_bf16",
    "linear_swiglu", "linear_argmax", "interleave_gate_up", "ABI_VERSION",
    "linear_bf16_static_scratch", "STATIC_SCRATCH_BYTES", "WORKSPACE_ZERO_BYTES",
    "linear_fp8_block128", "decode_stream", "decode_stream_workspace_bytes",
    "decode_stream_launches", "graph_cache_clear", "graph_cache_size", "set_wait_test",
    "set_override",
    "device_status", "exported_symbols", "header_symbols",
]

BF16 = 0
FP8_B128 = 1
KERNEL_AUTO, KERNEL_SIMT, KERNEL_MMA, KERNEL_TC = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libdecode_linear.so")
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "dl_linear.h")
_lock = threading.Lock()
_lib = None

_STATUS = {0: "DL_OK", 1: "DL_ERR_INVALID_ARG", 2: "DL_ERR_UNSUPPORTED_SHAPE",
           3: "DL_ERR_MISALIGNED", 4: "DL_ERR_WORKSPACE", 5: "DL_ERR_CUDA", 6: "DL_ERR_DEVICE"}


class DLError(RuntimeError):
    """A non-OK dl_status; ``.status`` holds the code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class _Layer(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("M", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("x", ctypes.c_void_p), ("W", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("act", ctypes.c_int)]

ABI_VERSION = 3   # DL_VERSION this binding marshals for


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load the shared library (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.dl_version.restype = i
        lib.dl_last_error.restype = ctypes.c_char_p
        lib.dl_workspace_bytes.argtypes = [i, i, i, i]
        lib.dl_workspace_bytes.restype = sz
        lib.dl_linear_bf16.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.dl_linear_bf16.restype = i
        lib.dl_linear_fp8_block128.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.dl_linear_fp8_block128.restype = i
        lib.dl_decode_stream.argtypes = [ctypes.POINTER(_Layer), i, vp, sz, vp, i]
        lib.dl_decode_stream.restype = i
        lib.dl_graph_cache_clear.restype = None
        lib.dl_graph_cache_size.restype = i
        lib.dl_set_wait_test.argtypes = [ctypes.c_longlong, i]
        lib.dl_set_wait_test.restype = i
        lib.dl_decode_stream_workspace_bytes.argtypes = [ctypes.POINTER(_Layer), i]
        lib.dl_decode_stream_workspace_bytes.restype = sz
        lib.dl_decode_stream_launches.argtypes = [ctypes.POINTER(_Layer), i, sz]
        lib.dl_decode_stream_launches.restype = i
        lib.dl_linear_swiglu.argtypes = [i, vp, vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.dl_linear_argmax.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, vp, sz, vp]
        lib.dl_linear_argmax.restype = i
        lib.dl_linear_swiglu.restype = i
        lib.dl_set_override.argtypes = [i, i, i]
        lib.dl_set_override.restype = i
        lib.dl_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.dl_device_status.restype = i
        if lib.dl_version() != ABI_VERSION:
            raise RuntimeError(f"{_LIB_PATH} is ABI version {lib.dl_version()}, this binding "
                               f"marshals version {ABI_VERSION}: rebuild the library")
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        raise DLError(status, load().dl_last_error().decode(errors="replace"))


def version() -> int:
    return load().dl_version()


def header_symbols() -> list[str]:
    """Function names declared in include/dl_linear.h."""
    text = open(_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dl_[a-z0-9_]+)\s*\(", text)))


def exported_symbols() -> list[str]:
    lib = load()
    return [s for s in header_symbols() if hasattr(lib, s)]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def workspace_bytes(M: int, N: int, K: int, dtype: int) -> int:
    """Workspace one call needs on the current device (0 = invalid shape)."""
    return int(load().dl_workspace_bytes(M, N, K, dtype))


class Workspace:
    """A device buffer for the arrival counters (its first WORKSPACE_ZERO_BYTES,
    zero-filled here once; every call leaves them zero) and the calls' scratch
    (split-K partial sums, the FP8 activation copy).  Do not share one
    Workspace between streams that may run at the same time.
    """

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = max(int(nbytes), 256)
        self.tensor = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        # the zeros must be in place before a kernel on any stream reads them
        torch.cuda.synchronize(self.tensor.device)

    @classmethod
    def for_shapes(cls, shapes, device="cuda"):
        """Workspace large enough for every (M, N, K, dtype) in `shapes`."""
        with torch.cuda.device(torch.device(device)):
            n = max(workspace_bytes(*s) for s in shapes)
        return cls(n, device)

    @classmethod
    def for_stream(cls, layers, device=None):
        """Workspace with which decode_stream makes the activation copies of all
        FP8 layers whose x no earlier layer writes in one launch at the start."""
        n = decode_stream_workspace_bytes(layers)
        return cls(n, device if device is not None else layers[0].x.device)

    def reset(self):
        self.tensor.zero_()
        torch.cuda.synchronize(self.tensor.device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())


_default_ws: dict = {}


def _workspace(ws, need: int, device):
    if ws is not None:
        return ws
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    cur = _default_ws.get(key)
    if cur is None or cur.nbytes < need:
        cur = Workspace(need, device)
        _default_ws[key] = cur
    return cur


def _out(out, out_f32, M, N, device):
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    _need(out, "out", torch.bfloat16, device)
    if out.numel() != M * N:
        raise ValueError("out must hold M*N elements")
    if out_f32 is not None:
        _need(out_f32, "out_f32", torch.float32, device)
        if out_f32.numel() != M * N:
            raise ValueError("out_f32 must hold M*N elements")
    return out


def linear_bf16(x, w, bias=None, *, out=None, out_f32=None, workspace: Workspace | None = None,
                stream=None):
    """out[M, N] (bf16) = x[M, K] . w[N, K]^T (+ bias[N]); bf16 weights."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    _need(w, "w", torch.bfloat16, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev)
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    M, K = x.shape
    N = w.shape[0]
    if bias is not None and bias.numel() != N:
        raise ValueError("bias must be [N]")
    out = _out(out, out_f32, M, N, dev)
    with torch.cuda.device(dev):
        need = workspace_bytes(M, N, K, BF16)
        ws = _workspace(workspace, need, dev)
        _check(load().dl_linear_bf16(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), _ptr(out_f32),
                                     M, N, K, ws.ptr, ws.nbytes, _stream(stream, dev)))
    return out


def linear_swiglu(x, w, scales=None, bias=None, *, out=None, out_f32=None,
                  workspace: Workspace | None = None, stream=None):
    """out[M, N/2] = silu(g) * u: gate_up projection with the SwiGLU epilogue.

    w: [N, K] bf16, or e4m3 codes (uint8 / float8_e4m3fn) with fp32 `scales`,
    its gate and up rows interleaved in groups of 16 (rows 16b..16b+7 gate,
    16b+8..16b+15 up, of outputs 8b..8b+7); see interleave_gate_up.
    """
    if isinstance(w, torch.Tensor) and w.dtype == torch.float8_e4m3fn:
        w = w.view(torch.uint8)
    _need(x, "x", torch.bfloat16)
    dev = x.device
    fp8 = scales is not None
    _need(w, "w", torch.uint8 if fp8 else torch.bfloat16, dev)
    if fp8:
        _need(scales, "scales", torch.float32, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev)
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    M, K = x.shape
    N = w.shape[0]
    if N % 16:
        raise ValueError("SwiGLU needs N % 16 == 0")
    out = _out(out, out_f32, M, N // 2, dev)
    dt = FP8_B128 if fp8 else BF16
    with torch.cuda.device(dev):
        ws = _workspace(workspace, workspace_bytes(M, N, K, dt), dev)
        _check(load().dl_linear_swiglu(dt, _ptr(x), _ptr(w), _ptr(scales), _ptr(bias), _ptr(out),
                                       _ptr(out_f32), M, N, K, ws.ptr, ws.nbytes, _stream(stream, dev)))
    return out


def linear_argmax(x, w, scales=None, bias=None, *, out_idx=None, out_max=None, out=None,
                  out_f32=None, workspace: Workspace | None = None, stream=None):
    """idx[M] (int32) = argmax over n of x . w^T (+ bias), lowest index among
    ties, decided on the fp32 values (NaN largest).  out_max (fp32 [M]) gets the
    largest value; out / out_f32 get the logits only if given."""
    if isinstance(w, torch.Tensor) and w.dtype == torch.float8_e4m3fn:
        w = w.view(torch.uint8)
    _need(x, "x", torch.bfloat16)
    dev = x.device
    fp8 = scales is not None
    _need(w, "w", torch.uint8 if fp8 else torch.bfloat16, dev)
    if fp8:
        _need(scales, "scales", torch.float32, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev)
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    M, K = x.shape
    N = w.shape[0]
    if out_idx is None:
        out_idx = torch.empty(M, dtype=torch.int32, device=dev)
    _need(out_idx, "out_idx", torch.int32, dev)
    if out_max is not None:
        _need(out_max, "out_max", torch.float32, dev)
    if out is not None:
        _need(out, "out", torch.bfloat16, dev)
    if out_f32 is not None:
        _need(out_f32, "out_f32", torch.float32, dev)
    dt = FP8_B128 if fp8 else BF16
    with torch.cuda.device(dev):
        ws = _workspace(workspace, workspace_bytes(M, N, K, dt), dev)
        _check(load().dl_linear_argmax(dt, _ptr(x), _ptr(w), _ptr(scales), _ptr(bias), _ptr(out_idx),
                                       _ptr(out_max), _ptr(out), _ptr(out_f32), M, N, K, ws.ptr,
                                       ws.nbytes, _stream(stream, dev)))
    return out_idx


def interleave_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """[I, K] gate and up matrices (any dtype) -> the [2I, K] row order of
    linear_swiglu: rows 16b..16b+7 = gate rows 8b..8b+7, rows 16b+8..16b+15 =
    the matching up rows.  I % 8 == 0.  A one-time layout step for weights
    (plain tensor indexing, not part of the decode path)."""
    if gate.shape != up.shape or gate.shape[0] % 8:
        raise ValueError("gate and up must have the same [I, K] shape, I % 8 == 0")
    I, K = gate.shape
    return torch.stack([gate.reshape(I // 8, 8, K), up.reshape(I // 8, 8, K)], dim=1).reshape(2 * I, K)


STATIC_SCRATCH_BYTES = 16 << 20   # DL_STATIC_SCRATCH_BYTES of include/dl_linear.h
WORKSPACE_ZERO_BYTES = 256 + 16384 * 4   # DL_WORKSPACE_ZERO_BYTES: zero before the first call


def linear_bf16_static_scratch(x, w, bias=None, *, out, out_f32=None, stream=None):
    """linear_bf16 through dl_linear_bf16_static_scratch: no workspace argument;
    the library's static device scratch (STATIC_SCRATCH_BYTES per device) holds
    the split-K state and nothing is allocated on the call path, so `out` (and
    `out_f32`, if wanted) must be passed in.  Calls that may overlap on the GPU
    share that scratch and race; calls ordered on one stream do not."""
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    _need(x, "x", torch.bfloat16)
    dev = x.device
    _need(w, "w", torch.bfloat16, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev)
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    M, K = x.shape
    N = w.shape[0]
    if bias is not None and bias.numel() != N:
        raise ValueError("bias must be [N]")
    out = _out(out, out_f32, M, N, dev)
    lib = load()
    fn = lib.dl_linear_bf16_static_scratch
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
    fn.restype = i
    with torch.cuda.device(dev):
        _check(fn(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), _ptr(out_f32), M, N, K,
                  _stream(stream, dev)))
    return out


def linear_fp8_block128(x, wq, scales, bias=None, *, out=None, out_f32=None,
                        workspace: Workspace | None = None, stream=None):
    """out[M, N] (bf16) = x . (e4m3(wq) * scales[n/128, k/128])^T (+ bias).

    wq: uint8 e4m3 codes [N, K] (a torch.float8_e4m3fn tensor is accepted and
    viewed as bytes); scales: fp32 [ceil(N/128), K/128].
    """
    if isinstance(wq, torch.Tensor) and wq.dtype == torch.float8_e4m3fn:
        wq = wq.view(torch.uint8)
    _need(x, "x", torch.bfloat16)
    dev = x.device
    _need(wq, "wq", torch.uint8, dev)
    _need(scales, "scales", torch.float32, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev)
    if x.dim() != 2 or wq.dim() != 2 or x.shape[1] != wq.shape[1]:
        raise ValueError("x must be [M, K] and wq [N, K]")
    M, K = x.shape
    N = wq.shape[0]
    if scales.numel() != ((N + 127) // 128) * ((K + 127) // 128):
        raise ValueError("scales must be [ceil(N/128), ceil(K/128)]")
    if bias is not None and bias.numel() != N:
        raise ValueError("bias must be [N]")
    out = _out(out, out_f32, M, N, dev)
    with torch.cuda.device(dev):
        need = workspace_bytes(M, N, K, FP8_B128)
        ws = _workspace(workspace, need, dev)
        _check(load().dl_linear_fp8_block128(_ptr(x), _ptr(wq), _ptr(scales), _ptr(bias),
                                             _ptr(out), _ptr(out_f32), M, N, K, ws.ptr,
                                             ws.nbytes, _stream(stream, dev)))
    return out


@dataclass
class Layer:
    """One entry of a decode weight stream (all tensors on one CUDA device)."""

    dtype: int
    x: torch.Tensor
    w: torch.Tensor
    y: torch.Tensor
    scales: torch.Tensor | None = None
    bias: torch.Tensor | None = None
    act: int = 0          # 1: SwiGLU epilogue (see linear_swiglu): y is [M, N/2];
                          # 2: argmax (see linear_argmax): y is int32 [M], no logits

    def shape(self):
        return (self.x.shape[0], self.w.shape[0], self.x.shape[1], self.dtype)


def _layer_struct(L: Layer) -> _Layer:
    M, N, K, dt = L.shape()
    w = L.w.view(torch.uint8) if L.w.dtype == torch.float8_e4m3fn else L.w
    for t, n in ((L.x, "x"), (w, "w"), (L.y, "y")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"layer {n} must be a contiguous CUDA tensor")
    return _Layer(dt, M, N, K, L.x.data_ptr(), w.data_ptr(),
                  None if L.scales is None else L.scales.data_ptr(),
                  None if L.bias is None else L.bias.data_ptr(), L.y.data_ptr(), int(L.act))


def decode_stream(layers, workspace: Workspace, *, use_graph: bool = False, stream=None):
    """Run the layers back to back on one stream (optionally as a cached CUDA graph)."""
    arr = (_Layer * max(1, len(layers)))(*[_layer_struct(L) for L in layers])
    dev = layers[0].x.device if layers else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(load().dl_decode_stream(arr, len(layers), workspace.ptr, workspace.nbytes,
                                       _stream(stream, dev), 1 if use_graph else 0))


def decode_stream_workspace_bytes(layers) -> int:
    """Workspace bytes for decode_stream over `layers` with the FP8 activation
    copies made without per-layer prep launches where possible: ahead for the
    layers whose x is ready at the start, by the layer before for a layer fed
    by a plain linear's whole y (see dl_linear.h)."""
    arr = (_Layer * max(1, len(layers)))(*[_layer_struct(L) for L in layers])
    dev = layers[0].x.device if layers else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        n = load().dl_decode_stream_workspace_bytes(arr, len(layers))
    if n == 0:
        raise ValueError("invalid layer list: " + load().dl_last_error().decode())
    return n


def decode_stream_launches(layers, workspace: Workspace) -> int:
    """Kernels one decode_stream call over `layers` enqueues with this workspace."""
    arr = (_Layer * max(1, len(layers)))(*[_layer_struct(L) for L in layers])
    dev = layers[0].x.device if layers else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        n = load().dl_decode_stream_launches(arr, len(layers), workspace.nbytes)
    if n < 0:
        raise ValueError("invalid layer list: " + load().dl_last_error().decode())
    return n


def graph_cache_clear():
    load().dl_graph_cache_clear()


def graph_cache_size() -> int:
    """Graphs currently cached by decode_stream(use_graph=True)."""
    return int(load().dl_graph_cache_size())


def set_wait_test(wait_limit_ns: int = 0, withhold_stage: int = 0):
    """Test hooks of the bounded device waits (see dl_set_wait_test): the wait
    limit of later launches and a stage CTA 0 withholds; (0, 0) turns them off."""
    _check(load().dl_set_wait_test(int(wait_limit_ns), int(withhold_stage)))


def set_override(kernel: int = 0, ctas_per_sm: int = 0, max_ctas: int = 0):
    """Force a kernel family / grid shape (0 = automatic).  Process-wide."""
    _check(load().dl_set_override(kernel, ctas_per_sm, max_ctas))


def device_status() -> int:
    """Synchronise, read and clear the device error word; returns it (0 = no error)."""
    flags = ctypes.c_uint(0)
    st = load().dl_device_status(ctypes.byref(flags))
    if st != 0 and st != 6:
        _check(st)
    return int(flags.value)
