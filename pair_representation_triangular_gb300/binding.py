"""Python binding of libtriattn (include/tri_attn.h): argument marshalling only.

Every function has the name and argument order of its C entry point; tensors
are passed as device (or host) pointers taken from torch tensors, and the
stream is a ``torch.cuda.Stream`` (or None for the current stream). No step of
the computation runs here. If the library is missing or cannot be loaded, the
first call raises ``RuntimeError`` (``OSError`` from ctypes for a library that
does not load): there is no fallback path. Calls that the library refuses raise
``TriAttnError`` with its status code.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

TRI_ATTN_F32 = 0
TRI_ATTN_BF16 = 1
TRI_ATTN_MASK_ROW_KEY = 0
TRI_ATTN_MASK_QUERY_KEY = 1
TRI_ATTN_STARTING_NODE = 0
TRI_ATTN_ENDING_NODE = 2        # OR-ed into the mode: attention along columns
TRI_ATTN_PATH_SIMT = 0
TRI_ATTN_PATH_TENSOR_CORE = 1

TRI_ATTN_OK = 0
TRI_ATTN_ERR_INVALID_ARG = 1
TRI_ATTN_ERR_UNSUPPORTED = 2
TRI_ATTN_ERR_CUDA = 3
TRI_ATTN_ERR_OOM = 4
TRI_ATTN_ERR_DEVICE_TIMEOUT = 5
TRI_ATTN_ERR_DEVICE_CHECK = 6

PARAM_ORDER = ("gamma", "beta", "Wq", "Wk", "Wv", "Wg", "bg", "Wb", "Wo", "bo")
_DTYPES = {TRI_ATTN_F32: torch.float32, TRI_ATTN_BF16: torch.bfloat16}

_lib = None


class TriAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tri_attn_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def exported_names(header: str | None = None) -> list[str]:
    """Entry points declared in include/tri_attn.h."""
    header = header or os.path.join(os.path.dirname(_build.PKG), "include", "tri_attn.h")
    with open(header) as f:
        return sorted(set(re.findall(r"\b(tri_attn_[a-z_]+)\s*\(", f.read())))


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libtriattn.so (built in-tree by ``build.build()``) and declare its ABI."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libtriattn is not built ({path} missing); run build.build() first")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    lib.tri_attn_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32] + [vp] * 11
    lib.tri_attn_forward.argtypes = [vp, vp, vp, vp, vp]
    lib.tri_attn_forward_host.argtypes = [vp, vp, vp, vp, vp]
    lib.tri_attn_sync_check.argtypes = [vp, vp]
    lib.tri_attn_destroy.argtypes = [vp]
    lib.tri_attn_status_string.argtypes = [i32]
    lib.tri_attn_status_string.restype = ctypes.c_char_p
    lib.tri_attn_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.tri_attn_set_wait_limit.argtypes = [vp, i64]
    lib.tri_attn_enable_kernel_timing.argtypes = [vp, i32]
    lib.tri_attn_debug_tensor.argtypes = [vp, ctypes.c_char_p, ctypes.POINTER(i64)]
    lib.tri_attn_kernel_path.argtypes = [vp]
    lib.tri_attn_kernel_path.restype = i32
    lib.tri_attn_debug_tensor.restype = vp
    lib.tri_attn_forward_noalloc.argtypes = [i32, i32, i32, i32, i32] + [vp] * 14
    lib.tri_attn_forward_noalloc.restype = i32
    lib.tri_attn_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float),
                                          ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i32)]
    for name in ("tri_attn_create", "tri_attn_forward", "tri_attn_forward_host",
                 "tri_attn_sync_check", "tri_attn_destroy", "tri_attn_workspace_bytes",
                 "tri_attn_set_wait_limit", "tri_attn_enable_kernel_timing",
                 "tri_attn_kernel_times"):
        getattr(lib, name).restype = i32
    if path == library_path():
        _lib = lib
    return lib


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> int:
    if status != TRI_ATTN_OK:
        raise TriAttnError(status, where)
    return status


def tri_attn_status_string(status: int) -> str:
    return load_library().tri_attn_status_string(status).decode()


def tri_attn_workspace_bytes(B, N, D, h, dtype) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().tri_attn_workspace_bytes(B, N, D, h, dtype, ctypes.byref(n)),
           "tri_attn_workspace_bytes")
    return n.value


def tri_attn_create(B, N, D, h, dtype, mode, params: dict, stream=None) -> ctypes.c_void_p:
    """``params``: device tensors gamma, beta, Wq, Wk, Wv, Wg, bg, Wb, Wo, bo of the
    handle's dtype (nn.Linear layout). Returns the opaque handle."""
    want = _DTYPES.get(dtype)
    ptrs = []
    for name in PARAM_ORDER:
        t = params[name]
        if want is not None and (t.dtype != want or not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous {want} CUDA tensor")
        ptrs.append(t.data_ptr())
    handle = ctypes.c_void_p()
    _check(load_library().tri_attn_create(ctypes.byref(handle), B, N, D, h, dtype, mode,
                                          *ptrs, _stream_ptr(stream)), "tri_attn_create")
    return handle


def tri_attn_forward(handle, stream, pair_repr: torch.Tensor, pair_mask: torch.Tensor,
                     out: torch.Tensor) -> None:
    _check(load_library().tri_attn_forward(handle, _stream_ptr(stream), pair_repr.data_ptr(),
                                           pair_mask.data_ptr(), out.data_ptr()),
           "tri_attn_forward")


def tri_attn_forward_host(handle, stream, pair_repr_host: torch.Tensor,
                          pair_mask_host: torch.Tensor, out_host: torch.Tensor) -> None:
    _check(load_library().tri_attn_forward_host(handle, _stream_ptr(stream),
                                                pair_repr_host.data_ptr(),
                                                pair_mask_host.data_ptr(), out_host.data_ptr()),
           "tri_attn_forward_host")


def tri_attn_sync_check(handle, stream=None) -> int:
    """Returns the status (does not raise), so callers can test device errors."""
    return load_library().tri_attn_sync_check(handle, _stream_ptr(stream))


def tri_attn_destroy(handle) -> None:
    _check(load_library().tri_attn_destroy(handle), "tri_attn_destroy")


def tri_attn_set_wait_limit(handle, spins: int) -> None:
    _check(load_library().tri_attn_set_wait_limit(handle, spins), "tri_attn_set_wait_limit")


def tri_attn_enable_kernel_timing(handle, enable: bool) -> None:
    _check(load_library().tri_attn_enable_kernel_timing(handle, int(enable)),
           "tri_attn_enable_kernel_timing")


def tri_attn_kernel_times(handle) -> list:
    """[(kernel name, ms), ...] for the most recent forward of the handle."""
    cap = 8
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = ctypes.c_int(cap)
    _check(load_library().tri_attn_kernel_times(handle, ms, names, ctypes.byref(n)),
           "tri_attn_kernel_times")
    return [(names[i].decode(), float(ms[i])) for i in range(n.value)]


def tri_attn_forward_noalloc(B, N, D, h, mode, params: dict, stream,
                             pair_repr: torch.Tensor, pair_mask: torch.Tensor,
                             out: torch.Tensor) -> None:
    """fp32 forward that allocates nothing on the device (see include/tri_attn.h):
    for callers that may not allocate; intermediates use the library's fixed
    16 MiB scratch, so problems beyond it raise TriAttnError (UNSUPPORTED)."""
    ptrs = [params[name].data_ptr() for name in PARAM_ORDER]
    _check(load_library().tri_attn_forward_noalloc(B, N, D, h, mode, *ptrs,
                                                   _stream_ptr(stream), pair_repr.data_ptr(),
                                                   pair_mask.data_ptr(), out.data_ptr()),
           "tri_attn_forward_noalloc")


def tri_attn_kernel_path(handle) -> int:
    return load_library().tri_attn_kernel_path(handle)


def tri_attn_debug_tensor(handle, name: str):
    """(device pointer, innermost row stride in elements) of an intermediate;
    (None, 0) for an unknown name."""
    ld = ctypes.c_longlong(0)
    ptr = load_library().tri_attn_debug_tensor(handle, name.encode(), ctypes.byref(ld))
    return ptr, ld.value


class _DeviceView:
    """A __cuda_array_interface__ view of library-owned device memory."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": shape,
                                         "typestr": typestr, "version": 2}


class TriangularAttention:
    """Owns one handle: ``TriangularAttention(B, N, D, h, dtype, mode, params)``,
    then ``forward(pair_repr, pair_mask)`` returns a new output tensor."""

    def __init__(self, B, N, D, h, dtype, mode, params, stream=None):
        self.B, self.N, self.D, self.h = B, N, D, h
        self.dtype, self.mode = dtype, mode
        self.torch_dtype = _DTYPES[dtype]
        self.handle = tri_attn_create(B, N, D, h, dtype, mode, params, stream)

    def _check_inputs(self, x, mask, out, device_side=True):
        shape = (self.B, self.N, self.N, self.D)
        if tuple(x.shape) != shape or x.dtype != self.torch_dtype or not x.is_contiguous():
            raise ValueError(f"pair_repr must be a contiguous {self.torch_dtype} tensor {shape}")
        if tuple(mask.shape) != shape[:3] or mask.dtype != torch.int32 or not mask.is_contiguous():
            raise ValueError(f"pair_mask must be a contiguous int32 tensor {shape[:3]}")
        if tuple(out.shape) != shape or out.dtype != self.torch_dtype or not out.is_contiguous():
            raise ValueError("out must match pair_repr")
        for t in (x, mask, out):
            if t.is_cuda != device_side:
                raise ValueError("tensors must all be on the " +
                                 ("device" if device_side else "host"))

    def forward(self, pair_repr, pair_mask, out=None, stream=None):
        if out is None:
            out = torch.empty_like(pair_repr)
        self._check_inputs(pair_repr, pair_mask, out, True)
        tri_attn_forward(self.handle, stream, pair_repr, pair_mask, out)
        return out

    __call__ = forward

    def forward_host(self, pair_repr, pair_mask, out, stream=None):
        self._check_inputs(pair_repr, pair_mask, out, False)
        tri_attn_forward_host(self.handle, stream, pair_repr, pair_mask, out)
        return out

    def intermediate(self, name: str) -> torch.Tensor:
        """Copy of an intermediate of the most recent forward (see
        tri_attn_debug_tensor): q, k, v, g, o as (B, N, N, D), on the
        tensor-core path of bf16 handles bf16 (v: fp16) with their raw bits
        reinterpreted, and fp32 on the SIMT path of fp32 handles;
        bias as (B, h, N, N) fp32. On the tensor-core path the plane the
        attention reads is stored in fp16 as log2(e) * (bias minus the largest
        kept entry of its (head, query) row), with -inf where the query-key
        mask drops a key; it is returned as stored, widened to fp32."""
        ptr, ld = tri_attn_debug_tensor(self.handle, name)
        if not ptr:
            raise KeyError(name)
        torch.cuda.synchronize()
        simt = tri_attn_kernel_path(self.handle) == TRI_ATTN_PATH_SIMT
        if name == "bias":
            ts = "<f4" if simt else "<f2"
            view = _DeviceView(ptr, (self.B, self.h, self.N, ld), ts)
            return torch.as_tensor(view, device="cuda")[..., :self.N].float()
        shape = (self.B, self.N, self.N, self.D)
        if simt:
            return torch.as_tensor(_DeviceView(ptr, shape, "<f4"), device="cuda").clone()
        raw = torch.as_tensor(_DeviceView(ptr, shape, "<i2"), device="cuda").clone()
        # v is fp16 on the tensor-core path (times a power of 2 that is 1 unless
        # the weights could drive |v| past 2^15), the others bf16.
        return raw.view(torch.float16 if name == "v" else torch.bfloat16)

    def sync_check(self, stream=None) -> int:
        return tri_attn_sync_check(self.handle, stream)

    def close(self):
        if self.handle is not None:
            tri_attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
