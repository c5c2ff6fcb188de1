"""GB300-native 4-bit mixture-of-experts FFN layer.

Python binding of libmoe.so: every entry point of include/moe.h under the same
name, doing argument marshalling only. All of the layer's work runs in the
library's CUDA kernels; torch is used for device memory and streams. There is
no fallback: if the library is missing, calls raise.

The layer follows "Optimizing on-device inference for Apple Silicon"
(Perplexity, 2026): 4-bit groupwise-affine experts (64 weights per bf16
scale/bias group), top-8-of-256 routing plus one shared expert, SwiGLU.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = 1
MOE_ERR_SHAPE = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_OPT_GEMV_MAX_ROWS = 1
MOE_OPT_FORCE_PATH = 2
MOE_OPT_KERNEL_TIMING = 3
MOE_OPT_GEMM_IMPL = 4
MOE_OPT_TEST_WAIT_CYCLES = 5
MOE_OPT_BLOCK_M = 6
MOE_OPT_DECODE_FUSED = 7
MOE_OPT_CHUNK_TOKENS = 8
MOE_OPT_HOST_SYNC_ROUTING = 9

PATH_AUTO, PATH_GEMV, PATH_GEMM = 0, 1, 2
GEMM_TENSOR_CORE, GEMM_CUDA_CORE, GEMM_TENSOR_CORE_SMEM = 0, 1, 2


class moe_qmatrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gate", moe_qmatrix), ("up", moe_qmatrix), ("down", moe_qmatrix),
                ("s_gate", moe_qmatrix), ("s_up", moe_qmatrix), ("s_down", moe_qmatrix)]


class moe_route_view(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("block_m", ctypes.c_int), ("max_blocks", ctypes.c_int),
                ("logits", ctypes.c_void_p), ("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("count", ctypes.c_void_p), ("off", ctypes.c_void_p), ("perm", ctypes.c_void_p),
                ("inv", ctypes.c_void_p), ("blocks", ctypes.c_void_p), ("n_blocks", ctypes.c_void_p),
                ("h", ctypes.c_void_p), ("y_acc", ctypes.c_void_p)]


# name -> (restype, argtypes), mirroring include/moe.h
_VP, _CI, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_W = ctypes.POINTER(moe_weights)
SIGNATURES = {
    "moe_workspace_size": (_SZ, [_W, _CI]),
    "moe_layer_forward": (_CI, [_W, _VP, _CI, _VP, _VP, _SZ, _VP]),
    "moe_layer_forward_static": (_CI, [_W, _VP, _CI, _VP, _VP]),
    "moe_get_device_status_static": (_CI, [_VP]),
    "moe_host_staging_size": (_SZ, [_W, _CI]),
    "moe_layer_forward_host": (_CI, [_W, _VP, _CI, _VP, _VP, _SZ, _VP]),
    "moe_route": (_CI, [_W, _VP, _CI, _VP, _SZ, _VP, ctypes.POINTER(moe_route_view)]),
    "moe_workspace_view": (_CI, [_W, _CI, _VP, _SZ, ctypes.POINTER(moe_route_view)]),
    "moe_get_device_status": (_CI, [_VP, _VP]),
    "moe_set_option": (_CI, [_CI, _CI]),
    "moe_get_option": (_CI, [_CI]),
    "moe_kernel_times": (_CI, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                               ctypes.POINTER(ctypes.c_int), _CI, ctypes.POINTER(ctypes.c_int)]),
    "moe_debug_dequant": (_CI, [ctypes.POINTER(moe_qmatrix), _CI, _CI, _CI, _VP, _VP]),
    "moe_expanded_weights_bytes": (_SZ, [_W]),
    "moe_layer_forward_expanded": (_CI, [_W, _VP, _CI, _VP, _VP, _SZ, _VP, _SZ, _VP]),
    "moe_last_launch_count": (_CI, []),
    "moe_status_string": (ctypes.c_char_p, [_CI]),
}

_lib = None


def lib():
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built ({LIB_PATH}); run bit_moe_expert_routing_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {moe_status_string(status)} ({status})")


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, what)


# --- the C entry points, same names --------------------------------------------------------

def moe_workspace_size(w: moe_weights, T: int) -> int:
    return lib().moe_workspace_size(ctypes.byref(w), T)


def moe_host_staging_size(w: moe_weights, T: int) -> int:
    return lib().moe_host_staging_size(ctypes.byref(w), T)


def moe_layer_forward(w, x_ptr, T, y_ptr, ws_ptr, ws_bytes, stream) -> int:
    return lib().moe_layer_forward(ctypes.byref(w), x_ptr, T, y_ptr, ws_ptr, ws_bytes, stream)


def moe_layer_forward_static(w, x_ptr, T, y_ptr, stream) -> int:
    """The layer with the library's fixed device scratch array as its
    workspace, for callers that cannot allocate device memory (include/moe.h
    says which)."""
    return lib().moe_layer_forward_static(ctypes.byref(w), x_ptr, T, y_ptr, stream)


def moe_get_device_status_static(stream) -> int:
    return lib().moe_get_device_status_static(stream)


def moe_expanded_weights_bytes(w: moe_weights) -> int:
    return lib().moe_expanded_weights_bytes(ctypes.byref(w))


def moe_layer_forward_expanded(w, x_ptr, T, y_ptr, ws_ptr, ws_bytes, wbuf_ptr, wbuf_bytes, stream) -> int:
    """The unfused form: a separate pass expands the selected experts'
    weights to bf16 in wbuf, then the GEMMs read them."""
    return lib().moe_layer_forward_expanded(ctypes.byref(w), x_ptr, T, y_ptr, ws_ptr, ws_bytes, wbuf_ptr, wbuf_bytes,
                                            stream)


def moe_layer_forward_host(w, x_host_ptr, T, y_host_ptr, ws_ptr, ws_bytes, stream) -> int:
    return lib().moe_layer_forward_host(ctypes.byref(w), x_host_ptr, T, y_host_ptr, ws_ptr, ws_bytes, stream)


def moe_route(w, x_ptr, T, ws_ptr, ws_bytes, stream, view: moe_route_view | None = None) -> int:
    return lib().moe_route(ctypes.byref(w), x_ptr, T, ws_ptr, ws_bytes, stream,
                           ctypes.byref(view) if view is not None else None)


def moe_workspace_view(w, T, ws_ptr, ws_bytes, view: moe_route_view) -> int:
    return lib().moe_workspace_view(ctypes.byref(w), T, ws_ptr, ws_bytes, ctypes.byref(view))


def moe_get_device_status(ws_ptr, stream) -> int:
    return lib().moe_get_device_status(ws_ptr, stream)


def moe_set_option(option: int, value: int) -> int:
    return lib().moe_set_option(option, value)


def moe_get_option(option: int) -> int:
    return lib().moe_get_option(option)


def moe_kernel_times(max_entries: int = 32) -> dict[str, tuple[float, int]]:
    """{kernel name: (total ms, launches)} since the previous call."""
    names = (ctypes.c_char_p * max_entries)()
    ms = (ctypes.c_float * max_entries)()
    cnt = (ctypes.c_int * max_entries)()
    n = ctypes.c_int(0)
    _check(lib().moe_kernel_times(names, ms, cnt, max_entries, ctypes.byref(n)), "moe_kernel_times")
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(n.value)}


def moe_debug_dequant(m: moe_qmatrix, expert, rows, K, out_ptr, stream) -> int:
    return lib().moe_debug_dequant(ctypes.byref(m), expert, rows, K, out_ptr, stream)


def moe_last_launch_count() -> int:
    return lib().moe_last_launch_count()


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


# --- torch helpers (allocation and streams only) ----------------------------------------

def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class DeviceLayer:
    """A layer's packed weights resident in device memory (torch tensors) and
    the moe_weights struct that points at them. `layer` is anything with the
    fields of synth.Layer (numpy arrays; bf16 as uint16 bit patterns)."""

    def __init__(self, layer, device="cuda"):
        import numpy as np
        import torch

        self.D, self.E, self.k, self.I = layer.D, layer.E, layer.k, layer.I
        self._t = []

        def up(arr, dtype):
            a = np.ascontiguousarray(arr)
            t = torch.from_numpy(a.view({np.uint32: np.int32, np.uint16: np.int16}.get(a.dtype.type, a.dtype)))
            t = t.to(device)
            self._t.append(t)
            return t

        def qm(m):
            c, s, b = up(m.codes, None), up(m.scales, None), up(m.biases, None)
            return moe_qmatrix(c.data_ptr(), s.data_ptr(), b.data_ptr())

        self.router_w = up(layer.router_w.astype(np.float32), None)
        self.router_bias = None if layer.router_bias is None else up(layer.router_bias.astype(np.float32), None)
        self.w = moe_weights(layer.D, layer.E, layer.k, layer.I, self.router_w.data_ptr(),
                             None if self.router_bias is None else self.router_bias.data_ptr(),
                             qm(layer.gate), qm(layer.up), qm(layer.down),
                             qm(layer.s_gate), qm(layer.s_up), qm(layer.s_down))

    def workspace_bytes(self, T: int, host_staging: bool = False) -> int:
        """Device bytes of the workspace for T tokens (one pass of at most the chunk size)."""
        n = moe_workspace_size(self.w, T)
        if n == 0:
            raise MoEError(MOE_ERR_ARG, "moe_workspace_size")
        return n + (moe_host_staging_size(self.w, T) if host_staging else 0)

    def workspace(self, T: int, host_staging: bool = False):
        import torch
        return torch.empty(self.workspace_bytes(T, host_staging), dtype=torch.uint8, device=self._t[0].device)

    def forward(self, x, y=None, workspace=None, stream=None):
        """x: bf16 [T, D] on the device. Returns y: bf16 [T, D]."""
        import torch
        T = x.shape[0]
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.shape[1] == self.D
        if y is None:
            y = torch.empty_like(x)
        if workspace is None:
            workspace = self.workspace(T)
        _check(moe_layer_forward(self.w, x.data_ptr(), T, y.data_ptr(), workspace.data_ptr(),
                                 workspace.numel(), _stream_ptr(stream)), "moe_layer_forward")
        return y

    def route(self, x, workspace, stream=None) -> moe_route_view:
        v = moe_route_view()
        _check(moe_route(self.w, x.data_ptr(), x.shape[0], workspace.data_ptr(), workspace.numel(),
                         _stream_ptr(stream), v), "moe_route")
        return v

    def view(self, T, workspace) -> moe_route_view:
        v = moe_route_view()
        _check(moe_workspace_view(self.w, T, workspace.data_ptr(), workspace.numel(), v), "moe_workspace_view")
        return v


def ws_tensor(workspace, ptr: int, shape, dtype):
    """A torch view of the workspace array at device pointer `ptr` (from a moe_route_view)."""
    import numpy as np
    import torch
    itemsize = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape))
    off = int(ptr) - workspace.data_ptr()
    assert 0 <= off and off + n * itemsize <= workspace.numel() and off % itemsize == 0
    return workspace[off:off + n * itemsize].view(dtype).reshape(shape)
