"""Python binding of libint8conv.so: INT8 2-D convolution forward propagation
with int32 results (or int8 after a rounding right shift) on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/int8conv.h``.  PyTorch provides
device memory and streams.  There is no CPU fallback: if the library is
missing or the device is not sm_103, calls raise.

The operation follows conv_fprop in the cuDNN documentation page
"Convolutions" (section "Convolution Fprop", "Python API" argument list):
image, weight, pre_padding, post_padding, stride, dilation, convolution_mode,
compute_data_type (INT32 only); ``padding`` is the symmetric overload.
Tensors are described by logical dims [N,C,H,W] / [K,C,R,S] plus per-dim
element strides, exactly what a torch tensor's ``size()``/``stride()`` give
(a channels_last tensor is NHWC in memory).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libint8conv.so")
_lib = None

CONV_INT8, CONV_INT32 = 1, 2
CROSS_CORRELATION, CONVOLUTION = 0, 1
ALGO_AUTO, ALGO_IMPLICIT_GEMM, ALGO_DIRECT_DP4A, ALGO_DIRECT_GENERIC = 0, 1, 2, 3
ALGO_IMPLICIT_GEMM_GLOBAL_LOADS = 4
EPILOGUE_BIAS, EPILOGUE_RELU, EPILOGUE_INT8_OUT = 1, 2, 4
ALGO_NAMES = {ALGO_IMPLICIT_GEMM: "implicit_gemm", ALGO_DIRECT_DP4A: "direct_dp4a",
              ALGO_DIRECT_GENERIC: "direct_generic",
              ALGO_IMPLICIT_GEMM_GLOBAL_LOADS: "implicit_gemm_global_loads"}

STATUS = {
    0: "CONV_OK", 1: "CONV_ERR_NULL_PTR", 2: "CONV_ERR_RANK", 3: "CONV_ERR_DTYPE",
    4: "CONV_ERR_SHAPE_MISMATCH", 5: "CONV_ERR_BAD_STRIDES", 6: "CONV_ERR_BUFFER_TOO_SMALL",
    7: "CONV_ERR_BAD_PARAM", 8: "CONV_ERR_OVERFLOW_RISK", 9: "CONV_ERR_UNSUPPORTED_COMPUTE",
    10: "CONV_ERR_ALIGNMENT", 11: "CONV_ERR_CUDA", 12: "CONV_ERR_DEVICE_TIMEOUT",
    13: "CONV_ERR_WORKSPACE", 14: "CONV_ERR_UNSUPPORTED_DEVICE", 15: "CONV_ERR_OVERLAP",
    16: "CONV_ERR_TOO_LARGE", 17: "CONV_ERR_STATIC_WORKSPACE_LIMIT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

EXPORTED_SYMBOLS = (
    "conv_params_init", "conv_params_set_symmetric_padding", "conv_tensor_desc_packed",
    "conv_fprop_output_dims", "conv_fprop_validate", "conv_fprop_plan", "conv_fprop_workspace_size",
    "conv_fprop_kernel_count", "conv_fprop_tile_shape",
    "conv_fprop", "conv_fprop_pack_filter", "conv_fprop_prepacked", "conv_fprop_static_workspace",
    "conv_fprop_host_buffer_size", "conv_fprop_host", "conv_device_status",
    "conv_selftest_wait_timeout", "conv_status_string", "conv_library_version",
    "conv_dgrad_workspace_size", "conv_dgrad", "conv_wgrad_workspace_size", "conv_wgrad",
    "conv_measure_peak_rates", "conv_shutdown", "conv_plan_cache_stats",
)


class PeakRates(ctypes.Structure):
    _fields_ = [("tcgen05_f16_tflops", ctypes.c_double), ("mma_sync_s8_tops", ctypes.c_double),
                ("mma_sync_f16_tflops", ctypes.c_double), ("dp4a_tops", ctypes.c_double),
                ("hbm_copy_gbs", ctypes.c_double), ("sm_mhz", ctypes.c_double)]


class ConvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {self.name}" if what else self.name)


class TensorDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("dims", ctypes.c_int64 * 4), ("strides", ctypes.c_int64 * 4),
                ("capacity_bytes", ctypes.c_uint64)]

    @classmethod
    def make(cls, dtype: int, dims: Sequence[int], strides: Sequence[int], capacity_bytes: int) -> "TensorDesc":
        d = cls()
        d.dtype, d.rank = dtype, 4
        for i in range(4):
            d.dims[i], d.strides[i] = int(dims[i]), int(strides[i])
        d.capacity_bytes = int(capacity_bytes)
        return d

    @classmethod
    def packed(cls, dtype: int, dims: Sequence[int], layout: str) -> "TensorDesc":
        d = cls()
        dd = (ctypes.c_int64 * 4)(*[int(v) for v in dims])
        _check(lib().conv_tensor_desc_packed(ctypes.byref(d), dtype, dd, layout.encode()), "packed descriptor")
        return d

    @classmethod
    def from_tensor(cls, t) -> "TensorDesc":
        import torch
        dtype = {torch.int8: CONV_INT8, torch.int32: CONV_INT32}.get(t.dtype, 0)
        cap = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
        return cls.make(dtype, tuple(t.shape), tuple(t.stride()), cap)

    @property
    def dims_t(self) -> Tuple[int, ...]:
        return tuple(self.dims)

    @property
    def strides_t(self) -> Tuple[int, ...]:
        return tuple(self.strides)


class Params(ctypes.Structure):
    _fields_ = [("pre_padding", ctypes.c_int64 * 2), ("post_padding", ctypes.c_int64 * 2),
                ("stride", ctypes.c_int64 * 2), ("dilation", ctypes.c_int64 * 2),
                ("mode", ctypes.c_int32), ("compute_dtype", ctypes.c_int32),
                ("epilogue", ctypes.c_uint32), ("algo", ctypes.c_int32),
                ("out_shift", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    @classmethod
    def make(cls, pre_padding=(0, 0), post_padding=(0, 0), stride=(1, 1), dilation=(1, 1),
             mode: int = CROSS_CORRELATION, bias: bool = False, relu: bool = False,
             algo: int = ALGO_AUTO, padding: Optional[Sequence[int]] = None,
             compute_dtype: int = CONV_INT32, out_shift: Optional[int] = None) -> "Params":
        """out_shift=None: int32 output; an integer s in 0..31: int8 output
        round(v / 2^s) (halves toward +inf) saturated to [-128, 127]."""
        p = cls()
        lib().conv_params_init(ctypes.byref(p))
        if padding is not None:
            pad = (ctypes.c_int64 * 2)(int(padding[0]), int(padding[1]))
            lib().conv_params_set_symmetric_padding(ctypes.byref(p), pad)
        else:
            for i in range(2):
                p.pre_padding[i], p.post_padding[i] = int(pre_padding[i]), int(post_padding[i])
        for i in range(2):
            p.stride[i], p.dilation[i] = int(stride[i]), int(dilation[i])
        p.mode = int(mode)
        p.compute_dtype = int(compute_dtype)
        p.epilogue = (EPILOGUE_BIAS if bias else 0) | (EPILOGUE_RELU if relu else 0)
        if out_shift is not None:
            p.epilogue |= EPILOGUE_INT8_OUT
            p.out_shift = int(out_shift)
        p.algo = int(algo)
        return p


def lib():
    """The loaded libint8conv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libint8conv.so is not built ({_LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(_LIB_PATH)
        P, D = ctypes.POINTER(Params), ctypes.POINTER(TensorDesc)
        i64p = ctypes.POINTER(ctypes.c_int64)
        L.conv_params_init.argtypes = [P]
        L.conv_params_init.restype = None
        L.conv_params_set_symmetric_padding.argtypes = [P, i64p]
        L.conv_params_set_symmetric_padding.restype = None
        L.conv_tensor_desc_packed.argtypes = [D, ctypes.c_int32, i64p, ctypes.c_char_p]
        L.conv_fprop_output_dims.argtypes = [D, D, P, i64p]
        L.conv_fprop_validate.argtypes = [D, D, D, P, ctypes.c_int64]
        L.conv_fprop_plan.argtypes = [D, D, D, P, ctypes.POINTER(ctypes.c_int32)]
        L.conv_fprop_workspace_size.argtypes = [D, D, D, P, ctypes.POINTER(ctypes.c_size_t)]
        L.conv_fprop_kernel_count.argtypes = [D, D, D, P, ctypes.POINTER(ctypes.c_int32)]
        L.conv_fprop_tile_shape.argtypes = [D, D, D, P, i64p]
        L.conv_fprop.argtypes = [D, ctypes.c_void_p, D, ctypes.c_void_p, D, ctypes.c_void_p, ctypes.c_void_p,
                                 P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.conv_fprop_pack_filter.argtypes = [D, D, ctypes.c_void_p, D, P, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p]
        L.conv_fprop_prepacked.argtypes = list(L.conv_fprop.argtypes)
        L.conv_fprop_static_workspace.argtypes = [D, ctypes.c_void_p, D, ctypes.c_void_p, D, ctypes.c_void_p,
                                                  ctypes.c_void_p, P, ctypes.c_void_p]
        L.conv_fprop_host_buffer_size.argtypes = [D, D, D, P, ctypes.POINTER(ctypes.c_size_t)]
        L.conv_fprop_host_buffer_size.restype = ctypes.c_int
        L.conv_fprop_host.argtypes = list(L.conv_fprop.argtypes)
        L.conv_fprop_host.restype = ctypes.c_int
        for name in ("conv_dgrad_workspace_size", "conv_wgrad_workspace_size"):
            getattr(L, name).argtypes = [D, D, D, P, ctypes.POINTER(ctypes.c_size_t)]
            getattr(L, name).restype = ctypes.c_int
        for name in ("conv_dgrad", "conv_wgrad"):
            getattr(L, name).argtypes = [D, ctypes.c_void_p, D, ctypes.c_void_p, D, ctypes.c_void_p, P,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
            getattr(L, name).restype = ctypes.c_int
        L.conv_measure_peak_rates.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PeakRates),
                                              ctypes.c_void_p]
        L.conv_measure_peak_rates.restype = ctypes.c_int
        L.conv_shutdown.argtypes = []
        L.conv_shutdown.restype = None
        u64p = ctypes.POINTER(ctypes.c_uint64)
        L.conv_plan_cache_stats.argtypes = [u64p, u64p, u64p, u64p]
        L.conv_plan_cache_stats.restype = ctypes.c_int
        L.conv_device_status.argtypes = [ctypes.c_void_p]
        L.conv_selftest_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
        L.conv_status_string.argtypes = [ctypes.c_int]
        L.conv_status_string.restype = ctypes.c_char_p
        L.conv_library_version.restype = ctypes.c_int32
        for name in ("conv_tensor_desc_packed", "conv_fprop_output_dims", "conv_fprop_validate",
                     "conv_fprop_plan", "conv_fprop_workspace_size", "conv_fprop", "conv_fprop_pack_filter",
                     "conv_fprop_prepacked", "conv_fprop_static_workspace", "conv_device_status",
                     "conv_selftest_wait_timeout"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, what: str = "") -> None:
    if status != 0:
        raise ConvError(status, what)


def status_string(status: int) -> str:
    return lib().conv_status_string(int(status)).decode()


def output_dims(xd: TensorDesc, wd: TensorDesc, p: Params) -> Tuple[int, int, int, int]:
    out = (ctypes.c_int64 * 4)()
    _check(lib().conv_fprop_output_dims(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(p), out), "output dims")
    return tuple(out)


def validate(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params, bias_elems: int = 0) -> int:
    """Status code of the host-side validation (0 = valid)."""
    return int(lib().conv_fprop_validate(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd),
                                         ctypes.byref(p), int(bias_elems)))


def plan(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params) -> int:
    out = ctypes.c_int32()
    _check(lib().conv_fprop_plan(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p),
                                 ctypes.byref(out)), "plan")
    return int(out.value)


def workspace_size(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params) -> int:
    out = ctypes.c_size_t()
    _check(lib().conv_fprop_workspace_size(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd),
                                           ctypes.byref(p), ctypes.byref(out)), "workspace size")
    return int(out.value)


def kernel_count(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params) -> int:
    """Kernels conv_fprop launches for this call (see the header)."""
    out = ctypes.c_int32()
    _check(lib().conv_fprop_kernel_count(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p),
                                         ctypes.byref(out)), "kernel count")
    return int(out.value)


def tile_shape(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params) -> tuple:
    """(pixels per tile, channels per tile, tiles, work units) of the
    implicit-GEMM convolution for this call (see the header)."""
    out = (ctypes.c_int64 * 4)()
    _check(lib().conv_fprop_tile_shape(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p), out),
           "tile shape")
    return tuple(int(v) for v in out)


def conv_fprop_raw(xd: TensorDesc, x_ptr: int, wd: TensorDesc, w_ptr: int, yd: TensorDesc, y_ptr: int,
                   bias_ptr: int, p: Params, workspace_ptr: int, workspace_bytes: int, stream: int) -> int:
    """Direct call of the C entry point with device addresses; returns the status."""
    return int(lib().conv_fprop(ctypes.byref(xd), x_ptr, ctypes.byref(wd), w_ptr, ctypes.byref(yd), y_ptr,
                                bias_ptr or None, ctypes.byref(p), workspace_ptr or None, int(workspace_bytes),
                                stream or None))


def pack_filter_raw(xd: TensorDesc, wd: TensorDesc, w_ptr: int, yd: TensorDesc, p: Params,
                    workspace_ptr: int, workspace_bytes: int, stream: int) -> int:
    """First half of conv_fprop: repack the filter into the workspace."""
    return int(lib().conv_fprop_pack_filter(ctypes.byref(xd), ctypes.byref(wd), w_ptr, ctypes.byref(yd),
                                            ctypes.byref(p), workspace_ptr or None, int(workspace_bytes),
                                            stream or None))


def conv_fprop_prepacked_raw(xd: TensorDesc, x_ptr: int, wd: TensorDesc, w_ptr: int, yd: TensorDesc, y_ptr: int,
                             bias_ptr: int, p: Params, workspace_ptr: int, workspace_bytes: int, stream: int) -> int:
    """Second half of conv_fprop: run from a workspace filled by pack_filter_raw."""
    return int(lib().conv_fprop_prepacked(ctypes.byref(xd), x_ptr, ctypes.byref(wd), w_ptr, ctypes.byref(yd),
                                          y_ptr, bias_ptr or None, ctypes.byref(p), workspace_ptr or None,
                                          int(workspace_bytes), stream or None))


def conv_fprop_static_workspace_raw(xd: TensorDesc, x_ptr: int, wd: TensorDesc, w_ptr: int, yd: TensorDesc,
                                    y_ptr: int, bias_ptr: int, p: Params, stream: int) -> int:
    """conv_fprop with the library's own static scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    return int(lib().conv_fprop_static_workspace(ctypes.byref(xd), x_ptr, ctypes.byref(wd), w_ptr, ctypes.byref(yd),
                                                 y_ptr, bias_ptr or None, ctypes.byref(p), stream or None))


def host_buffer_size(xd: TensorDesc, wd: TensorDesc, yd: TensorDesc, p: Params) -> int:
    out = ctypes.c_size_t()
    _check(lib().conv_fprop_host_buffer_size(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p),
                                             ctypes.byref(out)), "host buffer size")
    return int(out.value)


def conv_fprop_host_raw(xd: TensorDesc, x_host: int, wd: TensorDesc, w_host: int, yd: TensorDesc, y_host: int,
                        bias_host: int, p: Params, device_buffer: int, device_buffer_bytes: int, stream: int) -> int:
    """conv_fprop on host buffers (copies and compute pipelined by the library)."""
    return int(lib().conv_fprop_host(ctypes.byref(xd), x_host, ctypes.byref(wd), w_host, ctypes.byref(yd), y_host,
                                     bias_host or None, ctypes.byref(p), device_buffer or None,
                                     int(device_buffer_bytes), stream or None))


def conv_fprop_from_host(x, w, bias=None, *, out, device_buffer=None, stream=None, pre_padding=(0, 0),
                         post_padding=(0, 0), padding=None, stride=(1, 1), dilation=(1, 1),
                         mode: int = CROSS_CORRELATION, relu: bool = False, algo: int = ALGO_AUTO,
                         out_shift: Optional[int] = None):
    """conv_fprop on CPU tensors (pin them for overlapped copies); ``out`` is
    a CPU int32 tensor (int8 when ``out_shift`` is given).  Asynchronous on
    ``stream``; returns ``out``."""
    import torch
    p = Params.make(pre_padding, post_padding, stride, dilation, mode, bias is not None, relu, algo, padding,
                    out_shift=out_shift)
    xd, wd, yd = TensorDesc.from_tensor(x), TensorDesc.from_tensor(w), TensorDesc.from_tensor(out)
    need = host_buffer_size(xd, wd, yd, p)
    if device_buffer is None or device_buffer.numel() * device_buffer.element_size() < need:
        device_buffer = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream()
    st = conv_fprop_host_raw(xd, x.data_ptr(), wd, w.data_ptr(), yd, out.data_ptr(),
                             bias.data_ptr() if bias is not None else 0, p, device_buffer.data_ptr(),
                             device_buffer.numel() * device_buffer.element_size(), stream.cuda_stream)
    _check(st, "conv_fprop_host")
    return out


def measure_peak_rates(scratch_ptr: int, scratch_bytes: int, stream: int = 0) -> dict:
    """Measured rates of the int8-capable instruction routes and the copy
    bandwidth of the current device (see conv_measure_peak_rates)."""
    r = PeakRates()
    _check(lib().conv_measure_peak_rates(scratch_ptr or None, int(scratch_bytes), ctypes.byref(r), stream or None),
           "peak rates")
    return {name: float(getattr(r, name)) for name, _ in PeakRates._fields_}


def shutdown() -> None:
    """Empty the library's plan caches (conv_shutdown)."""
    lib().conv_shutdown()


def plan_cache_stats() -> dict:
    """Hit and miss counts of the plan and launch caches since load."""
    v = [ctypes.c_uint64() for _ in range(4)]
    _check(lib().conv_plan_cache_stats(*[ctypes.byref(x) for x in v]), "plan cache stats")
    return {"plan_hits": v[0].value, "plan_misses": v[1].value, "launch_hits": v[2].value,
            "launch_misses": v[3].value}


def device_status(stream: int = 0) -> int:
    return int(lib().conv_device_status(stream or None))


def selftest_wait_timeout(limit_us: int, stream: int = 0) -> int:
    return int(lib().conv_selftest_wait_timeout(int(limit_us), stream or None))


def conv_fprop(x, w, bias=None, *, pre_padding=(0, 0), post_padding=(0, 0), padding=None,
               stride=(1, 1), dilation=(1, 1), mode: int = CROSS_CORRELATION, relu: bool = False,
               algo: int = ALGO_AUTO, out=None, workspace=None, stream=None, out_shift: Optional[int] = None):
    """Y = conv_fprop(x, w) on the GPU.

    x: int8 CUDA tensor [N,C,H,W] with any strides; w: int8 [K,C,R,S]; bias:
    optional int32 [K]; out: optional int32 [N,K,P,Q] (any strides; default:
    the image's memory format), int8 when ``out_shift`` is given (the int32
    result after bias and ReLU, shifted right by out_shift with rounding and
    saturated).  Runs on ``stream`` (a torch.cuda.Stream; default the current
    stream).  Returns ``out``.
    """
    import torch
    if not (x.is_cuda and w.is_cuda):
        raise ValueError("x and w must be CUDA tensors")
    p = Params.make(pre_padding, post_padding, stride, dilation, mode, bias is not None, relu, algo, padding,
                    out_shift=out_shift)
    xd, wd = TensorDesc.from_tensor(x), TensorDesc.from_tensor(w)
    od = output_dims(xd, wd, p)
    if out is None:
        cl = x.dim() == 4 and x.is_contiguous(memory_format=torch.channels_last) and not x.is_contiguous()
        fmt = torch.channels_last if cl else torch.contiguous_format
        odt = torch.int32 if out_shift is None else torch.int8
        out = torch.empty(od, dtype=odt, device=x.device, memory_format=fmt)
    yd = TensorDesc.from_tensor(out)
    ws_bytes = workspace_size(xd, wd, yd, p)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    if bias is not None and (bias.dtype != torch.int32 or not bias.is_cuda or bias.numel() < od[1]
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous int32 CUDA tensor with K elements")
    st = conv_fprop_raw(xd, x.data_ptr(), wd, w.data_ptr(), yd, out.data_ptr(),
                        bias.data_ptr() if bias is not None else 0, p,
                        workspace.data_ptr() if ws_bytes else 0,
                        workspace.numel() * workspace.element_size() if ws_bytes else 0,
                        stream.cuda_stream)
    _check(st, "conv_fprop")
    return out


def dgrad_workspace_size(dyd: TensorDesc, wd: TensorDesc, dxd: TensorDesc, p: Params) -> int:
    out = ctypes.c_size_t()
    _check(lib().conv_dgrad_workspace_size(ctypes.byref(dyd), ctypes.byref(wd), ctypes.byref(dxd), ctypes.byref(p),
                                           ctypes.byref(out)), "dgrad workspace size")
    return int(out.value)


def wgrad_workspace_size(xd: TensorDesc, dyd: TensorDesc, dwd: TensorDesc, p: Params) -> int:
    out = ctypes.c_size_t()
    _check(lib().conv_wgrad_workspace_size(ctypes.byref(xd), ctypes.byref(dyd), ctypes.byref(dwd), ctypes.byref(p),
                                           ctypes.byref(out)), "wgrad workspace size")
    return int(out.value)


def _grad_params(pre_padding, post_padding, padding, stride, dilation, mode, algo):
    return Params.make(pre_padding, post_padding, stride, dilation, mode, False, False, algo, padding)


def conv_dgrad(dy, w, *, out, pre_padding=(0, 0), post_padding=(0, 0), padding=None, stride=(1, 1),
               dilation=(1, 1), mode: int = CROSS_CORRELATION, algo: int = ALGO_AUTO, workspace=None, stream=None):
    """Data gradient dX of conv_fprop: dy int8 CUDA tensor [N,K,P,Q] (the loss
    gradient), w int8 [K,C,R,S], out int32 [N,C,H,W] (any strides; H, W are
    the forward image size).  Parameters as for conv_fprop.  Returns ``out``."""
    import torch
    p = _grad_params(pre_padding, post_padding, padding, stride, dilation, mode, algo)
    dyd, wd, dxd = TensorDesc.from_tensor(dy), TensorDesc.from_tensor(w), TensorDesc.from_tensor(out)
    ws_bytes = dgrad_workspace_size(dyd, wd, dxd, p)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dy.device)
    if stream is None:
        stream = torch.cuda.current_stream(dy.device)
    st = lib().conv_dgrad(ctypes.byref(dyd), dy.data_ptr(), ctypes.byref(wd), w.data_ptr(), ctypes.byref(dxd),
                          out.data_ptr(), ctypes.byref(p), workspace.data_ptr() if ws_bytes else None,
                          ws_bytes if ws_bytes else 0, stream.cuda_stream or None)
    _check(st, "conv_dgrad")
    return out


def conv_wgrad(x, dy, *, out, pre_padding=(0, 0), post_padding=(0, 0), padding=None, stride=(1, 1),
               dilation=(1, 1), mode: int = CROSS_CORRELATION, algo: int = ALGO_AUTO, workspace=None, stream=None):
    """Weight gradient dW of conv_fprop: x int8 CUDA tensor [N,C,H,W], dy int8
    [N,K,P,Q] (the loss gradient), out int32 [K,C,R,S] (any strides; R, S are
    the forward filter size).  Parameters as for conv_fprop.  Returns ``out``."""
    import torch
    p = _grad_params(pre_padding, post_padding, padding, stride, dilation, mode, algo)
    xd, dyd, dwd = TensorDesc.from_tensor(x), TensorDesc.from_tensor(dy), TensorDesc.from_tensor(out)
    ws_bytes = wgrad_workspace_size(xd, dyd, dwd, p)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    st = lib().conv_wgrad(ctypes.byref(xd), x.data_ptr(), ctypes.byref(dyd), dy.data_ptr(), ctypes.byref(dwd),
                          out.data_ptr(), ctypes.byref(p), workspace.data_ptr() if ws_bytes else None,
                          ws_bytes if ws_bytes else 0, stream.cuda_stream or None)
    _check(st, "conv_wgrad")
    return out
