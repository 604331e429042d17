"""Python binding of libmq, the sm_103a quantized-weight prefill GEMM library.

Argument marshalling only: every step of decode and GEMM runs in the
library's CUDA kernels behind the C ABI in ``include/mq.h``.  The functions
keep the C names.  Tensors are torch CUDA tensors (PyTorch supplies device
memory and streams); the current torch stream is used when none is given.
If ``libmq.so`` is missing, the first call raises ImportError: there is no
CPU fallback.  (Importing the package alone does not load the library, so
the seeded input generator in ``synth`` stays usable without a build.)
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmq.so")

MQ_TYPE_F32, MQ_TYPE_F16, MQ_TYPE_BF16 = 0, 1, 30
MQ_TYPE_Q4_0, MQ_TYPE_Q5_0, MQ_TYPE_Q5_1, MQ_TYPE_Q8_0 = 2, 6, 7, 8
MQ_TYPE_Q4_K, MQ_TYPE_Q5_K, MQ_TYPE_Q6_K = 12, 13, 14
MQ_REG_NO_CACHE, MQ_REG_NO_KPAD, MQ_REG_KPAD, MQ_REG_E4M3 = 0x1, 0x2, 0x4, 0x8
STATUS = {0: "MQ_OK", -1: "MQ_ERR_INVALID", -2: "MQ_ERR_UNSUPPORTED_TYPE", -3: "MQ_ERR_SHAPE",
          -4: "MQ_ERR_ALIGN", -5: "MQ_ERR_NO_CACHE", -6: "MQ_ERR_OOM", -7: "MQ_ERR_CUDA",
          -8: "MQ_ERR_DEVICE", -9: "MQ_ERR_NO_DEVICE"}
# Every symbol include/mq.h declares.
EXPORTS = ("mq_register_weight", "mq_release_weight", "mq_weight_info", "mq_dequantize", "mq_gemm",
           "mq_gemm_fused", "mq_gemm_auto", "mq_get_m_gate", "mq_set_m_gate", "mq_reserve_workspace",
           "mq_stream_status", "mq_launch_count", "mq_error_string", "mq_last_error_detail", "mq_version",
           "mq_trace_enable", "mq_trace_count", "mq_trace_read", "mq_gemm_noalloc", "mq_gemm_grouped", "mq_gemm_fused_grouped", "mq_gemm_auto_grouped",
           "mq_gemm_scratch", "mq_quantize_e4m3", "mq_gemm_e4m3", "mq_weight_e4m3_info",
           "mq_gemm_e4m3_grouped", "mq_debug_schedule", "mq_debug_cvt_f16")
MQ_TRACE_GEMM_CACHED, MQ_TRACE_GEMM_FUSED, MQ_TRACE_DECODE = 1, 2, 3


class TraceRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("type", ctypes.c_int32), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("ms_main", ctypes.c_float),
                ("ms_aux", ctypes.c_float)]

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "mq_register_weight": ([ctypes.c_int, _P, _I64, _I64, ctypes.c_uint32, _P, ctypes.POINTER(_P)], ctypes.c_int),
        "mq_release_weight": ([_P], ctypes.c_int),
        "mq_weight_info": ([_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                            ctypes.POINTER(_P)], ctypes.c_int),
        "mq_dequantize": ([ctypes.c_int, _P, _I64, _I64, _P, _I64, _P], ctypes.c_int),
        "mq_gemm": ([_P, _P, _P, _I64, _P], ctypes.c_int),
        "mq_gemm_fused": ([_P, _P, _P, _I64, _P], ctypes.c_int),
        "mq_gemm_auto": ([_P, _P, _P, _I64, _P], ctypes.c_int),
        "mq_gemm_noalloc": ([_P, _P, _P, _I64, _P], ctypes.c_int),
        "mq_gemm_scratch": ([_P, _P, _P, _I64, _P, _I64, _P], ctypes.c_int),
        "mq_quantize_e4m3": ([_P, _I64, _I64, _I64, _P, _I64, _P, _P], ctypes.c_int),
        "mq_gemm_e4m3": ([_P, _P, _P, _P, _I64, _P], ctypes.c_int),
        "mq_gemm_e4m3_grouped": ([_P, _P, ctypes.POINTER(_P), ctypes.c_int, ctypes.POINTER(_P), _I64, _P],
                                 ctypes.c_int),
        "mq_weight_e4m3_info": ([_P, ctypes.POINTER(_I64), ctypes.POINTER(_P), ctypes.POINTER(_P)], ctypes.c_int),
        "mq_gemm_grouped": ([_P, ctypes.POINTER(_P), ctypes.c_int, ctypes.POINTER(_P), _I64, _P], ctypes.c_int),
        "mq_gemm_fused_grouped": ([_P, ctypes.POINTER(_P), ctypes.c_int, ctypes.POINTER(_P), _I64, _P], ctypes.c_int),
        "mq_gemm_auto_grouped": ([_P, ctypes.POINTER(_P), ctypes.c_int, ctypes.POINTER(_P), _I64, _P], ctypes.c_int),
        "mq_debug_schedule": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _I64, _P],
                              ctypes.c_int),
        "mq_debug_cvt_f16": ([ctypes.c_uint32, _I64, _P, _P], ctypes.c_int),
        "mq_get_m_gate": ([], _I64),
        "mq_set_m_gate": ([_I64], ctypes.c_int),
        "mq_reserve_workspace": ([_I64], ctypes.c_int),
        "mq_stream_status": ([_P], ctypes.c_int),
        "mq_launch_count": ([], _I64),
        "mq_error_string": ([ctypes.c_int], ctypes.c_char_p),
        "mq_last_error_detail": ([], ctypes.c_char_p),
        "mq_version": ([], ctypes.c_int),
        "mq_trace_enable": ([ctypes.c_int], ctypes.c_int),
        "mq_trace_count": ([], _I64),
        "mq_trace_read": ([_I64, ctypes.POINTER(TraceRecord)], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib_handle: ctypes.CDLL | None = None


def _lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use; ImportError if not built)."""
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


class MQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        detail = _lib().mq_last_error_detail().decode(errors="replace")
        super().__init__(f"{where}: {self.name} ({_lib().mq_error_string(code).decode()}): {detail}")


def _check(code: int, where: str) -> None:
    if code != 0:
        raise MQError(code, where)


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _ptr(t) -> int:
    return int(t.data_ptr()) if t is not None else 0


class Weight:
    """A registered weight.  Keeps a reference to the quantized bytes, which
    must stay unchanged while the handle lives (the fused path reads them on
    every call)."""

    def __init__(self, handle: int, qdata, qtype: int, N: int, K: int):
        self.handle = handle
        self.qdata = qdata
        self.qtype, self.N, self.K = qtype, N, K

    def info(self):
        n, k, ldk, cache = _I64(), _I64(), _I64(), _P()
        _check(_lib().mq_weight_info(self.handle, ctypes.byref(n), ctypes.byref(k), ctypes.byref(ldk),
                                  ctypes.byref(cache)), "mq_weight_info")
        return n.value, k.value, ldk.value, cache.value

    def cache_tensor(self):
        """The f16 cache as a torch view [N, ldk] (no copy; valid while the handle lives)."""
        import torch
        n, k, ldk, ptr = self.info()
        if not ptr:
            return None
        return _tensor_from_ptr(ptr, (n, ldk), torch.float16)

    def e4m3_tensors(self):
        """(codes uint8 [N, ldk8], scales float32 [N]) views of the e4m3 copy,
        or None without MQ_REG_E4M3."""
        import torch
        ldk8, codes, scales = _I64(), _P(), _P()
        _check(_lib().mq_weight_e4m3_info(self.handle, ctypes.byref(ldk8), ctypes.byref(codes), ctypes.byref(scales)),
               "mq_weight_e4m3_info")
        if not codes.value:
            return None
        n = self.info()[0]
        return (_tensor_from_ptr(codes.value, (n, ldk8.value), torch.uint8),
                _tensor_from_ptr(scales.value, (n,), torch.float32))

    def release(self) -> None:
        if self.handle:
            _check(_lib().mq_release_weight(self.handle), "mq_release_weight")
            self.handle = 0

    def __del__(self):
        try:
            if self.handle:
                _lib().mq_release_weight(self.handle)
        except Exception:
            pass


def _tensor_from_ptr(ptr: int, shape, dtype):
    """Zero-copy torch view of library-owned device memory."""
    import torch

    class _Holder:
        pass

    nbytes = 1
    for s in shape:
        nbytes *= s
    nbytes *= torch.empty((), dtype=dtype).element_size()
    h = _Holder()
    h.__cuda_array_interface__ = {
        "shape": tuple(shape), "typestr": {torch.float16: "<f2", torch.float32: "<f4", torch.uint8: "|u1"}[dtype],
        "data": (ptr, False), "version": 3, "strides": None,
    }
    return torch.as_tensor(h, device="cuda")


def mq_register_weight(qtype: int, qdata, N: int, K: int, flags: int = 0, stream=None) -> Weight:
    """qdata: torch uint8 CUDA tensor holding the flat block stream."""
    out = _P()
    _check(_lib().mq_register_weight(qtype, _ptr(qdata), N, K, flags, _stream(stream), ctypes.byref(out)),
           "mq_register_weight")
    return Weight(out.value, qdata, qtype, N, K)


def mq_dequantize(qtype: int, qdata, N: int, K: int, out, ldo: int | None = None, stream=None) -> None:
    _check(_lib().mq_dequantize(qtype, _ptr(qdata), N, K, _ptr(out), ldo if ldo is not None else K,
                             _stream(stream)), "mq_dequantize")


def mq_gemm(x, w: Weight, y, M: int | None = None, stream=None) -> None:
    _check(_lib().mq_gemm(_ptr(x), w.handle, _ptr(y), M if M is not None else x.shape[0], _stream(stream)),
           "mq_gemm")


def mq_gemm_fused(x, w: Weight, y, M: int | None = None, stream=None) -> None:
    _check(_lib().mq_gemm_fused(_ptr(x), w.handle, _ptr(y), M if M is not None else x.shape[0], _stream(stream)),
           "mq_gemm_fused")


def mq_gemm_auto(x, w: Weight, y, M: int | None = None, stream=None) -> None:
    _check(_lib().mq_gemm_auto(_ptr(x), w.handle, _ptr(y), M if M is not None else x.shape[0], _stream(stream)),
           "mq_gemm_auto")


def mq_gemm_grouped(x, ws, ys, M: int | None = None, stream=None) -> None:
    """One cached GEMM launch for weights sharing K and X: ys[g] = x . ws[g]^T."""
    if len(ws) != len(ys):
        raise ValueError(f"{len(ws)} weights but {len(ys)} outputs")
    n = len(ws)
    harr = (_P * n)(*[w.handle for w in ws])
    yarr = (_P * n)(*[_ptr(y) for y in ys])
    _check(_lib().mq_gemm_grouped(_ptr(x), harr, n, yarr, M if M is not None else x.shape[0], _stream(stream)),
           "mq_gemm_grouped")


def mq_gemm_fused_grouped(x, ws, ys, M: int | None = None, stream=None) -> None:
    """One fused GEMM launch for weights sharing K, X and block format: ys[g] = x . ws[g]^T."""
    if len(ws) != len(ys):
        raise ValueError(f"{len(ws)} weights but {len(ys)} outputs")
    n = len(ws)
    harr = (_P * n)(*[w.handle for w in ws])
    yarr = (_P * n)(*[_ptr(y) for y in ys])
    _check(_lib().mq_gemm_fused_grouped(_ptr(x), harr, n, yarr, M if M is not None else x.shape[0],
                                        _stream(stream)), "mq_gemm_fused_grouped")


def mq_gemm_auto_grouped(x, ws, ys, M: int | None = None, stream=None) -> None:
    """The M gate for a group: mq_gemm_fused_grouped below it, mq_gemm_grouped at and above it."""
    if len(ws) != len(ys):
        raise ValueError(f"{len(ws)} weights but {len(ys)} outputs")
    n = len(ws)
    harr = (_P * n)(*[w.handle for w in ws])
    yarr = (_P * n)(*[_ptr(y) for y in ys])
    _check(_lib().mq_gemm_auto_grouped(_ptr(x), harr, n, yarr, M if M is not None else x.shape[0],
                                       _stream(stream)), "mq_gemm_auto_grouped")


def mq_gemm_noalloc(x, w: Weight, y, M: int | None = None, stream=None) -> None:
    _check(_lib().mq_gemm_noalloc(_ptr(x), w.handle, _ptr(y), M if M is not None else x.shape[0],
                                  _stream(stream)), "mq_gemm_noalloc")


def mq_gemm_scratch(x, w: Weight, y, scratch, M: int | None = None, stream=None) -> None:
    """Per-call dequant into `scratch` (a CUDA tensor of at least 2*N*ldk
    bytes), then the cached GEMM on it."""
    nbytes = scratch.numel() * scratch.element_size()
    _check(_lib().mq_gemm_scratch(_ptr(x), w.handle, _ptr(y), M if M is not None else x.shape[0], _ptr(scratch),
                                  nbytes, _stream(stream)), "mq_gemm_scratch")


def mq_quantize_e4m3(x, dst, scales, stream=None) -> None:
    """Row-wise e4m3 quantization of f16 x [rows, K] into dst (uint8, [rows,
    >= K]) and scales (float32 [rows])."""
    rows, K = x.shape
    _check(_lib().mq_quantize_e4m3(_ptr(x), rows, K, x.stride(0), _ptr(dst), dst.stride(0), _ptr(scales),
                                   _stream(stream)), "mq_quantize_e4m3")


def mq_gemm_e4m3(x8, x_scale, w: Weight, y, M: int | None = None, stream=None) -> None:
    _check(_lib().mq_gemm_e4m3(_ptr(x8), _ptr(x_scale), w.handle, _ptr(y), M if M is not None else x8.shape[0],
                               _stream(stream)), "mq_gemm_e4m3")


def mq_gemm_e4m3_grouped(x8, x_scale, ws, ys, M: int | None = None, stream=None) -> None:
    """One e4m3 GEMM launch for weights sharing K and the quantized X."""
    if len(ws) != len(ys):
        raise ValueError(f"{len(ws)} weights but {len(ys)} outputs")
    n = len(ws)
    harr = (_P * n)(*[w.handle for w in ws])
    yarr = (_P * n)(*[_ptr(y) for y in ys])
    _check(_lib().mq_gemm_e4m3_grouped(_ptr(x8), _ptr(x_scale), harr, n, yarr, M if M is not None else x8.shape[0],
                                       _stream(stream)), "mq_gemm_e4m3_grouped")


def mq_debug_schedule(M: int, N: int, K: int, sms: int, path: int = 0, pair_clusters: int = 0):
    """(plan dict, units [n, 8] int32 array) of a GEMM launch as the kernels
    would run it (path 0 cached, 1 fused, 2 e4m3); host only."""
    import numpy as np
    plan = np.zeros(9, dtype=np.int64)
    count = ctypes.c_int64()
    _check(_lib().mq_debug_schedule(M, N, K, sms, path, pair_clusters, plan.ctypes.data, None, 0,
                                    ctypes.byref(count)), "mq_debug_schedule")
    units = np.zeros((max(count.value, 1), 8), dtype=np.int32)
    _check(_lib().mq_debug_schedule(M, N, K, sms, path, pair_clusters, plan.ctypes.data, units.ctypes.data,
                                    count.value, ctypes.byref(count)), "mq_debug_schedule")
    keys = ("bn", "pair", "split", "full_tiles", "tiles", "units", "grid", "ws_bytes", "kb_align")
    return dict(zip(keys, plan.tolist())), units[: count.value]


def mq_debug_cvt_f16(first: int, count: int, out, stream=None) -> None:
    """out (uint16 / int16 CUDA tensor of >= count elements) <- the f16 bits
    the decoders' f32 -> f16 step gives for binary32 patterns first ..
    first + count - 1."""
    _check(_lib().mq_debug_cvt_f16(first, count, _ptr(out), _stream(stream)), "mq_debug_cvt_f16")


def mq_get_m_gate() -> int:
    return int(_lib().mq_get_m_gate())


def mq_set_m_gate(m: int) -> None:
    _check(_lib().mq_set_m_gate(m), "mq_set_m_gate")


def mq_reserve_workspace(nbytes: int) -> None:
    _check(_lib().mq_reserve_workspace(nbytes), "mq_reserve_workspace")


def mq_stream_status(stream=None) -> None:
    _check(_lib().mq_stream_status(_stream(stream)), "mq_stream_status")


def mq_launch_count() -> int:
    return int(_lib().mq_launch_count())


def mq_version() -> int:
    return int(_lib().mq_version())


def mq_trace_enable(on: bool = True) -> None:
    _check(_lib().mq_trace_enable(1 if on else 0), "mq_trace_enable")


def mq_trace_records() -> list[dict]:
    """All records kept since the last mq_trace_enable(True)."""
    out = []
    rec = TraceRecord()
    for i in range(int(_lib().mq_trace_count())):
        _check(_lib().mq_trace_read(i, ctypes.byref(rec)), "mq_trace_read")
        out.append({f: getattr(rec, f) for f, _ in TraceRecord._fields_})
    return out
