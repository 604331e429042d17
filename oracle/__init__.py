"""CPU oracle for the GGUF quantized-weight prefill GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product path
(``quantized_weight_prefill_gguf_gb300``) never imports it and shares no code
with it; the two meet only through the seeded input generator module.

The arithmetic lives in plain C (``oracle.c``: binary16 conversion, block
decoders, f64 GEMM; ``encode.c``: field -> byte block encoders used by the
pin tests).  This module compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ("oracle.c", "encode.c")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC"]

# GGUF type ids and (elements per block, bytes per block).
F32, F16, BF16 = 0, 1, 30
Q4_0, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 6, 7, 8, 12, 13, 14
BLOCK = {F32: (1, 4), F16: (1, 2), BF16: (1, 2), Q4_0: (32, 18), Q5_0: (32, 22), Q5_1: (32, 24), Q8_0: (32, 34), Q4_K: (256, 144),
         Q5_K: (256, 176), Q6_K: (256, 210)}


def build(out: str | None = None, extra_flags: list[str] | None = None,
          src_dir: str | None = None) -> str:
    """Compile the oracle into a shared library and return its path."""
    src_dir = src_dir or HERE
    out = out or os.path.join(HERE, "liboracle.so")
    srcs = [os.path.join(src_dir, s) for s in SOURCES]
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), *srcs, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in SOURCES)


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        L = ctypes.CDLL(path)
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f32_to_f16_n.argtypes = [_P, _I64, _P]
        L.oracle_f16_to_f32_n.argtypes = [_P, _I64, _P]
        L.oracle_decode.argtypes = [ctypes.c_int, _P, _I64, _P]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_gemm_f64.argtypes = [_P, _I64, _I64, _P, _I64, _P]
        L.oracle_gemm_f64.restype = ctypes.c_int
        L.oracle_gemm_f64_sampled.argtypes = [_P, _I64, _P, _P, _P, _I64, _P]
        L.oracle_gemm_f64_sampled.restype = ctypes.c_int
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_quantize_e4m3_rows.argtypes = [_P, _I64, _I64, _I64, _P, _P]
        L.oracle_quantize_e4m3_rows.restype = ctypes.c_int
        L.oracle_gemm_e4m3_f64.argtypes = [_P, _P, _I64, _I64, _P, _P, _I64, _P]
        L.oracle_gemm_e4m3_f64.restype = ctypes.c_int
        L.oracle_gemm_e4m3_f64_sampled.argtypes = [_P, _P, _I64, _P, _P, _P, _P, _I64, _P]
        L.oracle_gemm_e4m3_f64_sampled.restype = ctypes.c_int
        L.oracle_pack_q8_0.argtypes = [ctypes.c_uint16, _P, _P]
        L.oracle_pack_q4_K.argtypes = [ctypes.c_uint16, ctypes.c_uint16, _P, _P, _P, _P]
        L.oracle_pack_q6_K.argtypes = [ctypes.c_uint16, _P, _P, _P]
        self.L = L

    # -- O1 -----------------------------------------------------------
    def f32_to_f16(self, a) -> np.ndarray:
        a = np.ascontiguousarray(a, dtype=np.float32)
        out = np.empty(a.shape, dtype=np.uint16)
        self.L.oracle_f32_to_f16_n(a.ctypes.data, a.size, out.ctypes.data)
        return out

    def f16_to_f32(self, h) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float32)
        self.L.oracle_f16_to_f32_n(h.ctypes.data, h.size, out.ctypes.data)
        return out

    # -- O2 -----------------------------------------------------------
    def decode(self, qtype: int, qbytes) -> np.ndarray:
        """Decode a flat block stream; returns the f16 bit patterns (uint16)."""
        qk, bb = BLOCK[qtype]
        q = np.ascontiguousarray(qbytes, dtype=np.uint8).reshape(-1)
        if q.size % bb:
            raise ValueError("byte count is not a whole number of blocks")
        nb = q.size // bb
        out = np.empty(nb * qk, dtype=np.uint16)
        rc = self.L.oracle_decode(qtype, q.ctypes.data, nb, out.ctypes.data)
        if rc:
            raise ValueError(f"oracle_decode failed: {rc}")
        return out

    def decode_matrix(self, qtype: int, qbytes, N: int, K: int) -> np.ndarray:
        """W[N,K] as f16 bits, the flat stream read row-major."""
        return self.decode(qtype, qbytes)[: N * K].reshape(N, K)

    # -- O4 -----------------------------------------------------------
    def gemm_f64(self, X16, W16) -> np.ndarray:
        """Y = X . W^T with f64 accumulation; X16 [M,K], W16 [N,K] are f16 bits."""
        X16 = np.ascontiguousarray(X16, dtype=np.uint16)
        W16 = np.ascontiguousarray(W16, dtype=np.uint16)
        M, K = X16.shape
        N, K2 = W16.shape
        assert K == K2
        Y = np.empty((M, N), dtype=np.float64)
        rc = self.L.oracle_gemm_f64(X16.ctypes.data, M, K, W16.ctypes.data, N, Y.ctypes.data)
        if rc:
            raise MemoryError("oracle_gemm_f64 failed")
        return Y

    def gemm_f64_sampled(self, X16, W16, mi, ni) -> np.ndarray:
        X16 = np.ascontiguousarray(X16, dtype=np.uint16)
        W16 = np.ascontiguousarray(W16, dtype=np.uint16)
        mi = np.ascontiguousarray(mi, dtype=np.int64)
        ni = np.ascontiguousarray(ni, dtype=np.int64)
        K = X16.shape[1]
        assert W16.shape[1] == K and mi.shape == ni.shape
        assert mi.size == 0 or (mi.min() >= 0 and mi.max() < X16.shape[0])
        assert ni.size == 0 or (ni.min() >= 0 and ni.max() < W16.shape[0])
        out = np.empty(mi.size, dtype=np.float64)
        rc = self.L.oracle_gemm_f64_sampled(X16.ctypes.data, K, W16.ctypes.data,
                                            mi.ctypes.data, ni.ctypes.data, mi.size,
                                            out.ctypes.data)
        if rc:
            raise MemoryError("oracle_gemm_f64_sampled failed")
        return out

    # -- O5 -----------------------------------------------------------
    def f32_to_e4m3(self, x) -> np.ndarray:
        """e4m3 codes of binary32 values (round to nearest even, clamp to 448)."""
        x = np.asarray(x, dtype=np.float32).reshape(-1)
        return np.array([self.L.oracle_f32_to_e4m3(float(v)) for v in x], dtype=np.uint8)

    def e4m3_to_f64(self, codes) -> np.ndarray:
        codes = np.asarray(codes, dtype=np.uint8).reshape(-1)
        return np.array([self.L.oracle_e4m3_to_f64(int(c)) for c in codes], dtype=np.float64)

    def quantize_e4m3_rows(self, X16):
        """Row-wise e4m3 quantization of f16 bits [rows, K]: (codes [rows, K]
        uint8, scales [rows] float32)."""
        X16 = np.ascontiguousarray(X16, dtype=np.uint16)
        rows, K = X16.shape
        q = np.empty((rows, K), dtype=np.uint8)
        sc = np.empty(rows, dtype=np.float32)
        self.L.oracle_quantize_e4m3_rows(X16.ctypes.data, rows, K, K, q.ctypes.data, sc.ctypes.data)
        return q, sc

    def gemm_e4m3_f64(self, X8, sx, W8, sw) -> np.ndarray:
        """Y = (x8 . w8^T) * sw[n] * sx[m] in f64."""
        X8 = np.ascontiguousarray(X8, dtype=np.uint8)
        W8 = np.ascontiguousarray(W8, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = X8.shape
        N, K2 = W8.shape
        assert K == K2 and sx.size == M and sw.size == N
        Y = np.empty((M, N), dtype=np.float64)
        self.L.oracle_gemm_e4m3_f64(X8.ctypes.data, sx.ctypes.data, M, K, W8.ctypes.data, sw.ctypes.data, N,
                                    Y.ctypes.data)
        return Y

    def gemm_e4m3_f64_sampled(self, X8, sx, W8, sw, mi, ni) -> np.ndarray:
        X8 = np.ascontiguousarray(X8, dtype=np.uint8)
        W8 = np.ascontiguousarray(W8, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        mi = np.ascontiguousarray(mi, dtype=np.int64)
        ni = np.ascontiguousarray(ni, dtype=np.int64)
        K = X8.shape[1]
        assert W8.shape[1] == K and mi.shape == ni.shape
        assert mi.size == 0 or (mi.min() >= 0 and mi.max() < X8.shape[0])
        assert ni.size == 0 or (ni.min() >= 0 and ni.max() < W8.shape[0])
        out = np.empty(mi.size, dtype=np.float64)
        self.L.oracle_gemm_e4m3_f64_sampled(X8.ctypes.data, sx.ctypes.data, K, W8.ctypes.data, sw.ctypes.data,
                                            mi.ctypes.data, ni.ctypes.data, mi.size, out.ctypes.data)
        return out

    def num_threads(self) -> int:
        return int(self.L.oracle_num_threads())

    # -- O3 (encoders, tests only) ------------------------------------
    def pack_q8_0(self, d: int, q) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.int8)
        assert q.size == 32
        out = np.zeros(34, dtype=np.uint8)
        self.L.oracle_pack_q8_0(int(d), q.ctypes.data, out.ctypes.data)
        return out

    def pack_q4_K(self, d: int, dmin: int, sc, m, q) -> np.ndarray:
        sc = np.ascontiguousarray(sc, dtype=np.uint8)
        m = np.ascontiguousarray(m, dtype=np.uint8)
        q = np.ascontiguousarray(q, dtype=np.uint8)
        assert sc.size == 8 and m.size == 8 and q.size == 256
        out = np.zeros(144, dtype=np.uint8)
        self.L.oracle_pack_q4_K(int(d), int(dmin), sc.ctypes.data, m.ctypes.data,
                                q.ctypes.data, out.ctypes.data)
        return out

    def pack_q6_K(self, d: int, sc, q6) -> np.ndarray:
        sc = np.ascontiguousarray(sc, dtype=np.int8)
        q6 = np.ascontiguousarray(q6, dtype=np.int8)
        assert sc.size == 16 and q6.size == 256
        out = np.zeros(210, dtype=np.uint8)
        self.L.oracle_pack_q6_K(int(d), sc.ctypes.data, q6.ctypes.data, out.ctypes.data)
        return out


_cached: Oracle | None = None


def load() -> Oracle:
    """The oracle library, compiled on first use if missing or stale."""
    global _cached
    if _cached is None:
        path = os.path.join(HERE, "liboracle.so")
        if _stale(path):
            build(path)
        _cached = Oracle(path)
    return _cached
