"""The C-ABI library loads and exports what include/mq.h declares; argument
validation that needs no device; the product path and the oracle stay
apart.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_weight_prefill_gguf_gb300")


@pytest.fixture(scope="module")
def lib():
    from quantized_weight_prefill_gguf_gb300 import _build
    _build.build()
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq._lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mq_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mq_register_weight", "mq_gemm", "mq_gemm_fused", "mq_gemm_auto",
                     "mq_dequantize", "mq_release_weight", "mq_stream_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import quantized_weight_prefill_gguf_gb300 as mq
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mq.h but not exported"
    assert sorted(mq.EXPORTS) == names


def test_error_strings(lib):
    import quantized_weight_prefill_gguf_gb300 as mq
    for code in mq.STATUS:
        s = lib.mq_error_string(code).decode()
        assert s and s != "unknown status"
    assert lib.mq_version() >= 100


def test_host_validation_without_device(lib):
    """Checks that run before any device work return their codes."""
    out = ctypes.c_void_p()
    assert lib.mq_register_weight(10, ctypes.c_void_p(16), 256, 256, 0, None, ctypes.byref(out)) == -2
    assert b"type id 10" in lib.mq_last_error_detail()
    assert lib.mq_register_weight(12, None, 256, 256, 0, None, ctypes.byref(out)) == -1
    assert lib.mq_register_weight(12, ctypes.c_void_p(16), 256, 100, 0, None, ctypes.byref(out)) == -3
    assert lib.mq_register_weight(12, ctypes.c_void_p(16), 3, 264, 0, None, ctypes.byref(out)) == -3
    assert lib.mq_register_weight(12, ctypes.c_void_p(18), 256, 256, 0, None, ctypes.byref(out)) == -4
    assert lib.mq_register_weight(12, ctypes.c_void_p(16), 256, 256, 0x80, None, ctypes.byref(out)) == -1
    assert lib.mq_register_weight(12, ctypes.c_void_p(16), 256, 256, 0, None, None) == -1
    # a handle that was never registered is rejected without being dereferenced
    assert lib.mq_gemm(ctypes.c_void_p(16), ctypes.c_void_p(0x1234), ctypes.c_void_p(16), 8, None) == -1
    assert lib.mq_release_weight(ctypes.c_void_p(0x1234)) == -1
    assert lib.mq_set_m_gate(0) == -1
    # the default gate is the measured fused/cached crossover (fused up to M = 128)
    if not os.environ.get("MQ_M_GATE"):
        assert lib.mq_get_m_gate() == 129
    assert lib.mq_reserve_workspace(-1) == -1
    # grouped entry points: null arrays, count out of range, stale member handles
    P = ctypes.c_void_p
    ys = (P * 2)(16, 32)
    for fn in (lib.mq_gemm_grouped, lib.mq_gemm_fused_grouped, lib.mq_gemm_auto_grouped):
        assert fn(P(16), None, 2, ys, 8, None) == -1
        assert fn(P(16), (P * 2)(0x1234, 0x1234), 2, None, 8, None) == -1
        assert fn(P(16), (P * 2)(0x1234, 0x1234), 0, ys, 8, None) == -1
        assert fn(P(16), (P * 2)(0x1234, 0x1234), 5, ys, 8, None) == -1
        assert fn(P(16), (P * 2)(0x1234, 0x1234), 2, ys, 8, None) == -1


def test_product_and_oracle_share_nothing():
    """The package never imports or loads the oracle, and the oracle never
    imports the package; only the generator module is shared."""
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+quantized_weight_prefill_gguf_gb300", text, flags=re.M), f
            assert "#include \"mq" not in text and "libmq" not in text, f
