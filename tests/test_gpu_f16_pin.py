"""Device half of the binary16 pin: all 2^32 binary32 bit patterns through
the decoders' own f32 -> f16 step on the GPU (the packed round-to-nearest-
even conversion that every decoder and the fused GEMM's on-chip decode end
with), compared with the oracle's conversion, which the CPU suite pins
exhaustively against the compiler's _Float16 ("05 · 8p — Persistent f16
weight cache + fused dequant-in-GEMM", section 3.3 Pitfalls: the fused and
cached decodes must round through the same path).

Bit for bit for every non-NaN input (signed zeros, subnormals, ties,
overflow to infinity included); a NaN input must give an f16 NaN (its
payload is not part of the contract).  Chunks of 2^28 patterns keep the
device and host buffers at 512 MB."""
import numpy as np
import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def test_device_f16_rounding_exhaustive(orc):
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    out = torch.empty(CHUNK, dtype=torch.int16, device="cuda")
    host = torch.empty(CHUNK, dtype=torch.int16).pin_memory()
    total_nan = 0
    for c in range((1 << 32) // CHUNK):
        first = c * CHUNK
        mq.mq_debug_cvt_f16(first, CHUNK, out)
        host.copy_(out)
        mq.mq_stream_status()
        got = host.numpy().view(np.uint16)
        pats = np.arange(first, first + CHUNK, dtype=np.uint64).astype(np.uint32)
        ref = orc.f32_to_f16(pats.view(np.float32))
        is_nan = ((pats & 0x7F800000) == 0x7F800000) & ((pats & 0x007FFFFF) != 0)
        bad = np.flatnonzero((got != ref) & ~is_nan)
        assert bad.size == 0, (f"pattern 0x{int(pats[bad[0]]):08x}: device 0x{int(got[bad[0]]):04x}, "
                               f"oracle 0x{int(ref[bad[0]]):04x} ({bad.size} mismatches in chunk {c})")
        gn = got[is_nan]
        assert np.all(((gn & 0x7C00) == 0x7C00) & ((gn & 0x03FF) != 0)), f"chunk {c}: NaN input gave a non-NaN"
        total_nan += int(is_nan.sum())
    assert total_nan == 2 * ((1 << 23) - 1)   # every NaN pattern was seen


def test_debug_cvt_argument_checks():
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    out = torch.empty(16, dtype=torch.int16, device="cuda")
    with pytest.raises(mq.MQError) as e:
        mq.mq_debug_cvt_f16(1, 4, out)
    assert e.value.name == "MQ_ERR_SHAPE"
    with pytest.raises(mq.MQError) as e:
        mq.mq_debug_cvt_f16(0xFFFFFFFE, 4, out)
    assert e.value.name == "MQ_ERR_SHAPE"
    mq.mq_debug_cvt_f16(0x3C000000, 2, out)   # 2^-7 and its successor: f16 0x2000, 0x2000
    mq.mq_stream_status()
    assert out[:2].cpu().numpy().view(np.uint16).tolist() == [0x2000, 0x2000]
