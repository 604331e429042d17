"""mq_gemm_noalloc: the cached GEMM whose split-K scratch is a static device
array, for callers that cannot allocate device memory (graph capture in
global mode, engines whose pool owns the device, latency-critical paths).

Called through the C ABI and compared with mq_gemm's output, within the
GEMM tolerance of the other tests, on two calls in a row (the shared scratch
keeps the previous call's contents, which must not leak into the next
result).  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _call(L, x, h, y, M):
    return L.mq_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(h.handle),
                             ctypes.c_void_p(y.data_ptr()), M, None)


@pytest.mark.parametrize("N,K,M", [
    (512, 3584, 2048),   # the 7B k/v shape: split-K over the static scratch
    (384, 1024, 300),    # split-K with ragged M
    (1024, 2048, 96),
])
def test_noalloc_matches_mq_gemm(N, K, M):
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    L = mq._lib()
    g = synth.rng(N + K + M)
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    x = dev(synth.activations(g, M, K))
    y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mq.mq_gemm(x, h, y_ref, M)
    mq.mq_stream_status()
    ref = y_ref.cpu().numpy()
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L, x, h, y, M) == 0, L.mq_last_error_detail()
        mq.mq_stream_status()
        assert_gemm_close(y.cpu().numpy(), ref, f"noalloc call {call} N={N} K={K} M={M}")
    # a different problem in between, then the first again: no stale scratch
    x2 = dev(synth.activations(g, 64, K))
    y2 = torch.empty((64, N), dtype=torch.float32, device="cuda")
    assert _call(L, x2, h, y2, 64) == 0
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert _call(L, x, h, y, M) == 0
    mq.mq_stream_status()
    assert_gemm_close(y.cpu().numpy(), ref, "noalloc after another problem")
    h.release()


def test_noalloc_rejects_oversized_scratch():
    """A split plan larger than the 16 MiB static scratch is refused with a
    clear message (the 7B q/o shape at M = 2048 needs about 18.9 MB)."""
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    L = mq._lib()
    g = synth.rng(3)
    N = K = 3584
    M = 2048
    h = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, N, K)), N, K)
    x = dev(synth.activations(g, M, K))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert _call(L, x, h, y, M) == -3
    assert b"static scratch holds" in L.mq_last_error_detail()
    h.release()
