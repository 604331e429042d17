"""mq_gemm_noalloc: the cached GEMM whose split-K scratch is a static device
array, for callers that cannot allocate device memory (runtimes whose own
pool owns the device's memory, latency-critical paths that must not risk an
allocation's implicit synchronization).

Called through the C ABI.  Two noalloc calls in a row come first (so the
file also passes alone in a fresh process, before anything else has set up
the library's workspace), then each result is compared with mq_gemm's output
and with the f64 oracle on sampled outputs, within the GEMM tolerance of the
other tests.  The shared scratch keeps the previous call's contents, which
must not leak into the next result.  A call on a fresh weight must leave the
device's free memory unchanged.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
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
def test_noalloc_matches_mq_gemm_and_oracle(N, K, M, orc):
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    L = mq._lib()
    g = synth.rng(N + K + M)
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    xh = synth.activations(g, M, K)
    x = dev(xh)
    outs = []
    for call in range(2):   # two noalloc calls in a row, before any mq_gemm
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L, x, h, y, M) == 0, L.mq_last_error_detail()
        mq.mq_stream_status()
        outs.append(y.cpu().numpy())
    y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mq.mq_gemm(x, h, y_ref, M)
    mq.mq_stream_status()
    ref = y_ref.cpu().numpy()
    mi, ni = sample_indices(M, N, 2000, seed=N + M)
    w16 = orc.decode_matrix(synth.Q4_K, data, N, K)
    ref_s = orc.gemm_f64_sampled(xh.view(np.uint16), w16, mi, ni)
    for call, out in enumerate(outs):
        assert_gemm_close(out, ref, f"noalloc call {call} vs mq_gemm, N={N} K={K} M={M}")
        assert_gemm_close(out[mi, ni], ref_s, f"noalloc call {call} vs oracle, N={N} K={K} M={M}")
    # a different problem in between, then the first again: no stale scratch
    x2 = dev(synth.activations(g, 64, K))
    y2 = torch.empty((64, N), dtype=torch.float32, device="cuda")
    assert _call(L, x2, h, y2, 64) == 0
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert _call(L, x, h, y, M) == 0
    mq.mq_stream_status()
    assert_gemm_close(y.cpu().numpy(), ref, "noalloc after another problem")
    h.release()


def test_noalloc_leaves_free_memory_unchanged():
    """A call on a freshly registered weight (same shape as an earlier call,
    so no kernel is loaded for the first time) takes no device memory."""
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    L = mq._lib()
    N, K, M = 512, 3584, 2048
    g = synth.rng(11)
    x = dev(synth.activations(g, M, K))
    ya = torch.empty((M, N), dtype=torch.float32, device="cuda")
    yb = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ha = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, N, K)), N, K)
    assert _call(L, x, ha, ya, M) == 0, L.mq_last_error_detail()
    mq.mq_stream_status()
    hb = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, N, K)), N, K)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert _call(L, x, hb, yb, M) == 0, L.mq_last_error_detail()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes across one noalloc call"
    mq.mq_stream_status()
    assert np.all(np.isfinite(yb.cpu().numpy()))
    ha.release()
    hb.release()


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
