"""Host-side failure paths on a GPU machine: every one is caught before any
kernel runs and reported with its status code; nothing here faults the GPU.
Also: a full pipeline of two dependent GEMMs with no host read between them,
and workspace reservation before capturing calls in a CUDA graph."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def test_error_codes():
    torch = torch_cuda()
    mq = _mq()
    L = mq._lib()
    g = synth.rng(1)
    N, K = 128, 512
    q = dev(synth.weight_bytes(g, synth.Q4_K, N, K))
    x = dev(synth.activations(g, 8, K))
    y = torch.empty((8, N), dtype=torch.float32, device="cuda")
    out = ctypes.c_void_p()
    # misaligned qdata / x / y
    assert L.mq_register_weight(12, q.data_ptr() + 2, N, K, 0, None, ctypes.byref(out)) == -4
    h = mq.mq_register_weight(synth.Q4_K, q, N, K)
    assert L.mq_gemm(x.data_ptr() + 2, h.handle, y.data_ptr(), 8, None) == -4
    assert L.mq_gemm(x.data_ptr(), h.handle, y.data_ptr() + 4, 8, None) == -4
    assert L.mq_gemm(x.data_ptr(), h.handle, y.data_ptr(), 0, None) == -3
    # no cache
    hn = mq.mq_register_weight(synth.Q4_K, q, N, K, flags=mq.MQ_REG_NO_CACHE)
    assert L.mq_gemm(x.data_ptr(), hn.handle, y.data_ptr(), 8, None) == -5
    assert b"MQ_REG_NO_CACHE" in L.mq_last_error_detail()
    # released handle
    stale = h.handle
    h.release()
    assert L.mq_gemm(x.data_ptr(), stale, y.data_ptr(), 8, None) == -1
    assert L.mq_release_weight(stale) == -1
    # fused path needs K % 64 == 0
    q8 = dev(synth.weight_bytes(g, synth.Q8_0, 64, 96))
    h8 = mq.mq_register_weight(synth.Q8_0, q8, 64, 96)
    x8 = dev(synth.activations(g, 4, 96))
    y8 = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    assert L.mq_gemm_fused(x8.data_ptr(), h8.handle, y8.data_ptr(), 4, None) == -3
    # mq_gemm_auto on that handle takes the cached path
    mq.mq_gemm_auto(x8, h8, y8)
    mq.mq_stream_status()
    assert mq.mq_stream_status() is None


def test_forced_allocation_failure():
    """MQ_FAULT_ALLOC=1 makes the cache allocation fail: registration returns
    MQ_ERR_OOM early and leaves nothing allocated (run in a child process so
    the environment variable does not leak)."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import torch, ctypes\n"
        "import quantized_weight_prefill_gguf_gb300 as mq\n"
        "q = torch.zeros(144 * 4, dtype=torch.uint8, device='cuda')\n"
        "out = ctypes.c_void_p()\n"
        "rc = mq._lib().mq_register_weight(12, q.data_ptr(), 4, 256, 0, None, ctypes.byref(out))\n"
        "print(rc, out.value, mq._lib().mq_last_error_detail().decode())\n"
        "rc2 = mq._lib().mq_register_weight(12, q.data_ptr(), 4, 256, 1, None, ctypes.byref(out))\n"
        "print(rc2)\n"
    ) % ROOT
    env = dict(os.environ, MQ_FAULT_ALLOC="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    first, second = r.stdout.strip().splitlines()[-2:]
    assert first.startswith("-6 None") and "f16 cache" in first
    assert second.strip() == "0"      # a cache-less registration allocates nothing and succeeds


@pytest.mark.parametrize("M", [64, 300])
def test_dependent_chain_and_graph_capture(orc, M):
    """Two dependent GEMMs (the second consumes the first's output, cast to
    f16 on the device) with no host read in between, then the same pair
    replayed from a CUDA graph after reserving the workspace.  M = 64 runs
    the cached GEMM as multicast CTA pairs, M = 300 as 2-SM MMAs."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(8)
    N1, K1, N2 = 512, 1024, 256
    d1 = synth.weight_bytes(g, synth.Q4_K, N1, K1)
    d2 = synth.weight_bytes(g, synth.Q6_K, N2, N1)
    x = synth.activations(g, M, K1)
    h1 = mq.mq_register_weight(synth.Q4_K, dev(d1), N1, K1)
    h2 = mq.mq_register_weight(synth.Q6_K, dev(d2), N2, N1)
    xd = dev(x)
    y1 = torch.empty((M, N1), dtype=torch.float32, device="cuda")
    y2 = torch.empty((M, N2), dtype=torch.float32, device="cuda")
    mq.mq_reserve_workspace(64 << 20)

    def chain(stream=None):
        mq.mq_gemm(xd, h1, y1, M, stream)
        x2 = (y1 * 0.05).half()
        mq.mq_gemm_fused(x2, h2, y2, M, stream)
        return x2

    x2 = chain()
    mq.mq_stream_status()
    W1 = orc.decode_matrix(synth.Q4_K, d1, N1, K1)
    W2 = orc.decode_matrix(synth.Q6_K, d2, N2, N1)
    assert_gemm_close(y1.cpu().numpy(), orc.gemm_f64(x.view(np.uint16), W1), "chain 1")
    x2h = x2.cpu().numpy()
    assert_gemm_close(y2.cpu().numpy(), orc.gemm_f64(x2h.view(np.uint16), W2), "chain 2")

    ref2 = y2.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        chain(s)   # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            chain(s)
    y2.zero_()
    graph.replay()
    torch.cuda.synchronize()
    mq.mq_stream_status()
    assert torch.equal(y2, ref2)


@pytest.mark.parametrize("path", ["cached", "fused", "cached_2sm", "e4m3_2sm"])
def test_bounded_wait_timeout_recovers(orc, monkeypatch, path):
    """A producer that never delivers (injected from the host): every
    consumer's bounded wait runs out after about a second, the kernel exits
    cleanly (TMEM freed; both CTAs of a pair meet at the final cluster
    barrier), mq_stream_status reports MQ_ERR_DEVICE, and the context stays
    usable -- the next call is correct.  No GPU fault.  M = 48 runs the
    multicast CTA pairs, M = 300 the 2-SM MMAs."""
    import time
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(12)
    N, K = 256, 512
    M = 300 if path.endswith("2sm") else 48
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    x = dev(synth.activations(g, M, K))
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K, flags=mq.MQ_REG_E4M3)
    if path == "e4m3_2sm":
        x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        mq.mq_quantize_e4m3(x, x8, sx)

        def fn(_x, hh, yy, mm):
            mq.mq_gemm_e4m3(x8, sx, hh, yy, mm)
    else:
        fn = mq.mq_gemm_fused if path == "fused" else mq.mq_gemm
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    mq.mq_stream_status()
    monkeypatch.setenv("MQ_INJECT_PRODUCER_STALL", "1")
    t0 = time.time()
    fn(x, h, y, M)
    with pytest.raises(mq.MQError) as ei:
        mq.mq_stream_status()
    assert ei.value.code == -8 and "timed out" in str(ei.value)
    assert time.time() - t0 < 60
    monkeypatch.delenv("MQ_INJECT_PRODUCER_STALL")
    mq.mq_stream_status()   # status word was cleared by the failing read
    fn(x, h, y, M)
    mq.mq_stream_status()
    if path == "e4m3_2sm":
        codes, scales = h.e4m3_tensors()
        y_ref = orc.gemm_e4m3_f64(x8.cpu().numpy(), sx.cpu().numpy(), codes.cpu().numpy()[:, :K],
                                  scales.cpu().numpy())
        del codes, scales
    else:
        y_ref = orc.gemm_f64(x.cpu().numpy().view(np.uint16), orc.decode_matrix(synth.Q4_K, data, N, K))
    assert_gemm_close(y.cpu().numpy(), y_ref, f"{path} after a timed-out call")
