"""Sizes at the edges of what the library plans for, against the oracle on
sampled outputs (corners and tile edges included): a long token axis
(M = 32768, 128 token tiles of 256), a long reduction axis (K = 65536: 256
K steps, split over K at small M), a single weight row tile with a ragged
tail (N = 1, the smallest registrable weight; N = 129), and the smallest K
the fused path takes (K = 64 on a 32-element format).  Each runs the paths a
caller would reach for it (cached, fused, the M gate)."""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _run_sampled(orc, qtype, N, K, M, paths, seed, count=2000):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(seed)
    data = synth.weight_bytes(g, qtype, N, K)
    xh = synth.activations(g, M, K)
    x = dev(xh)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    W16 = orc.decode_matrix(qtype, data, N, K)
    mi, ni = sample_indices(M, N, count, seed=seed)
    ref = orc.gemm_f64_sampled(xh.view(np.uint16), W16, mi, ni)
    for name in paths:
        fn = {"cached": mq.mq_gemm, "fused": mq.mq_gemm_fused, "auto": mq.mq_gemm_auto}[name]
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        fn(x, h, y, M)
        mq.mq_stream_status()
        yh = y.cpu().numpy()
        assert np.all(np.isfinite(yh)), f"{name} {N}x{K} M={M}: non-finite output"
        assert_gemm_close(yh[mi, ni], ref, f"{name} {synth.TYPE_NAME[qtype]} {N}x{K} M={M}")
        del y
    h.release()


def test_long_token_axis(orc):
    """M = 32768 on the 7B k/v shape (128 token tiles, many waves)."""
    _run_sampled(orc, synth.Q4_K, 512, 3584, 32768, ("cached", "auto"), seed=1)


@pytest.mark.parametrize("M", [1, 40, 300])
def test_long_reduction_axis(orc, M):
    """K = 65536 (256 K steps; 256 raw chunks on the fused path), N = 384:
    three row tiles, so small M is split over K."""
    _run_sampled(orc, synth.Q4_K, 384, 65536, M, ("cached", "fused", "auto"), seed=2 + M)


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q8_0, 1, 1024),     # one weight row: a tile that is almost all tail
    (synth.Q6_K, 129, 2048),   # one full row tile and a one-row tail
    (synth.Q4_0, 64, 64),      # the fused path's smallest K (one 64-wide K step)
])
@pytest.mark.parametrize("M", [1, 257])
def test_degenerate_shapes(orc, qtype, N, K, M):
    _run_sampled(orc, qtype, N, K, M, ("cached", "fused", "auto"), seed=N + K + M, count=500)
