"""Cached-path GEMM (tcgen05, f16 cache) against the oracle's f64 GEMM.

Small and ragged shapes are compared element by element over the whole
output; the full-size workloads at sampled outputs (the oracle computes each
sampled Y[m,n] as its own f64 dot product).  Also: the one-hot identity
(Y = W^T exactly), bitwise determinism including the split-K path, and the
M tail / N tail / K tail of every tile width.
"""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def run(fn, xdev, h, M, N):
    torch = torch_cuda()
    mq = _mq()
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fn(xdev, h, y, M)
    mq.mq_stream_status()
    return y


def full_case(orc, qtype, N, K, M, seed, fn_name="mq_gemm", flags=0):
    mq = _mq()
    g = synth.rng(seed)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K, flags=flags)
    y = run(getattr(mq, fn_name), dev(x), h, M, N).cpu().numpy()
    W = orc.decode_matrix(qtype, data, N, K)
    y_ref = orc.gemm_f64(x.view(np.uint16), W)
    assert_gemm_close(y, y_ref, f"{fn_name} {synth.TYPE_NAME[qtype]} M={M} N={N} K={K}")
    h.release()
    return y


def test_c0_cached(orc):
    weights, xs = synth.workload("q4k_896", seed=0)
    w = weights[0]
    x = xs[w.K]
    mq = _mq()
    h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
    y = run(mq.mq_gemm, dev(x), h, x.shape[0], w.N).cpu().numpy()
    y_ref = orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(w.qtype, w.data, w.N, w.K))
    assert_gemm_close(y, y_ref, "q4k_896 cached")


@pytest.mark.parametrize("M", [1, 17, 32, 33, 64, 65, 100, 128, 129, 255, 256, 300, 513])
def test_tile_widths_and_m_tail(orc, M):
    full_case(orc, synth.Q4_K, 384, 512, M, seed=M)


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q8_0, 200, 136),    # N tail, K not a multiple of 64
    (synth.Q8_0, 132, 72),
    (synth.Q6_K, 257, 768),
    (synth.Q4_K, 128, 4096),   # K-padded cache (ldk = K + 64)
    (synth.Q8_0, 1, 3584),     # a single weight row
])
def test_ragged_shapes(orc, qtype, N, K):
    for M in (5, 130):
        full_case(orc, qtype, N, K, M, seed=N + K + M)


def test_split_k_underfilled(orc):
    """k/v-shaped weight (N=512): 4 x 8 tiles underfill the GPU, so K is
    split and the partial planes reduced in fixed order."""
    y1 = full_case(orc, synth.Q4_K, 512, 3584, 2048, seed=3)
    # bitwise deterministic from call to call
    mq = _mq()
    g = synth.rng(3)
    data = synth.weight_bytes(g, synth.Q4_K, 512, 3584)
    x = synth.activations(g, 2048, 3584)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), 512, 3584)
    xd = dev(x)
    ya = run(mq.mq_gemm, xd, h, 2048, 512).cpu().numpy()
    yb = run(mq.mq_gemm, xd, h, 2048, 512).cpu().numpy()
    assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))
    assert np.array_equal(ya.view(np.uint32), y1.view(np.uint32))


def test_one_hot_identity(orc):
    """X = identity rows: every output is one product W[n,k]*1, exact in f32,
    so Y must equal the oracle's decoded W^T bit for bit (K-padded cache)."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(11)
    N, K = 384, 1024
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    x = np.eye(K, dtype=np.float16)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    y = run(mq.mq_gemm, dev(x), h, K, N).cpu().numpy()
    W = orc.f16_to_f32(orc.decode_matrix(synth.Q4_K, data, N, K))
    assert np.array_equal(y, W.T)
    del torch


@pytest.mark.parametrize("workload", ["qwen2.5-7b_layer", "llama3.1-8b_layer", "q8_0_pair"])
def test_full_size_sampled(orc, workload):
    """Every GEMM of the workload at its full size, M as in the workload,
    checked at ~2000 sampled outputs (corners and tile edges included)."""
    mq = _mq()
    weights, xs = synth.workload(workload, seed=0)
    for M in synth.WORKLOADS[workload][1]:
        for w in weights:
            x = xs[w.K][:M]
            h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
            y = run(mq.mq_gemm, dev(x), h, M, w.N).cpu().numpy()
            mi, ni = sample_indices(M, w.N, 2000, seed=w.N + M)
            W = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
            ref = orc.gemm_f64_sampled(x.view(np.uint16), W, mi, ni)
            assert_gemm_close(y[mi, ni], ref, f"{workload} {w.name} M={M}")
            assert np.all(np.isfinite(y))
            h.release()


def test_matches_cublas_on_cache(orc):
    """Off-path cross-check: cuBLAS (torch.matmul) on the same f16 cache."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(21)
    N, K, M = 1024, 2048, 256
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    x = dev(synth.activations(g, M, K))
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    y = run(mq.mq_gemm, x, h, M, N)
    wc = h.cache_tensor()[:, :K]
    yc = torch.matmul(x.float(), wc.float().t())
    rel = (torch.linalg.norm(y - yc) / torch.linalg.norm(yc)).item()
    assert rel < 1e-5, rel
