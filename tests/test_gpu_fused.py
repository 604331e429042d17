"""Fused dequant-in-GEMM and the M gate against the oracle.

The one-hot identity makes the fused path's on-chip decode observable:
with X = identity rows every output is a single product 1 * W[n,k], exact in
f32, so Y must equal the oracle's decoded W^T -- the same f16 values the
cache holds ("05 · 8p", section 3.3: fused and cached must round the same
way).  The rest compares Y with the oracle's f64 GEMM within tolerance.
"""
import os

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
    return y.cpu().numpy()


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q4_K, 896, 896),     # the 896x896 workload: odd rows start mid-block
    (synth.Q4_K, 256, 1024),
    (synth.Q6_K, 200, 768),     # 210-byte blocks, 2-byte aligned; N tail
    (synth.Q6_K, 64, 576),      # K % 256 != 0: chunks straddle blocks
    (synth.Q8_0, 130, 512),     # 34-byte blocks
    (synth.Q8_0, 64, 448),
])
def test_one_hot_fused_equals_decode(orc, qtype, N, K):
    mq = _mq()
    g = synth.rng(N + K)
    data = synth.weight_bytes(g, qtype, N, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    x = dev(np.eye(K, dtype=np.float16))
    W = orc.f16_to_f32(orc.decode_matrix(qtype, data, N, K))
    yf = run(mq.mq_gemm_fused, x, h, K, N)
    assert np.array_equal(yf, W.T), "fused on-chip decode differs from the oracle's decode"
    yc = run(mq.mq_gemm, x, h, K, N)
    assert np.array_equal(yc, yf), "fused and cached paths decode differently"


def test_c0_fused(orc):
    weights, xs = synth.workload("q4k_896", seed=0)
    w = weights[0]
    x = xs[w.K]
    mq = _mq()
    h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K, flags=mq.MQ_REG_NO_CACHE)
    assert h.cache_tensor() is None
    y = run(mq.mq_gemm_fused, dev(x), h, x.shape[0], w.N)
    y_ref = orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(w.qtype, w.data, w.N, w.K))
    assert_gemm_close(y, y_ref, "q4k_896 fused")


@pytest.mark.parametrize("M", [1, 7, 32, 33, 100, 129, 300])
@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K, synth.Q8_0])
def test_fused_shapes(orc, qtype, M):
    mq = _mq()
    N, K = 320, 1536
    g = synth.rng(M * 31 + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K, flags=mq.MQ_REG_NO_CACHE)
    y = run(mq.mq_gemm_fused, dev(x), h, M, N)
    y_ref = orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K))
    assert_gemm_close(y, y_ref, f"fused {synth.TYPE_NAME[qtype]} M={M}")


def test_small_m_sweep_sampled(orc):
    """gate/up (Q4_K 18944x3584) and down (Q6_K 3584x18944) of the 7B layer
    through the fused path at every M of the sweep, sampled outputs; down at
    small M runs split-K (28 row tiles)."""
    mq = _mq()
    weights, xs = synth.workload("small_m_sweep", seed=0)
    for w in weights:
        if w.name == "up":
            continue
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K, flags=mq.MQ_REG_NO_CACHE)
        W = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
        for M in synth.WORKLOADS["small_m_sweep"][1]:
            x = xs[w.K][:M]
            y = run(mq.mq_gemm_fused, dev(x), h, M, w.N)
            mi, ni = sample_indices(M, w.N, 1500, seed=M)
            ref = orc.gemm_f64_sampled(x.view(np.uint16), W, mi, ni)
            assert_gemm_close(y[mi, ni], ref, f"fused {w.name} M={M}")
            assert np.all(np.isfinite(y))
        h.release()


def test_fused_deterministic_split():
    mq = _mq()
    g = synth.rng(77)
    N, K, M = 3584, 18944, 16
    data = synth.weight_bytes(g, synth.Q6_K, N, K)
    h = mq.mq_register_weight(synth.Q6_K, dev(data), N, K, flags=mq.MQ_REG_NO_CACHE)
    x = dev(synth.activations(g, M, K))
    a = run(mq.mq_gemm_fused, x, h, M, N)
    b = run(mq.mq_gemm_fused, x, h, M, N)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gate_dispatch(orc):
    """mq_gemm_auto: fused below the gate, cached at and above it; both
    within tolerance.  A handle without a cache always goes fused."""
    mq = _mq()
    g = synth.rng(5)
    N, K = 256, 1024
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    x = synth.activations(g, 160, K)
    W = orc.decode_matrix(synth.Q4_K, data, N, K)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    hn = mq.mq_register_weight(synth.Q4_K, dev(data), N, K, flags=mq.MQ_REG_NO_CACHE)
    old = mq.mq_get_m_gate()
    try:
        mq.mq_set_m_gate(100)
        assert mq.mq_get_m_gate() == 100
        for M in (16, 99, 100, 160):
            y_ref = orc.gemm_f64(x[:M].view(np.uint16), W)
            for handle in (h, hn):
                n0 = mq.mq_launch_count()
                y = run(mq.mq_gemm_auto, dev(x[:M]), handle, M, N)
                assert mq.mq_launch_count() > n0
                assert_gemm_close(y, y_ref, f"auto M={M}")
    finally:
        mq.mq_set_m_gate(old)


@pytest.mark.parametrize("qtype,N,K", [(synth.Q4_K, 256, 1024), (synth.Q6_K, 136, 1536), (synth.Q8_0, 128, 768)])
def test_raw_paths_agree(orc, qtype, N, K, monkeypatch):
    """Block-aligned weights are read through row-class tensor maps; with
    MQ_RAW_TMA=0 the same weight takes the per-row bulk-copy path.  Both
    must decode to the oracle's values (one-hot identity)."""
    mq = _mq()
    g = synth.rng(N * 7 + K)
    data = synth.weight_bytes(g, qtype, N, K)
    q = dev(data)
    W = orc.f16_to_f32(orc.decode_matrix(qtype, data, N, K))
    x = dev(np.eye(K, dtype=np.float16))
    h_tma = mq.mq_register_weight(qtype, q, N, K, flags=mq.MQ_REG_NO_CACHE)
    monkeypatch.setenv("MQ_RAW_TMA", "0")
    h_bulk = mq.mq_register_weight(qtype, q, N, K, flags=mq.MQ_REG_NO_CACHE)
    monkeypatch.delenv("MQ_RAW_TMA")
    for h in (h_tma, h_bulk):
        y = run(mq.mq_gemm_fused, x, h, K, N)
        assert np.array_equal(y, W.T)


def test_default_gate_boundary(orc):
    """With the default gate (the measured crossover, 129 tokens) mq_gemm_auto
    launches the fused kernel at M = 128 and the cached kernel at M = 129,
    read from the launch trace; both results within tolerance."""
    torch = torch_cuda()
    mq = _mq()
    if os.environ.get("MQ_M_GATE"):
        pytest.skip("MQ_M_GATE overrides the default gate")
    assert mq.mq_get_m_gate() == 129
    g = synth.rng(17)
    N, K = 384, 1024
    data = synth.weight_bytes(g, synth.Q4_K, N, K)
    h = mq.mq_register_weight(synth.Q4_K, dev(data), N, K)
    W = orc.decode_matrix(synth.Q4_K, data, N, K)
    x = synth.activations(g, 129, K)
    for M, want in ((128, mq.MQ_TRACE_GEMM_FUSED), (129, mq.MQ_TRACE_GEMM_CACHED)):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        mq.mq_trace_enable(True)
        mq.mq_gemm_auto(dev(x[:M]), h, y, M)
        mq.mq_stream_status()
        kinds = {r["kind"] for r in mq.mq_trace_records()}
        mq.mq_trace_enable(False)
        assert kinds == {want}, f"M={M}: trace kinds {kinds}"
        assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x[:M].view(np.uint16), W), f"auto M={M}")
    h.release()
