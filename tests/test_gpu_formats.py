"""Q4_0, Q5_0, Q5_1 and Q5_K through every path (load-time decode into the
cache, cached GEMM, fused dequant-in-GEMM on both raw-read paths) against
the oracle.

Decodes are compared bit for bit: each block definition fixes one f16 value
per element.  The one-hot identity (X = identity rows, so Y = W^T exactly in
f32) makes the fused path's on-chip decode observable.  GEMMs are compared
with the oracle's f64 result within the shared tolerance.
"""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, check_cache, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu

NEW = [synth.Q4_0, synth.Q5_0, synth.Q5_1, synth.Q5_K]


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


def test_more_formats_cache_bit_exact(orc):
    """Every weight of the more-formats workload (each format at the 7B gate
    18944 x 3584 and down 3584 x 18944 shapes) decodes bit for bit."""
    weights, _ = synth.workload("more_formats", seed=0, max_m=1)
    assert sorted({w.qtype for w in weights}) == sorted(NEW)
    for w in weights:
        want = w.K + 64 if (2 * w.K) % 2048 == 0 else w.K
        check_cache(orc, w, expect_ldk=want)


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q4_0, 1, 32), (synth.Q4_0, 4, 40), (synth.Q4_0, 1000, 24), (synth.Q4_0, 257, 96),
    (synth.Q5_0, 1, 32), (synth.Q5_0, 4, 40), (synth.Q5_0, 333, 96),
    (synth.Q5_1, 1, 32), (synth.Q5_1, 12, 56), (synth.Q5_1, 129, 160),
    (synth.Q5_K, 1, 256), (synth.Q5_K, 3, 256), (synth.Q5_K, 8, 896),    # rows starting mid-block
    (synth.Q5_K, 66, 128), (synth.Q5_K, 5, 512), (synth.Q5_K, 33, 2304),
])
def test_ragged_streams(orc, qtype, N, K):
    g = synth.rng(N * 1000 + K + qtype)
    check_cache(orc, synth.Weight("w", qtype, N, K, synth.weight_bytes(g, qtype, N, K)))


@pytest.mark.parametrize("qtype", NEW)
def test_kpad_and_row_stride(orc, qtype):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(40 + qtype)
    w = synth.Weight("w", qtype, 256, 1024, synth.weight_bytes(g, qtype, 256, 1024))
    check_cache(orc, w, expect_ldk=1088)
    check_cache(orc, w, flags=mq.MQ_REG_NO_KPAD, expect_ldk=1024)
    N, K, ldo = 96, 1280, 1352
    data = synth.weight_bytes(g, qtype, N, K)
    out = torch.full((N, ldo), -7.0, dtype=torch.float16, device="cuda")
    mq.mq_dequantize(qtype, dev(data), N, K, out, ldo)
    mq.mq_stream_status()
    o = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(o[:, :K], orc.decode_matrix(qtype, data, N, K))
    assert np.all(out[:, K:].cpu().numpy() == -7.0), "columns past K must be left untouched"


def test_signed_zero_and_subnormals(orc):
    """Blocks whose decoded values include -0.0 and f16 subnormals."""
    from oracle_pins import MINUS_ONE, ONE, q40_bytes, q50_bytes, q51_bytes, q5k_bytes
    cases = [
        (synth.Q4_0, np.concatenate([q40_bytes(MINUS_ONE, [0x88] * 16),                 # d * 0 = -0
                                     q40_bytes(0x0001, list(range(0, 256, 16)))])),     # k * 2^-24
        (synth.Q5_0, np.concatenate([q50_bytes(MINUS_ONE, 0xFFFFFFFF, [0x00] * 16),     # q = 16
                                     q50_bytes(0x0003, 0x12345678, list(range(16)))])),
        (synth.Q5_1, np.concatenate([q51_bytes(MINUS_ONE, 0x8000, 0, [0] * 16),         # -1*0 + -0
                                     q51_bytes(0x0001, 0x0002, 0xA5A5A5A5, list(range(16)))])),
        (synth.Q5_K, np.concatenate([q5k_bytes(MINUS_ONE, ONE, [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1],
                                               [0] * 32, [0] * 128),
                                     q5k_bytes(0x0001, 0x0001, list(range(1, 13)), list(range(32)),
                                               list(range(128)))])),
    ]
    for qtype, data in cases:
        qk, _ = synth.BLOCK[qtype]
        check_cache(orc, synth.Weight("w", qtype, 2, qk, data))
        ref = orc.decode(qtype, data)
        assert np.any(ref == 0x8000), synth.TYPE_NAME[qtype]
        assert np.any(((ref & 0x7C00) == 0) & ((ref & 0x3FF) != 0)), synth.TYPE_NAME[qtype]


@pytest.mark.parametrize("qtype", NEW)
@pytest.mark.parametrize("N,K,M", [(200, 768, 5), (384, 512, 130), (128, 4096, 33)])
def test_cached_gemm(orc, qtype, N, K, M):
    mq = _mq()
    g = synth.rng(N + K + M + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    y = run(mq.mq_gemm, dev(x), h, M, N)
    assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      f"cached {synth.TYPE_NAME[qtype]} {N}x{K} M={M}")
    h.release()


@pytest.mark.parametrize("qtype", NEW)
@pytest.mark.parametrize("N,K", [(256, 1024), (200, 768), (130, 640), (64, 576)])
def test_one_hot_fused_equals_decode(orc, qtype, N, K, monkeypatch):
    """Block-aligned rows (K % 256 == 0) go through the row tensor maps and,
    with MQ_RAW_TMA=0, through the per-row bulk copies; K = 640 / 576 rows
    start inside Q5_K blocks and always take the bulk path.  Every path
    must decode to the oracle's values, and cached == fused."""
    mq = _mq()
    g = synth.rng(N * 3 + K + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    q = dev(data)
    W = orc.f16_to_f32(orc.decode_matrix(qtype, data, N, K))
    x = dev(np.eye(K, dtype=np.float16))
    h = mq.mq_register_weight(qtype, q, N, K)
    monkeypatch.setenv("MQ_RAW_TMA", "0")
    h_bulk = mq.mq_register_weight(qtype, q, N, K, flags=mq.MQ_REG_NO_CACHE)
    monkeypatch.delenv("MQ_RAW_TMA")
    yf = run(mq.mq_gemm_fused, x, h, K, N)
    assert np.array_equal(yf, W.T), "fused on-chip decode differs from the oracle's decode"
    assert np.array_equal(run(mq.mq_gemm_fused, x, h_bulk, K, N), W.T), "bulk-copy raw path differs"
    assert np.array_equal(run(mq.mq_gemm, x, h, K, N), yf), "fused and cached paths decode differently"


@pytest.mark.parametrize("qtype", NEW)
@pytest.mark.parametrize("M", [1, 32, 33, 129])
def test_fused_shapes(orc, qtype, M):
    mq = _mq()
    N, K = 320, 1536
    g = synth.rng(M * 31 + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K, flags=mq.MQ_REG_NO_CACHE)
    y = run(mq.mq_gemm_fused, dev(x), h, M, N)
    assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      f"fused {synth.TYPE_NAME[qtype]} M={M}")


def test_more_formats_full_size_sampled(orc):
    """Each more-formats weight at full size: fused at M = 32 (the small
    workload M; down runs split-K) and cached at M = 2048, ~1500 sampled
    outputs each."""
    mq = _mq()
    weights, xs = synth.workload("more_formats", seed=0)
    mq.mq_reserve_workspace(64 << 20)
    for w in weights:
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
        W = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
        for M, fn in ((32, mq.mq_gemm_fused), (2048, mq.mq_gemm)):
            x = xs[w.K][:M]
            y = run(fn, dev(x), h, M, w.N)
            assert np.all(np.isfinite(y))
            mi, ni = sample_indices(M, w.N, 1500, seed=M + w.qtype)
            ref = orc.gemm_f64_sampled(x.view(np.uint16), W, mi, ni)
            assert_gemm_close(y[mi, ni], ref, f"{w.name} M={M}")
        h.release()
