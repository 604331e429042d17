"""Float weights (F32 / F16 / BF16, rows padded by one 128-byte line when an
f16 row is a multiple of 2048 bytes) and the per-call scratch mode
(mq_gemm_scratch), against the oracle.

The f16 form of a float weight is fixed element by element (round to
nearest even; F16 is the element itself), so the cache is compared bit for
bit.  The scratch mode decodes into caller memory and runs the cached GEMM
on it, so its Y must equal mq_gemm's bit for bit.
"""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, check_cache, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu

FLOATS = [synth.F32, synth.F16, synth.BF16]
ALL_TYPES = FLOATS + [synth.Q4_0, synth.Q5_0, synth.Q5_1, synth.Q8_0, synth.Q4_K, synth.Q5_K, synth.Q6_K]


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


@pytest.mark.parametrize("qtype", FLOATS)
@pytest.mark.parametrize("N,K", [(64, 4096), (33, 3584), (5, 8), (3, 1048), (17, 2048)])
def test_float_cache_bit_exact(orc, qtype, N, K):
    g = synth.rng(N + K + qtype)
    w = synth.Weight("w", qtype, N, K, synth.weight_bytes(g, qtype, N, K))
    want = K + 64 if (2 * K) % 2048 == 0 else K
    check_cache(orc, w, expect_ldk=want)
    mq = _mq()
    check_cache(orc, w, flags=mq.MQ_REG_NO_KPAD, expect_ldk=K)
    check_cache(orc, w, flags=mq.MQ_REG_KPAD, expect_ldk=K + 64)


def test_f16_read_in_place(orc):
    """An F16 weight whose rows need no padding is its own cache: no copy,
    and releasing the handle leaves the caller's tensor alone."""
    mq = _mq()
    g = synth.rng(3)
    N, K = 96, 3584
    data = synth.weight_bytes(g, synth.F16, N, K)
    q = dev(data)
    for flags in (0, mq.MQ_REG_NO_CACHE):
        h = mq.mq_register_weight(synth.F16, q, N, K, flags=flags)
        n, k, ldk, ptr = h.info()
        assert (ldk, ptr) == (K, q.data_ptr())
        h.release()
    assert np.array_equal(q.cpu().numpy(), data), "release must not touch the caller's weight"
    h = mq.mq_register_weight(synth.F16, q, N, K, flags=mq.MQ_REG_KPAD)
    assert h.info()[3] != q.data_ptr() and h.info()[2] == K + 64   # padded copy
    h.release()


def test_float_registration_errors():
    import ctypes
    mq = _mq()
    L = mq._lib()
    g = synth.rng(4)
    for qt in (synth.F32, synth.BF16):
        q = dev(synth.weight_bytes(g, qt, 8, 64))
        out = ctypes.c_void_p()
        assert L.mq_register_weight(qt, q.data_ptr(), 8, 64, mq.MQ_REG_NO_CACHE, None, ctypes.byref(out)) == -1
        assert b"MQ_REG_NO_CACHE" in L.mq_last_error_detail()


def test_float_nan_inf(orc):
    """NaN elements stay NaN (payload not compared), infinities and values
    past the f16 range become infinities, the rest bit for bit."""
    torch = torch_cuda()
    mq = _mq()
    f32 = np.array([np.nan, np.inf, -np.inf, 70000.0, -65520.0, 65519.0, 1e-8, -0.0] * 4, dtype="<f4")
    bf = (f32.view("<u4") >> 16).astype("<u2")
    for qt, raw in ((synth.F32, f32.view(np.uint8)), (synth.BF16, bf.view(np.uint8))):
        h = mq.mq_register_weight(qt, dev(raw), 4, 8)
        mq.mq_stream_status()
        got = h.cache_tensor().cpu().numpy().view(np.uint16)[:, :8].reshape(-1)
        ref = orc.decode(qt, raw)
        nan_g = ((got & 0x7C00) == 0x7C00) & ((got & 0x3FF) != 0)
        nan_r = ((ref & 0x7C00) == 0x7C00) & ((ref & 0x3FF) != 0)
        assert np.array_equal(nan_g, nan_r) and nan_r.sum() == 4
        assert np.array_equal(got[~nan_r], ref[~nan_r])
        h.release()
    del torch


@pytest.mark.parametrize("qtype", FLOATS)
@pytest.mark.parametrize("M", [1, 130])
def test_float_gemms(orc, qtype, M):
    """mq_gemm, mq_gemm_fused and mq_gemm_auto on a float weight are the
    same cached GEMM: equal to each other and within tolerance of the
    oracle; a group of float weights too."""
    mq = _mq()
    N, K = 256, 2048
    g = synth.rng(M + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    data2 = synth.weight_bytes(g, qtype, 128, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    h2 = mq.mq_register_weight(qtype, dev(data2), 128, K)
    xd = dev(x)
    yc = run(mq.mq_gemm, xd, h, M, N)
    assert np.array_equal(run(mq.mq_gemm_fused, xd, h, M, N), yc)
    assert np.array_equal(run(mq.mq_gemm_auto, xd, h, M, N), yc)
    assert_gemm_close(yc, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      f"{synth.TYPE_NAME[qtype]} M={M}")
    torch = torch_cuda()
    ys = [torch.empty((M, n), dtype=torch.float32, device="cuda") for n in (N, 128)]
    mq.mq_gemm_grouped(xd, [h, h2], ys, M)
    mq.mq_stream_status()
    assert_gemm_close(ys[0].cpu().numpy(), orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      "group member 0")
    assert_gemm_close(ys[1].cpu().numpy(), orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data2, 128, K)),
                      "group member 1")


def test_float_one_hot(orc):
    mq = _mq()
    g = synth.rng(12)
    N, K = 192, 1024
    for qt in FLOATS:
        data = synth.weight_bytes(g, qt, N, K)
        h = mq.mq_register_weight(qt, dev(data), N, K)
        y = run(mq.mq_gemm, dev(np.eye(K, dtype=np.float16)), h, K, N)
        assert np.array_equal(y, orc.f16_to_f32(orc.decode_matrix(qt, data, N, K)).T)
        h.release()


def test_float_layer_padded_equals_unpadded(orc):
    """The Llama-3.1-8B-shaped float weights at M = 512: the padded copy
    (default) and the unpadded layout give the same Y bit for bit (only the
    row stride differs), within tolerance of the oracle at sampled outputs."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = synth.workload("float_layer", seed=0)
    M = 512
    for w in weights:
        q = dev(w.data)
        hp = mq.mq_register_weight(w.qtype, q, w.N, w.K)
        hu = mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=mq.MQ_REG_NO_KPAD)
        assert hp.info()[2] == w.K + 64 and hu.info()[2] == w.K
        x = dev(xs[w.K][:M])
        yp = run(mq.mq_gemm, x, hp, M, w.N)
        yu = run(mq.mq_gemm, x, hu, M, w.N)
        assert np.array_equal(yp.view(np.uint32), yu.view(np.uint32)), w.name
        mi, ni = sample_indices(M, w.N, 1500, seed=w.N)
        ref = orc.gemm_f64_sampled(xs[w.K][:M].view(np.uint16), orc.decode_matrix(w.qtype, w.data, w.N, w.K), mi, ni)
        assert_gemm_close(yp[mi, ni], ref, w.name)
        hp.release()
        hu.release()
    del torch


@pytest.mark.parametrize("qtype", ALL_TYPES)
def test_scratch_equals_cached(orc, qtype):
    """mq_gemm_scratch decodes into the caller's scratch (which then holds
    the oracle's decode in the cache layout) and gives mq_gemm's Y bit for
    bit; a handle without a cache works too."""
    torch = torch_cuda()
    mq = _mq()
    N, K, M = 320, 2048, 200
    g = synth.rng(50 + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    x = dev(synth.activations(g, M, K))
    q = dev(data)
    h = mq.mq_register_weight(qtype, q, N, K)
    ldk = h.info()[2]
    scratch = torch.full((N, ldk), -3.0, dtype=torch.float16, device="cuda")
    yc = run(mq.mq_gemm, x, h, M, N)
    ys = run(lambda xx, hh, yy, mm: mq.mq_gemm_scratch(xx, hh, yy, scratch, mm), x, h, M, N)
    assert np.array_equal(ys.view(np.uint32), yc.view(np.uint32))
    got = scratch.cpu().numpy().view(np.uint16)[:, :K]
    assert np.array_equal(got, orc.decode_matrix(qtype, data, N, K))
    if qtype not in (synth.F32, synth.BF16):
        hn = mq.mq_register_weight(qtype, q, N, K, flags=mq.MQ_REG_NO_CACHE)
        if hn.info()[2] == ldk:
            yn = run(lambda xx, hh, yy, mm: mq.mq_gemm_scratch(xx, hh, yy, scratch, mm), x, hn, M, N)
            assert np.array_equal(yn.view(np.uint32), yc.view(np.uint32))
        hn.release()
    h.release()


def test_scratch_errors():
    import ctypes
    torch = torch_cuda()
    mq = _mq()
    L = mq._lib()
    g = synth.rng(8)
    N, K, M = 128, 1024, 8
    h = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, N, K)), N, K)
    ldk = h.info()[2]
    x = dev(synth.activations(g, M, K))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.empty((N, ldk), dtype=torch.float16, device="cuda")
    assert L.mq_gemm_scratch(x.data_ptr(), h.handle, y.data_ptr(), M, s.data_ptr(), 2 * N * ldk - 2, None) == -3
    assert L.mq_gemm_scratch(x.data_ptr(), h.handle, y.data_ptr(), M, None, 2 * N * ldk, None) == -1
    assert L.mq_gemm_scratch(x.data_ptr(), h.handle, y.data_ptr(), M, s.data_ptr() + 2, 2 * N * ldk, None) == -4
    mq.mq_stream_status()
    h.release()
