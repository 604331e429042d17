"""The cached and 8-bit GEMMs' two output paths give the same Y bit for bit:
TMA stores of staged 128-row boxes (the default, clipped at the output's
extents) and plain per-lane stores (MQ_TMA_Y=0, and what an output whose
N % 4 != 0 always takes: its row stride is no TMA stride; Y itself must be
16-byte aligned for every GEMM entry point).  Shapes cover each kernel form
(2-SM pairs at 256-token tiles, multicast pairs at 128, single CTAs at 32),
ragged token tails inside a box, a grouped launch and a row count that is
not a multiple of 4; one case is also held against the f64 oracle."""
import os

import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _with_tma_y(on, fn):
    old = os.environ.get("MQ_TMA_Y")
    os.environ["MQ_TMA_Y"] = "1" if on else "0"
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["MQ_TMA_Y"]
        else:
            os.environ["MQ_TMA_Y"] = old


def _run(torch, mq, x, h, M, N):
    """mq_gemm into a fresh NaN-filled Y."""
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mq.mq_gemm(x, h, y, M)
    mq.mq_stream_status()
    return y.cpu().numpy()


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q4_K, 512, 1024, 300),   # 256-token 2-SM tiles; 44-token tail (a box cut at M)
    (synth.Q4_K, 384, 1024, 100),   # 128-token tiles (CTA pairs); tail of 100
    (synth.Q6_K, 256, 512, 20),     # 32-token tiles, single CTAs; box cut at 20 tokens
    (synth.Q8_0, 130, 1024, 300),   # N % 4 != 0: plain stores either way
    (synth.Q4_K, 1024, 2048, 2048),  # full waves, no tails
])
def test_tma_store_matches_plain_stores(qtype, N, K, M):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N + K + M)
    h = mq.mq_register_weight(qtype, dev(synth.weight_bytes(g, qtype, N, K)), N, K)
    x = dev(synth.activations(g, M, K))
    y_tma = _with_tma_y(True, lambda: _run(torch, mq, x, h, M, N))
    y_plain = _with_tma_y(False, lambda: _run(torch, mq, x, h, M, N))
    assert np.all(np.isfinite(y_tma)), "TMA-stored output has unwritten (NaN) entries"
    assert np.array_equal(y_tma.view(np.uint32), y_plain.view(np.uint32))
    h.release()


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q8_0, 132, 1024, 300),   # a 128-row box cut at row 132
    (synth.Q4_0, 4, 1024, 257),     # a 4-row weight: one box, 124 rows clipped
])
def test_tma_store_partial_row_tiles(orc, qtype, N, K, M):
    """Whole tiles (split-K off, so the few tiles are not split over K) whose
    last 128-row box runs past N: the TMA store must clip at row N, equal the
    plain stores bit for bit and match the oracle."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N + M)
    data = synth.weight_bytes(g, qtype, N, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    xh = synth.activations(g, M, K)
    x = dev(xh)
    old = os.environ.get("MQ_SPLITK")
    os.environ["MQ_SPLITK"] = "0"
    try:
        y_tma = _with_tma_y(True, lambda: _run(torch, mq, x, h, M, N))
        y_plain = _with_tma_y(False, lambda: _run(torch, mq, x, h, M, N))
    finally:
        if old is None:
            del os.environ["MQ_SPLITK"]
        else:
            os.environ["MQ_SPLITK"] = old
    assert np.all(np.isfinite(y_tma))
    assert np.array_equal(y_tma.view(np.uint32), y_plain.view(np.uint32))
    ref = orc.gemm_f64(xh.view(np.uint16), orc.decode_matrix(qtype, data, N, K))
    assert_gemm_close(y_tma, ref, f"{synth.TYPE_NAME[qtype]} N={N} M={M}, TMA-stored")
    h.release()


def test_grouped_tma_store_matches_plain_and_oracle(orc):
    """Two members in one grouped launch (each with its own output map); the
    second member is also held against the f64 oracle on sampled outputs."""
    torch = torch_cuda()
    mq = _mq()
    K, M = 1024, 300
    Ns = (256, 512)
    g = synth.rng(9)
    datas = [synth.weight_bytes(g, synth.Q4_K, n, K) for n in Ns]
    hs = [mq.mq_register_weight(synth.Q4_K, dev(d), n, K) for d, n in zip(datas, Ns)]
    xh = synth.activations(g, M, K)
    x = dev(xh)

    def run():
        ys = [torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda") for n in Ns]
        mq.mq_gemm_grouped(x, hs, ys, M)
        mq.mq_stream_status()
        return [y.cpu().numpy() for y in ys]

    ys_tma = _with_tma_y(True, run)
    ys_plain = _with_tma_y(False, run)
    for a, b in zip(ys_tma, ys_plain):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    N = Ns[1]
    mi, ni = sample_indices(M, N, 1500, seed=3)
    ref = orc.gemm_f64_sampled(xh.view(np.uint16), orc.decode_matrix(synth.Q4_K, datas[1], N, K), mi, ni)
    assert_gemm_close(ys_tma[1][mi, ni], ref, "grouped member 1, TMA-stored")
    for h in hs:
        h.release()


def test_e4m3_tma_store_matches_plain_stores():
    torch = torch_cuda()
    mq = _mq()
    N, K, M = 512, 1024, 300
    g = synth.rng(13)
    h = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, N, K)), N, K,
                              flags=mq.MQ_REG_E4M3)
    x = dev(synth.activations(g, M, K))
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(x, x8, sx)

    def run():
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        mq.mq_gemm_e4m3(x8, sx, h, y, M)
        mq.mq_stream_status()
        return y.cpu().numpy()

    a = _with_tma_y(True, run)
    b = _with_tma_y(False, run)
    assert np.all(np.isfinite(a))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    h.release()
