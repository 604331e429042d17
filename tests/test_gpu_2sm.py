"""2-SM MMAs (the default for 256-token tiles; set explicitly here): a CTA
pair computes 256 x 256 tiles with
tcgen05.mma.cta_group::2, each CTA staging its own weight rows and half of
the tokens.  Every case is checked against the oracle: an odd count of
weight-row tiles (phantom tile), split-K tails, M tails inside a 256-token
tile, a grouped launch, and the e4m3 kernel."""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


@pytest.fixture
def two_sm(monkeypatch):
    monkeypatch.setenv("MQ_2SM", "1")
    yield
    monkeypatch.delenv("MQ_2SM")


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q4_K, 256, 512, 256),      # one pair tile
    (synth.Q4_K, 384, 1024, 300),     # phantom tile, M tail
    (synth.Q6_K, 512, 3584, 2048),    # split-K tail
    (synth.Q8_0, 3584, 1024, 700),
])
def test_2sm_matches_oracle(orc, two_sm, qtype, N, K, M):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N + K + M + 7)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    mq.mq_reserve_workspace(64 << 20)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mq.mq_gemm(dev(x), h, y, M)
    mq.mq_stream_status()
    assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      f"2sm {synth.TYPE_NAME[qtype]} {N}x{K} M={M}")
    h.release()


def test_2sm_group_and_e4m3(orc, two_sm):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(33)
    K, M = 1024, 512
    shapes = [(synth.Q4_K, 640), (synth.Q4_K, 256), (synth.Q4_K, 256)]
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in shapes]
    hs = [mq.mq_register_weight(qt, dev(d), N, K, flags=mq.MQ_REG_E4M3) for (qt, N), d in zip(shapes, datas)]
    x = synth.activations(g, M, K)
    xd = dev(x)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in shapes]
    mq.mq_gemm_grouped(xd, hs, ys, M)
    mq.mq_stream_status()
    for (qt, N), d, y in zip(shapes, datas, ys):
        assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qt, d, N, K)),
                          f"group N={N}")
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(xd, x8, sx)
    ys8 = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in shapes]
    mq.mq_gemm_e4m3_grouped(x8, sx, hs, ys8, M)
    mq.mq_stream_status()
    X8, SX = x8.cpu().numpy(), sx.cpu().numpy()
    for h, y in zip(hs, ys8):
        codes, scales = h.e4m3_tensors()
        ref = orc.gemm_e4m3_f64(X8, SX, codes.cpu().numpy()[:, :K], scales.cpu().numpy())
        del codes, scales
        assert_gemm_close(y.cpu().numpy(), ref, "e4m3 group")
    for h in hs:
        h.release()


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q8_0, 512, 64, 1024),      # one K step per unit: the first stages span six units
    (synth.Q4_K, 8192, 256, 2048),    # four K steps, ~3.4 units per pair: accumulator hand-off
    (synth.Q8_0, 512, 1056, 512),     # last K step half past K (zero-filled boxes, full byte count)
    (synth.Q8_0, 768, 1024, 257),     # second token tile holds one token
    (synth.F16, 256, 4096, 256),      # rows padded to K + 64
    (synth.BF16, 640, 1024, 512),     # padded rows, odd pair-row count (phantom tile)
])
def test_2sm_edge_shapes(orc, two_sm, qtype, N, K, M):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N * 3 + K + M)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    mq.mq_reserve_workspace(64 << 20)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mq.mq_gemm(dev(x), h, y, M)
    mq.mq_stream_status()
    assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qtype, data, N, K)),
                      f"2sm {synth.TYPE_NAME[qtype]} {N}x{K} M={M}")
    h.release()


@pytest.mark.parametrize("N,K,M", [(512, 1056, 512), (1280, 128, 768)])
def test_2sm_e4m3_k_tails(orc, two_sm, N, K, M):
    """The e4m3 kernel's 128-element K steps: a partial last step (1056 =
    8.25 steps) and a single step per unit."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N + K * 5 + M)
    data = synth.weight_bytes(g, synth.Q8_0, N, K)
    h = mq.mq_register_weight(synth.Q8_0, dev(data), N, K, flags=mq.MQ_REG_E4M3)
    xd = dev(synth.activations(g, M, K))
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(xd, x8, sx)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mq.mq_gemm_e4m3(x8, sx, h, y, M)
    mq.mq_stream_status()
    codes, scales = h.e4m3_tensors()
    ref = orc.gemm_e4m3_f64(x8.cpu().numpy(), sx.cpu().numpy(), codes.cpu().numpy()[:, :K], scales.cpu().numpy())
    del codes, scales
    assert_gemm_close(y.cpu().numpy(), ref, f"e4m3 2sm {N}x{K} M={M}")
    h.release()
