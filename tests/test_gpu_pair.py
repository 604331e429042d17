"""Multicast CTA pairs (the default below 256-token tiles; MQ_PAIR=0 turns
them off): clusters of two CTAs that share each token tile,
multicast into both.  Every case runs with pairs on and off; both must
match the oracle, and where the two plans split K the same way (no split)
the outputs must agree bit for bit (each tile's arithmetic is unchanged).
Covers an odd number of weight-row tiles (a phantom tile in the last
pair), grouped launches, split-K tails, M tails and the e4m3 kernel."""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _run(monkeypatch, pair, fn):
    # MQ_2SM=0: 256-token tiles use the multicast pairs too (2-SM MMAs, the
    # default there, have their own tests)
    monkeypatch.setenv("MQ_PAIR", "1" if pair else "0")
    monkeypatch.setenv("MQ_2SM", "0")
    out = fn()
    monkeypatch.delenv("MQ_PAIR")
    monkeypatch.delenv("MQ_2SM")
    return out


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q4_K, 384, 1024, 300),     # 3 weight-row tiles: the second pair has a phantom tile
    (synth.Q4_K, 512, 3584, 2048),    # 4 x 8 tiles: split-K tail
    (synth.Q6_K, 256, 768, 100),      # BN = 128, M tail
    (synth.Q8_0, 1024, 512, 64),      # BN = 64
    (synth.Q4_K, 3584, 3584, 2048),   # the 7B o shape
])
def test_pair_matches_oracle(orc, monkeypatch, qtype, N, K, M):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(N + K + M)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K)
    xd = dev(x)
    mq.mq_reserve_workspace(64 << 20)

    def call():
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        mq.mq_gemm(xd, h, y, M)
        mq.mq_stream_status()
        return y.cpu().numpy()
    y1, y0 = _run(monkeypatch, True, call), _run(monkeypatch, False, call)
    W = orc.decode_matrix(qtype, data, N, K)
    ref = orc.gemm_f64(x.view(np.uint16), W) if M * N <= 4_000_000 else None
    if ref is not None:
        assert_gemm_close(y1, ref, "pair")
    assert_gemm_close(y1, y0, "pair vs single")
    h.release()


def test_pair_group_and_e4m3(orc, monkeypatch):
    """q|k|v-like group (4608 rows = 36 tiles) and gate-like e4m3 weights."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(21)
    K, M = 1024, 512
    shapes = [(synth.Q4_K, 640), (synth.Q4_K, 256), (synth.Q4_K, 256)]
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in shapes]
    hs = [mq.mq_register_weight(qt, dev(d), N, K, flags=mq.MQ_REG_E4M3) for (qt, N), d in zip(shapes, datas)]
    x = synth.activations(g, M, K)
    xd = dev(x)
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(xd, x8, sx)

    def grouped():
        ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in shapes]
        mq.mq_gemm_grouped(xd, hs, ys, M)
        mq.mq_stream_status()
        return [y.cpu().numpy() for y in ys]

    def grouped8():
        ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in shapes]
        mq.mq_gemm_e4m3_grouped(x8, sx, hs, ys, M)
        mq.mq_stream_status()
        return [y.cpu().numpy() for y in ys]
    for (qt, N), d, y in zip(shapes, datas, _run(monkeypatch, True, grouped)):
        assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qt, d, N, K)), f"group N={N}")
    X8, SX = x8.cpu().numpy(), sx.cpu().numpy()
    for h, y in zip(hs, _run(monkeypatch, True, grouped8)):
        codes, scales = h.e4m3_tensors()
        ref = orc.gemm_e4m3_f64(X8, SX, codes.cpu().numpy()[:, :K], scales.cpu().numpy())
        del codes, scales
        assert_gemm_close(y, ref, "e4m3 group")
    for h in hs:
        h.release()
