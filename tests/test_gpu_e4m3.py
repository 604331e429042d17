"""The 8-bit (e4m3) variant against the oracle.

Its own contract: row quantization (codes and scales) is compared bit for
bit -- both sides take the same binary32 steps and the same e4m3 rounding --
and the GEMM against the oracle's exact f64 product of the quantized
operands within the f32-accumulation tolerance (products of two e4m3 values
are exact in f32).  The distance to the f16 result is the quantization
error; it is checked against a loose bound and reported, not asserted
tightly.
"""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def quantize(x16, ld=None, ldo=None):
    """GPU quantization of f16 rows; returns (codes [rows, K], scales)."""
    torch = torch_cuda()
    mq = _mq()
    rows, K = x16.shape
    ld = ld or K
    ldo = ldo or K
    src = torch.zeros((rows, ld), dtype=torch.float16, device="cuda")
    src[:, :K] = dev(x16)
    dst = torch.full((rows, ldo), 0xA5, dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(src[:, :K], dst, sc)
    mq.mq_stream_status()
    d = dst.cpu().numpy()
    if ldo > K:
        assert np.all(d[:, K:] == 0xA5), "columns past K must be left untouched"
    return d[:, :K], sc.cpu().numpy()


@pytest.mark.parametrize("rows,K,ld,ldo", [(37, 3584, None, None), (5, 16, None, None), (64, 1040, 1048, 1056),
                                           (300, 512, None, None)])
def test_quantize_bit_exact(orc, rows, K, ld, ldo):
    g = synth.rng(rows + K)
    x = synth.activations(g, rows, K)
    q, sc = quantize(x, ld, ldo)
    qr, scr = orc.quantize_e4m3_rows(x.view(np.uint16))
    assert np.array_equal(sc.view(np.uint32), scr.view(np.uint32)), "scales differ"
    bad = np.argwhere(q != qr)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0].tolist()}: 0x{q[tuple(bad[0])]:02x} " \
                          f"vs 0x{qr[tuple(bad[0])]:02x}"


def test_quantize_special_rows(orc):
    """All-zero rows, a row whose amax is 448, f16 subnormals, the f16
    maximum, signed zeros, and values that land on e4m3 ties."""
    K = 32
    rows = [np.zeros(K), np.full(K, -0.0), np.linspace(-448, 448, K), np.linspace(-3, 3, K) * 2.0 ** -20,
            np.array([65504.0] + [1.0] * (K - 1)), np.array([1.765625, 1.32421875] + [0.0] * (K - 2)),
            np.array([448.0, 1.0625, 1.1875, 232.0, 464.0 / 2, -0.0] + [0.5] * (K - 6))]
    x = np.array(rows, dtype=np.float16)
    q, sc = quantize(x)
    qr, scr = orc.quantize_e4m3_rows(x.view(np.uint16))
    assert np.array_equal(sc.view(np.uint32), scr.view(np.uint32))
    assert np.array_equal(q, qr)
    assert q[5, 1] == 0x7A   # the binary32 tie that tells RN32(448/amax) from 1/s


@pytest.mark.parametrize("qtype,N,K", [(synth.Q4_K, 384, 1024), (synth.Q6_K, 200, 768), (synth.Q8_0, 136, 2048),
                                       (synth.F16, 256, 4096)])
def test_weight_copy_bit_exact(orc, qtype, N, K):
    """MQ_REG_E4M3 quantizes each cache row: codes and scales equal the
    oracle's quantization of the oracle's decode; pad columns are zero."""
    mq = _mq()
    g = synth.rng(N * K + qtype)
    data = synth.weight_bytes(g, qtype, N, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K, flags=mq.MQ_REG_E4M3)
    mq.mq_stream_status()
    codes, scales = h.e4m3_tensors()
    codes = codes.cpu().numpy()
    qr, scr = orc.quantize_e4m3_rows(orc.decode_matrix(qtype, data, N, K))
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), scr.view(np.uint32))
    assert np.array_equal(codes[:, :K], qr)
    assert codes.shape[1] == (K + 128 if K % 2048 == 0 else K)
    assert np.all(codes[:, K:] == 0)
    h.release()


def _e4m3_case(orc, qtype, N, K, M, seed):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(seed)
    data = synth.weight_bytes(g, qtype, N, K)
    x = synth.activations(g, M, K)
    h = mq.mq_register_weight(qtype, dev(data), N, K, flags=mq.MQ_REG_E4M3)
    xd = dev(x)
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(xd, x8, sx)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mq.mq_gemm_e4m3(x8, sx, h, y, M)
    mq.mq_stream_status()
    codes, scales = h.e4m3_tensors()   # views of library memory: copy before release
    W8 = codes.cpu().numpy()[:, :K]
    SW = scales.cpu().numpy()
    Y = y.cpu().numpy()
    yf = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mq.mq_gemm(xd, h, yf, M)
    mq.mq_stream_status()
    del codes, scales
    h.release()
    return x8.cpu().numpy(), sx.cpu().numpy(), W8, SW, Y, yf.cpu().numpy()


@pytest.mark.parametrize("M", [1, 33, 130, 300])
@pytest.mark.parametrize("qtype,N,K", [(synth.Q4_K, 384, 1024), (synth.Q6_K, 200, 768), (synth.Q8_0, 256, 528)])
def test_gemm_matches_oracle(orc, qtype, N, K, M):
    """Tile-width and M tails, N tails, K not a multiple of the 128-element
    stage (528: the last stage is zero-filled), split-K tails."""
    X8, sx, W8, sw, Y, Yf = _e4m3_case(orc, qtype, N, K, M, seed=M + N + K)
    assert_gemm_close(Y, orc.gemm_e4m3_f64(X8, sx, W8, sw), f"e4m3 {synth.TYPE_NAME[qtype]} M={M}")
    rel = np.linalg.norm(Y - Yf) / np.linalg.norm(Yf)
    assert rel < 0.1, f"quantization error {rel:.3f} vs the f16 path"


@pytest.mark.parametrize("members,K,M", [
    ([(synth.Q4_K, 384), (synth.Q4_K, 128), (synth.Q4_K, 128)], 512, 64),    # one launch
    ([(synth.Q4_K, 1024), (synth.Q6_K, 512)], 768, 256),                     # split-K tail inside the group
    ([(synth.Q4_K, 200), (synth.Q8_0, 128)], 512, 48),                       # N % 128 != 0: one after another
])
def test_grouped_matches_oracle(orc, members, K, M):
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(K + M)
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in members]
    hs = [mq.mq_register_weight(qt, dev(d), N, K, flags=mq.MQ_REG_E4M3) for (qt, N), d in zip(members, datas)]
    x = dev(synth.activations(g, M, K))
    x8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    mq.mq_quantize_e4m3(x, x8, sx)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in members]
    mq.mq_gemm_e4m3_grouped(x8, sx, hs, ys, M)
    mq.mq_stream_status()
    X8, SX = x8.cpu().numpy(), sx.cpu().numpy()
    for i, (h, y) in enumerate(zip(hs, ys)):
        codes, scales = h.e4m3_tensors()
        ref = orc.gemm_e4m3_f64(X8, SX, codes.cpu().numpy()[:, :K], scales.cpu().numpy())
        assert_gemm_close(y.cpu().numpy(), ref, f"member {i}")
        del codes, scales
    for h in hs:
        h.release()


def test_layer_full_size_sampled(orc):
    """Every GEMM of the 7B layer at M = 2048 through the e4m3 path, ~1500
    sampled outputs each against the oracle; the relative distance to the
    f16 path is reported."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = synth.workload("qwen2.5-7b_layer", seed=0)
    M = 2048
    mq.mq_reserve_workspace(64 << 20)
    errs = {}
    for w in weights:
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K, flags=mq.MQ_REG_E4M3)
        x = xs[w.K][:M]
        xd = dev(x)
        x8 = torch.empty((M, w.K), dtype=torch.uint8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        mq.mq_quantize_e4m3(xd, x8, sx)
        y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        yf = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        mq.mq_gemm_e4m3(x8, sx, h, y, M)
        mq.mq_gemm(xd, h, yf, M)
        mq.mq_stream_status()
        codes, scales = h.e4m3_tensors()
        W8 = codes.cpu().numpy()[:, :w.K]
        Y = y.cpu().numpy()
        mi, ni = sample_indices(M, w.N, 1500, seed=w.N)
        ref = orc.gemm_e4m3_f64_sampled(x8.cpu().numpy(), sx.cpu().numpy(), W8, scales.cpu().numpy(), mi, ni)
        assert_gemm_close(Y[mi, ni], ref, f"e4m3 {w.name}")
        errs[w.name] = float(np.linalg.norm(Y - yf.cpu().numpy()) / np.linalg.norm(yf.cpu().numpy()))
        h.release()
    print("relative distance to the f16 path:", errs)
    assert max(errs.values()) < 0.1


def test_e4m3_errors():
    import ctypes
    torch = torch_cuda()
    mq = _mq()
    L = mq._lib()
    g = synth.rng(9)
    data = dev(synth.weight_bytes(g, synth.Q8_0, 64, 264))
    out = ctypes.c_void_p()
    # K % 16 != 0, and no cache, are refused with MQ_REG_E4M3
    assert L.mq_register_weight(synth.Q8_0, data.data_ptr(), 64, 264, mq.MQ_REG_E4M3, None, ctypes.byref(out)) == -1
    d2 = dev(synth.weight_bytes(g, synth.Q4_K, 128, 512))
    assert L.mq_register_weight(synth.Q4_K, d2.data_ptr(), 128, 512, mq.MQ_REG_E4M3 | mq.MQ_REG_NO_CACHE, None,
                                ctypes.byref(out)) == -1
    h = mq.mq_register_weight(synth.Q4_K, d2, 128, 512)   # no e4m3 copy
    x8 = torch.zeros((8, 512), dtype=torch.uint8, device="cuda")
    sx = torch.ones(8, dtype=torch.float32, device="cuda")
    y = torch.empty((8, 128), dtype=torch.float32, device="cuda")
    assert L.mq_gemm_e4m3(x8.data_ptr(), sx.data_ptr(), h.handle, y.data_ptr(), 8, None) == -5
    assert L.mq_gemm_e4m3(x8.data_ptr(), None, h.handle, y.data_ptr(), 8, None) == -1
    xf = torch.zeros((8, 520), dtype=torch.float16, device="cuda")
    assert L.mq_quantize_e4m3(xf.data_ptr(), 8, 520, 520, x8.data_ptr(), 512, sx.data_ptr(), None) == -3
    mq.mq_stream_status()
    h.release()
