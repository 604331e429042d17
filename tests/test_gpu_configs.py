"""The Q8_0 pair (3584 x 18944 and 18944 x 3584 at M = 128 and 1024) and the
Llama-3.1-8B-shaped layer (all Q4_K, M = 512) through every path the
library dispatches them to, at full size.

Small shapes passing proves little about the real ones ("79 · Phase-8
coverage & first-measurement batch", section 6 Lessons: test the real
shapes; section 3.6: the misaligned 34-byte Q8_0 loads only showed at model
shapes).  Here the fused path, the M gate (mq_gemm_auto, with the path it
took read from the launch trace) and the grouped launches the benchmark
uses are each compared with the f64 oracle on ~2000 sampled outputs
(corners and tile edges included), and a one-hot K slice through the fused
path at full N shows its on-chip decode equals the oracle's decode bit for
bit, at the start, the middle and the end of K.
"""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _traced(fn):
    """Run fn() with the library's trace on; the kinds of the launches."""
    mq = _mq()
    mq.mq_trace_enable(True)
    try:
        fn()
        mq.mq_stream_status()
        return [r["kind"] for r in mq.mq_trace_records()]
    finally:
        mq.mq_trace_enable(False)


def _check_sampled(orc, x, W16, y, what, seed):
    M, N = y.shape
    mi, ni = sample_indices(M, N, 2000, seed=seed)
    ref = orc.gemm_f64_sampled(x.view(np.uint16), W16, mi, ni)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    assert_gemm_close(y[mi, ni], ref, what)


@pytest.fixture(scope="module")
def q8_pair():
    return synth.workload("q8_0_pair", seed=0)


@pytest.fixture(scope="module")
def llama():
    return synth.workload("llama3.1-8b_layer", seed=0)


@pytest.mark.parametrize("M", [128, 1024])
def test_q8_0_pair_fused_and_auto(orc, q8_pair, M):
    torch = torch_cuda()
    mq = _mq()
    weights, xs = q8_pair
    gate = mq.mq_get_m_gate()
    for w in weights:
        x = xs[w.K][:M]
        xd = dev(x)
        W16 = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
        assert h.info()[2] == w.K, "K = 18944 / 3584 take the no-pad branch"
        y = torch.full((M, w.N), float("nan"), dtype=torch.float32, device="cuda")
        kinds = _traced(lambda: mq.mq_gemm_fused(xd, h, y, M))
        assert kinds == [mq.MQ_TRACE_GEMM_FUSED]
        _check_sampled(orc, x, W16, y.cpu().numpy(), f"q8_0 {w.N}x{w.K} fused M={M}", w.N + M)
        y.fill_(float("nan"))
        kinds = _traced(lambda: mq.mq_gemm_auto(xd, h, y, M))
        want = mq.MQ_TRACE_GEMM_FUSED if M < gate else mq.MQ_TRACE_GEMM_CACHED
        assert kinds == [want], f"M={M} gate={gate}: auto took {kinds}"
        _check_sampled(orc, x, W16, y.cpu().numpy(), f"q8_0 {w.N}x{w.K} auto M={M}", w.N + M + 1)
        h.release()


@pytest.mark.parametrize("name", ["w1", "w2"])
def test_q8_0_pair_one_hot_slices(orc, q8_pair, name):
    """X = one-hot rows over a 256-wide K slice: Y[i, n] = W[n, k0 + i]
    exactly, through the fused path at full N (and equal to the cached
    path), for slices at the start, middle and end of K."""
    torch = torch_cuda()
    mq = _mq()
    weights, _ = q8_pair
    w = next(v for v in weights if v.name == name)
    W = orc.f16_to_f32(orc.decode_matrix(w.qtype, w.data, w.N, w.K))
    h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
    S = 256
    for k0 in (0, (w.K // 2) // 256 * 256, w.K - S):
        x = np.zeros((S, w.K), dtype=np.float16)
        x[np.arange(S), k0 + np.arange(S)] = 1.0
        xd = dev(x)
        yf = torch.full((S, w.N), float("nan"), dtype=torch.float32, device="cuda")
        mq.mq_gemm_fused(xd, h, yf, S)
        yc = torch.full((S, w.N), float("nan"), dtype=torch.float32, device="cuda")
        mq.mq_gemm(xd, h, yc, S)
        mq.mq_stream_status()
        yf, yc = yf.cpu().numpy(), yc.cpu().numpy()
        want = W[:, k0:k0 + S].T
        bad = np.argwhere(yf != want)
        assert bad.size == 0, f"{name} k0={k0}: fused decode differs at {bad[0].tolist()}"
        assert np.array_equal(yc, yf), f"{name} k0={k0}: cached and fused differ"
    h.release()


def test_llama_layer_fused_and_auto(orc, llama):
    """Every GEMM of the layer at M = 512 through the fused path and the M
    gate (which takes the cached path at 512 with the default gate)."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = llama
    M = synth.WORKLOADS["llama3.1-8b_layer"][1][0]
    gate = mq.mq_get_m_gate()
    for w in weights:
        x = xs[w.K][:M]
        xd = dev(x)
        W16 = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
        assert h.info()[2] == w.K + 64, "K = 4096 / 14336 rows alias at 2048 bytes: padded"
        for fn, want in ((mq.mq_gemm_fused, mq.MQ_TRACE_GEMM_FUSED),
                         (mq.mq_gemm_auto, mq.MQ_TRACE_GEMM_FUSED if M < gate else mq.MQ_TRACE_GEMM_CACHED)):
            y = torch.full((M, w.N), float("nan"), dtype=torch.float32, device="cuda")
            kinds = _traced(lambda: fn(xd, h, y, M))
            assert kinds == [want], f"{w.name}: {fn.__name__} launched {kinds}"
            _check_sampled(orc, x, W16, y.cpu().numpy(), f"llama {w.name} {fn.__name__} M={M}", w.N + 7)
        h.release()


def test_llama_layer_grouped_launches(orc, llama):
    """The layer as the benchmark launches it: q|k|v and gate|up grouped,
    o and down single, through the fused grouped path, the cached grouped
    path and the grouped M gate; every member against the oracle."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = llama
    M = synth.WORKLOADS["llama3.1-8b_layer"][1][0]
    by = {w.name: w for w in weights}
    hs = {w.name: mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K) for w in weights}
    W16 = {w.name: orc.decode_matrix(w.qtype, w.data, w.N, w.K) for w in weights}
    for grp in (("q", "k", "v"), ("gate", "up")):
        K = by[grp[0]].K
        x = xs[K][:M]
        xd = dev(x)
        for fn in (mq.mq_gemm_fused_grouped, mq.mq_gemm_grouped, mq.mq_gemm_auto_grouped):
            ys = [torch.full((M, by[n].N), float("nan"), dtype=torch.float32, device="cuda") for n in grp]
            kinds = _traced(lambda: fn(xd, [hs[n] for n in grp], ys, M))
            assert len(kinds) == 1, f"{'|'.join(grp)} {fn.__name__}: {len(kinds)} launches, want one"
            for n, y in zip(grp, ys):
                _check_sampled(orc, x, W16[n], y.cpu().numpy(), f"llama {n} in {'|'.join(grp)} {fn.__name__}",
                               by[n].N + 3)
    for h in hs.values():
        h.release()


def test_llama_one_hot_slices_fused(orc, llama):
    """One-hot K slices through the fused path on the padded-cache weights
    (gate 14336 x 4096 and down 4096 x 14336): bit-exact decode at the
    start, middle and end of K, equal to the cached path."""
    torch = torch_cuda()
    mq = _mq()
    weights, _ = llama
    S = 256
    for w in (v for v in weights if v.name in ("gate", "down")):
        W = orc.f16_to_f32(orc.decode_matrix(w.qtype, w.data, w.N, w.K))
        h = mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K)
        for k0 in (0, (w.K // 2) // 256 * 256, w.K - S):
            x = np.zeros((S, w.K), dtype=np.float16)
            x[np.arange(S), k0 + np.arange(S)] = 1.0
            xd = dev(x)
            yf = torch.full((S, w.N), float("nan"), dtype=torch.float32, device="cuda")
            yc = torch.full((S, w.N), float("nan"), dtype=torch.float32, device="cuda")
            mq.mq_gemm_fused(xd, h, yf, S)
            mq.mq_gemm(xd, h, yc, S)
            mq.mq_stream_status()
            yf, yc = yf.cpu().numpy(), yc.cpu().numpy()
            assert np.array_equal(yf, W[:, k0:k0 + S].T), f"{w.name} k0={k0}: fused decode differs"
            assert np.array_equal(yc, yf), f"{w.name} k0={k0}: cached and fused differ"
        h.release()
