"""Grouped fused GEMM (mq_gemm_fused_grouped): several weights of one block
format that share K and X, decoded on chip in one launch, each member's
output against the oracle.  One-hot rows of X make the on-chip decode of
every member observable bit for bit.  Covers both raw-read paths (row tensor
maps, and per-row bulk copies when rows start inside blocks), a split-K tail
inside a group, M tails, the 7B q|k|v and gate|up groups at small M, the
one-after-another fallbacks and the argument errors."""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _run(xd, hs, members, M):
    torch = torch_cuda()
    mq = _mq()
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in members]
    n0 = mq.mq_launch_count()
    mq.mq_gemm_fused_grouped(xd, hs, ys, M)
    mq.mq_stream_status()
    return [y.cpu().numpy() for y in ys], mq.mq_launch_count() - n0


def _register(members, K, seed, flags=None):
    mq = _mq()
    flags = mq.MQ_REG_NO_CACHE if flags is None else flags
    g = synth.rng(seed)
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in members]
    hs = [mq.mq_register_weight(qt, dev(d), N, K, flags=flags) for (qt, N), d in zip(members, datas)]
    return g, datas, hs


@pytest.mark.parametrize("members,K,M", [
    ([(synth.Q4_K, 384), (synth.Q4_K, 128), (synth.Q4_K, 128)], 1024, 1),     # q|k|v-like
    ([(synth.Q4_K, 384), (synth.Q4_K, 128), (synth.Q4_K, 128)], 1024, 33),
    ([(synth.Q6_K, 256), (synth.Q6_K, 512)], 2048, 100),                      # 210-byte blocks
    ([(synth.Q8_0, 128), (synth.Q8_0, 256), (synth.Q8_0, 128), (synth.Q8_0, 384)], 512, 17),   # 4 members
    ([(synth.Q4_K, 256), (synth.Q4_K, 128)], 896, 40),                         # rows start inside blocks: bulk copies
    ([(synth.Q5_K, 1024), (synth.Q5_K, 1024)], 3584, 8),                       # split-K tail inside the group
])
def test_fused_group_matches_oracle(orc, members, K, M):
    g, datas, hs = _register(members, K, seed=K + M + len(members))
    x = synth.activations(g, M, K)
    ys, launches = _run(dev(x), hs, members, M)
    assert 1 <= launches <= 2, f"{launches} launches for one group"
    for i, ((qt, N), d, y) in enumerate(zip(members, datas, ys)):
        W = orc.decode_matrix(qt, d, N, K)
        assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), W), f"member {i} {synth.TYPE_NAME[qt]} N={N} M={M}")
    for h in hs:
        h.release()


@pytest.mark.parametrize("members,K", [
    ([(synth.Q4_K, 256), (synth.Q4_K, 128), (synth.Q4_K, 128)], 512),
    ([(synth.Q6_K, 128), (synth.Q6_K, 256)], 512),
    ([(synth.Q4_K, 128), (synth.Q4_K, 256)], 896),      # bulk-copy path
])
def test_fused_group_one_hot_equals_decode(orc, members, K):
    """X = identity: every member's Y is its decoded W^T, bit for bit."""
    g, datas, hs = _register(members, K, seed=K * 7 + len(members))
    ys, _ = _run(dev(np.eye(K, dtype=np.float16)), hs, members, K)
    for i, ((qt, N), d, y) in enumerate(zip(members, datas, ys)):
        W = orc.f16_to_f32(orc.decode_matrix(qt, d, N, K))
        assert np.array_equal(y, W.T), f"member {i}: on-chip decode differs from the oracle's"
    for h in hs:
        h.release()


@pytest.mark.parametrize("names,M", [(("q", "k", "v"), 1), (("q", "k", "v"), 32), (("gate", "up"), 32)])
def test_layer_groups_small_m_sampled(orc, names, M):
    """The 7B layer's q|k|v and gate|up groups at small M, sampled outputs
    against the oracle; the same outputs as one mq_gemm_fused per member up
    to f32 summation order."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = synth.workload("qwen2.5-7b_layer", seed=0)
    ws = [w for w in weights if w.name in names]
    hs = [mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K, flags=mq.MQ_REG_NO_CACHE) for w in ws]
    x = xs[ws[0].K][:M]
    xd = dev(x)
    ys, launches = _run(xd, hs, [(w.qtype, w.N) for w in ws], M)
    assert launches <= 2
    for w, h, y in zip(ws, hs, ys):
        mi, ni = sample_indices(M, w.N, 1500, seed=w.N + M)
        W = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
        assert_gemm_close(y[mi, ni], orc.gemm_f64_sampled(x.view(np.uint16), W, mi, ni), f"{w.name} M={M}")
        y1 = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        mq.mq_gemm_fused(xd, h, y1, M)
        mq.mq_stream_status()
        assert_gemm_close(y1.cpu().numpy()[mi, ni], orc.gemm_f64_sampled(x.view(np.uint16), W, mi, ni),
                          f"{w.name} single M={M}")
    for h in hs:
        h.release()


def test_fused_group_fallbacks(orc, monkeypatch):
    """N % 128 != 0, or members whose raw rows are read differently (one
    registered with MQ_RAW_TMA=0), run one after another; float weights take
    the grouped cached GEMM."""
    K, M = 512, 24
    members = [(synth.Q4_K, 200), (synth.Q4_K, 128)]
    g, datas, hs = _register(members, K, seed=11)
    x = synth.activations(g, M, K)
    ys, launches = _run(dev(x), hs, members, M)
    assert launches >= 2
    for (qt, N), d, y in zip(members, datas, ys):
        assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qt, d, N, K)), f"fallback N={N}")
    for h in hs:
        h.release()

    mq = _mq()
    members = [(synth.Q4_K, 256), (synth.Q4_K, 128)]
    g = synth.rng(12)
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in members]
    monkeypatch.setenv("MQ_RAW_TMA", "0")
    h0 = mq.mq_register_weight(members[0][0], dev(datas[0]), members[0][1], K, flags=mq.MQ_REG_NO_CACHE)
    monkeypatch.delenv("MQ_RAW_TMA")
    h1 = mq.mq_register_weight(members[1][0], dev(datas[1]), members[1][1], K, flags=mq.MQ_REG_NO_CACHE)
    ys, launches = _run(dev(x), [h0, h1], members, M)
    assert launches >= 2
    for (qt, N), d, y in zip(members, datas, ys):
        assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qt, d, N, K)), f"raw paths N={N}")
    h0.release()
    h1.release()

    members = [(synth.F16, 256), (synth.F16, 128)]
    g, datas, hs = _register(members, K, seed=13, flags=0)
    ys, _ = _run(dev(x), hs, members, M)
    for (qt, N), d, y in zip(members, datas, ys):
        assert_gemm_close(y, orc.gemm_f64(x.view(np.uint16), orc.decode_matrix(qt, d, N, K)), f"float N={N}")
    for h in hs:
        h.release()


def test_fused_group_errors():
    torch = torch_cuda()
    mq = _mq()
    L = mq._lib()
    g = synth.rng(21)
    ha = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, 128, 512)), 128, 512,
                               flags=mq.MQ_REG_NO_CACHE)
    hb = mq.mq_register_weight(synth.Q8_0, dev(synth.weight_bytes(g, synth.Q8_0, 128, 512)), 128, 512,
                               flags=mq.MQ_REG_NO_CACHE)
    hc = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, 128, 1024)), 128, 1024,
                               flags=mq.MQ_REG_NO_CACHE)
    x = torch.zeros((8, 512), dtype=torch.float16, device="cuda")
    y0 = torch.empty((8, 128), dtype=torch.float32, device="cuda")
    y1 = torch.empty((8, 128), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    yarr = (P * 2)(y0.data_ptr(), y1.data_ptr())
    n0 = mq.mq_launch_count()
    assert L.mq_gemm_fused_grouped(x.data_ptr(), (P * 2)(ha.handle, hb.handle), 2, yarr, 8, None) == -1   # types
    assert L.mq_gemm_fused_grouped(x.data_ptr(), (P * 2)(ha.handle, hc.handle), 2, yarr, 8, None) == -3   # K
    assert L.mq_gemm_fused_grouped(x.data_ptr(), (P * 2)(ha.handle, ha.handle), 0, yarr, 8, None) == -1   # count
    assert L.mq_gemm_fused_grouped(x.data_ptr(), (P * 2)(ha.handle, ha.handle), 5, yarr, 8, None) == -1
    assert L.mq_gemm_fused_grouped(x.data_ptr(), None, 2, yarr, 8, None) == -1
    assert mq.mq_launch_count() == n0, "nothing is launched when an argument check fails"
    mq.mq_stream_status()
    for h in (ha, hb, hc):
        h.release()


def test_auto_grouped_gate(orc):
    """mq_gemm_auto_grouped: one fused launch below the gate, the grouped
    cached GEMM at and above it (seen in the launch trace); a member without
    an f16 cache sends the group to the fused path at any M."""
    torch = torch_cuda()
    mq = _mq()
    K = 512
    members = [(synth.Q4_K, 256), (synth.Q4_K, 128)]
    g, datas, hs = _register(members, K, seed=31, flags=0)
    hn = mq.mq_register_weight(members[1][0], dev(datas[1]), members[1][1], K, flags=mq.MQ_REG_NO_CACHE)
    x = synth.activations(g, 160, K)
    refs = [orc.decode_matrix(qt, d, N, K) for (qt, N), d in zip(members, datas)]
    old = mq.mq_get_m_gate()
    try:
        mq.mq_set_m_gate(100)
        for M, group, want in ((16, hs, mq.MQ_TRACE_GEMM_FUSED), (99, hs, mq.MQ_TRACE_GEMM_FUSED),
                               (100, hs, mq.MQ_TRACE_GEMM_CACHED), (160, hs, mq.MQ_TRACE_GEMM_CACHED),
                               (160, [hs[0], hn], mq.MQ_TRACE_GEMM_FUSED)):
            ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in members]
            mq.mq_trace_enable(True)
            mq.mq_gemm_auto_grouped(dev(x[:M]), group, ys, M)
            mq.mq_stream_status()
            kinds = {r["kind"] for r in mq.mq_trace_records()}
            mq.mq_trace_enable(False)
            assert kinds == {want}, f"M={M}: trace kinds {kinds}"
            for i, (y, W) in enumerate(zip(ys, refs)):
                assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x[:M].view(np.uint16), W), f"auto M={M} member {i}")
    finally:
        mq.mq_set_m_gate(old)
    for h in hs + [hn]:
        h.release()
