"""Grouped cached GEMM (mq_gemm_grouped): several weights that share K and X
in one launch, each member's output against the oracle.  Covers a split-K
tail inside a group, members of different block formats, the sampled
full-size q|k|v and gate|up groups of the 7B layer, the one-after-another
fallback (a member N not a multiple of 128), and the argument errors."""
import numpy as np
import pytest

from gpu_util import assert_gemm_close, dev, sample_indices, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


def _mq():
    import quantized_weight_prefill_gguf_gb300 as mq
    return mq


def _group_case(orc, members, K, M, seed):
    """members: list of (qtype, N).  Runs the group and checks every output
    in full against the oracle."""
    torch = torch_cuda()
    mq = _mq()
    g = synth.rng(seed)
    datas = [synth.weight_bytes(g, qt, N, K) for qt, N in members]
    hs = [mq.mq_register_weight(qt, dev(d), N, K) for (qt, N), d in zip(members, datas)]
    x = synth.activations(g, M, K)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _, N in members]
    mq.mq_gemm_grouped(dev(x), hs, ys, M)
    mq.mq_stream_status()
    for i, ((qt, N), d, y) in enumerate(zip(members, datas, ys)):
        W = orc.decode_matrix(qt, d, N, K)
        assert_gemm_close(y.cpu().numpy(), orc.gemm_f64(x.view(np.uint16), W), f"member {i} N={N} M={M}")
    for h in hs:
        h.release()


@pytest.mark.parametrize("members,K,M", [
    ([(synth.Q4_K, 384), (synth.Q4_K, 128), (synth.Q4_K, 128)], 512, 64),     # q|k|v-like, one wave
    ([(synth.Q4_K, 1024), (synth.Q6_K, 512)], 768, 256),                      # split-K tail inside the group
    ([(synth.Q8_0, 256), (synth.Q4_K, 256), (synth.Q6_K, 128), (synth.Q4_K, 640)], 1024, 200),  # 4 members, M tail
    ([(synth.Q4_K, 256)], 512, 33),                                            # group of one
])
def test_group_matches_oracle(orc, members, K, M):
    _group_case(orc, members, K, M, seed=K + M + len(members))


def test_group_fallback_when_n_not_tile_multiple(orc):
    """A member with N % 128 != 0 makes the members run one after another."""
    _group_case(orc, [(synth.Q4_K, 200), (synth.Q4_K, 128)], 512, 48, seed=5)


@pytest.mark.parametrize("names", [("q", "k", "v"), ("gate", "up")])
def test_layer_groups_full_size_sampled(orc, names):
    """The 7B layer's q|k|v and gate|up groups at M = 2048, ~2000 sampled
    outputs per member against the oracle."""
    torch = torch_cuda()
    mq = _mq()
    weights, xs = synth.workload("qwen2.5-7b_layer", seed=0)
    ws = [w for w in weights if w.name in names]
    K = ws[0].K
    M = 2048
    x = xs[K][:M]
    hs = [mq.mq_register_weight(w.qtype, dev(w.data), w.N, w.K) for w in ws]
    ys = [torch.empty((M, w.N), dtype=torch.float32, device="cuda") for w in ws]
    mq.mq_reserve_workspace(64 << 20)
    mq.mq_gemm_grouped(dev(x), hs, ys, M)
    mq.mq_stream_status()
    for w, y in zip(ws, ys):
        yh = y.cpu().numpy()
        assert np.all(np.isfinite(yh))
        mi, ni = sample_indices(M, w.N, 2000, seed=w.N)
        ref = orc.gemm_f64_sampled(x.view(np.uint16), orc.decode_matrix(w.qtype, w.data, w.N, w.K), mi, ni)
        assert_gemm_close(yh[mi, ni], ref, f"group {names} member {w.name}")
    for h in hs:
        h.release()


def test_group_errors():
    import ctypes
    torch = torch_cuda()
    mq = _mq()
    L = mq._lib()
    g = synth.rng(3)
    a = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, 128, 512)), 128, 512)
    b = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, 128, 768)), 128, 768)
    c = mq.mq_register_weight(synth.Q4_K, dev(synth.weight_bytes(g, synth.Q4_K, 128, 512)), 128, 512,
                              flags=mq.MQ_REG_NO_CACHE)
    x = dev(synth.activations(g, 8, 512))
    y0 = torch.empty((8, 128), dtype=torch.float32, device="cuda")
    y1 = torch.empty((8, 128), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p

    def call(hs, ys, count=None):
        n = len(hs)
        return L.mq_gemm_grouped(x.data_ptr(), (P * n)(*[h.handle for h in hs]), n if count is None else count,
                                 (P * n)(*[t.data_ptr() for t in ys]), 8, None)

    assert call([a, b], [y0, y1]) == -3                       # K differs
    assert call([a, c], [y0, y1]) == -5                       # member without a cache
    assert call([a, a], [y0, y1], count=0) == -1              # empty group
    assert call([a] * 5, [y0] * 5) == -1                      # more than 4 members
    assert L.mq_gemm_grouped(x.data_ptr(), None, 1, None, 8, None) == -1
    mq.mq_stream_status()
    for h in (a, b, c):
        h.release()
