"""GPU block decoders against the oracle, bit for bit (sm_103a, through the C ABI).

The f16 cache must equal the oracle's decode of the same bytes exactly: the
block definitions fix one f16 value per element (f32 arithmetic, one round
to nearest even).  Covers every workload's weights at full size, the K-pad
branch (pad columns +0.0), ragged flat streams, and mq_dequantize with a
caller-chosen row stride.
"""
import numpy as np
import pytest

from gpu_util import check_cache, dev, torch_cuda
from quantized_weight_prefill_gguf_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload", ["q4k_896", "qwen2.5-7b_layer", "llama3.1-8b_layer", "q8_0_pair"])
def test_cache_bit_exact(orc, workload):
    weights, _ = synth.workload(workload, seed=0, max_m=1)
    for w in weights:
        want = w.K + 64 if (2 * w.K) % 2048 == 0 else w.K
        check_cache(orc, w, expect_ldk=want)


def test_kpad_flags(orc):
    g = synth.rng(5)
    w = synth.Weight("w", synth.Q4_K, 256, 1024, synth.weight_bytes(g, synth.Q4_K, 256, 1024))
    import quantized_weight_prefill_gguf_gb300 as mq
    check_cache(orc, w, expect_ldk=1088)
    check_cache(orc, w, flags=mq.MQ_REG_NO_KPAD, expect_ldk=1024)
    w2 = synth.Weight("w", synth.Q6_K, 64, 768, synth.weight_bytes(g, synth.Q6_K, 64, 768))
    check_cache(orc, w2, flags=mq.MQ_REG_KPAD, expect_ldk=832)


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q4_K, 3, 256), (synth.Q4_K, 8, 896), (synth.Q4_K, 66, 128),     # rows starting mid-block
    (synth.Q6_K, 1, 256), (synth.Q6_K, 5, 512), (synth.Q6_K, 10, 384),     # odd block counts: tail bytes
    (synth.Q8_0, 1, 32), (synth.Q8_0, 4, 40), (synth.Q8_0, 1000, 24),     # K % 32 != 0, tiny K
    (synth.Q8_0, 257, 96), (synth.Q6_K, 33, 2304),
])
def test_ragged_streams(orc, qtype, N, K):
    g = synth.rng(N * 1000 + K)
    w = synth.Weight("w", qtype, N, K, synth.weight_bytes(g, qtype, N, K))
    check_cache(orc, w)


def test_dequantize_row_stride(orc):
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    g = synth.rng(9)
    N, K, ldo = 96, 1280, 1352
    for qtype in (synth.Q4_K, synth.Q6_K, synth.Q8_0):
        data = synth.weight_bytes(g, qtype, N, K)
        out = torch.full((N, ldo), -7.0, dtype=torch.float16, device="cuda")
        mq.mq_dequantize(qtype, dev(data), N, K, out, ldo)
        mq.mq_stream_status()
        o = out.cpu().numpy().view(np.uint16)
        assert np.array_equal(o[:, :K], orc.decode_matrix(qtype, data, N, K))
        assert np.all(out[:, K:].cpu().numpy() == -7.0), "columns past K must be left untouched"


def test_signed_zero_and_subnormals(orc):
    """Blocks whose decoded values include -0.0 and f16 subnormals: the GPU
    keeps both (no flush to zero, sign of zero kept)."""
    from oracle_pins import q4k_bytes, q6k_bytes, QH_ZERO, MINUS_ONE, ONE
    blocks4 = [q4k_bytes(MINUS_ONE, ONE, [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], [0] * 128),   # all -0
               q4k_bytes(0x0001, 0x0001, [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12], list(range(128)))]
    data4 = np.concatenate(blocks4)
    w4 = synth.Weight("w", synth.Q4_K, 2, 256, data4)
    check_cache(orc, w4)
    data6 = np.concatenate([q6k_bytes([0] * 128, QH_ZERO, [5, -5] * 8, ONE),
                            q6k_bytes(list(range(128)), list(range(64)), list(range(-8, 8)), 0x0003)])
    w6 = synth.Weight("w", synth.Q6_K, 2, 256, data6)
    check_cache(orc, w6)
    ref6 = orc.decode(synth.Q6_K, data6)
    assert np.any(ref6 == 0x8000) and np.any((ref6 & 0x7C00) == 0)
