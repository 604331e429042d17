"""Shared helpers for the GPU parity tests."""
from __future__ import annotations

import numpy as np
import pytest

from quantized_weight_prefill_gguf_gb300.synth import TYPE_NAME

# Tolerance for GEMM outputs against the oracle's f64 result: relative
# Frobenius error <= 1e-3 and max abs error <= 5e-3 * max|Y_ref|.  f16 x f16
# products are exact in f32, so the kernels' only error is f32 accumulation
# (about sqrt(K) * 2^-24 relative), far inside this bound.
REL_FROB = 1e-3
MAX_ABS_REL = 5e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_gemm_close(y, y_ref, what=""):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    diff = y - y_ref
    nref = np.linalg.norm(y_ref)
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    scale = np.abs(y_ref).max()
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= REL_FROB, f"{what}: relative Frobenius error {rel:.3e} > {REL_FROB}"
    assert mx <= MAX_ABS_REL * max(scale, 1e-30), f"{what}: max abs error {mx:.3e} > {MAX_ABS_REL}*{scale:.3e}"
    return rel, mx


def sample_indices(M, N, count, seed=0):
    """Sampled (m, n) output positions: the four corners, tile edges, and
    uniform random picks."""
    g = np.random.Generator(np.random.PCG64(seed))
    pts = [(0, 0), (M - 1, N - 1), (0, N - 1), (M - 1, 0)]
    for m in (127, 128, 255, 256, M // 2):
        for n in (127, 128, N // 2, N - 129):
            if 0 <= m < M and 0 <= n < N:
                pts.append((m, n))
    mi = np.concatenate([np.array([p[0] for p in pts]), g.integers(0, M, count)])
    ni = np.concatenate([np.array([p[1] for p in pts]), g.integers(0, N, count)])
    return mi.astype(np.int64), ni.astype(np.int64)


def check_cache(orc, w, flags=0, expect_ldk=None):
    """Registers weight w and compares its f16 cache with the oracle's
    decode bit for bit; pad columns (ldk > K) must hold +0.0."""
    torch = torch_cuda()
    import quantized_weight_prefill_gguf_gb300 as mq
    q = dev(w.data)
    h = mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=flags)
    mq.mq_stream_status()
    n, k, ldk, _ = h.info()
    assert (n, k) == (w.N, w.K)
    if expect_ldk is not None:
        assert ldk == expect_ldk
    cache = h.cache_tensor().cpu().numpy().view(np.uint16)
    ref = orc.decode_matrix(w.qtype, w.data, w.N, w.K)
    got = cache[:, : w.K]
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (f"{TYPE_NAME[w.qtype]} {w.N}x{w.K}: {len(bad)} mismatches, first at "
                           f"{bad[0].tolist()}: got 0x{int(got[tuple(bad[0])]):04x} want 0x{int(ref[tuple(bad[0])]):04x}")
    if ldk > w.K:
        assert np.all(cache[:, w.K:] == 0), "pad columns must hold +0.0"
    h.release()
    del torch
