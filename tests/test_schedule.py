"""Host logic: the GEMM work plan and the unit schedule the kernels run.

mq_debug_schedule plans a launch and lists every unit each CTA runs, using
the kernels' own schedule code (no device needed).  For many shapes, with
single CTAs and with CTA pairs, and for the cached, fused and e4m3 paths:

* every tile's K steps are covered exactly once (whole, or by the split
  parts in order, with no gap or overlap);
* tile_coords places the tiles on distinct (weight-row tile, token tile)
  positions covering the grid (plus one phantom weight-row tile per token
  tile when pairs meet an odd count);
* split units use slots [0, tiles - full_tiles), parts [0, split), and the
  workspace the plan asks for holds them;
* the two CTAs of a pair run the same K-ranges in the same order, on
  adjacent weight-row tiles of the same token tile;
* the grid stays within the SMs (or resident clusters), every CTA has work,
  and the fused path's split boundaries fall on whole 256-element chunks.
"""
import itertools

import numpy as np
import pytest

import quantized_weight_prefill_gguf_gb300 as mq

SHAPES = [(1, 18944, 3584), (33, 512, 3584), (256, 4608, 3584), (2048, 37888, 3584), (2048, 3584, 18944),
          (2048, 512, 3584), (300, 200, 768), (130, 384, 1024), (4096, 128, 4096), (513, 1000, 520)]


def _check(M, N, K, sms, path, pc):
    plan, units = mq.mq_debug_schedule(M, N, K, sms, path, pc)
    kstep = 128 if path == 2 else 64
    kblocks = -(-K // kstep)
    bn = plan["bn"]
    m_tiles = -(-M // bn)
    n_tiles = -(-N // 128)
    pair = plan["pair"]
    assert pair == (1 if pc > 0 and path != 1 else 0)
    tiles, full, split = plan["tiles"], plan["full_tiles"], plan["split"]
    assert tiles == (2 * m_tiles * (-(-n_tiles // 2)) if pair else m_tiles * n_tiles)
    assert units.shape[0] == plan["units"] * (2 if pair else 1)
    assert 0 < plan["grid"] <= (2 * pc if pair else sms)
    if pair:
        assert plan["grid"] % 2 == 0
    # every CTA has work
    assert set(units[:, 0].tolist()) == set(range(plan["grid"]))
    # tiles placed on distinct positions covering the grid
    pos = {}
    for t, nt, mt in units[:, 1:4].tolist():
        pos.setdefault(t, (nt, mt))
        assert pos[t] == (nt, mt)
    assert sorted(pos) == list(range(tiles))
    cells = sorted(pos.values())
    assert len(set(cells)) == tiles
    assert all(0 <= mt < m_tiles for _, mt in cells)
    n_extent = n_tiles + (n_tiles % 2 if pair else 0)
    assert all(0 <= nt < n_extent for nt, _ in cells)
    assert len(cells) == n_extent * m_tiles
    # K coverage per tile
    by_tile = {}
    for cta, t, nt, mt, kb0, kb1, part, slot in units.tolist():
        by_tile.setdefault(t, []).append((kb0, kb1, part, slot))
    for t, parts in by_tile.items():
        parts.sort()
        if t < full:
            assert parts == [(0, kblocks, -1, 0)], (t, parts)
        else:
            assert [p[2] for p in parts] == list(range(split))
            assert parts[0][0] == 0 and parts[-1][1] == kblocks
            for a, b in zip(parts, parts[1:]):
                assert a[1] == b[0] and a[0] < a[1]
            assert all(p[3] == t - full for p in parts)
            if plan["kb_align"] > 1:
                assert all(p[0] % plan["kb_align"] == 0 for p in parts)
    if split > 1:
        assert plan["ws_bytes"] >= (tiles - full) * split * bn * 128 * 4
    # pairs: the two CTAs of a cluster run the same K-ranges on adjacent tiles
    if pair:
        seq = {}
        for cta, t, nt, mt, kb0, kb1, part, slot in units.tolist():
            seq.setdefault(cta, []).append((t, nt, mt, kb0, kb1, part))
        for c in range(0, plan["grid"], 2):
            a, b = seq[c], seq[c + 1]
            assert len(a) == len(b)
            for x, y in zip(a, b):
                assert x[3:] == y[3:] and y[0] == x[0] + 1 and y[1] == x[1] + 1 and y[2] == x[2]
                assert x[1] % 2 == 0


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("path,pc", [(0, 0), (0, 74), (0, 76), (1, 0), (2, 0), (2, 76)])
def test_schedule_invariants(M, N, K, path, pc):
    for sms in (148, 152):
        _check(M, N, K, sms, path, pc)


def test_schedule_random_shapes():
    g = np.random.Generator(np.random.PCG64(5))
    for _ in range(300):
        M = int(g.integers(1, 5000))
        N = int(g.integers(1, 40000))
        K = int(g.integers(1, 300)) * 64
        sms = int(g.choice([8, 37, 148, 152]))
        path = int(g.integers(0, 3))
        pc = int(g.choice([0, 3, sms // 2]))
        _check(M, N, K, sms, path, pc)


def test_schedule_bad_args():
    import ctypes
    L = mq._lib()
    plan = np.zeros(9, dtype=np.int64)
    n = ctypes.c_int64()
    assert L.mq_debug_schedule(0, 10, 64, 148, 0, 0, plan.ctypes.data, None, 0, ctypes.byref(n)) == -1
    assert L.mq_debug_schedule(10, 10, 64, 148, 3, 0, plan.ctypes.data, None, 0, ctypes.byref(n)) == -1
