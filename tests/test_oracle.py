"""The CPU oracle against its pins (CPU only)."""
import os
import subprocess

import numpy as np
import pytest

import oracle_pins
from oracle_pins import ALL_PINS

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_f16_exhaustive(orc, tmp_path):
    """All 2^32 binary32 inputs against the compiler's _Float16 conversion."""
    exe = str(tmp_path / "pin_f16")
    subprocess.run(["gcc", "-O2", "-fopenmp", os.path.join(HERE, "pin_f16_exhaustive.c"),
                    orc.path, "-o", exe, f"-Wl,-rpath,{os.path.dirname(orc.path)}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "narrow_mismatches=0 widen_mismatches=0" in r.stdout


def test_block_counts_match_workloads():
    """Flat-stream block counts of the workloads: the 896x896 Q4_K weight is
    3136 super-blocks, so rows of 896 elements share blocks (odd rows start
    at element 128 of a super-block)."""
    from quantized_weight_prefill_gguf_gb300 import synth
    assert synth.nblocks(synth.Q4_K, 896, 896) == 3136
    assert synth.nblocks(synth.Q6_K, 3584, 18944) == 3584 * 74
    assert synth.nblocks(synth.Q8_0, 3584, 18944) == 2121728
    assert synth.nblocks(synth.Q8_0, 18944, 3584) == 2121728


def test_flat_stream_rows_share_blocks(orc):
    """Decoding the 896x896 stream as one flat sequence and reading it
    row-major is the same as decoding block by block: row 1 starts at element
    128 of block 3 (896 = 3.5 * 256)."""
    from quantized_weight_prefill_gguf_gb300 import synth
    g = synth.rng(0)
    q = synth.weight_bytes(g, synth.Q4_K, 896, 896)
    W = orc.decode_matrix(synth.Q4_K, q, 896, 896)
    blk3 = orc.decode(synth.Q4_K, q[3 * 144: 4 * 144])
    assert np.array_equal(W[0, 768:896], blk3[:128])
    assert np.array_equal(W[1, 0:128], blk3[128:])


def test_generator_is_deterministic():
    from quantized_weight_prefill_gguf_gb300 import synth
    a, xa = synth.workload("q4k_896", seed=0)
    b, xb = synth.workload("q4k_896", seed=0)
    assert np.array_equal(a[0].data, b[0].data)
    assert np.array_equal(xa[896], xb[896])
    assert a[0].data.size == 3136 * 144


def test_generator_field_ranges(orc):
    """The generated fields follow the recipe: Q4_K d in [2e-4,1e-3] and dmin
    in [0,5e-4] (to f16 rounding), Q8_0 quants never -128, decoded Q6_K
    magnitudes below 1e-3*128*32."""
    from quantized_weight_prefill_gguf_gb300 import synth
    g = synth.rng(1)
    q4 = synth.q4_K_blocks(g, 1000).reshape(1000, 144)
    d = q4[:, 0:2].copy().view("<f2").astype(np.float64).reshape(-1)
    dmin = q4[:, 2:4].copy().view("<f2").astype(np.float64).reshape(-1)
    assert d.min() >= 1.99e-4 and d.max() <= 1.001e-3
    assert dmin.min() >= 0 and dmin.max() <= 5.001e-4
    q8 = synth.q8_0_blocks(g, 1000).reshape(1000, 34)
    assert q8[:, 2:].view(np.int8).min() >= -127
    q6 = synth.q6_K_blocks(g, 1000)
    y = orc.f16_to_f32(orc.decode(synth.Q6_K, q6))
    assert np.all(np.isfinite(y)) and np.abs(y).max() <= 1.001e-3 * 128 * 32
