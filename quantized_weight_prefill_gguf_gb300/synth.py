"""Seeded synthetic inputs: GGUF-style quantized weights and f16 activations.

This module only draws random numbers and lays them into block bytes at the
fields' byte offsets.  It holds none of the method's arithmetic (no
decoding, no GEMM) and imports neither the CUDA library nor the oracle, so
both sides can be fed the same bytes.

Recipe (numpy ``Generator(PCG64(seed))``, one generator per workload, weights
drawn in the listed order, then the activations):

* Q4_K block (144 B): d ~ U[2e-4, 1e-3] and dmin ~ U[0, 5e-4], each rounded
  to f16 and stored little-endian at bytes 0 and 2; the 12 packed scale/min
  bytes and the 128 nibble bytes are uniform random bytes, so every 6-bit
  scale and min is uniform on {0..63} and every nibble on {0..15}.
* Q6_K block (210 B): ql (128 B) and qh (64 B) uniform bytes, 16 int8 scales
  uniform on {-128..127}, d ~ U[2e-4, 1e-3] as f16 at byte 208.
* Q8_0 block (34 B): d ~ U[1e-3, 5e-3] as f16 at byte 0, 32 int8 quants
  uniform on {-127..127}.
* Q4_0 block (18 B): d ~ U[1e-3, 5e-3] as f16 at byte 0, 16 nibble bytes.
* Q5_0 block (22 B): d ~ U[1e-3, 5e-3] as f16 at byte 0, the 4-byte qh bit
  plane at byte 2, 16 nibble bytes at byte 6 (all uniform bytes).
* Q5_1 block (24 B): d ~ U[5e-4, 2e-3] and m ~ U[-2e-2, 0] as f16 at bytes
  0 and 2, qh at byte 4, 16 nibble bytes at byte 8.
* Q5_K block (176 B): d, dmin as Q4_K at bytes 0 and 2, 12 scale/min bytes
  at 4, 32 qh bytes at 16, 128 nibble bytes at 48 (uniform bytes).
* Float weights: values ~ N(0, 0.02) drawn in f32; F32 stores them, F16
  stores them rounded to f16 (numpy's conversion), BF16 stores the upper
  16 bits of each f32 draw (the distribution is defined that way: no
  rounding step).
* Activations X[M,K] ~ N(0,1) in f32, rounded to f16.

Draw order inside a weight: Q4_K d, dmin, scale bytes, nibble bytes;
Q6_K ql, qh, scales, d; Q8_0 d, quants; Q4_0 d, nibbles; Q5_0 d, qh,
nibbles; Q5_1 d, m, qh, nibbles; Q5_K d, dmin, scale bytes, qh, nibbles.
Field values are drawn for all blocks of the weight at once.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F32, F16, BF16 = 0, 1, 30
Q4_0, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 6, 7, 8, 12, 13, 14
BLOCK = {F32: (1, 4), F16: (1, 2), BF16: (1, 2), Q4_0: (32, 18), Q5_0: (32, 22), Q5_1: (32, 24), Q8_0: (32, 34), Q4_K: (256, 144),
         Q5_K: (256, 176), Q6_K: (256, 210)}
TYPE_NAME = {F32: "f32", F16: "f16", BF16: "bf16", Q4_0: "q4_0", Q5_0: "q5_0", Q5_1: "q5_1", Q8_0: "q8_0", Q4_K: "q4_K", Q5_K: "q5_K",
             Q6_K: "q6_K"}


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f16_le_bytes(v: np.ndarray) -> np.ndarray:
    """[n] float values -> [n, 2] little-endian f16 bytes."""
    return v.astype(np.float16).astype("<f2").view(np.uint8).reshape(-1, 2)


def q4_K_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(2e-4, 1e-3, nblocks)
    dmin = g.uniform(0.0, 5e-4, nblocks)
    scales = g.integers(0, 256, (nblocks, 12), dtype=np.uint8)
    qs = g.integers(0, 256, (nblocks, 128), dtype=np.uint8)
    b = np.empty((nblocks, 144), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:4] = _f16_le_bytes(dmin)
    b[:, 4:16] = scales
    b[:, 16:144] = qs
    return b.reshape(-1)


def q6_K_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    ql = g.integers(0, 256, (nblocks, 128), dtype=np.uint8)
    qh = g.integers(0, 256, (nblocks, 64), dtype=np.uint8)
    sc = g.integers(-128, 128, (nblocks, 16), dtype=np.int16).astype(np.int8)
    d = g.uniform(2e-4, 1e-3, nblocks)
    b = np.empty((nblocks, 210), dtype=np.uint8)
    b[:, 0:128] = ql
    b[:, 128:192] = qh
    b[:, 192:208] = sc.view(np.uint8)
    b[:, 208:210] = _f16_le_bytes(d)
    return b.reshape(-1)


def q8_0_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(1e-3, 5e-3, nblocks)
    q = g.integers(-127, 128, (nblocks, 32), dtype=np.int16).astype(np.int8)
    b = np.empty((nblocks, 34), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:34] = q.view(np.uint8)
    return b.reshape(-1)


def q4_0_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(1e-3, 5e-3, nblocks)
    qs = g.integers(0, 256, (nblocks, 16), dtype=np.uint8)
    b = np.empty((nblocks, 18), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:18] = qs
    return b.reshape(-1)


def q5_0_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(1e-3, 5e-3, nblocks)
    qh = g.integers(0, 256, (nblocks, 4), dtype=np.uint8)
    qs = g.integers(0, 256, (nblocks, 16), dtype=np.uint8)
    b = np.empty((nblocks, 22), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:6] = qh
    b[:, 6:22] = qs
    return b.reshape(-1)


def q5_1_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(5e-4, 2e-3, nblocks)
    m = g.uniform(-2e-2, 0.0, nblocks)
    qh = g.integers(0, 256, (nblocks, 4), dtype=np.uint8)
    qs = g.integers(0, 256, (nblocks, 16), dtype=np.uint8)
    b = np.empty((nblocks, 24), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:4] = _f16_le_bytes(m)
    b[:, 4:8] = qh
    b[:, 8:24] = qs
    return b.reshape(-1)


def q5_K_blocks(g: np.random.Generator, nblocks: int) -> np.ndarray:
    d = g.uniform(2e-4, 1e-3, nblocks)
    dmin = g.uniform(0.0, 5e-4, nblocks)
    scales = g.integers(0, 256, (nblocks, 12), dtype=np.uint8)
    qh = g.integers(0, 256, (nblocks, 32), dtype=np.uint8)
    qs = g.integers(0, 256, (nblocks, 128), dtype=np.uint8)
    b = np.empty((nblocks, 176), dtype=np.uint8)
    b[:, 0:2] = _f16_le_bytes(d)
    b[:, 2:4] = _f16_le_bytes(dmin)
    b[:, 4:16] = scales
    b[:, 16:48] = qh
    b[:, 48:176] = qs
    return b.reshape(-1)


def f32_elems(g: np.random.Generator, n: int) -> np.ndarray:
    return g.normal(0.0, 0.02, n).astype("<f4").view(np.uint8)


def f16_elems(g: np.random.Generator, n: int) -> np.ndarray:
    return g.normal(0.0, 0.02, n).astype(np.float32).astype("<f2").view(np.uint8)


def bf16_elems(g: np.random.Generator, n: int) -> np.ndarray:
    upper = (g.normal(0.0, 0.02, n).astype("<f4").view("<u4") >> 16).astype("<u2")
    return upper.view(np.uint8)


_DRAW = {F32: f32_elems, F16: f16_elems, BF16: bf16_elems, Q4_K: q4_K_blocks, Q6_K: q6_K_blocks, Q8_0: q8_0_blocks, Q4_0: q4_0_blocks, Q5_0: q5_0_blocks,
         Q5_1: q5_1_blocks, Q5_K: q5_K_blocks}


def nblocks(qtype: int, N: int, K: int) -> int:
    qk, _ = BLOCK[qtype]
    if (N * K) % qk:
        raise ValueError(f"N*K={N * K} is not a whole number of {qk}-element blocks")
    return N * K // qk


def weight_bytes(g: np.random.Generator, qtype: int, N: int, K: int) -> np.ndarray:
    """Flat block stream of a weight W[N,K] (element (n,k) = flat n*K+k)."""
    return _DRAW[qtype](g, nblocks(qtype, N, K))


def activations(g: np.random.Generator, M: int, K: int) -> np.ndarray:
    """X[M,K] ~ N(0,1) rounded to f16 (numpy float16 array)."""
    return g.standard_normal((M, K), dtype=np.float32).astype(np.float16)


@dataclass
class Weight:
    name: str
    qtype: int
    N: int
    K: int
    data: np.ndarray  # uint8 flat block stream


# Layer shapes (name, type, N rows = output features, K = input features).
QWEN25_7B = [("q", Q4_K, 3584, 3584), ("k", Q4_K, 512, 3584), ("v", Q4_K, 512, 3584),
             ("o", Q4_K, 3584, 3584), ("gate", Q4_K, 18944, 3584),
             ("up", Q4_K, 18944, 3584), ("down", Q6_K, 3584, 18944)]
LLAMA31_8B = [("q", Q4_K, 4096, 4096), ("k", Q4_K, 1024, 4096), ("v", Q4_K, 1024, 4096),
              ("o", Q4_K, 4096, 4096), ("gate", Q4_K, 14336, 4096),
              ("up", Q4_K, 14336, 4096), ("down", Q4_K, 4096, 14336)]
Q8_0_PAIR = [("w1", Q8_0, 3584, 18944), ("w2", Q8_0, 18944, 3584)]
SINGLE_896 = [("w", Q4_K, 896, 896)]
# The other block formats (Q4_0 / Q5_0 / Q5_1 / Q5_K), each at the 7B gate
# (18944 x 3584) and down (3584 x 18944) shapes.
# Float weights at the Llama-3.1-8B layer's shapes (K = 4096 and 14336 rows
# are multiples of 2048 bytes in f16, so their copies are row-padded).
FLOAT_LAYER = [(f"{TYPE_NAME[t]}_{nm}", t, n, k) for t in (F16, BF16)
               for nm, n, k in (("q", 4096, 4096), ("gate", 14336, 4096), ("down", 4096, 14336))]
MORE_FORMATS = [(f"{TYPE_NAME[t]}_{nm}", t, n, k) for t in (Q4_0, Q5_0, Q5_1, Q5_K)
                for nm, n, k in (("gate", 18944, 3584), ("down", 3584, 18944))]

WORKLOADS = {
    # name: (weights, token counts M)
    "q4k_896": (SINGLE_896, [128]),
    "qwen2.5-7b_layer": (QWEN25_7B, [2048]),
    "llama3.1-8b_layer": (LLAMA31_8B, [512]),
    "q8_0_pair": (Q8_0_PAIR, [128, 1024]),
    "more_formats": (MORE_FORMATS, [32, 2048]),
    "float_layer": (FLOAT_LAYER, [512]),
    "small_m_sweep": ([w for w in QWEN25_7B if w[0] in ("gate", "up", "down")],
                      [1, 8, 32, 128, 129, 192, 256, 512, 2048]),
}


def workload(name: str, seed: int = 0, max_m: int | None = None):
    """Weights of a named workload and one activation matrix per distinct K.

    Returns (weights, xs) where xs maps K -> X[max(M), K] (f16).  Smaller M
    use the leading rows.  Draw order: every weight in list order, then one
    X per distinct K in order of first appearance.
    """
    shapes, ms = WORKLOADS[name]
    g = rng(seed)
    weights = [Weight(n, t, N, K, weight_bytes(g, t, N, K)) for (n, t, N, K) in shapes]
    M = max_m if max_m is not None else max(ms)
    xs = {}
    for w in weights:
        if w.K not in xs:
            xs[w.K] = activations(g, M, w.K)
    return weights, xs
