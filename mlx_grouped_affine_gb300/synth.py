"""Seeded synthetic inputs for MLX grouped affine quantization.

This module only draws random numbers; it holds none of the method's
arithmetic (no unpacking, no dequantization, no matmul), so both the CUDA
path and the CPU oracle may use it.

* Codes uniform on [0, 2^bits - 1] packed LSB-first into uint32 words are
  drawn as uniformly random words: every bit of the packed stream is an
  independent fair bit, which is exactly a row of independent uniform codes.
* bf16 values are drawn in fp32 and keep their top 16 bits; fp16 values are
  numpy's float16 conversion of the fp32 draws; fp32 values are the draws.
* Scales are uniform on [lo, hi]; biases are -scale * 2^(bits-1) plus
  N(0, sigma) noise, so that dequantized weights are centred on zero.
* x is N(0, 1) in bf16; row indices are uniform on [0, table_rows).

Every generator takes an integer seed and uses numpy's PCG64.
"""
from dataclasses import dataclass

import numpy as np


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _top16(values):
    """bf16 bit patterns: the top half of the fp32 bit patterns."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def as_dtype(values, dtype):
    """fp32 draws stored as dtype: "f32" float32 values, "bf16" the top 16
    bits, "f16" the bit patterns of numpy's float16 conversion."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    if dtype == "f32":
        return v
    if dtype == "bf16":
        return _top16(v)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    raise ValueError(dtype)


@dataclass
class QuantWeight:
    """A packed weight: the packed codes, scales and biases, host arrays."""
    packed: np.ndarray   # uint32 [rows, cols*bits/32]
    scales: np.ndarray   # [rows, cols/group_size]: bf16 bit patterns (uint16) by default
    biases: np.ndarray   # same dtype as scales
    rows: int
    cols: int
    bits: int
    group_size: int
    sb_dtype: str = "bf16"   # "bf16", "f16" (uint16 patterns) or "f32" (float32)

    @property
    def nbytes(self):
        return self.packed.nbytes + self.scales.nbytes + self.biases.nbytes


def random_words(g, rows, cols, bits):
    assert (cols * bits) % 32 == 0
    return g.integers(0, 1 << 32, size=(rows, cols * bits // 32), dtype=np.uint32)


def quant_weight(seed, rows, cols, bits, group_size, scale_lo=0.002, scale_hi=0.02,
                 bias_sigma=1e-3):
    """A [rows, cols] weight with the value law described in the module doc."""
    g = rng(seed)
    packed = random_words(g, rows, cols, bits)
    groups = cols // group_size
    s = g.uniform(scale_lo, scale_hi, size=(rows, groups)).astype(np.float32)
    b = (-s * np.float32(2 ** (bits - 1))
         + g.normal(0.0, bias_sigma, size=(rows, groups)).astype(np.float32))
    return QuantWeight(packed, _top16(s), _top16(b), rows, cols, bits, group_size)


def quant_weight_typed(seed, rows, cols, bits, group_size, sb_dtype, scale_lo=0.002,
                       scale_hi=0.02, bias_sigma=1e-3):
    """quant_weight's law with the scales and biases stored as sb_dtype (the
    same draws: for "bf16" this is quant_weight itself)."""
    g = rng(seed)
    packed = random_words(g, rows, cols, bits)
    groups = cols // group_size
    s = g.uniform(scale_lo, scale_hi, size=(rows, groups)).astype(np.float32)
    b = (-s * np.float32(2 ** (bits - 1))
         + g.normal(0.0, bias_sigma, size=(rows, groups)).astype(np.float32))
    return QuantWeight(packed, as_dtype(s, sb_dtype), as_dtype(b, sb_dtype), rows, cols, bits,
                       group_size, sb_dtype)


def x_typed(seed, M, K, dtype):
    """x [M, K] N(0, 1) stored as dtype (x_bf16's draws)."""
    g = rng(seed)
    return as_dtype(g.standard_normal(size=(M, K)).astype(np.float32), dtype)


def x_bf16(seed, M, K):
    """x bf16 bit patterns [M, K], N(0, 1)."""
    g = rng(seed)
    return _top16(g.standard_normal(size=(M, K)).astype(np.float32))


def indices(seed, n, table_rows):
    return rng(seed).integers(0, table_rows, size=n, dtype=np.uint32)


def pr1_weight(seed=0):
    """The small reference case: W [256, 512] at 4 bits, group 64, scales on
    [0.005, 0.02], biases -8*scale + N(0, 0.001)."""
    return quant_weight(seed, 256, 512, 4, 64, scale_lo=0.005, scale_hi=0.02,
                        bias_sigma=1e-3)


# Named workloads, by what they are.  Each entry gives the shapes and laws the
# tests and the benchmark draw their inputs from.
DECODE_SHAPE = (4096, 4096)                 # W [N, K]; x [M, K], M in 1, 4, 8, 16
DECODE_M = (1, 4, 8, 16)
ODD_SHAPE = (11008, 4096)                   # W [N, K] at 1, 2, 3, 5, 6 bits
ODD_BITS = (1, 2, 3, 5, 6)
ODD_GROUPS = (32, 128)
ROWS_TABLE = (128256, 4096)                 # embedding table at 4 bits, group 64
ROWS_GATHER = 4096
PREFILL = dict(M=2048, N=14336, K=4096)     # 4 bits, group 64; also W stored [K, N]
SWEEP_SHAPES = ((4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336))
SWEEP_M = (1, 16, 128, 2048)
SWEEP_BITS = (4, 8)
