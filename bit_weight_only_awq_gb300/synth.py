"""Seeded synthetic inputs for the AWQ W4A16 / W4A8 linear layer.

This module only draws random numbers and holds workload shape tables; it
contains none of the layer's arithmetic (no packing, dequantization or
products).  Tests, the bench harness and the oracle-side checks all draw their
inputs from here, so the CUDA path and the oracle always see the same bytes.

Distributions (the synthetic stand-in for trained checkpoints, which the
pages benchmark but which are not available here):

* 4-bit weight codes and zero points uniform on 0..15.  The eight nibbles of a
  packed int32 are independent and uniform exactly when the 32-bit word is
  uniform, so packed ``qweight`` / ``qzeros`` words are drawn as uniform
  32-bit integers directly.
* scales fp16, uniform on [0.002, 0.02] (W4A16) or [0.001, 0.01] (W4A8
  per-channel), rounded to fp16.
* activations fp16, standard normal, rounded to fp16 (``with_x=False`` leaves them out, for a caller
  that draws them itself).
"""

from __future__ import annotations

import numpy as np

GROUP_SIZE = 128

# Llama-2-7B linear shapes (K, N) used for the decode (M <= 8) sweep.
LLAMA2_7B_DECODE = (
    ("qkv", 4096, 12288),
    ("o_proj", 4096, 4096),
    ("gate_up", 4096, 22016),
    ("down", 11008, 4096),
)
DECODE_M = (1, 2, 4, 8)

# Mistral-7B (GQA) linear shapes (K, N) used for the prefill sweep.
MISTRAL_7B_PREFILL = (
    ("qkv", 4096, 6144),
    ("o_proj", 4096, 4096),
    ("gate_up", 4096, 28672),
    ("down", 14336, 4096),
)
PREFILL_M = (256, 1024, 4096, 8192)

# Llama-3.1-8B decoder-layer linear stack, swept over the batch size.
LLAMA31_8B_STACK = (
    ("qkv", 4096, 6144),
    ("o_proj", 4096, 4096),
    ("gate_up", 4096, 28672),
    ("down", 14336, 4096),
)
CROSSOVER_M = (1, 8, 16, 64, 256, 1024)

# W4A8 GEMM shape and token counts.
W4A8_SHAPE = (21760, 8192)  # (K, N)
W4A8_M = (1, 16, 64, 256, 1024, 4096)


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def random_words(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """Uniform 32-bit words viewed as int32 (eight independent uniform nibbles each), from random bytes."""
    return np.frombuffer(rng.bytes(rows * cols * 4), dtype=np.int32).reshape(rows, cols).copy()


def random_codes(rows: int, cols: int, seed: int, high: int = 16) -> np.ndarray:
    """Codes uniform on 0..high-1 as uint8 [rows, cols] (high may exceed 16 to exercise clamping)."""
    return rng_for(seed).integers(0, high, size=(rows, cols), dtype=np.int64).astype(np.uint8)


def activations(rng: np.random.Generator, m: int, k: int) -> np.ndarray:
    return rng.standard_normal((m, k), dtype=np.float32).astype(np.float16)


def awq_problem(m: int, k: int, n: int, seed: int, group_size: int = GROUP_SIZE,
                symmetric: bool = False, with_x: bool = True) -> dict:
    """Inputs of one W4A16 AWQ linear call.

    Returns a dict with ``x`` fp16 [M, K], ``qweight`` int32 [K, N/8],
    ``qzeros`` int32 [K/g, N/8] (None when symmetric), ``scales`` fp16 [K/g, N].
    """
    if n % 8 or k % group_size:
        raise ValueError("N must be a multiple of 8 and K a multiple of the group size")
    rng = rng_for(seed)
    qweight = random_words(rng, k, n // 8)
    qzeros = None if symmetric else random_words(rng, k // group_size, n // 8)
    scales = rng.uniform(0.002, 0.02, size=(k // group_size, n)).astype(np.float16)
    x = activations(rng, m, k) if with_x else None
    return {"x": x, "qweight": qweight, "qzeros": qzeros, "scales": scales,
            "group_size": group_size}


def w4a8_problem(m: int, k: int, n: int, seed: int, with_x: bool = True) -> dict:
    """Inputs of one W4A8 call: fp16 activations, packed u = q + 8 weights, fp16 channel scales."""
    if n % 8:
        raise ValueError("N must be a multiple of 8")
    rng = rng_for(seed)
    wq = random_words(rng, k, n // 8)
    s_ch = rng.uniform(0.001, 0.01, size=(n,)).astype(np.float16)
    x = activations(rng, m, k) if with_x else None
    return {"x": x, "wq": wq, "s_ch": s_ch}


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Synthetic bf16 inputs: the upper 16 bits of each float32 (truncation), as uint16 bit patterns.

    Any bf16 value is a valid input; truncation is the input recipe here, not the layer's rounding.
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def awq_problem_bf16(m: int, k: int, n: int, seed: int, group_size: int = GROUP_SIZE,
                     symmetric: bool = False, with_x: bool = True) -> dict:
    """Inputs of one bf16 W4A16 AWQ linear call: the W4A16 recipe with bf16 activations
    (N(0, 1)) and bf16 scales (U[0.002, 0.02]), both as uint16 bit patterns."""
    if n % 8 or k % group_size:
        raise ValueError("N must be a multiple of 8 and K a multiple of the group size")
    rng = rng_for(seed)
    qweight = random_words(rng, k, n // 8)
    qzeros = None if symmetric else random_words(rng, k // group_size, n // 8)
    scales = to_bf16_bits(rng.uniform(0.002, 0.02, size=(k // group_size, n)))
    x = to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32)) if with_x else None
    return {"x": x, "qweight": qweight, "qzeros": qzeros, "scales": scales, "group_size": group_size}


def w4a8_group_problem(m: int, k: int, n: int, seed: int, group_size: int = GROUP_SIZE,
                       with_x: bool = True) -> dict:
    """Inputs of one per-group W4A8 call: fp16 activations, packed u = q + 8 weights, integer group
    factors s3 uniform on 1..16 (fp16 [K/g, N]) and fp16 channel scales s2 uniform on [1e-4, 1e-3]."""
    if n % 8 or k % group_size:
        raise ValueError("N must be a multiple of 8 and K a multiple of the group size")
    rng = rng_for(seed)
    wq = random_words(rng, k, n // 8)
    s3 = rng.integers(1, 17, size=(k // group_size, n)).astype(np.float16)
    s2 = rng.uniform(0.0001, 0.001, size=(n,)).astype(np.float16)
    x = activations(rng, m, k) if with_x else None
    return {"x": x, "wq": wq, "s3": s3, "s2": s2, "group_size": group_size}
