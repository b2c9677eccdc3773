"""Seeded synthetic inputs for the bitmap-encoded sparse matmul.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no encoding, no decoding, no products).  Both the CPU
oracle and the CUDA path take their inputs from here, so a parity test feeds
the same bytes to each side.

Recipes (all numpy ``Generator(PCG64(seed))``):

* fp16 weights ``W[M][K]``: N(0, 0.02) drawn in fp32, rounded to fp16.
* Masks, one of
  - ``"bernoulli"``: i.i.d. zero with probability ``s``;
  - ``"uniform"``: a uniformly random subset of exactly ``round(s*M*K)``
    positions is zeroed;
  - ``"magnitude"``: the ``round(s*M*K)`` smallest ``|w|`` are zeroed, ties
    broken by linear index (lowest index zeroed first).  This is the shape of
    magnitude pruning named on the SPDP page (section 3.2) without needing
    trained weights.
* int8 weights: nonzeros uniform in [-127, 127] without 0, then a uniform
  exact-count mask.
* Activations ``X[N][K]`` (K contiguous, the ``[tokens, features]`` layout):
  fp16 N(0, 1), or int8 uniform in [-127, 127].
* Post-ReLU decode activations: ``max(0, z)``, ``z ~ N(-1.0364, 1)``, so about
  85% of the entries are exactly zero (1.0364 is the 0.85 quantile of N(0,1)).
* Per-row scales: U(0.001, 0.01) fp32.

Arrays are returned as numpy arrays: fp16 data as ``uint16`` bit patterns
(the encoder works on raw bits), int8 as ``int8``.
"""
from __future__ import annotations

import numpy as np

RELU_SHIFT = -1.0364  # -Phi^{-1}(0.85): P(z <= 0) = 0.85 for z ~ N(-1.0364, 1)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f16_bits(a32: np.ndarray) -> np.ndarray:
    return a32.astype(np.float16).view(np.uint16)


def _exact_count_mask(g: np.random.Generator, size: int, n_zero: int) -> np.ndarray:
    """Boolean array with exactly ``n_zero`` True entries at uniform positions."""
    zero = np.zeros(size, dtype=bool)
    if n_zero <= 0:
        return zero
    if n_zero >= size:
        zero[:] = True
        return zero
    keys = g.random(size, dtype=np.float32)
    # ties in float32 keys are broken by index inside argpartition's result set
    idx = np.argpartition(keys, n_zero - 1)[:n_zero]
    zero[idx] = True
    return zero


def _magnitude_mask(bits: np.ndarray, n_zero: int) -> np.ndarray:
    """Zero the ``n_zero`` smallest |w| (fp16 bits), ties by linear index."""
    flat = bits.reshape(-1)
    mag = flat & np.uint16(0x7FFF)  # |w| as bits; order of bits == order of values
    zero = np.zeros(flat.size, dtype=bool)
    if n_zero <= 0:
        return zero
    if n_zero >= flat.size:
        zero[:] = True
        return zero
    tau = np.partition(mag, n_zero - 1)[n_zero - 1]
    below = mag < tau
    zero |= below
    need = n_zero - int(below.sum())
    if need > 0:
        ties = np.flatnonzero(mag == tau)[:need]
        zero[ties] = True
    return zero


def weights_f16(M: int, K: int, sparsity: float, mask: str, seed: int,
                std: float = 0.02) -> np.ndarray:
    """fp16 weight bits ``uint16[M][K]`` with the requested zero mask."""
    g = rng(seed)
    w = _f16_bits(g.standard_normal((M, K), dtype=np.float32) * np.float32(std))
    n_zero = int(round(sparsity * M * K))
    if mask == "bernoulli":
        zero = g.random((M, K), dtype=np.float32) < np.float32(sparsity)
    elif mask == "uniform":
        zero = _exact_count_mask(g, M * K, n_zero).reshape(M, K)
    elif mask == "magnitude":
        zero = _magnitude_mask(w, n_zero).reshape(M, K)
    elif mask == "none":
        zero = np.zeros((M, K), dtype=bool)
    else:
        raise ValueError(f"unknown mask {mask!r}")
    w[zero] = 0
    return w


def weights_i8(M: int, K: int, sparsity: float, seed: int) -> np.ndarray:
    """int8 weights: nonzeros uniform in [-127,127]\\{0}, exact-count uniform mask."""
    g = rng(seed)
    mag = g.integers(1, 128, size=(M, K), dtype=np.int16)
    sign = g.integers(0, 2, size=(M, K), dtype=np.int16) * 2 - 1
    w = (mag * sign).astype(np.int8)
    zero = _exact_count_mask(g, M * K, int(round(sparsity * M * K))).reshape(M, K)
    w[zero] = 0
    return w


def weights_int(M: int, K: int, bits: int, sparsity: float, seed: int, exact: bool = True) -> np.ndarray:
    """int8 containers of b-bit weights: nonzeros uniform over the signed
    b-bit range without 0; an exact-count uniform mask, or (exact=False) an
    i.i.d. Bernoulli(sparsity) one."""
    g = rng(seed)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    w = g.integers(lo, hi, size=(M, K), dtype=np.int8)   # lo .. hi - 1
    w[w >= 0] += 1                                       # skip 0: lo .. -1, 1 .. hi
    if exact:
        zero = _exact_count_mask(g, M * K, int(round(sparsity * M * K))).reshape(M, K)
    else:
        zero = g.random((M, K), dtype=np.float32) < sparsity
    w[zero] = 0
    return w


def activations_int(N: int, K: int, bits: int, seed: int) -> np.ndarray:
    """int8 containers of b-bit activations, uniform over the signed range."""
    g = rng(seed)
    return g.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=(N, K), dtype=np.int16).astype(np.int8)


def activations_f16(N: int, K: int, seed: int) -> np.ndarray:
    """fp16 bits ``uint16[N][K]``, N(0, 1)."""
    g = rng(seed)
    return _f16_bits(g.standard_normal((N, K), dtype=np.float32))


def activations_relu_f16(K: int, seed: int, shift: float = RELU_SHIFT) -> np.ndarray:
    """fp16 bits ``uint16[K]``: ``max(0, z)``, ``z ~ N(shift, 1)`` (~85% zeros)."""
    g = rng(seed)
    z = g.standard_normal(K, dtype=np.float32) + np.float32(shift)
    return _f16_bits(np.maximum(z, np.float32(0.0)))


def activations_i8(N: int, K: int, seed: int) -> np.ndarray:
    g = rng(seed)
    return g.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8)


def row_scales(M: int, seed: int) -> np.ndarray:
    g = rng(seed)
    return g.uniform(0.001, 0.01, size=M).astype(np.float32)


def small_int_f16(shape, lo: int, hi: int, seed: int, sparsity: float = 0.0) -> np.ndarray:
    """fp16 bits of small integers in [lo, hi], with an i.i.d. zero mask.

    With |w|, |x| <= 8 and K <= 256 every partial sum of a product is an
    integer below 2^11, so fp16 and fp32 represent it exactly and the result
    of ``W x`` has exactly one correct fp16 value.
    """
    g = rng(seed)
    v = g.integers(lo, hi + 1, size=shape).astype(np.float32)
    if sparsity > 0:
        v[g.random(shape) < sparsity] = 0
    return _f16_bits(v)


def seed_for(config: int, variant: int) -> int:
    """Seed convention: 1000 + 10*config + variant."""
    return 1000 + 10 * config + variant
