"""Counter-based random numbers shared by the host and the device weight fill.

Every synthetic expert weight is a pure function of (key, flat index), so the
host can regenerate any expert slice that the GPU filled, bit for bit, without
copying anything back from the device.

The mixing function is SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014): the i-th output of a
generator seeded with ``s`` is ``mix64(s + (i + 1) * GOLDEN)`` with the
finaliser below.  We use it in counter mode.  ``workload/fill.cu`` implements
the same definition in CUDA; ``tests/test_workload.py`` checks the two agree.

Value maps (all exact in their storage type, so no rounding mode is involved):

* ``grid8``: top byte ``b`` of the hash -> ``(2b - 255) * 2^-13``.  Odd
  integers in [-255, 255] scaled by a power of two: exactly representable in
  bf16 (8 significant bits) and fp32.  Standard deviation about 0.018.
* ``e4m3``: top byte of the hash taken as an OCP FP8 E4M3 code; the two NaN
  codes (S.1111.111) are replaced by the code one below (+-448).
* ``scale``: fp32 ``(1 + f * 2^-23) * 2^-SCALE_EXP`` with ``f`` the 23 bits
  below the top byte; exact in fp32.
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

# Scale exponent for the FP8 block scales: |e4m3| <= 448, the code mix has
# an rms near 100, so 2^-13 brings the effective weights to O(0.02).
SCALE_EXP = 13

KIND_GRID8_BF16 = 0
KIND_GRID8_F32 = 1
KIND_E4M3 = 2
KIND_SCALE_F32 = 3


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """Key of one named stream: the (stream+1)-th SplitMix64 output of ``seed``."""
    return mix64_int(seed + (stream + 1) * GOLDEN)


def hash_at(key: int, idx: np.ndarray) -> np.ndarray:
    """``mix64(key + (idx + 1) * GOLDEN)`` for a uint64 index array."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = idx + np.uint64(1)
        z *= np.uint64(GOLDEN)
        z += np.uint64(key)
        t = z >> np.uint64(30)
        z ^= t
        z *= np.uint64(MIX1)
        np.right_shift(z, np.uint64(27), out=t)
        z ^= t
        z *= np.uint64(MIX2)
        np.right_shift(z, np.uint64(31), out=t)
        z ^= t
    return z


def grid8_values(h: np.ndarray) -> np.ndarray:
    """fp32 values of the ``grid8`` map (exact in bf16 too)."""
    b = (h >> np.uint64(56)).astype(np.int64)
    return ((2 * b - 255).astype(np.float32) * np.float32(2.0 ** -13)).astype(np.float32)


def grid8_bf16_bits(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of the ``grid8`` map."""
    v = grid8_values(h)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e4m3_codes(h: np.ndarray) -> np.ndarray:
    c = (h >> np.uint64(56)).astype(np.uint8)
    nan = (c & np.uint8(0x7F)) == np.uint8(0x7F)
    c = c.copy()
    c[nan] ^= np.uint8(1)
    return c


def scale_values(h: np.ndarray) -> np.ndarray:
    f = ((h >> np.uint64(33)) & np.uint64(0x7FFFFF)).astype(np.float64)
    v = (1.0 + f * 2.0 ** -23) * 2.0 ** -SCALE_EXP
    return v.astype(np.float32)


def fill_host(kind: int, key: int, idx0: int, n: int, chunk: int = 1 << 20) -> np.ndarray:
    """Host twin of the device fill: elements ``idx0 .. idx0+n-1`` of a stream.

    Returns uint16 (bf16 bits), float32 or uint8 (e4m3 codes) by ``kind``.
    Works in chunks so the uint64 temporaries stay small.
    """
    dt = {KIND_GRID8_BF16: np.uint16, KIND_GRID8_F32: np.float32, KIND_E4M3: np.uint8,
          KIND_SCALE_F32: np.float32}
    if kind not in dt:
        raise ValueError(f"unknown fill kind {kind}")
    out = np.empty(n, dtype=dt[kind])
    fn = {KIND_GRID8_BF16: grid8_bf16_bits, KIND_GRID8_F32: grid8_values, KIND_E4M3: e4m3_codes,
          KIND_SCALE_F32: scale_values}[kind]
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        out[a:b] = fn(hash_at(key, np.arange(idx0 + a, idx0 + b, dtype=np.uint64)))
    return out
