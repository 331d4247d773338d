"""Test-side Q4_K *packer*: chosen fields -> 144 block bytes.

Written from the GGUF Q4_K super-block description (the format named by the
"UD-Q4_K_XL" distribution in "Layer Package Repository Spec", section
"Repository Identity"), independently of the oracle's unpacker, so that a
pack -> unpack round trip pins the oracle's reading of the layout:

  [d: binary16][dmin: binary16][12 scale bytes][128 quant bytes]
  scale bytes: bytes 0-3 carry sc_0..sc_3 in their low 6 bits and the top two
  bits of sc_4..sc_7 in their high 2 bits; bytes 4-7 do the same for the mins;
  bytes 8-11 carry the low 4 bits of sc_4..sc_7 (low nibble) and of m_4..m_7
  (high nibble).
  quant bytes: chunk c (bytes 32c..32c+31) holds weights 64c..64c+31 in its low
  nibbles and weights 64c+32..64c+63 in its high nibbles.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def pack_scales(sc, m) -> bytes:
    assert len(sc) == 8 and len(m) == 8
    assert all(0 <= v < 64 for v in list(sc) + list(m))
    out = bytearray(12)
    for i in range(4):
        out[i] = (sc[i] & 0x3F) | ((sc[i + 4] >> 4) << 6)
        out[i + 4] = (m[i] & 0x3F) | ((m[i + 4] >> 4) << 6)
        out[i + 8] = (sc[i + 4] & 0x0F) | ((m[i + 4] & 0x0F) << 4)
    return bytes(out)


def pack_quants(q) -> bytes:
    assert len(q) == 256 and all(0 <= v < 16 for v in q)
    out = bytearray(128)
    for c in range(4):
        for l in range(32):
            out[32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return bytes(out)


def pack_block(d_bits: int, dmin_bits: int, sc, m, q) -> bytes:
    head = int(d_bits).to_bytes(2, "little") + int(dmin_bits).to_bytes(2, "little")
    blk = head + pack_scales(sc, m) + pack_quants(q)
    assert len(blk) == 144
    return blk


def half_bits(value: float) -> int:
    """binary16 bits of a value (numpy's round-to-nearest-even conversion)."""
    return int(np.array([value], dtype=np.float16).view(np.uint16)[0])


def half_fraction(bits: int) -> Fraction:
    """Exact rational value of binary16 bits, via numpy's decoder (library)."""
    v = np.array([bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
    return Fraction(float(v))


def exact_weights(d_bits: int, dmin_bits: int, sc, m, q) -> list[Fraction]:
    """Weights of a block from its fields, in exact rationals."""
    d = half_fraction(d_bits)
    dmin = half_fraction(dmin_bits)
    return [d * sc[i // 32] * q[i] - dmin * m[i // 32] for i in range(256)]


def random_fields(rng: np.random.Generator):
    d_bits = half_bits(rng.uniform(1e-3, 2e-2))
    dmin_bits = half_bits(rng.uniform(1e-3, 2e-2))
    sc = [int(v) for v in rng.integers(0, 64, 8)]
    m = [int(v) for v in rng.integers(0, 64, 8)]
    q = [int(v) for v in rng.integers(0, 16, 256)]
    return d_bits, dmin_bits, sc, m, q
