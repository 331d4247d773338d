"""Test-side packers for the other k-quant super-blocks: chosen fields -> block
bytes, written from the GGUF k-quant format descriptions (the q2_K / q3_K
routed-down recipes and the Q5_K / Q6_K tensors of "_XL" mixes named in "Layer
Package Repository Spec", section "Policy Resolution") byte by byte,
independently of the oracle's per-weight unpacking, so that a pack -> unpack
round trip pins the oracle's reading of each layout.  Each packer also states
the exact weights of its block.

Weight i of a 256-weight super-block belongs to sub-block i // 16 (q2_K, q3_K,
Q6_K: 16 sub-blocks of 16) or i // 32 (Q5_K: 8 of 32).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from _q4k_fields import half_bits, half_fraction, pack_scales


def _h(bits: int) -> bytes:
    return int(bits).to_bytes(2, "little")


def pack_q2k(d_bits, dmin_bits, sc, m, q) -> bytes:
    """sc, m: 16 values 0..15; q: 256 values 0..3.
    [16 scale bytes: sc | m << 4][64 quant bytes][d][dmin]; quant byte 32h + l
    holds, in bit pairs 0-1, 2-3, 4-5, 6-7, weights 128h + l, 128h + 32 + l,
    128h + 64 + l, 128h + 96 + l."""
    assert len(sc) == 16 and len(m) == 16 and len(q) == 256
    scales = bytes((sc[j] & 15) | ((m[j] & 15) << 4) for j in range(16))
    qs = bytearray(64)
    for h in range(2):
        for l in range(32):
            qs[32 * h + l] = sum((q[128 * h + 32 * g + l] & 3) << (2 * g) for g in range(4))
    blk = scales + bytes(qs) + _h(d_bits) + _h(dmin_bits)
    assert len(blk) == 84
    return blk


def exact_q2k(d_bits, dmin_bits, sc, m, q):
    d, dmin = half_fraction(d_bits), half_fraction(dmin_bits)
    return [d * sc[i // 16] * q[i] - dmin * m[i // 16] for i in range(256)]


def pack_q3k(d_bits, sc, q) -> bytes:
    """sc: 16 six-bit values 0..63 (the weight uses sc - 32); q: 256 values -4..3
    stored as u = q + 4: the low two bits of u in the quant bytes (laid out as
    q2_K's), the top bit of u in the mask bytes (mask byte l, bit 4h + g, for
    weight 128h + 32g + l).  Scale bytes: low nibbles of sc_0..7 in the low
    nibbles of bytes 0..7, of sc_8..15 in their high nibbles; the top two bits
    of sc_j in bits 2(j // 4) of byte 8 + j % 4."""
    assert len(sc) == 16 and len(q) == 256
    u = [v + 4 for v in q]
    assert all(0 <= v < 8 for v in u) and all(0 <= v < 64 for v in sc)
    hm = bytearray(32)
    qs = bytearray(64)
    for h in range(2):
        for g in range(4):
            for l in range(32):
                uv = u[128 * h + 32 * g + l]
                qs[32 * h + l] |= (uv & 3) << (2 * g)
                hm[l] |= (uv >> 2) << (4 * h + g)
    s = bytearray(12)
    for j in range(16):
        if j < 8:
            s[j] |= sc[j] & 15
        else:
            s[j - 8] |= (sc[j] & 15) << 4
        s[8 + j % 4] |= (sc[j] >> 4) << (2 * (j // 4))
    blk = bytes(hm) + bytes(qs) + bytes(s) + _h(d_bits)
    assert len(blk) == 110
    return blk


def exact_q3k(d_bits, sc, q):
    d = half_fraction(d_bits)
    return [d * (sc[i // 16] - 32) * q[i] for i in range(256)]


def pack_q5k(d_bits, dmin_bits, sc, m, q) -> bytes:
    """sc, m: 8 six-bit values (packed as Q4_K's); q: 256 values 0..31.
    [d][dmin][12 scale bytes][32 high-bit bytes][128 nibble bytes]: nibble byte
    32c + l holds the low 4 bits of weights 64c + l (low nibble) and 64c + 32 + l
    (high nibble); high-bit byte l holds bit 4 of weight 64c + 32e + l in bit
    2c + e."""
    assert len(q) == 256 and all(0 <= v < 32 for v in q)
    qh = bytearray(32)
    qs = bytearray(128)
    for c in range(4):
        for l in range(32):
            lo, hi = q[64 * c + l], q[64 * c + 32 + l]
            qs[32 * c + l] = (lo & 15) | ((hi & 15) << 4)
            qh[l] |= ((lo >> 4) << (2 * c)) | ((hi >> 4) << (2 * c + 1))
    blk = _h(d_bits) + _h(dmin_bits) + pack_scales(sc, m) + bytes(qh) + bytes(qs)
    assert len(blk) == 176
    return blk


def exact_q5k(d_bits, dmin_bits, sc, m, q):
    d, dmin = half_fraction(d_bits), half_fraction(dmin_bits)
    return [d * sc[i // 32] * q[i] - dmin * m[i // 32] for i in range(256)]


def pack_q6k(d_bits, sc, q) -> bytes:
    """sc: 16 int8 scales; q: 256 values -32..31 stored as u = q + 32 (6 bits).
    [128 low-nibble bytes][64 high-bit bytes][16 scale bytes][d]: for half h,
    position l and quarter e (weight 128h + 32e + l): the low 4 bits of u go to
    byte 64h + l + 32(e % 2), low nibble for e < 2, high nibble for e >= 2; the
    top 2 bits of u go to bits 2e, 2e + 1 of byte 128 + 32h + l."""
    assert len(sc) == 16 and len(q) == 256
    u = [v + 32 for v in q]
    assert all(0 <= v < 64 for v in u) and all(-128 <= v < 128 for v in sc)
    ql = bytearray(128)
    qh = bytearray(64)
    for h in range(2):
        for e in range(4):
            for l in range(32):
                uv = u[128 * h + 32 * e + l]
                ql[64 * h + l + 32 * (e % 2)] |= (uv & 15) << (0 if e < 2 else 4)
                qh[32 * h + l] |= (uv >> 4) << (2 * e)
    scales = bytes((v + 256) % 256 for v in sc)
    blk = bytes(ql) + bytes(qh) + scales + _h(d_bits)
    assert len(blk) == 210
    return blk


def exact_q6k(d_bits, sc, q):
    d = half_fraction(d_bits)
    return [d * sc[i // 16] * q[i] for i in range(256)]


def random_block(fmt: int, rng: np.random.Generator):
    """(block bytes, exact weights as Fractions) for format id fmt."""
    d = half_bits(rng.uniform(1e-3, 2e-2))
    dm = half_bits(rng.uniform(1e-3, 2e-2))
    if fmt == 2:
        sc, m = [int(v) for v in rng.integers(0, 16, 16)], [int(v) for v in rng.integers(0, 16, 16)]
        q = [int(v) for v in rng.integers(0, 4, 256)]
        return pack_q2k(d, dm, sc, m, q), exact_q2k(d, dm, sc, m, q)
    if fmt == 3:
        sc = [int(v) for v in rng.integers(0, 64, 16)]
        q = [int(v) for v in rng.integers(-4, 4, 256)]
        return pack_q3k(d, sc, q), exact_q3k(d, sc, q)
    if fmt == 5:
        sc, m = [int(v) for v in rng.integers(0, 64, 8)], [int(v) for v in rng.integers(0, 64, 8)]
        q = [int(v) for v in rng.integers(0, 32, 256)]
        return pack_q5k(d, dm, sc, m, q), exact_q5k(d, dm, sc, m, q)
    if fmt == 6:
        sc = [int(v) for v in rng.integers(-128, 128, 16)]
        q = [int(v) for v in rng.integers(-32, 32, 256)]
        return pack_q6k(d, sc, q), exact_q6k(d, sc, q)
    raise ValueError(fmt)


def frac_to_f64(ws) -> np.ndarray:
    return np.array([float(Fraction(v)) for v in ws], dtype=np.float64)
