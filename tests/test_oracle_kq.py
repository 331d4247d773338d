"""Pins of the oracle's other k-quant formats (q2_K, q3_K, Q5_K, Q6_K).

The pages name these formats and print none of their bytes; the oracle reads
them as the GGUF k-quant super-blocks.  These tests pin that reading against
things other than itself: an independent byte-wise packer (round trip against
exact rational weights), Q5_K against the pinned Q4_K (identical when every
fifth bit is clear), q3_K against q2_K (identical for non-negative quants with
matching scales and zero mins), single-weight probes of every position,
numpy's own rounding, and a library matmul.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from _kq_fields import (exact_q2k, exact_q3k, frac_to_f64, pack_q2k, pack_q3k, pack_q5k, pack_q6k,
                        random_block)
from _q4k_fields import half_bits, pack_block, random_fields

FMTS = (2, 3, 5, 6)


@pytest.mark.parametrize("fmt", FMTS)
def test_pack_unpack_round_trip_is_exact(fmt):
    rng = np.random.default_rng(100 + fmt)
    blocks, want = [], []
    for _ in range(24):
        b, w = random_block(fmt, rng)
        blocks.append(b)
        want.append(frac_to_f64(w))
    raw = np.frombuffer(b"".join(blocks), np.uint8)
    got = oracle.kq_dequant_f64(fmt, raw, 24, 256)
    assert np.array_equal(got, np.stack(want))
    # the same blocks as 3 rows of 8 super-blocks (row layout)
    got2 = oracle.kq_dequant_f64(fmt, raw, 3, 2048)
    assert np.array_equal(got2.reshape(24, 256), np.stack(want))


def test_q5k_with_clear_fifth_bits_equals_q4k():
    rng = np.random.default_rng(110)
    q4, q5 = [], []
    for _ in range(16):
        d, dm, sc, m, q = random_fields(rng)           # q in 0..15
        q4.append(pack_block(d, dm, sc, m, q))
        q5.append(pack_q5k(d, dm, sc, m, q))
    a = oracle.dequant_f64(np.frombuffer(b"".join(q4), np.uint8), 16, 256)
    b = oracle.kq_dequant_f64(5, np.frombuffer(b"".join(q5), np.uint8), 16, 256)
    assert np.array_equal(a, b)
    # and the Q4_K id of the generic path is the Q4_K oracle itself
    c = oracle.kq_dequant_f64(4, np.frombuffer(b"".join(q4), np.uint8), 16, 256)
    assert np.array_equal(a, c)


def test_q3k_with_set_mask_bits_equals_q2k_with_matching_scales():
    # q3_K weight d (sc3 - 32) q for q >= 0 (mask bit set, low bits = q) equals
    # q2_K weight d sc2 q - 0 * m with sc2 = sc3 - 32 in 1..15
    rng = np.random.default_rng(111)
    for _ in range(8):
        d = half_bits(rng.uniform(1e-3, 2e-2))
        sc2 = [int(v) for v in rng.integers(1, 16, 16)]
        q = [int(v) for v in rng.integers(0, 4, 256)]
        b2 = pack_q2k(d, half_bits(0.0), sc2, [0] * 16, q)
        b3 = pack_q3k(d, [v + 32 for v in sc2], q)
        w2 = oracle.kq_dequant_f64(2, np.frombuffer(b2, np.uint8), 1, 256)
        w3 = oracle.kq_dequant_f64(3, np.frombuffer(b3, np.uint8), 1, 256)
        assert np.array_equal(w2, w3)
        assert np.array_equal(w2[0], frac_to_f64(exact_q2k(d, half_bits(0.0), sc2, [0] * 16, q)))
        assert np.array_equal(w3[0], frac_to_f64(exact_q3k(d, [v + 32 for v in sc2], q)))


def _probe_blocks(fmt):
    """Block i: every weight zero except weight i (value d * 1 * 1)."""
    d = half_bits(0.5)
    out = []
    for i in range(256):
        if fmt == 2:
            q = [0] * 256
            q[i] = 1
            out.append(pack_q2k(d, half_bits(0.0), [1] * 16, [0] * 16, q))
        elif fmt == 3:
            q = [0] * 256
            q[i] = 1
            out.append(pack_q3k(d, [33] * 16, q))
        elif fmt == 5:
            q = [0] * 256
            q[i] = 1
            out.append(pack_q5k(d, half_bits(0.0), [1] * 8, [0] * 8, q))
        else:
            q = [0] * 256
            q[i] = 1
            out.append(pack_q6k(d, [1] * 16, q))
    return np.frombuffer(b"".join(out), np.uint8)


@pytest.mark.parametrize("fmt", FMTS)
def test_single_weight_probes_land_at_their_position(fmt):
    w = oracle.kq_dequant_f64(fmt, _probe_blocks(fmt), 256, 256)
    assert np.array_equal(w, np.eye(256) * 0.5)


@pytest.mark.parametrize("fmt", FMTS)
def test_fp32_and_bf16_are_the_rounded_exact_weights(fmt):
    rng = np.random.default_rng(120 + fmt)
    raw = np.frombuffer(b"".join(random_block(fmt, rng)[0] for _ in range(32)), np.uint8)
    e = oracle.kq_dequant_f64(fmt, raw, 4, 2048)
    f = oracle.kq_dequant_f32(fmt, raw, 4, 2048)
    assert np.array_equal(f, e.astype(np.float32))
    import torch
    bf = oracle.kq_dequant_bf16(fmt, raw, 4, 2048)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, want)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_matches_library_matmul(fmt):
    rng = np.random.default_rng(130 + fmt)
    n, k = 12, 1024
    raw = np.frombuffer(b"".join(random_block(fmt, rng)[0] for _ in range(n * k // 256)), np.uint8)
    x = rng.standard_normal((3, k)).astype(np.float32)
    import torch
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    y, s = oracle.kq_gemv(fmt, raw, n, k, xbits)
    w = oracle.kq_dequant_f64(fmt, raw, n, k)
    xf = xb.to(torch.float64).numpy()
    assert np.all(np.abs(y - xf @ w.T) <= 1e-12 * (np.abs(xf) @ np.abs(w).T) + 1e-300)
    assert np.allclose(s, np.abs(xf) @ np.abs(w).T, rtol=1e-12, atol=0)
