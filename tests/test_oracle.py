"""Pins for the CPU oracle: each check ties it to something other than itself
(library decoders, exact rationals, closed forms, invariants, an independent
packer), chosen so that a dropped term, a wrong shift, sign or index fails.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from _q4k_fields import (exact_weights, half_bits, half_fraction, pack_block, pack_quants,
                         pack_scales, random_fields)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4k_handbuilt.txt")


# ---------------------------------------------------------------- scalar decoders

def test_fp16_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_matches_torch_for_every_bit_pattern():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b) & 0xFFFF) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_to_bf16_rne_matches_torch_including_ties():
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(4000).astype(np.float32))
    # exact ties between two bf16 values (dropped half == 0x8000), both parities
    for kept in (0x3F80, 0x3F81, 0x4000, 0x4001, 0xBF80, 0xBF81, 0x7F7F, 0x0001, 0x0080):
        u = np.array([(kept << 16) | 0x8000], dtype=np.uint32)
        vals.append(u.view(np.float32)[0])
        u2 = np.array([(kept << 16) | 0x7FFF, (kept << 16) | 0x8001], dtype=np.uint32)
        vals.extend(u2.view(np.float32))
    vals += [np.float32(0.0), np.float32(-0.0), np.float32(np.inf), np.float32(-np.inf),
             np.float32(3.4e38), np.float32(1e-40)]
    arr = np.array(vals, dtype=np.float32)
    ref = torch.from_numpy(arr).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in arr], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- layout

def test_scale_unpack_round_trip_every_value_every_slot():
    rng = np.random.default_rng(1)
    for slot in range(16):
        for v in range(64):
            sc = [int(a) for a in rng.integers(0, 64, 8)]
            m = [int(a) for a in rng.integers(0, 64, 8)]
            if slot < 8:
                sc[slot] = v
            else:
                m[slot - 8] = v
            got_sc, got_m = oracle.unpack_scales(pack_scales(sc, m))
            assert got_sc == sc and got_m == m, (slot, v)


def test_quant_positions_round_trip():
    rng = np.random.default_rng(2)
    for _ in range(20):
        q = [int(a) for a in rng.integers(0, 16, 256)]
        qs = pack_quants(q)
        assert [oracle.quant(qs, i) for i in range(256)] == q


def test_quant_single_nonzero_lands_at_its_index():
    for i in range(256):
        q = [0] * 256
        q[i] = 15
        qs = pack_quants(q)
        got = [oracle.quant(qs, t) for t in range(256)]
        assert got == q, i


def _golden_blocks():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, d, dm, sc, m, rule, hexb, _ = [c.strip() for c in line.split("|")]
            rows.append((name, int(d, 16), int(dm, 16), [int(v) for v in sc.split(",")],
                         [int(v) for v in m.split(",")], rule, bytes.fromhex(hexb)))
    return rows


def _closed_form(name, i, sc, m):
    j = i // 32
    F = Fraction
    if name == "ramp":
        return F((j + 1) * (i % 16) - j)
    if name == "max_scales":
        return F(63, 16) * (15 - i % 16) - F(63, 32)
    if name == "high_bits_only":
        return F(0) if j < 4 else F(48 * ((7 * i) % 16) - 48)
    if name == "low_bits_only":
        return F(3 * sc[j] - 2 * m[j])
    if name == "subnormal_d":
        return F(1, 1 << 24) * (j + 1) * (i % 16) - F(1023, 1 << 24) * (8 - j)
    if name == "zero":
        return F(0)
    if name == "negative_d":
        return F(-(i % 16)) + F(1, 2)
    raise KeyError(name)


@pytest.mark.parametrize("row", _golden_blocks(), ids=lambda r: r[0])
def test_handbuilt_blocks_dequantize_to_closed_form(row):
    name, d, dm, sc, m, rule, blk = row
    q = [eval(rule, {}, {"i": i}) % 16 for i in range(256)]
    assert pack_block(d, dm, sc, m, q) == blk          # fixture consistent with its fields
    w = oracle.dequant_f64(np.frombuffer(blk, np.uint8), 1, 256)[0]
    for i in range(256):
        assert Fraction(float(w[i])) == _closed_form(name, i, sc, m), (name, i)


def test_random_blocks_exact_against_rationals():
    rng = np.random.default_rng(3)
    for _ in range(25):
        fields = random_fields(rng)
        blk = pack_block(*fields)
        w = oracle.dequant_f64(np.frombuffer(blk, np.uint8), 1, 256)[0]
        ref = exact_weights(*fields)
        assert all(Fraction(float(a)) == b for a, b in zip(w, ref))


def test_fp32_and_bf16_outputs_are_one_rounding_of_the_exact_value():
    w = synth.q4k_weight(6, 512, seed=11).numpy()
    exact = oracle.dequant_f64(w, 6, 512)
    f32 = oracle.dequant_f32(w, 6, 512)
    assert np.array_equal(f32, exact.astype(np.float32))       # numpy RNE cast
    bf = oracle.dequant_bf16(w, 6, 512)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, ref)
    # every exact value is representable in 22 bits or fewer: fp32 rounding is
    # the only rounding, and for these generated fields it is exact
    assert np.array_equal(f32.astype(np.float64), exact)


# ---------------------------------------------------------------- contraction

def _x_bits(x_bf16: torch.Tensor) -> np.ndarray:
    return x_bf16.view(torch.int16).numpy().view(np.uint16)


def _x_f64(x_bf16: torch.Tensor) -> np.ndarray:
    return x_bf16.to(torch.float64).numpy()


def test_gemv_exact_rational_brute_force_tiny():
    for n, k, batch in ((1, 256, 1), (3, 256, 2), (2, 512, 3)):
        w = synth.q4k_weight(n, k, seed=100 + n + k).numpy()
        x = synth.bf16_normal((batch, k), seed=200 + batch)
        y, s = oracle.gemv(w, n, k, _x_bits(x))
        wq = oracle.dequant_f64(w, n, k)
        xf = _x_f64(x)
        for b in range(batch):
            for r in range(n):
                exact = sum(Fraction(float(wq[r, i])) * Fraction(float(xf[b, i])) for i in range(k))
                mag = sum(abs(Fraction(float(wq[r, i])) * Fraction(float(xf[b, i]))) for i in range(k))
                assert abs(Fraction(float(y[b, r])) - exact) <= Fraction(1, 10**12) * mag
                assert abs(Fraction(float(s[b, r])) - mag) <= Fraction(1, 10**12) * mag


def test_gemv_reduces_to_library_matmul():
    n, k, batch = 37, 1024, 4
    w = synth.q4k_weight(n, k, seed=5).numpy()
    x = synth.bf16_normal((batch, k), seed=6)
    y, s = oracle.gemv(w, n, k, _x_bits(x))
    wq = oracle.dequant_f64(w, n, k)
    ref = _x_f64(x) @ wq.T
    mag = np.abs(_x_f64(x)) @ np.abs(wq).T
    assert np.all(np.abs(y - ref) <= 1e-12 * mag)
    assert np.allclose(s, mag, rtol=1e-12, atol=0)


def test_gemv_unit_vector_picks_a_column_exactly():
    n, k = 9, 512
    w = synth.q4k_weight(n, k, seed=8).numpy()
    wq = oracle.dequant_f64(w, n, k)
    for col in (0, 1, 31, 32, 255, 256, 300, 511):
        x = torch.zeros((1, k), dtype=torch.bfloat16)
        x[0, col] = 1.0
        y, _ = oracle.gemv(w, n, k, _x_bits(x))
        assert np.array_equal(y[0], wq[:, col])


def test_gemv_zero_quant_rows_closed_form():
    rng = np.random.default_rng(9)
    blocks, mins = [], []
    for _ in range(2):                                # one row, k = 512
        d, dm, sc, m, _q = random_fields(rng)
        blocks.append(pack_block(d, dm, sc, m, [0] * 256))
        mins.append([half_fraction(dm) * mj for mj in m])
    w = np.frombuffer(b"".join(blocks), np.uint8)
    x = synth.bf16_normal((1, 512), seed=10)
    xf = [Fraction(float(v)) for v in _x_f64(x)[0]]
    expect = -sum(mins[b][j] * sum(xf[256 * b + 32 * j: 256 * b + 32 * j + 32])
                  for b in range(2) for j in range(8))
    y, _ = oracle.gemv(w, 1, 512, _x_bits(x))
    mag = sum(abs(mins[b][i // 32 % 8] * xf[256 * b + i % 256]) for b in range(2) for i in range(256))
    assert abs(Fraction(float(y[0, 0])) - expect) <= Fraction(1, 10**12) * mag


def test_gemv_homogeneous_in_powers_of_two():
    n, k = 11, 768
    w = synth.q4k_weight(n, k, seed=12).numpy()
    x = synth.bf16_normal((1, k), seed=13)
    y1, _ = oracle.gemv(w, n, k, _x_bits(x))
    for e in range(-3, 4):
        a = 2.0 ** e
        ya, _ = oracle.gemv(w, n, k, _x_bits((x.float() * a).to(torch.bfloat16)))
        assert np.array_equal(ya, y1 * a)


def test_gemv_row_subset_matches_full():
    n, k = 20, 256
    w = synth.q4k_weight(n, k, seed=14).numpy()
    x = synth.bf16_normal((2, k), seed=15)
    y, s = oracle.gemv(w, n, k, _x_bits(x))
    rows = [19, 0, 7, 7]
    ys, ss = oracle.gemv(w, n, k, _x_bits(x), rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(ss, s[:, rows])


def test_gemv_f64_abs_branch_matches_library():
    # oracle_gemv_f64 with use_abs: |W| x, the scale of the MoE error bounds.
    # Against numpy on the oracle's exact weights (pinned above); a dropped
    # fabs would give W |x| instead, which differs on rows with mixed signs.
    n, k = 13, 512
    w = synth.q4k_weight(n, k, seed=31).numpy()
    wq = oracle.dequant_f64(w, n, k)
    xa = np.abs(np.random.default_rng(32).standard_normal((3, k)))
    got = oracle.gemv_f64(w, n, k, xa, use_abs=True)
    assert np.allclose(got, xa @ np.abs(wq).T, rtol=1e-12, atol=0)
    plain = oracle.gemv_f64(w, n, k, xa)
    assert np.all(np.abs(plain - xa @ wq.T) <= 1e-12 * (xa @ np.abs(wq).T))
    assert np.all(got > np.abs(plain))      # mixed-sign rows: |W||x| > |W x|


def _cancel_fields(rng, sc_c_m=((2, 4, 4), (6, 7, 21), (8, 15, 60), (14, 9, 63), (5, 0, 0))):
    """Block fields whose weights are all exactly zero: d = 2^-6, dmin = 2^-5,
    and in every sub-block q = c with d sc c = dmin m (sc c = 2 m)."""
    picks = [sc_c_m[int(i)] for i in rng.integers(0, len(sc_c_m), 8)]
    sc = [p[0] for p in picks]
    m = [p[2] for p in picks]
    q = [picks[i // 32][1] for i in range(256)]
    return half_bits(2.0 ** -6), half_bits(2.0 ** -5), sc, m, q


def test_cancelling_blocks_are_exactly_zero():
    rng = np.random.default_rng(33)
    rows = [b"".join(pack_block(*_cancel_fields(rng)) for _ in range(2)) for _ in range(3)]
    w = np.frombuffer(b"".join(rows), np.uint8)
    assert np.all(oracle.dequant_f64(w, 3, 512) == 0.0)
    for fields in (_cancel_fields(rng) for _ in range(4)):
        assert all(v == 0 for v in exact_weights(*fields))
    y, s = oracle.gemv(w, 3, 512, _x_bits(synth.bf16_normal((2, 512), seed=34)))
    assert np.all(y == 0.0) and np.all(s == 0.0)


# ---------------------------------------------------------------- fused gate/up

def test_glu_is_silu_of_gate_times_up():
    # against two oracle GEMVs (pinned above) and the logistic function of a
    # library; x small enough that g lies in SiLU's curved region
    from scipy.special import expit
    n, k, batch = 23, 768, 3
    wg = synth.q4k_weight(n, k, seed=35).numpy()
    wu = synth.q4k_weight(n, k, seed=36).numpy()
    x = _x_bits(synth.bf16_normal((batch, k), seed=37, sigma=0.02))
    h, g, u, sg, su = oracle.gemv_glu(wg, wu, n, k, x)
    g2, sg2 = oracle.gemv(wg, n, k, x)
    u2, su2 = oracle.gemv(wu, n, k, x)
    assert np.array_equal(g, g2) and np.array_equal(u, u2)
    assert np.array_equal(sg, sg2) and np.array_equal(su, su2)
    assert np.allclose(h, g2 * expit(g2) * u2, rtol=1e-13, atol=0)
    assert np.abs(g).min() < 4.0 and np.abs(g).max() > 0.1   # the curved region is exercised


def test_glu_zero_gate_gives_exact_zero_and_large_gate_gives_up():
    # gate rows of zero weights: silu(0) = 0; gate rows of one large positive
    # weight against x = e_0: silu(g) = g (1 - O(e^-g)), so h = g u
    rng = np.random.default_rng(38)
    k = 256
    zero = pack_block(0, 0, [1] * 8, [0] * 8, [0] * 256)
    big = pack_block(half_bits(1.0), 0, [63] * 8, [0] * 8, [15] + [0] * 255)   # w_0 = 945
    up_blocks = [pack_block(*random_fields(rng)) for _ in range(2)]
    wg = np.frombuffer(zero + big, np.uint8)
    wu = np.frombuffer(b"".join(up_blocks), np.uint8)
    x = torch.zeros((1, k), dtype=torch.bfloat16)
    x[0, 0] = 1.0
    h, g, u, _, _ = oracle.gemv_glu(wg, wu, 2, k, _x_bits(x))
    assert h[0, 0] == 0.0 and g[0, 0] == 0.0
    assert g[0, 1] == 945.0 and h[0, 1] == 945.0 * u[0, 1]


# ---------------------------------------------------------------- RMSNorm prologue

def _signs(shape, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.where(rng.random(shape) < 0.5, -1.0, 1.0).astype(np.float32)).to(
        torch.bfloat16)


def test_rmsnorm_with_unit_rms_and_unit_gamma_is_the_plain_projection():
    # x = +-1 everywhere, eps = 0: mean x^2 = 1, rinv = 1, xh = x exactly
    n, k = 24, 512
    w = synth.q4k_weight(n, k, seed=70).numpy()
    x = _signs((3, k), 71)
    y, s, rinv = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), np.ones(k, np.float32), 0.0)
    y0, s0 = oracle.gemv(w, n, k, _x_bits(x))
    assert np.all(rinv == 1.0)
    assert np.array_equal(y, y0) and np.array_equal(s, s0)


def test_rmsnorm_is_invariant_to_scaling_x_by_a_power_of_two():
    n, k = 20, 768
    w = synth.q4k_weight(n, k, seed=72).numpy()
    x = synth.bf16_normal((2, k), seed=73)
    gamma = np.random.default_rng(74).uniform(0.5, 1.5, k).astype(np.float32)
    y1, s1, r1 = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), gamma, 0.0)
    y4, s4, r4 = oracle.rmsnorm_gemv(w, n, k, _x_bits(x * 4), gamma, 0.0)
    assert np.array_equal(r4 * 4, r1)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)


def test_rmsnorm_single_nonzero_activation_closed_form():
    # x = a e_j, eps = 0: rinv = sqrt(k) / |a|, so y = sign(a) sqrt(k) gamma_j W[:, j]
    n, k, j = 16, 512, 137
    w = synth.q4k_weight(n, k, seed=75).numpy()
    gamma = np.random.default_rng(76).uniform(-2, 2, k).astype(np.float32)
    x = torch.zeros((2, k), dtype=torch.bfloat16)
    x[0, j] = -3.0
    x[1, j] = 0.015625
    y, s, rinv = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), gamma, 0.0)
    col = oracle.dequant_f64(w, n, k)[:, j]
    assert np.allclose(rinv, [np.sqrt(k) / 3.0, np.sqrt(k) / 0.015625], rtol=1e-15)
    want = np.sqrt(k) * float(gamma[j]) * col
    assert np.allclose(y[0], -want, rtol=1e-14, atol=0) and np.allclose(y[1], want, rtol=1e-14, atol=0)
    assert np.allclose(s[0], np.abs(want), rtol=1e-14, atol=0)


def test_rmsnorm_eps_closed_form_and_linearity_in_gamma():
    n, k = 12, 256
    w = synth.q4k_weight(n, k, seed=77).numpy()
    x = torch.full((1, k), 0.5, dtype=torch.bfloat16)            # mean x^2 = 0.25
    g1 = np.random.default_rng(78).uniform(-1, 1, k).astype(np.float32)
    g2 = np.random.default_rng(79).uniform(-1, 1, k).astype(np.float32)
    eps = 1e-2
    y1, s1, r = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), g1, eps)
    assert np.isclose(r[0], 1.0 / np.sqrt(0.25 + float(np.float32(eps))), rtol=1e-15)
    y2, s2, _ = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), g2, eps)
    y12, _, _ = oracle.rmsnorm_gemv(w, n, k, _x_bits(x), (g1 + g2).astype(np.float32), eps)
    # g1 + g2 is rounded to fp32 once: 2^-24 of |g1| + |g2| per entry
    assert np.all(np.abs(y12 - (y1 + y2)) <= 1e-6 * (s1 + s2))


# ---------------------------------------------------------------- MoE

def _moe_case(E=4, H=256, F=512, T=3, K=2, seed=20):
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=seed).numpy().reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=seed + 1).numpy().reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=seed + 2).numpy().reshape(-1)
    x = synth.bf16_normal((T, H), seed=seed + 3)
    ids, wts = synth.zipf_routing(T, E, K, seed=seed + 4)
    return dict(wg=wg, wu=wu, wd=wd, stride=stride, E=E, H=H, F=F, x=x, ids=ids.numpy(),
                wts=wts.numpy())


def _run_moe(c, **kw):
    args = dict(c)
    args.update(kw)
    return oracle.moe(args["wg"], args["wu"], args["wd"], args["stride"], args["E"], args["H"],
                      args["F"], _x_bits(args["x"]), args["ids"], args["wts"], return_stages=True,
                      weighted_down=args.get("weighted_down", False))


def test_moe_matches_library_composition():
    from scipy.special import expit
    c = _moe_case()
    y, (g, u, h) = _run_moe(c)
    E, H, F = c["E"], c["H"], c["F"]
    Wg = oracle.dequant_f64(c["wg"], E * F, H).reshape(E, F, H)
    Wu = oracle.dequant_f64(c["wu"], E * F, H).reshape(E, F, H)
    Wd = oracle.dequant_f64(c["wd"], E * H, F).reshape(E, H, F)
    xf = _x_f64(c["x"])
    T, K = c["ids"].shape
    yref = np.zeros((T, H))
    for t in range(T):
        for j in range(K):
            e = c["ids"][t, j]
            gg = Wg[e] @ xf[t]
            uu = Wu[e] @ xf[t]
            hh = gg * expit(gg) * uu
            assert np.allclose(g[t * K + j], gg, rtol=1e-12, atol=1e-12)
            assert np.allclose(u[t * K + j], uu, rtol=1e-12, atol=1e-12)
            assert np.allclose(h[t * K + j], hh, rtol=1e-12, atol=1e-12)
            yref[t] += float(c["wts"][t, j]) * (Wd[e] @ hh)
    assert np.allclose(y, yref, rtol=1e-10, atol=1e-10)


def test_moe_relabelling_experts_leaves_output_unchanged():
    c = _moe_case(seed=30)
    y, _ = _run_moe(c)
    E = c["E"]
    perm = np.array([2, 0, 3, 1])                      # new slot p holds old expert perm[p]
    inv = np.argsort(perm)
    s = c["stride"]

    def permute(w):
        return np.concatenate([w[perm[p] * s:(perm[p] + 1) * s] for p in range(E)])

    y2, _ = _run_moe(c, wg=permute(c["wg"]), wu=permute(c["wu"]), wd=permute(c["wd"]),
                     ids=inv[c["ids"]].astype(np.int32))
    assert np.array_equal(y, y2)


def test_moe_identical_experts_reduce_to_one_dense_ffn():
    c = _moe_case(seed=40)
    s = c["stride"]
    E = c["E"]
    same = dict(wg=np.tile(c["wg"][:s], E), wu=np.tile(c["wu"][:s], E), wd=np.tile(c["wd"][:s], E))
    y, _ = _run_moe(c, **same)
    one = dict(ids=np.zeros_like(c["ids"])[:, :1], wts=np.ones((c["ids"].shape[0], 1), np.float32))
    y1, _ = _run_moe(c, **same, **one)
    # softmax weights sum to one up to fp32 rounding
    wsum = c["wts"].astype(np.float64).sum(axis=1, keepdims=True)
    assert np.allclose(y, y1 * wsum, rtol=1e-12, atol=1e-12)
    assert np.allclose(wsum, 1.0, atol=1e-6)


def test_moe_zero_gate_gives_zero_and_bad_ids_contribute_nothing():
    c = _moe_case(seed=50)
    zero_gate = np.zeros_like(c["wg"])                # d = dmin = 0: every gate weight is 0
    y, (g, u, h) = _run_moe(c, wg=zero_gate)
    assert np.all(g == 0) and np.all(h == 0) and np.all(y == 0)
    ids = c["ids"].copy()
    ids[0, 0] = c["E"]                                 # out of range
    ids[1, 1] = -1
    y_bad, _ = _run_moe(c, ids=ids)
    keep = np.ones_like(c["wts"])
    keep[0, 0] = 0
    keep[1, 1] = 0
    y_ref, _ = _run_moe(c, wts=(c["wts"] * keep).astype(np.float32))
    assert np.allclose(y_bad, y_ref, rtol=0, atol=1e-12)


def test_moe_weighted_down_with_unit_weights_is_the_plain_form_bit_for_bit():
    # r = 1: r h = h and 1 * p = p exactly, so both orders give the same bits
    c = _moe_case(seed=60)
    ones = np.ones_like(c["wts"])
    y0, st0 = _run_moe(c, wts=ones)
    y1, st1 = _run_moe(c, wts=ones, weighted_down=True)
    assert np.array_equal(y0, y1)
    for a, b in zip(st0, st1):
        assert np.array_equal(a, b)


def test_moe_weighted_down_matches_library_composition_and_the_plain_form():
    # Wd (r h) summed over slots, composed here from the dequantized matrices;
    # the same as sum r (Wd h) up to fp64 rounding (Wd is linear); the staged
    # h is the unweighted silu(g) u
    from scipy.special import expit
    c = _moe_case(seed=61, T=4, K=3, E=5)
    y, (g, u, h) = _run_moe(c, weighted_down=True)
    y_plain, (_, _, h_plain) = _run_moe(c)
    E, H, F = c["E"], c["H"], c["F"]
    Wg = oracle.dequant_f64(c["wg"], E * F, H).reshape(E, F, H)
    Wu = oracle.dequant_f64(c["wu"], E * F, H).reshape(E, F, H)
    Wd = oracle.dequant_f64(c["wd"], E * H, F).reshape(E, H, F)
    xf = _x_f64(c["x"])
    T, K = c["ids"].shape
    yref = np.zeros((T, H))
    scale = np.zeros((T, H))
    for t in range(T):
        for j in range(K):
            e = c["ids"][t, j]
            r = float(c["wts"][t, j])
            gg, uu = Wg[e] @ xf[t], Wu[e] @ xf[t]
            hh = gg * expit(gg) * uu
            yref[t] += Wd[e] @ (r * hh)
            scale[t] += abs(r) * (np.abs(Wd[e]) @ np.abs(hh))
    assert np.array_equal(h, h_plain)
    assert np.all(np.abs(y - yref) <= 1e-12 * scale + 1e-300)
    assert np.all(np.abs(y - y_plain) <= 1e-12 * scale + 1e-300)
    assert not np.array_equal(y, y_plain) or np.all(c["wts"] == 1)   # a distinct path


# ---------------------------------------------------------------- generator sanity

def test_generator_fields_have_the_stated_distributions():
    w = synth.q4k_weight(64, 4096, seed=60).numpy().reshape(-1, 144)
    d = w[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    assert d.min() >= 1e-3 - 1e-6 and d.max() <= 2e-2 + 1e-5
    scs = np.array([oracle.unpack_scales(b[4:16]) for b in w[:200]])
    assert scs.min() == 0 and scs.max() == 63
    wn = synth.q4k_weight(16, 4096, seed=61, quants="normal").numpy().reshape(-1, 144)
    q = np.concatenate([wn[:, 16:] & 15, wn[:, 16:] >> 4], axis=1).astype(np.float64)
    assert abs(q.mean() - 8.0) < 0.05 and 2.5 < q.std() < 3.2
    ids, wts = synth.zipf_routing(16, 128, 8, seed=62)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert np.allclose(wts.double().sum(1).numpy(), 1.0, atol=1e-6)
