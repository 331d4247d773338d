"""Parity edge cases of the fp32-accumulate decode paths (batch 1, batched,
fused gate/up) and of the prefill GEMM, against the oracle.

Weights that cancel: a Q4_K weight is exactly zero when d sc_j q = dmin m_j.
  * Rows whose every weight cancels have sum |w||x| = 0, so the per-element
    bound 2e-3 * sum |w||x| demands an exact 0.
  * Rows that cancel except for one weight must come out as that one product,
    to within 2e-3 of it, however large the rest of x is.
Activations at the edges of bf16:
  * entries spanning 2^-60 .. 2^60 inside one super-block;
  * bf16 subnormals mixed with normal values;
  * |x| near 2^100;
  * one huge entry at a position whose weight is exactly zero in every row,
    beside small entries that carry all of the row's sum.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_bound, xbits
from _q4k_fields import half_bits, pack_block, random_fields

pytestmark = pytest.mark.gpu
TOL = 2e-3

# (sc, c, m) with sc * c = 2 m: with d = 2^-6 and dmin = 2^-5, d sc c = dmin m.
CANCEL = ((2, 4, 4), (6, 7, 21), (8, 15, 60), (14, 9, 63), (5, 0, 0), (12, 5, 30), (4, 1, 2))


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _cancel_block(rng, one_off=None):
    """A super-block whose weights are all exactly zero; with one_off = i,
    weight i gets q = c + 1 (or c - 1 at c = 15), the only nonzero weight."""
    picks = [CANCEL[int(j)] for j in rng.integers(0, len(CANCEL), 8)]
    sc = [p[0] for p in picks]
    m = [p[2] for p in picks]
    q = [picks[i // 32][1] for i in range(256)]
    if one_off is not None:
        q[one_off] = q[one_off] + 1 if q[one_off] < 15 else 14
    return pack_block(half_bits(2.0 ** -6), half_bits(2.0 ** -5), sc, m, q)


def _matrix(rows):
    return torch.frombuffer(bytearray(b"".join(rows)), dtype=torch.uint8).view(len(rows), -1)


def _cancel_matrix(k, seed):
    """Rows 0 mod 3: all weights cancel; 1 mod 3: cancel except one weight;
    2 mod 3: random fields."""
    rng = np.random.default_rng(seed)
    nsb = k // 256
    rows = []
    for r in range(48):
        kind = r % 3
        if kind == 0:
            rows.append(b"".join(_cancel_block(rng) for _ in range(nsb)))
        elif kind == 1:
            hit = int(rng.integers(0, k))
            rows.append(b"".join(_cancel_block(rng, hit - 256 * b if hit // 256 == b else None)
                                 for b in range(nsb)))
        else:
            rows.append(b"".join(pack_block(*random_fields(rng)) for _ in range(nsb)))
    return _matrix(rows)


def _gemv(q4k, w, n, k, x, flags=0):
    y = q4k.q4k_gemv_ex(w.to(DEV), n, k, x.to(DEV), flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("batch", [1, 2, 4, 16])
@pytest.mark.parametrize("k", [256, 1280, 5120])
def test_cancelling_rows_give_exact_zero(q4k, batch, k):
    w = _cancel_matrix(k, seed=k + batch)
    n = w.shape[0]
    x = synth.bf16_normal((batch, k), seed=7 * k + batch)
    y = _gemv(q4k, w, n, k, x, flags=1)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    assert np.all(s[:, 0::3] == 0.0) and np.all(yref[:, 0::3] == 0.0)
    assert np.all(y[:, 0::3] == 0.0), "rows whose weights all cancel must be exactly 0"
    check_bound(y, yref, s, TOL, f"cancel k{k} b{batch}")


@pytest.mark.parametrize("batch", [1, 3, 16])
def test_cancelling_gate_rows_give_exact_zero_through_glu(q4k, batch):
    k = 1280
    wg = _cancel_matrix(k, seed=91)
    wu = synth.q4k_weight(wg.shape[0], k, seed=92)
    n = wg.shape[0]
    x = synth.bf16_normal((batch, k), seed=93)
    h = q4k.q4k_gemv_glu(wg.to(DEV), wu.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    h = h.cpu().numpy()
    assert np.all(h[:, 0::3] == 0.0)                 # g = 0 exactly, silu(0) = 0
    from test_gemv import check_glu
    check_glu(h, wg, wu, n, k, x, f"glu cancel b{batch}")


def _zero_weight_at(k, n, pos, seed):
    """Random rows in which weight `pos` is exactly zero in every row: its
    sub-block gets d sc c = dmin m with q = c at pos; every other field random."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n):
        blocks = []
        for b in range(k // 256):
            d, dm, sc, m, q = random_fields(rng)
            if b == pos // 256:
                j = (pos % 256) // 32
                scj, c, mj = CANCEL[int(rng.integers(0, 4))]
                d, dm = half_bits(2.0 ** -6), half_bits(2.0 ** -5)
                sc[j], m[j] = scj, mj
                q[pos % 256] = c
            blocks.append(pack_block(d, dm, sc, m, q))
        rows.append(b"".join(blocks))
    return _matrix(rows)


def _bf16_from(values: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(values.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 16])
def test_huge_activation_at_a_zero_weight(q4k, batch):
    k, n, pos = 1024, 40, 300
    w = _zero_weight_at(k, n, pos, seed=11)
    rng = np.random.default_rng(12)
    xv = rng.standard_normal((batch, k)) * 2.0 ** -40
    xv[:, pos] = 2.0 ** 100
    x = _bf16_from(xv)
    y = _gemv(q4k, w, n, k, x)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    assert np.all(s < 1e-6)                           # the huge entry meets only zero weights
    check_bound(y, yref, s, TOL, f"huge at zero weight b{batch}")


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 16])
def test_activations_spanning_2e_minus60_to_2e60(q4k, batch):
    k, n = 2048, 64
    w = synth.q4k_weight(n, k, seed=13, quants="normal")
    rng = np.random.default_rng(14)
    xv = rng.standard_normal((batch, k)) * 2.0 ** rng.integers(-60, 61, (batch, k))
    x = _bf16_from(xv)
    y = _gemv(q4k, w, n, k, x, flags=1)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y, yref, s, TOL, f"wide range b{batch}")
    # the same with the large entries only at positions whose weights are zero
    pos = 777
    w2 = _zero_weight_at(k, n, pos, seed=15)
    xv2 = rng.standard_normal((batch, k)) * 2.0 ** rng.integers(-60, -20, (batch, k))
    xv2[:, pos] = 2.0 ** 60
    x2 = _bf16_from(xv2)
    y2 = _gemv(q4k, w2, n, k, x2)
    yref2, s2 = oracle.gemv(w2.numpy(), n, k, xbits(x2))
    check_bound(y2, yref2, s2, TOL, f"wide range, big at zero weight b{batch}")


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_activations_near_2e100_and_bf16_subnormals(q4k, batch):
    k, n = 1536, 50
    w = synth.q4k_weight(n, k, seed=16, quants="normal")
    rng = np.random.default_rng(17)
    big = rng.standard_normal((batch, k)) * 2.0 ** 100
    x = _bf16_from(big)
    y = _gemv(q4k, w, n, k, x)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y, yref, s, TOL, f"2^100 b{batch}")
    # bf16 subnormals (|x| < 2^-126) among normal values
    bits = rng.integers(1, 0x7F, (batch, k)).astype(np.uint16)          # subnormal patterns
    bits |= (rng.integers(0, 2, (batch, k)).astype(np.uint16) << 15)
    xs = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).clone()
    normal = synth.bf16_normal((batch, k), seed=18)
    mix = torch.where(torch.from_numpy(rng.random((batch, k)) < 0.5), xs, normal)
    y2 = _gemv(q4k, w, n, k, mix)
    yref2, s2 = oracle.gemv(w.numpy(), n, k, xbits(mix))
    check_bound(y2, yref2, s2, TOL, f"subnormals mixed b{batch}")


@pytest.mark.parametrize("case", ["wide", "subnormal_mix", "big"])
def test_gemm_activation_edges(q4k, case):
    m, n, k = 130, 256, 1024
    w = synth.q4k_weight(n, k, seed=19, quants="normal")
    rng = np.random.default_rng(20)
    if case == "wide":
        xv = rng.standard_normal((m, k)) * 2.0 ** rng.integers(-60, 61, (m, k))
        x = _bf16_from(xv)
    elif case == "big":
        x = _bf16_from(rng.standard_normal((m, k)) * 2.0 ** 100)
    else:
        bits = rng.integers(1, 0x7F, (m, k)).astype(np.uint16)
        xs = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).clone()
        x = torch.where(torch.from_numpy(rng.random((m, k)) < 0.5), xs,
                        synth.bf16_normal((m, k), seed=21))
    y = q4k.q4k_gemm(w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y.float().cpu().numpy(), yref, s, 1e-2, f"gemm {case}")


def test_moe_cancelling_rows(q4k):
    # experts whose gate rows 0 mod 3 and down rows 0 mod 3 cancel exactly:
    # g is exactly 0 there (read back from the workspace), and the hidden rows
    # whose down rows cancel in every expert come out as exactly 0
    from test_moe import _gpu_stages
    E, H, F, T, K = 4, 512, 768, 6, 2
    nsb_h, nsb_f = H // 256, F // 256
    rng = np.random.default_rng(40)

    def mat(rows, nsb):
        out = []
        for r in range(rows):
            if r % 3 == 0:
                out.append(b"".join(_cancel_block(rng) for _ in range(nsb)))
            else:
                out.append(b"".join(pack_block(*random_fields(rng)) for _ in range(nsb)))
        return b"".join(out)

    wg = torch.frombuffer(bytearray(b"".join(mat(F, nsb_h) for _ in range(E))), dtype=torch.uint8)
    wu = synth.q4k_weight(E * F, H, seed=41).reshape(-1)
    wd = torch.frombuffer(bytearray(b"".join(mat(H, nsb_f) for _ in range(E))), dtype=torch.uint8)
    x = synth.bf16_normal((T, H), seed=42)
    ids, wts = synth.zipf_routing(T, E, K, seed=43)
    c = dict(wg=wg, wu=wu, wd=wd, stride=F * nsb_h * 144, E=E, H=H, F=F, x=x)
    y, tj, st = _gpu_stages(q4k, c, ids, wts)
    assert np.all(st["g"][:, 0::3] == 0.0) and np.all(st["h"][:, 0::3] == 0.0)
    assert np.all(y[:, 0::3] == 0.0)
    from test_moe import _bound, _check
    yref, bound = _bound(c, ids, wts, list(range(T)))
    _check(y, yref, bound, "moe cancel")

