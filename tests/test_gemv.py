"""q4k_gemv (decode, batch 1..16) on the GPU against the oracle.

Bound: |y - y_ref| <= 2e-3 * sum_k |w_k||x_k| per element (fp32-accumulate
path).  Shapes span several row tiles, ragged row tails and split-K slices;
the full-size 27B-class projections are checked on sampled rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_bound, xbits
from _q4k_fields import pack_block, random_fields

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _run(q4k, w, n, k, x, flags=0):
    y = q4k.q4k_gemv_ex(w.to(DEV), n, k, x.to(DEV), flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    return y.cpu().numpy()


CASES = [(1, 256, 1), (7, 512, 1), (129, 1280, 1), (597, 5120, 1), (33, 17408, 1),
         (4096, 4096, 1), (1000, 2560, 2), (597, 5120, 3), (300, 4096, 4), (130, 1536, 8),
         (129, 5120, 9), (597, 5120, 16), (40, 8192, 16)]


# flags 0: plain launches; Q4K_FLAG_OVERLAP_WEIGHTS: programmatic dependent
# launch (weights streamed before the dependency wait).
FLAGS = [0, 1]


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("n,k,batch", CASES)
def test_gemv_matches_oracle(q4k, n, k, batch, flags):
    w = synth.q4k_weight(n, k, seed=1000 + n + k + batch, quants="normal" if n % 2 else "uniform")
    x = synth.bf16_normal((batch, k), seed=2000 + n + batch)
    y = _run(q4k, w, n, k, x, flags)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y, yref, s, TOL, f"gemv {n}x{k} b{batch} flags{flags}")


@pytest.mark.parametrize("n,k", [(16 * 152 * 2 + 5, 1280), (5000, 2560), (16 * 152, 256), (3000, 17408)])
def test_gemv_many_row_tiles(q4k, n, k):
    # many row tiles (more than one per SM), ragged last tile, both launch modes
    w = synth.q4k_weight(n, k, seed=n + k, quants="normal")
    x = synth.bf16_normal((1, k), seed=n + 7)
    y = _run(q4k, w, n, k, x, flags=1)
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(y, yref, s, TOL, f"overlap {n}x{k}")
    y0 = _run(q4k, w, n, k, x, flags=0)
    check_bound(y0, yref, s, TOL, f"per-tile {n}x{k}")


@pytest.mark.parametrize("batch,flags", [(1, 0), (1, 1), (4, 1), (16, 0)])
def test_gemv_seq_matches_oracle_and_single_calls(q4k, batch, flags):
    # one q4k_gemv_seq call over projections of different shapes (an empty one
    # among them) equals the oracle, and equals q4k_gemv_ex called per op
    shapes = [(700, 1280), (0, 512), (2048, 4096), (129, 5120), (4096, 2304)]
    ws, xs, ys = [], [], []
    for i, (n, k) in enumerate(shapes):
        ws.append(synth.q4k_weight(max(n, 1), k, seed=3100 + i, quants="normal"))
        xs.append(synth.bf16_normal((batch, k), seed=3200 + i))
        ys.append(torch.full((batch, max(n, 1)), 7.0, device=DEV))
    dw, dx = [w.to(DEV) for w in ws], [x.to(DEV) for x in xs]
    ops = q4k.gemv_ops([(w, n, k, x, y) for w, (n, k), x, y in zip(dw, shapes, dx, ys)])
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    for i, ((n, k), w, x, y) in enumerate(zip(shapes, ws, xs, ys)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
            continue
        yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
        check_bound(y.cpu().numpy(), yref, s, TOL, f"seq op {i} {n}x{k} b{batch}")
        single = _run(q4k, w, n, k, x, flags)
        assert np.array_equal(single, y.cpu().numpy()), f"seq op {i} differs from a single call"


def test_gemv_overlap_chain_reads_the_previous_output(q4k):
    # y1 = W1 x0; x1 = bf16(y1) by a torch kernel; y2 = W2 x1, all queued on
    # one stream with programmatic dependent launch: the second projection
    # must see x1 as written, even though its weights stream early.
    n1, k1, n2 = 2048, 1024, 700
    w1 = synth.q4k_weight(n1, k1, seed=21).to(DEV)
    w2 = synth.q4k_weight(n2, n1, seed=22).to(DEV)
    x0 = synth.bf16_normal((1, k1), seed=23).to(DEV)
    flags = q4k.Q4K_FLAG_OVERLAP_WEIGHTS
    for _ in range(3):
        y1 = q4k.q4k_gemv_ex(w1, n1, k1, x0, flags)
        x1 = (y1 * 0.05).to(torch.bfloat16)
        y2 = q4k.q4k_gemv_ex(w2, n2, n1, x1, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    yref1, s1 = oracle.gemv(w1.cpu().numpy(), n1, k1, xbits(x0.cpu()))
    check_bound(y1.cpu().numpy(), yref1, s1, TOL, "chain first")
    yref2, s2 = oracle.gemv(w2.cpu().numpy(), n2, n1, xbits(x1.cpu()))
    check_bound(y2.cpu().numpy(), yref2, s2, TOL, "chain second")


@pytest.mark.parametrize("batch", [1, 5, 16])
def test_gemv_strided_x_and_y(q4k, batch):
    n, k = 77, 1024
    w = synth.q4k_weight(n, k, seed=3)
    xs = synth.bf16_normal((batch, k + 64), seed=4).to(DEV)
    x = xs[:, 8:8 + k]                                   # ldx = k + 64, offset 16 bytes
    out = torch.full((batch, n + 5), float("nan"), device=DEV)
    q4k.q4k_gemv(w.to(DEV), n, k, x, out=out[:, :n])
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[:, n:]))                  # nothing written past the row
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(got[:, :n], yref, s, TOL, "strided")


def test_gemv_zero_quant_rows_and_zero_blocks(q4k):
    rng = np.random.default_rng(11)
    k = 1024
    rows = []
    for r in range(40):
        blks = []
        for b in range(k // 256):
            d, dm, sc, m, q = random_fields(rng)
            if r % 3 == 0:
                q = [0] * 256                            # zero quants: w = -dmin*m
            if r % 5 == 0:
                d, dm = 0, 0                             # zero block: w = 0
            blks.append(pack_block(d, dm, sc, m, q))
        rows.append(b"".join(blks))
    n = len(rows)
    w = torch.frombuffer(bytearray(b"".join(rows)), dtype=torch.uint8).view(n, -1)
    for batch in (1, 4):
        x = synth.bf16_normal((batch, k), seed=12 + batch)
        y = _run(q4k, w, n, k, x)
        yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
        check_bound(y, yref, s, TOL, f"zero-quant b{batch}")
        assert np.all(y[:, ::5] == 0.0)                  # d = dmin = 0 rows are exactly 0


def test_gemv_unit_vectors_pick_columns(q4k):
    n, k = 64, 768
    w = synth.q4k_weight(n, k, seed=13)
    wq = oracle.dequant_f64(w.numpy(), n, k)
    cols = [0, 2, 31, 32, 100, 255, 256, 511, 767]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    y = _run(q4k, w, n, k, x)
    for i, c in enumerate(cols):
        assert np.allclose(y[i], wq[:, c], rtol=1e-6, atol=1e-6)
    y1 = _run(q4k, w, n, k, x[3:4])
    assert np.allclose(y1[0], wq[:, cols[3]], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("batch,flags", [(1, 0), (1, 1), (6, 0)])
def test_gemv_homogeneous_and_deterministic_bitwise(q4k, batch, flags):
    n, k = 300, 2048
    w = synth.q4k_weight(n, k, seed=14).to(DEV)
    x = synth.bf16_normal((batch, k), seed=15).to(DEV)
    y1 = q4k.q4k_gemv_ex(w, n, k, x, flags).clone()
    y1b = q4k.q4k_gemv_ex(w, n, k, x, flags).clone()
    y2 = q4k.q4k_gemv_ex(w, n, k, (x.float() * 4).to(torch.bfloat16), flags)
    torch.cuda.synchronize()
    assert torch.equal(y1, y1b)
    assert torch.equal(y2, y1 * 4)


def test_gemv_zero_activations(q4k):
    n, k = 50, 512
    w = synth.q4k_weight(n, k, seed=16)
    y = _run(q4k, w, n, k, torch.zeros((2, k), dtype=torch.bfloat16))
    assert np.all(y == 0.0)


# 27B-class dense decoder layer shapes (hidden 5120): QKV, O, gate/up, down.
LAYER = [(10240, 5120), (5120, 8192), (17408, 5120), (5120, 17408)]


@pytest.mark.parametrize("n,k", LAYER)
@pytest.mark.parametrize("batch,flags", [(1, 0), (1, 1), (4, 0), (16, 0)])
def test_gemv_full_size_sampled_rows(q4k, n, k, batch, flags):
    w = synth.q4k_weight(n, k, seed=n * 3 + k, quants="normal", device=DEV)
    x = synth.bf16_normal((batch, k), seed=n + batch, device=DEV)
    y = q4k.q4k_gemv_ex(w, n, k, x, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    rows = np.sort(np.random.default_rng(n + k).choice(n, 96, replace=False))
    rows = np.unique(np.concatenate([rows, [0, n - 1]]))
    wsub = w[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    yref, s = oracle.gemv(wsub, len(rows), k, xbits(x))
    check_bound(y[:, torch.from_numpy(rows).to(DEV)].cpu().numpy(), yref, s, TOL,
                f"full {n}x{k} b{batch} flags{flags}")
