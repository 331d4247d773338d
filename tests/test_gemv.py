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
         (4096, 4096, 1), (1000, 2560, 2), (597, 5120, 3), (300, 4096, 4), (1, 256, 2),
         (17, 768, 3), (33, 17408, 4), (4901, 1280, 2), (4901, 2304, 3), (39000, 256, 2),
         (29200, 512, 3), (130, 1536, 8),
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


@pytest.mark.parametrize("batch,flags", [(1, 0), (1, 1), (2, 1), (3, 0), (4, 1), (5, 1), (16, 0)])
def test_gemv_seq_matches_oracle(q4k, batch, flags):
    # one q4k_gemv_seq call over projections of different shapes (an empty one
    # and a fused gate/up op among them) matches the oracle; a second call gives
    # bitwise the same result
    shapes = [(700, 1280), (0, 512), (2048, 4096), (129, 5120), (4096, 2304), (333, 1536)]
    glu = {5}
    ws, wus, xs, ys = [], [], [], []
    for i, (n, k) in enumerate(shapes):
        ws.append(synth.q4k_weight(max(n, 1), k, seed=3100 + i, quants="normal"))
        wus.append(synth.q4k_weight(max(n, 1), k, seed=3300 + i) if i in glu else None)
        xs.append(synth.bf16_normal((batch, k), seed=3200 + i, sigma=0.05 if i in glu else 1.0))
        ys.append(torch.full((batch, max(n, 1)), 7.0, device=DEV))
    dw, dx = [w.to(DEV) for w in ws], [x.to(DEV) for x in xs]
    dwu = [None if w is None else w.to(DEV) for w in wus]
    tup = []
    for w, wu, (n, k), x, y in zip(dw, dwu, shapes, dx, ys):
        tup.append((w, n, k, x, y) if wu is None else (w, n, k, x, y, wu))
    ops = q4k.gemv_ops(tup)
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    first = [y.clone() for y in ys]
    for i, ((n, k), w, wu, x, y) in enumerate(zip(shapes, ws, wus, xs, ys)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
            continue
        if wu is None:
            yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
            check_bound(y.cpu().numpy(), yref, s, TOL, f"seq op {i} {n}x{k} b{batch}")
        else:
            check_glu(y.cpu().numpy(), w, wu, n, k, x, f"seq glu op {i} {n}x{k} b{batch}")
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    for a, b in zip(first, ys):
        assert torch.equal(a, b), "a sequence is deterministic"


@pytest.mark.parametrize("batch,flags,count", [(1, 1, 170), (1, 0, 341), (2, 1, 170), (4, 1, 200)])
def test_gemv_seq_several_launches(q4k, batch, flags, count):
    # at batch 1..4 a launch takes Q4K_SEQ_MATRICES_PER_LAUNCH weight matrices
    # (a fused gate/up op counts two): sequences of 170-341 small ops (empty
    # ops and fused gate/up ops among them) run as two or three launches, and
    # every op matches the oracle
    rng = np.random.default_rng(4100 + count + batch)
    shapes = [(int(rng.integers(0, 48)), int(rng.choice([256, 512, 768]))) for _ in range(count)]
    glu = {i for i in range(count) if i % 7 == 3}
    mats = sum((2 if i in glu else 1) for i, (n, _) in enumerate(shapes) if n > 0)
    assert mats > q4k.Q4K_SEQ_MATRICES_PER_LAUNCH
    ws, wus, xs, ys, tup = [], [], [], [], []
    for i, (n, k) in enumerate(shapes):
        w = synth.q4k_weight(max(n, 1), k, seed=6100 + i, quants="normal")
        wu = synth.q4k_weight(max(n, 1), k, seed=6400 + i) if i in glu else None
        x = synth.bf16_normal((batch, k), seed=6700 + i, sigma=0.05 if i in glu else 1.0)
        y = torch.full((batch, max(n, 1)), 7.0, device=DEV)
        ws.append(w)
        wus.append(wu)
        xs.append(x)
        ys.append(y)
        dw, dx = w.to(DEV), x.to(DEV)
        tup.append((dw, n, k, dx, y) if wu is None else (dw, n, k, dx, y, wu.to(DEV)))
    ops = q4k.gemv_ops(tup)
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    for i, ((n, k), w, wu, x, y) in enumerate(zip(shapes, ws, wus, xs, ys)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
        elif wu is None:
            yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
            check_bound(y.cpu().numpy(), yref, s, TOL, f"seq op {i} {n}x{k} b{batch}")
        else:
            check_glu(y.cpu().numpy(), w, wu, n, k, x, f"seq glu op {i} {n}x{k} b{batch}")


@pytest.mark.parametrize("batch,flags", [(6, 1), (16, 0)])
def test_gemv_seq_64_row_tiles_several_launches(q4k, batch, flags):
    # batch 5..16 with enough 64-row tiles to fill the GPU and more than
    # Q4K_SEQ_MATRICES_PER_LAUNCH weight matrices (fused gate/up ops count
    # two): the 64-row tile kernel runs two launches; every op matches the
    # oracle and an empty op writes nothing
    count = 170
    rng = np.random.default_rng(4300 + batch)
    # about 2000 tiles of 64 rows: at least two per resident CTA at batch 5..16
    shapes = [(int(rng.integers(700, 1000)), int(rng.choice([256, 512]))) for _ in range(count)]
    shapes[5] = (0, 256)
    glu = {i for i in range(count) if i % 7 == 3}
    mats = sum((2 if i in glu else 1) for i, (n, _) in enumerate(shapes) if n > 0)
    assert mats > q4k.Q4K_SEQ_MATRICES_PER_LAUNCH
    ws, wus, xs, ys, tup = [], [], [], [], []
    for i, (n, k) in enumerate(shapes):
        w = synth.q4k_weight(max(n, 1), k, seed=6900 + i, quants="normal")
        wu = synth.q4k_weight(max(n, 1), k, seed=7900 + i) if i in glu else None
        x = synth.bf16_normal((batch, k), seed=8900 + i, sigma=0.05 if i in glu else 1.0)
        y = torch.full((batch, max(n, 1)), 7.0, device=DEV)
        ws.append(w)
        wus.append(wu)
        xs.append(x)
        ys.append(y)
        dw, dx = w.to(DEV), x.to(DEV)
        tup.append((dw, n, k, dx, y) if wu is None else (dw, n, k, dx, y, wu.to(DEV)))
    ops = q4k.gemv_ops(tup)
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    for i, ((n, k), w, wu, x, y) in enumerate(zip(shapes, ws, wus, xs, ys)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
        elif wu is None:
            yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
            check_bound(y.cpu().numpy(), yref, s, TOL, f"wide seq op {i} {n}x{k} b{batch}")
        else:
            check_glu(y.cpu().numpy(), w, wu, n, k, x, f"wide seq glu op {i} {n}x{k} b{batch}")


@pytest.mark.parametrize("batch,flags", [(5, 1), (8, 0), (9, 1), (16, 1)])
def test_gemv_seq_persistent_64_row_tiles(q4k, batch, flags):
    # batch 5..16 with enough 64-row tiles to fill the GPU (at least two per
    # resident CTA) runs as one persistent launch: ragged row tails, an empty
    # op, a fused gate/up op and strided x / y among the ops; every row is
    # checked against the oracle
    shapes = [(40000, 256), (0, 512), (30001, 512), (20000, 512), (9000, 768)]
    glu = {3}
    ws, wus, xs, xviews, ys, yviews = [], [], [], [], [], []
    for i, (n, k) in enumerate(shapes):
        ws.append(synth.q4k_weight(max(n, 1), k, seed=5100 + i, quants="normal"))
        wus.append(synth.q4k_weight(max(n, 1), k, seed=5300 + i) if i in glu else None)
        if i == 4:  # strided: ldx = k + 64 (offset 16 bytes), ldy = n + 3
            xb = synth.bf16_normal((batch, k + 64), seed=5200 + i).to(DEV)
            xs.append(xb)
            xviews.append(xb[:, 8:8 + k])
            yb = torch.full((batch, n + 3), float("nan"), device=DEV)
            ys.append(yb)
            yviews.append(yb[:, :n])
        else:
            x = synth.bf16_normal((batch, k), seed=5200 + i, sigma=0.05 if i in glu else 1.0).to(DEV)
            xs.append(x)
            xviews.append(x)
            y = torch.full((batch, max(n, 1)), 7.0, device=DEV)
            ys.append(y)
            yviews.append(y)
    tup = []
    for w, wu, (n, k), x, y in zip(ws, wus, shapes, xviews, yviews):
        dw = w.to(DEV)
        tup.append((dw, n, k, x, y) if wu is None else (dw, n, k, x, y, wu.to(DEV)))
    ops = q4k.gemv_ops(tup)
    q4k.q4k_gemv_seq(ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    for i, ((n, k), w, wu, x, y) in enumerate(zip(shapes, ws, wus, xviews, yviews)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
            continue
        if wu is None:
            yref, s = oracle.gemv(w.numpy(), n, k, xbits(x.cpu()))
            check_bound(y.cpu().numpy(), yref, s, TOL, f"wide op {i} {n}x{k} b{batch}")
        else:
            check_glu(y.cpu().numpy(), w, wu, n, k, x.cpu(), f"wide glu op {i} {n}x{k} b{batch}")
    assert bool(torch.isnan(ys[4][:, shapes[4][0]:]).all()), "nothing written past a row"


def check_glu(h, wg, wu, n, k, x, what):
    """h = silu(g) u against the oracle, with g and u each within the GEMV
    bound: |dh| <= 1.1 dg |u| + |silu(g)| du + 1.1 dg du + 2^-20 |h| (the last
    term covers fp32 rounding of the SiLU and the product)."""
    href, g, u, sg, su = oracle.gemv_glu(wg.numpy(), wu.numpy(), n, k, xbits(x))
    dg, du = TOL * sg, TOL * su
    sgl = g / (1.0 + np.exp(-np.clip(g, -700, 700)))
    bound = 1.1 * dg * np.abs(u) + np.abs(sgl) * du + 1.1 * dg * du + 2.0 ** -20 * np.abs(href)
    err = np.abs(np.asarray(h, np.float64) - href)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} outside, worst {np.max(err - bound)}"


@pytest.mark.parametrize("n,k,batch", [(1, 256, 1), (77, 1024, 1), (1000, 2560, 1), (1000, 2560, 2),
                                       (77, 1024, 3), (300, 4096, 4), (130, 1536, 8), (129, 5120, 9),
                                       (597, 5120, 16)])
@pytest.mark.parametrize("sigma", [1.0, 0.02])
def test_gemv_glu_matches_oracle(q4k, n, k, batch, sigma):
    # sigma 0.02: g in SiLU's curved region; 1.0: g large, SiLU near identity / 0
    wg = synth.q4k_weight(n, k, seed=4100 + n + k, quants="normal")
    wu = synth.q4k_weight(n, k, seed=4200 + n + k)
    x = synth.bf16_normal((batch, k), seed=4300 + batch, sigma=sigma)
    h = q4k.q4k_gemv_glu(wg.to(DEV), wu.to(DEV), n, k, x.to(DEV), q4k.Q4K_FLAG_OVERLAP_WEIGHTS)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    check_glu(h.cpu().numpy(), wg, wu, n, k, x, f"glu {n}x{k} b{batch} sigma {sigma}")


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_gemv_glu_27b_gate_up_full_size_sampled_rows(q4k, batch):
    # the 27B-class gate/up pair (5120 -> 17408), sampled rows
    n, k = 17408, 5120
    wg = synth.q4k_weight(n, k, seed=4401, quants="normal", device=DEV)
    wu = synth.q4k_weight(n, k, seed=4402, quants="normal", device=DEV)
    x = synth.bf16_normal((batch, k), seed=4403, sigma=0.02, device=DEV)
    h = q4k.q4k_gemv_glu(wg, wu, n, k, x)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    rows = np.unique(np.concatenate([np.random.default_rng(4404).choice(n, 64, replace=False),
                                     [0, n - 1]]))
    ri = torch.from_numpy(rows).to(DEV)
    check_glu(h[:, ri].cpu().numpy(), wg[ri].cpu(), wu[ri].cpu(), len(rows), k, x.cpu(),
              f"27b glu b{batch}")


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_gemv_seq_graph_replay_matches_oracle(q4k, batch):
    # 27B-class layers' five projections as one q4k_gemv_seq call with
    # programmatic dependent launch, captured in a CUDA graph; the graph is
    # replayed twice with x rewritten in between, and every replay's results
    # match the oracle on sampled rows (batch 16: two layers, which is enough
    # 64-row tiles for the persistent launch)
    shapes = [(10240, 5120), (5120, 8192), (17408, 5120), (17408, 5120), (5120, 17408)]
    if batch == 16:
        shapes = shapes * 2
    ws = [synth.q4k_weight(n, k, seed=4500 + i, quants="normal", device=DEV)
          for i, (n, k) in enumerate(shapes)]
    xs = [torch.empty((batch, k), dtype=torch.bfloat16, device=DEV) for _, k in shapes]
    ys = [torch.empty((batch, n), dtype=torch.float32, device=DEV) for n, _ in shapes]
    ops = q4k.gemv_ops([(w, n, k, x, y) for w, (n, k), x, y in zip(ws, shapes, xs, ys)])
    stream = torch.cuda.Stream(device=DEV)
    for x in xs:
        x.normal_()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        q4k.q4k_gemv_seq(ops, batch, q4k.Q4K_FLAG_OVERLAP_WEIGHTS, stream=stream)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        q4k.q4k_gemv_seq(ops, batch, q4k.Q4K_FLAG_OVERLAP_WEIGHTS, stream=stream)
    rng = np.random.default_rng(4600)
    for rep in range(2):
        for i, x in enumerate(xs):
            x.copy_(synth.bf16_normal(x.shape, seed=4700 + 10 * rep + i, device=DEV))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert q4k.q4k_get_device_error() == 0
        for i, ((n, k), w, x, y) in enumerate(zip(shapes, ws, xs, ys)):
            rows = np.unique(np.concatenate([rng.choice(n, 48, replace=False), [0, n - 1]]))
            ri = torch.from_numpy(rows).to(DEV)
            yref, s = oracle.gemv(w[ri].cpu().numpy(), len(rows), k, xbits(x))
            check_bound(y[:, ri].cpu().numpy(), yref, s, TOL, f"replay {rep} op {i}")


def test_gemv_rejects_memory_of_the_host(q4k):
    # a pinned host buffer is not device memory of the current device: the call
    # fails with Q4K_ERR_MEMORY and launches nothing
    n, k = 64, 512
    w = synth.q4k_weight(n, k, seed=4800).to(DEV)
    xh = synth.bf16_normal((1, k), seed=4801).pin_memory()
    y = torch.full((1, n), 3.0, device=DEV)
    L = q4k.lib()
    st = L.q4k_gemv(w.data_ptr(), n, k, xh.data_ptr(), 1, k, y.data_ptr(), n, None)
    assert st == 8
    wh = w.cpu().pin_memory()
    xd = xh.to(DEV)
    assert L.q4k_gemv(wh.data_ptr(), n, k, xd.data_ptr(), 1, k, y.data_ptr(), n, None) == 8
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())


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


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 16])
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


@pytest.mark.parametrize("batch,flags", [(1, 0), (1, 1), (3, 1), (6, 0)])
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
