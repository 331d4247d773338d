"""The other k-quant formats (q2_K, q3_K, Q5_K, Q6_K) on the GPU against the
oracle: dequantization bit-exact (fp32: the exact weight rounded once; bf16:
that, rounded to nearest even), the decode projection within 2e-3 * sum|w||x|
per element, and one-hot activations that must return the oracle's fp32
weights exactly."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_bound, xbits

pytestmark = pytest.mark.gpu
FMTS = (2, 3, 5, 6)
TOL = 2e-3


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(1, 256), (7, 1024), (33, 5120), (3, 17408)])
def test_kq_dequant_bit_exact(q4k, fmt, n, k):
    w = synth.kq_weight(fmt, n, k, seed=fmt * 100 + n + k)
    got32 = q4k.q4k_kq_dequant(fmt, w.to(DEV), n, k).cpu().numpy()
    got16 = q4k.q4k_kq_dequant(fmt, w.to(DEV), n, k, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    assert np.array_equal(got32.view(np.uint32), oracle.kq_dequant_f32(fmt, w.numpy(), n, k).view(np.uint32))
    bits = got16.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, oracle.kq_dequant_bf16(fmt, w.numpy(), n, k))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 9, 16])
@pytest.mark.parametrize("n,k", [(37, 256), (130, 2560), (64, 17408)])
def test_kq_gemv_matches_oracle(q4k, fmt, batch, n, k):
    w = synth.kq_weight(fmt, n, k, seed=fmt * 1000 + batch * 7 + n + k)
    x = synth.bf16_normal((batch, k), seed=fmt + batch + k)
    y = q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x))
    check_bound(y.cpu().numpy().astype(np.float64), yref, s, TOL, f"kq{fmt} b{batch} {n}x{k}")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_gemv_one_hot_returns_the_fp32_weights(q4k, fmt):
    # x = e_i (one nonzero of value 1): every product but one is zero, so y is
    # exactly the weight column, as the fp32 dequantization rounds it
    n, k = 40, 1024
    w = synth.kq_weight(fmt, n, k, seed=fmt + 500)
    cols = [0, 7, 8, 15, 16, 31, 32, 63, 64, 127, 128, 255, 256, 511, 777, 1023]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16)
    for b, c in enumerate(cols):
        x[b, c] = 1.0
    wf = oracle.kq_dequant_f32(fmt, w.numpy(), n, k)
    for lo in range(0, len(cols), 16):
        y = q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x[lo:lo + 16].to(DEV))
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        for b, c in enumerate(cols[lo:lo + 16]):
            assert np.array_equal(got[b], wf[:, c]), f"fmt {fmt} column {c}"


def test_kq_gemv_strided_io_and_q4k_route(q4k):
    n, k, batch = 96, 1536, 5
    for fmt in (3, 4):
        w = (synth.kq_weight(fmt, n, k, seed=600 + fmt) if fmt != 4
             else synth.q4k_weight(n, k, seed=604))
        xs = synth.bf16_normal((batch, k + 64), seed=601).to(DEV)
        x = xs[:, 32:32 + k]
        out = torch.full((batch, n + 8), float("nan"), dtype=torch.float32, device=DEV)
        q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x, out=out[:, :n])
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isnan(got[:, n:]))
        yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x.cpu()))
        check_bound(got[:, :n].astype(np.float64), yref, s, TOL, f"strided kq{fmt}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(5120, 17408), (4096, 1536)])
def test_kq_gemv_full_size_sampled(q4k, fmt, n, k):
    # the 27B-class down projection, and one routed expert's down projection
    # of the 235B-class MoE (the q2_K / q3_K routed-down recipes)
    w = synth.kq_weight(fmt, n, k, seed=700 + fmt + n, device=DEV)
    x = synth.bf16_normal((1, k), seed=701 + fmt)
    y = q4k.q4k_kq_gemv(fmt, w, n, k, x.to(DEV))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(n).choice(n, 48, replace=False),
                                     [0, 1, n - 2, n - 1]]))
    wsub = w[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    yref, s = oracle.kq_gemv(fmt, wsub, len(rows), k, xbits(x))
    check_bound(y.cpu().numpy()[:, rows].astype(np.float64), yref, s, TOL, f"full kq{fmt} {n}x{k}")


def test_kq_gemv_longest_row_and_host_memory_rejected(q4k):
    # Q6_K at the longest K whose 8 row buffers fit in shared memory (138 super-blocks)
    n, k = 5, 35328
    w = synth.kq_weight(6, n, k, seed=800)
    x = synth.bf16_normal((2, k), seed=801)
    y = q4k.q4k_kq_gemv(6, w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    yref, s = oracle.kq_gemv(6, w.numpy(), n, k, xbits(x))
    check_bound(y.cpu().numpy().astype(np.float64), yref, s, TOL, "Q6_K longest row")
    # weights in host memory: refused before anything runs (Q4K_ERR_MEMORY)
    wh = w.pin_memory()
    with pytest.raises(q4k.Q4KError) as ei:
        q4k.q4k_kq_gemv(6, wh, n, k, x.to(DEV))
    assert ei.value.status == 8


def _cancel_matrix(fmt, k, seed):
    """Rows of q2_K, q3_K, Q5_K or Q6_K blocks; every third row has all weights
    exactly 0 (q2_K, Q5_K: d sc q = dmin m with q = c for every weight of every
    sub-block, Q5_K's c up to 31 so that the fifth quant bit is set; q3_K,
    Q6_K: every quant at its zero point), the others random."""
    from _kq_fields import pack_q2k, pack_q3k, pack_q5k, pack_q6k, random_block
    from _q4k_fields import half_bits
    rng = np.random.default_rng(seed)
    rows = []
    for r in range(30):
        blks = []
        for _ in range(k // 256):
            if r % 3 == 0:
                # d = 1/64, sc = 2 (ds = 1/32); dmin = 1/32, m = c: w = (q - c)/32
                if fmt == 6:  # no min term: every quant at the zero point (u = 32)
                    sc = [int(v) for v in rng.integers(-128, 128, 16)]
                    blks.append(pack_q6k(half_bits(rng.uniform(1e-3, 2e-2)), sc, [0] * 256))
                elif fmt == 3:  # no min term: every quant at the zero point (u = 4)
                    sc = [int(v) for v in rng.integers(0, 64, 16)]
                    blks.append(pack_q3k(half_bits(rng.uniform(1e-3, 2e-2)), sc, [0] * 256))
                elif fmt == 5:
                    c = [int(v) for v in rng.integers(0, 32, 8)]
                    q = [c[i // 32] for i in range(256)]
                    blks.append(pack_q5k(half_bits(1 / 64), half_bits(1 / 32), [2] * 8, c, q))
                else:
                    c = [int(v) for v in rng.integers(0, 4, 16)]
                    q = [c[i // 16] for i in range(256)]
                    blks.append(pack_q2k(half_bits(1 / 64), half_bits(1 / 32), [2] * 16, c, q))
            else:
                blks.append(random_block(fmt, rng)[0])
        rows.append(b"".join(blks))
    return torch.frombuffer(bytearray(b"".join(rows)), dtype=torch.uint8).view(len(rows), -1)


@pytest.mark.parametrize("fmt", [2, 3, 5, 6])
@pytest.mark.parametrize("k", [256, 1280, 5120])
def test_cancelling_rows_give_exact_zero_at_batch_1(q4k, fmt, k):
    # batch 1 runs q2_K, Q5_K (offset form, c up to 4 and 32), q3_K and Q6_K
    # (exact q - 4, q - 32) on the tensor cores: rows whose weights are all zero
    # must come out exactly 0, the rest within the bound
    w = _cancel_matrix(fmt, k, seed=k + fmt)
    n = w.shape[0]
    x = synth.bf16_normal((1, k), seed=3 * k + fmt)
    y = q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    got = y.cpu().numpy().astype(np.float64)
    yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x))
    assert np.all(s[:, 0::3] == 0.0) and np.all(yref[:, 0::3] == 0.0)
    assert np.all(got[:, 0::3] == 0.0), f"kq{fmt}: rows whose weights all cancel must be exactly 0"
    check_bound(got, yref, s, TOL, f"kq{fmt} cancel k{k}")


@pytest.mark.parametrize("fmt", [2, 3, 5, 6])
@pytest.mark.parametrize("batch", [2, 3, 4])
@pytest.mark.parametrize("k", [256, 5120])
def test_cancelling_rows_give_exact_zero_at_batch_2_to_4(q4k, fmt, batch, k):
    # batch 2..4 runs on the tensor cores too (MMA columns = (sub-block slot,
    # batch row)): rows whose weights all cancel come out exactly 0 for every
    # batch row, the rest within the bound
    w = _cancel_matrix(fmt, k, seed=k + 10 * fmt + batch)
    n = w.shape[0]
    x = synth.bf16_normal((batch, k), seed=5 * k + batch + fmt)
    y = q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    got = y.cpu().numpy().astype(np.float64)
    yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x))
    assert np.all(s[:, 0::3] == 0.0) and np.all(yref[:, 0::3] == 0.0)
    assert np.all(got[:, 0::3] == 0.0), f"kq{fmt} b{batch}: rows whose weights all cancel must be exactly 0"
    check_bound(got, yref, s, TOL, f"kq{fmt} cancel k{k} b{batch}")


@pytest.mark.parametrize("fmt", [2, 3, 5, 6])
@pytest.mark.parametrize("n,k", [(4901, 1280), (16 * 152 * 2 + 3, 512), (3, 3 * 256), (1000, 17408)])
def test_batch_1_tensor_core_formats_many_shapes(q4k, fmt, n, k):
    # many 16-row tiles (more than one per warp) with a ragged last tile, a
    # single odd row count with an odd number of super-blocks (q2_K, q3_K and
    # Q6_K rows then start at every 4- or 2-byte offset mod 16), and long rows
    # (many ring turns)
    w = synth.kq_weight(fmt, n, k, seed=900 + n + fmt)
    x = synth.bf16_normal((1, k), seed=901 + fmt)
    y = q4k.q4k_kq_gemv(fmt, w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x))
    check_bound(y.cpu().numpy().astype(np.float64), yref, s, TOL, f"kq{fmt} b1 {n}x{k}")


@pytest.mark.parametrize("fmt", [2, 3, 5, 6])
@pytest.mark.parametrize("batch,flags,count", [(1, 1, 12), (1, 0, 175), (3, 0, 5)])
def test_kq_gemv_seq_matches_oracle(q4k, fmt, batch, flags, count):
    # one q4k_kq_gemv_seq call over projections of different shapes (empty
    # ops, single rows, odd super-block counts and ragged tiles among them):
    # at batch 1 one or two persistent launches, at batch 3 one launch per op;
    # every op matches the oracle and an empty op writes nothing
    rng = np.random.default_rng(7100 + 10 * fmt + count)
    shapes = [(int(rng.choice([0, 1, 17, 40, 129, 700])), int(rng.choice([256, 768, 1280])))
              for _ in range(count)]
    shapes[0] = (333, 2304)
    ws, xs, ys, tup = [], [], [], []
    for i, (n, k) in enumerate(shapes):
        w = synth.kq_weight(fmt, max(n, 1), k, seed=7200 + 7 * i + fmt)
        x = synth.bf16_normal((batch, k), seed=7300 + i)
        y = torch.full((batch, max(n, 1)), 7.0, device=DEV)
        ws.append(w)
        xs.append(x)
        ys.append(y)
        tup.append((w.to(DEV), n, k, x.to(DEV), y))
    ops = q4k.gemv_ops(tup)
    q4k.q4k_kq_gemv_seq(fmt, ops, batch, flags)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    for i, ((n, k), w, x, y) in enumerate(zip(shapes, ws, xs, ys)):
        if n == 0:
            assert bool((y == 7.0).all()), "an empty op writes nothing"
            continue
        yref, s = oracle.kq_gemv(fmt, w.numpy(), n, k, xbits(x))
        check_bound(y.cpu().numpy().astype(np.float64), yref, s, TOL, f"kq{fmt} seq op {i} {n}x{k} b{batch}")
