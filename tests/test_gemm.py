"""q4k_gemm (prefill, tcgen05) on the GPU against the oracle.

Bound (bf16 tensor-core path): per element |y - y_ref| <= 1e-2 * sum_k |w_k||x_k|,
and normwise ||Y - Y_ref||_F <= 1e-2 ||Y_ref||_F.  A tighter check ties the
weight tiles to round-to-nearest-even bf16 of the exact weights: against the
fp64 product of the oracle's bf16-dequantized weights the only remaining errors
are fp32 accumulation and the final bf16 rounding of Y.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_bound, xbits

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _bf16_to_f64(a_u16: np.ndarray) -> np.ndarray:
    return (a_u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check(q4k, w, n, k, x, sigma_note=""):
    y = q4k.q4k_gemm(w.to(DEV), n, k, x.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    got = y.float().cpu().numpy().astype(np.float64)
    yref, s = oracle.gemv(w.cpu().numpy(), n, k, xbits(x))
    check_bound(got, yref, s, TOL, f"gemm m{x.shape[0]} n{n} k{k} {sigma_note}")
    nrm = np.linalg.norm(got - yref) / max(np.linalg.norm(yref), 1e-300)
    assert nrm <= TOL, nrm
    # tiles are RNE-bf16 of the exact weights: compare with the fp64 product of
    # those bf16 weights; remaining error = fp32 accumulation + bf16 output
    wb = _bf16_to_f64(oracle.dequant_bf16(w.cpu().numpy(), n, k))
    xf = x.to(torch.float64).cpu().numpy()
    yb = xf @ wb.T
    mag = np.abs(xf) @ np.abs(wb).T
    err = np.abs(got - yb)
    assert np.all(err <= 2.0 ** -8 * np.abs(yb) + 1e-5 * mag + 1e-30), float(np.max(err - 2.0 ** -8 * np.abs(yb)))
    return got


# Few output tiles with enough K take the cluster split-K path, K split 2, 3 or 4
# ways (uneven ranges included), alone or with X shared by pairs of weight tiles:
# (128, 256, 1024) 1x2, (512, 384, 2048) 1x4, (64, 300, 1792) 1x3, (700, 130, 2560)
# 1x4, (513, 1024, 1536) 2x3, (256, 2048, 5120) 2x4, (64, 7680, 1024) 2x2.
CASES = [(1, 128, 256), (77, 200, 512), (128, 256, 1024), (512, 384, 2048), (600, 130, 768),
         (513, 1024, 1536), (256, 2048, 5120), (64, 300, 1792), (700, 130, 2560),
         (64, 7680, 1024)]


@pytest.mark.parametrize("m,n,k", CASES)
def test_gemm_matches_oracle(q4k, m, n, k):
    w = synth.q4k_weight(n, k, seed=m + n + k, quants="normal" if n % 3 else "uniform")
    x = synth.bf16_normal((m, k), seed=m * 3 + k, sigma=0.5)
    _check(q4k, w, n, k, x)


def test_gemm_strided_io(q4k):
    m, n, k = 100, 256, 512
    w = synth.q4k_weight(n, k, seed=5)
    xs = synth.bf16_normal((m, k + 32), seed=6, sigma=0.5).to(DEV)
    x = xs[:, 16:16 + k]
    out = torch.full((m, n + 8), float("nan"), dtype=torch.bfloat16, device=DEV)
    q4k.q4k_gemm(w.to(DEV), n, k, x, out=out[:, :n])
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    assert np.all(np.isnan(got[:, n:]))
    yref, s = oracle.gemv(w.numpy(), n, k, xbits(x))
    check_bound(got[:, :n].astype(np.float64), yref, s, TOL, "strided gemm")


def test_gemm_row_matches_gemv(q4k):
    m, n, k = 64, 384, 1024
    w = synth.q4k_weight(n, k, seed=7).to(DEV)
    x = synth.bf16_normal((m, k), seed=8, sigma=0.5).to(DEV)
    yg = q4k.q4k_gemm(w, n, k, x).float()
    yv = q4k.q4k_gemv(w, n, k, x[:16])
    torch.cuda.synchronize()
    _, s = oracle.gemv(w.cpu().numpy(), n, k, xbits(x[:16]))
    diff = (yg[:16] - yv).abs().cpu().numpy()
    assert np.all(diff <= (1e-2 + 2e-3) * s)


def test_gemm_deterministic(q4k):
    m, n, k = 300, 512, 1024
    w = synth.q4k_weight(n, k, seed=9).to(DEV)
    x = synth.bf16_normal((m, k), seed=10, sigma=0.5).to(DEV)
    a = q4k.q4k_gemm(w, n, k, x).clone()
    b = q4k.q4k_gemm(w, n, k, x)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# 512-token prefill on the 27B-class gate (5120 -> 17408) and down (17408 -> 5120)
@pytest.mark.parametrize("n,k", [(17408, 5120), (5120, 17408)])
def test_gemm_full_size_sampled(q4k, n, k):
    m = 512
    w = synth.q4k_weight(n, k, seed=n + k, quants="normal", device=DEV)
    x = synth.bf16_normal((m, k), seed=n, sigma=0.5, device=DEV)
    y = q4k.q4k_gemm(w, n, k, x)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    rows = np.unique(np.concatenate([np.random.default_rng(n).choice(n, 40, replace=False),
                                     [0, 127, 128, n - 1]]))
    idx = torch.from_numpy(rows).to(DEV)
    wsub = w[idx].cpu().numpy()
    yref, s = oracle.gemv(wsub, len(rows), k, xbits(x))
    got = y[:, idx].float().cpu().numpy().astype(np.float64)
    check_bound(got, yref, s, TOL, f"full gemm {n}x{k}")


def test_gemm_chain_reads_the_previous_output(q4k):
    # Y1 = X0 W1^T and Y2 = Y1 W2^T queued back to back on one stream (the
    # GEMM is launched as a programmatic dependent of the kernel before it):
    # the second GEMM must see Y1 complete, so Y2 equals the same GEMM run on a
    # copy of Y1 taken after a synchronize (the kernel is deterministic).
    m, k0, n1, n2 = 700, 1024, 2048, 640
    w1 = synth.q4k_weight(n1, k0, seed=41, quants="normal").to(DEV)
    w2 = synth.q4k_weight(n2, n1, seed=42, quants="normal").to(DEV)
    x0 = synth.bf16_normal((m, k0), seed=43, sigma=0.5).to(DEV)
    for _ in range(3):
        y1 = q4k.q4k_gemm(w1, n1, k0, x0)
        y2 = q4k.q4k_gemm(w2, n2, n1, y1)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    y1c = y1.clone()
    torch.cuda.synchronize()
    ref = q4k.q4k_gemm(w2, n2, n1, y1c)
    torch.cuda.synchronize()
    assert torch.equal(y2, ref)


def test_gemm_rejects_memory_of_the_host(q4k):
    # the GEMM multicasts X within a cluster through a tensor map over x: a
    # pinned host buffer (not device memory of the current device) as x, w or
    # y fails with Q4K_ERR_MEMORY and launches nothing, with and without the
    # RMSNorm prologue
    m, n, k = 128, 256, 512
    w = synth.q4k_weight(n, k, seed=4900).to(DEV)
    x = synth.bf16_normal((m, k), seed=4901)
    xh = x.pin_memory()
    xd = x.to(DEV)
    y = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    gamma = torch.ones(k, dtype=torch.float32, device=DEV)
    rinv = torch.full((m,), 5.0, dtype=torch.float32, device=DEV)
    L = q4k.lib()
    assert L.q4k_gemm(w.data_ptr(), n, k, xh.data_ptr(), m, k, y.data_ptr(), n, None) == 8
    wh = w.cpu().pin_memory()
    assert L.q4k_gemm(wh.data_ptr(), n, k, xd.data_ptr(), m, k, y.data_ptr(), n, None) == 8
    yh = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    assert L.q4k_gemm(w.data_ptr(), n, k, xd.data_ptr(), m, k, yh.data_ptr(), n, None) == 8
    assert L.q4k_gemm_rmsnorm(w.data_ptr(), n, k, xh.data_ptr(), m, k, gamma.data_ptr(), 1e-6,
                              rinv.data_ptr(), y.data_ptr(), n, None) == 8
    torch.cuda.synchronize()
    assert bool((y == 3.0).all()) and bool((rinv == 5.0).all())
