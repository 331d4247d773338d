"""q4k_gemm_rmsnorm (prefill projection with a fused RMSNorm prologue) on the
GPU against the oracle.

Bound: the q4k_gemm bound on the normalised input, per element
|y - y_ref| <= 1e-2 * sum_k |w_k| |xh_k| with xh = x * rinv * gamma from the
oracle (fp64), and normwise 1e-2.  rinv against the oracle's: the fp32 sum of
k squares (thread-strided over 256 threads, a 5-step butterfly, then 8 warp
sums: at most k/2048 + 13 roundings of a sum of positive terms) plus the
division and square root, relative error <= (k/2048 + 16) * 2^-24.
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
EPS = 1e-6


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _inputs(m, k, seed):
    """x rows N(0, 0.5^2) times 2^u, u uniform in [-8, 8] per token (so 1/rms
    spans 2^16), and gamma uniform in [-2, 2] (signs included)."""
    rng = np.random.default_rng(seed)
    x = synth.bf16_normal((m, k), seed=seed, sigma=0.5)
    scale = torch.from_numpy(2.0 ** rng.integers(-8, 9, (m, 1))).to(torch.float32)
    x = (x.float() * scale).to(torch.bfloat16)
    gamma = torch.from_numpy(rng.uniform(-2.0, 2.0, k).astype(np.float32))
    return x, gamma


def _run(q4k, w, n, k, x, gamma, eps=EPS):
    y, rinv = q4k.q4k_gemm_rmsnorm(w.to(DEV), n, k, x.to(DEV), gamma.to(DEV), eps)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    return y.float().cpu().numpy().astype(np.float64), rinv.cpu().numpy().astype(np.float64)


def _check(got, rinv, w, n, k, x, gamma, what, eps=EPS):
    yref, s, rref = oracle.rmsnorm_gemv(w.cpu().numpy(), n, k, xbits(x), gamma.numpy(), eps)
    rtol = (k / 2048 + 16) * 2.0 ** -24
    assert np.all(np.abs(rinv - rref) <= rtol * rref), f"{what}: rinv"
    check_bound(got, yref, s, TOL, what)
    nrm = np.linalg.norm(got - yref) / max(np.linalg.norm(yref), 1e-300)
    assert nrm <= TOL, nrm


# The q4k_gemm shapes: one CTA per tile (KS = 1) and the cluster split-K
# path with K split 2, 3 or 4 ways, with and without X shared by pairs.
CASES = [(1, 128, 256), (77, 200, 512), (128, 256, 1024), (512, 384, 2048), (600, 130, 768),
         (513, 1024, 1536), (256, 2048, 5120), (64, 300, 1792), (700, 130, 2560),
         (64, 7680, 1024)]


@pytest.mark.parametrize("m,n,k", CASES)
def test_gemm_rmsnorm_matches_oracle(q4k, m, n, k):
    w = synth.q4k_weight(n, k, seed=m + n + k + 1, quants="normal" if n % 3 else "uniform")
    x, gamma = _inputs(m, k, seed=m * 5 + k)
    got, rinv = _run(q4k, w, n, k, x, gamma)
    _check(got, rinv, w, n, k, x, gamma, f"gemm_rmsnorm m{m} n{n} k{k}")


def test_gemm_rmsnorm_zero_row_unit_gamma_and_eps(q4k):
    # a token row of zeros: rinv = 1/sqrt(eps), y = 0 exactly; gamma = 1 and
    # x = +-1 with eps = 0: rinv = 1 and the result is q4k_gemm's, bit for bit
    m, n, k = 40, 256, 1024
    w = synth.q4k_weight(n, k, seed=60)
    x, gamma = _inputs(m, k, seed=61)
    x[7] = 0
    got, rinv = _run(q4k, w, n, k, x, gamma, eps=0.25)
    assert rinv[7] == 2.0 and np.all(got[7] == 0.0)
    _check(got, rinv, w, n, k, x, gamma, "zero row", eps=0.25)
    signs = torch.where(torch.from_numpy(np.random.default_rng(62).random((m, k)) < 0.5), -1.0,
                        1.0).to(torch.bfloat16)
    got1, rinv1 = _run(q4k, w, n, k, signs, torch.ones(k), eps=0.0)
    plain = q4k.q4k_gemm(w.to(DEV), n, k, signs.to(DEV))
    torch.cuda.synchronize()
    assert np.all(rinv1 == 1.0)
    assert np.array_equal(got1, plain.float().cpu().numpy().astype(np.float64))


def test_gemm_rmsnorm_deterministic(q4k):
    m, n, k = 300, 512, 1024
    w = synth.q4k_weight(n, k, seed=63).to(DEV)
    x, gamma = _inputs(m, k, seed=64)
    x, gamma = x.to(DEV), gamma.to(DEV)
    a, ra = q4k.q4k_gemm_rmsnorm(w, n, k, x, gamma, EPS)
    a, ra = a.clone(), ra.clone()
    b, rb = q4k.q4k_gemm_rmsnorm(w, n, k, x, gamma, EPS)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ra, rb)


# 512-token prefill, 27B-class gate (5120 -> 17408: one CTA per tile, pairs
# sharing X) and down (17408 -> 5120: K split 3 ways), sampled rows
@pytest.mark.parametrize("n,k", [(17408, 5120), (5120, 17408)])
def test_gemm_rmsnorm_full_size_sampled(q4k, n, k):
    m = 512
    w = synth.q4k_weight(n, k, seed=n + k + 2, quants="normal", device=DEV)
    x, gamma = _inputs(m, k, seed=n + 3)
    y, rinv = q4k.q4k_gemm_rmsnorm(w, n, k, x.to(DEV), gamma.to(DEV), EPS)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    rows = np.unique(np.concatenate([np.random.default_rng(n).choice(n, 40, replace=False),
                                     [0, 127, 128, n - 1]]))
    idx = torch.from_numpy(rows).to(DEV)
    got = y[:, idx].float().cpu().numpy().astype(np.float64)
    _check(got, rinv.cpu().numpy().astype(np.float64), w[idx], len(rows), k, x, gamma,
           f"full gemm_rmsnorm {n}x{k}")


def test_gemm_rmsnorm_reads_the_previous_output(q4k):
    # Y1 = q4k_gemm(X0), then the normed projection of Y1 queued right behind
    # it (its rinv kernel and GEMM are programmatic dependents): both must see
    # Y1 complete, so the result equals a run on a copy of Y1 taken after a
    # synchronize.
    m, k0, n1, n2 = 700, 1024, 2048, 640
    w1 = synth.q4k_weight(n1, k0, seed=65, quants="normal").to(DEV)
    w2 = synth.q4k_weight(n2, n1, seed=66, quants="normal").to(DEV)
    x0 = synth.bf16_normal((m, k0), seed=67, sigma=0.5).to(DEV)
    gamma = torch.from_numpy(np.random.default_rng(68).uniform(0.5, 1.5, n1).astype(np.float32)).to(DEV)
    for _ in range(3):
        y1 = q4k.q4k_gemm(w1, n1, k0, x0)
        y2, r2 = q4k.q4k_gemm_rmsnorm(w2, n2, n1, y1, gamma, EPS)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    y1c = y1.clone()
    torch.cuda.synchronize()
    ref, rref = q4k.q4k_gemm_rmsnorm(w2, n2, n1, y1c, gamma, EPS)
    torch.cuda.synchronize()
    assert torch.equal(y2, ref) and torch.equal(r2, rref)
