"""q4k_dequant on the GPU against the oracle: bit-exact fp32 and bf16."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV
from _q4k_fields import pack_block, random_fields

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


@pytest.mark.parametrize("n,k,quants", [(1, 256, "uniform"), (7, 512, "normal"),
                                        (129, 1280, "uniform"), (300, 4096, "normal")])
def test_dequant_fp32_bit_exact(q4k, n, k, quants):
    w = synth.q4k_weight(n, k, seed=n * 7 + k, quants=quants)
    got = q4k.q4k_dequant(w.to(DEV), n, k).cpu().numpy()
    ref = oracle.dequant_f32(w.numpy(), n, k)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n,k", [(3, 256), (65, 2048)])
def test_dequant_bf16_bit_exact(q4k, n, k):
    w = synth.q4k_weight(n, k, seed=n + k)
    got = q4k.q4k_dequant(w.to(DEV), n, k, out_dtype=torch.bfloat16).cpu()
    ref = oracle.dequant_bf16(w.numpy(), n, k)
    assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), ref)


def test_dequant_handbuilt_and_extreme_fields(q4k):
    rng = np.random.default_rng(5)
    blocks = [random_fields(rng) for _ in range(30)]
    # extremes: max scales/mins, subnormal and negative d, zero block
    blocks.append((0x7BFF, 0x7BFF, [63] * 8, [63] * 8, [15] * 256))
    blocks.append((0x0001, 0x0001, [63] * 8, [0] * 8, list(range(16)) * 16))
    blocks.append((0xBC00, 0x3C00, list(range(8)), list(range(8, 16)), [7] * 256))
    blocks.append((0, 0, [0] * 8, [0] * 8, [0] * 256))
    raw = b"".join(pack_block(*b) for b in blocks)
    n = len(blocks)
    w = torch.frombuffer(bytearray(raw), dtype=torch.uint8).view(n, 144)
    got = q4k.q4k_dequant(w.to(DEV), n, 256).cpu().numpy()
    ref = oracle.dequant_f32(w.numpy(), n, 256)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_full_size_projection_sampled(q4k):
    # a 27B-class gate projection (17408 x 5120), every block checked on sampled rows
    n, k = 17408, 5120
    w = synth.q4k_weight(n, k, seed=77, quants="normal", device=DEV)
    got = q4k.q4k_dequant(w, n, k)
    rows = np.random.default_rng(0).choice(n, 64, replace=False)
    rows.sort()
    wc = w[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    ref = oracle.dequant_f32(wc, len(rows), k)
    assert np.array_equal(got[torch.from_numpy(rows).to(DEV)].cpu().numpy().view(np.uint32),
                          ref.view(np.uint32))


def test_dequant_4096x4096_every_block(q4k):
    # the 4096 x 4096 single-matrix workload (uniform quants), every block in
    # fp32 and bf16 against the oracle, bit for bit
    n = k = 4096
    w = synth.q4k_weight(n, k, seed=1000)
    d32 = q4k.q4k_dequant(w.to(DEV), n, k)
    d16 = q4k.q4k_dequant(w.to(DEV), n, k, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(d32.cpu().numpy(), oracle.dequant_f32(w.numpy(), n, k))
    got16 = d16.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got16, oracle.dequant_bf16(w.numpy(), n, k))

