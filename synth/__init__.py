"""Seeded synthetic inputs for the Q4_K projection path.

This module is the only code that both the CUDA path's tests/benchmark and the
CPU oracle consume.  It draws random fields and lays them into bytes; it holds
none of the method's arithmetic (no unpacking, no dequantization, no
contraction).  Every tensor is drawn from a torch generator seeded from
(base seed, tensor id), on the CPU or on a CUDA device.

Weights: each 144-byte Q4_K super-block gets
  * d and dmin drawn uniform in [lo, hi] in fp64 and rounded to binary16;
  * 12 uniformly random scale bytes.  The 96 bits of those bytes hold the
    eight 6-bit scales and eight 6-bit mins exactly once each, so uniform
    random bytes give independent scales/mins uniform in [0, 63];
  * 128 quant bytes.  "uniform": uniformly random bytes, i.e. independent
    4-bit quants uniform in [0, 15].  "normal": 256 independent draws of
    clip(round(8 + 3 z), 0, 15), z ~ N(0, 1), two per byte (low and high
    nibble).  The quants are independent and identically distributed, so
    which draw lands in which nibble does not change the distribution.
Activations: fp32 N(0, sigma) draws rounded to bf16 (round to nearest even).
Routing: top-k expert ids per token without replacement, expert popularity
Zipf(s) over a seeded random ranking of the experts; router weights are the
softmax over the token's k slots of N(0, 1) logits.
"""
from __future__ import annotations

import hashlib

import torch

Q4K_VALUES = 256
Q4K_BYTES = 144


def derive_seed(base: int, *ids) -> int:
    """A 63-bit seed for tensor `ids` of a workload seeded with `base`."""
    h = hashlib.sha256(repr((int(base),) + tuple(ids)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def q4k_weight(n: int, k: int, seed: int, quants: str = "uniform", device="cpu",
               d_range=(1e-3, 2e-2), chunk_blocks: int = 1 << 20) -> torch.Tensor:
    """An n x k Q4_K matrix as a uint8 tensor of shape [n, k/256*144]."""
    if k % Q4K_VALUES:
        raise ValueError("k must be a multiple of 256")
    if quants not in ("uniform", "normal"):
        raise ValueError(quants)
    nsb = n * (k // Q4K_VALUES)
    out = torch.empty((nsb, Q4K_BYTES), dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    lo, hi = d_range
    for start in range(0, nsb, chunk_blocks):
        cnt = min(chunk_blocks, nsb - start)
        blk = out[start:start + cnt]
        dd = torch.rand((cnt, 2), generator=g, dtype=torch.float64, device=device)
        dd = (lo + (hi - lo) * dd).to(torch.float16)           # RNE to binary16
        blk[:, 0:4] = dd.contiguous().view(torch.uint8).view(cnt, 4)
        blk[:, 4:16] = torch.randint(0, 256, (cnt, 12), generator=g, dtype=torch.uint8,
                                     device=device)
        if quants == "uniform":
            blk[:, 16:] = torch.randint(0, 256, (cnt, 128), generator=g, dtype=torch.uint8,
                                        device=device)
        else:
            z = torch.randn((cnt, 256), generator=g, dtype=torch.float32, device=device)
            q = torch.clamp(torch.round(8.0 + 3.0 * z), 0, 15).to(torch.uint8)
            blk[:, 16:] = q[:, :128] | (q[:, 128:] << 4)
    return out.view(n, (k // Q4K_VALUES) * Q4K_BYTES)


# Other k-quant super-blocks: bytes per block and the byte offsets of their
# binary16 scale fields (every other byte of a block is a valid field value).
KQ_LAYOUT = {2: (84, (80, 82)), 3: (110, (108,)), 4: (144, (0, 2)), 5: (176, (0, 2)),
             6: (210, (208,))}


def kq_weight(fmt: int, n: int, k: int, seed: int, device="cpu", d_range=(1e-3, 2e-2),
              chunk_blocks: int = 1 << 20) -> torch.Tensor:
    """An n x k matrix of k-quant format id fmt (2 q2_K, 3 q3_K, 4 Q4_K, 5 Q5_K,
    6 Q6_K) as uint8 [n, k/256 * block bytes]: uniform random bytes, with each
    binary16 scale field drawn uniformly in d_range."""
    if k % Q4K_VALUES:
        raise ValueError("k must be a multiple of 256")
    bb, halves = KQ_LAYOUT[fmt]
    nsb = n * (k // Q4K_VALUES)
    out = torch.empty((nsb, bb), dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    lo, hi = d_range
    for start in range(0, nsb, chunk_blocks):
        cnt = min(chunk_blocks, nsb - start)
        blk = out[start:start + cnt]
        blk[:] = torch.randint(0, 256, (cnt, bb), generator=g, dtype=torch.uint8, device=device)
        for off in halves:
            dd = torch.rand((cnt, 1), generator=g, dtype=torch.float64, device=device)
            dd = (lo + (hi - lo) * dd).to(torch.float16)
            blk[:, off:off + 2] = dd.contiguous().view(torch.uint8).view(cnt, 2)
    return out.view(n, (k // Q4K_VALUES) * bb)


def bf16_normal(shape, seed: int, sigma: float = 1.0, device="cpu") -> torch.Tensor:
    """bf16 activations: fp32 N(0, sigma) draws rounded to nearest-even bf16."""
    g = _gen(seed, device)
    v = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    return (v * sigma).to(torch.bfloat16)


def zipf_routing(n_tokens: int, n_experts: int, top_k: int, seed: int, s: float = 1.1):
    """(ids int32 [T, k], weights float32 [T, k]) drawn on the CPU."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(n_experts, generator=g)                 # rank -> expert id
    ranks = torch.arange(1, n_experts + 1, dtype=torch.float64)
    p = ranks.pow(-s)
    p = p / p.sum()
    picks = torch.stack([torch.multinomial(p, top_k, replacement=False, generator=g)
                         for _ in range(n_tokens)]) if n_tokens else torch.empty((0, top_k),
                                                                                 dtype=torch.long)
    ids = perm[picks].to(torch.int32)
    logits = torch.randn((n_tokens, top_k), generator=g, dtype=torch.float64)
    wts = torch.softmax(logits, dim=1).to(torch.float32)
    return ids.contiguous(), wts.contiguous()


def as_u16(x_bf16: torch.Tensor) -> torch.Tensor:
    """Reinterpret a bf16 tensor's bits as int16->uint16-compatible numpy input."""
    return x_bf16.contiguous().view(torch.int16)
