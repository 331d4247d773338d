"""q4k_moe_prefill (routed-expert FFN for token blocks, grouped tcgen05 GEMMs)
on the GPU against the oracle's MoE.

Bound, stage by stage (the GEMM bound 1e-2 * sum |w||x| on each grouped GEMM's
own input; g, u, h and the down outputs in bf16):
  dg = 1e-2 |Wg||x|,  du = 1e-2 |Wu||x|
  dh0 = 1.1 dg |u| + |silu(g)| du + 1.1 dg du          (|silu'| <= 1.1)
  dh  = dh0 + 2^-8 (|h| + dh0)                          (h rounded to bf16)
  |dy| <= sum_j |r_j| (1e-2 |Wd| (|h| + dh) + |Wd| dh) + 1e-5 sum_j |r_j| |Wd| |h|
(the last term covers the fp32 weighted sum).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, xbits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _make(E, H, F, T, K, seed, device="cpu"):
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=seed, device=device).reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=seed + 1, device=device).reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=seed + 2, device=device).reshape(-1)
    x = synth.bf16_normal((T, H), seed=seed + 3)
    ids, wts = synth.zipf_routing(T, E, K, seed=seed + 4)
    return dict(wg=wg, wu=wu, wd=wd, stride=stride, E=E, H=H, F=F, x=x, ids=ids, wts=wts)


def _gpu(q4k, c, ids=None, wts=None):
    ids = c["ids"] if ids is None else ids
    wts = c["wts"] if wts is None else wts
    y = q4k.q4k_moe_prefill(c["wg"].to(DEV), c["wu"].to(DEV), c["wd"].to(DEV), c["stride"], c["E"],
                            c["H"], c["F"], c["x"].to(DEV), ids.to(DEV), wts.to(DEV))
    torch.cuda.synchronize()
    err = q4k.q4k_get_device_error()
    return y.cpu().numpy().astype(np.float64), err


def _bound(c, ids, wts, tokens):
    E, H, F, s = c["E"], c["H"], c["F"], c["stride"]
    wg, wu, wd = (c[k].cpu().numpy() for k in ("wg", "wu", "wd"))
    xb = xbits(c["x"])
    xf = c["x"].to(torch.float64).numpy()
    ids_n = ids.numpy()
    wts_n = wts.numpy().astype(np.float64)
    yref = oracle.moe(wg, wu, wd, s, E, H, F, xb[tokens], ids_n[tokens],
                      wts_n[tokens].astype(np.float32))
    bound = np.zeros((len(tokens), H))
    for ti, t in enumerate(tokens):
        for j in range(ids_n.shape[1]):
            e = int(ids_n[t, j])
            if e < 0 or e >= E:
                continue
            ge, ue, de = (m[e * s:(e + 1) * s] for m in (wg, wu, wd))
            g = oracle.gemv_f64(ge, F, H, xf[t])[0]
            u = oracle.gemv_f64(ue, F, H, xf[t])[0]
            dg = 1e-2 * oracle.gemv_f64(ge, F, H, np.abs(xf[t]), use_abs=True)[0]
            du = 1e-2 * oracle.gemv_f64(ue, F, H, np.abs(xf[t]), use_abs=True)[0]
            sg = g / (1.0 + np.exp(-np.clip(g, -700.0, 700.0)))
            h = sg * u
            dh0 = 1.1 * dg * np.abs(u) + np.abs(sg) * du + 1.1 * dg * du
            dh = dh0 + 2.0 ** -8 * (np.abs(h) + dh0)
            awd_h = oracle.gemv_f64(de, H, F, np.abs(h), use_abs=True)[0]
            awd_dh = oracle.gemv_f64(de, H, F, dh, use_abs=True)[0]
            r = abs(wts_n[t, j])
            bound[ti] += r * (1e-2 * (awd_h + awd_dh) + awd_dh + 1e-5 * awd_h)
    return yref, bound


def _check(y, yref, bound, what):
    err = np.abs(y - yref)
    bad = ~(err <= bound + 1e-30)
    assert not bad.any(), f"{what}: {bad.sum()} outside, worst {np.max(err - bound)}"


@pytest.mark.parametrize("E,H,F,T,K", [(8, 256, 256, 1, 1), (8, 512, 512, 40, 2),
                                       (16, 1024, 512, 96, 4), (4, 512, 768, 300, 3)])
def test_moe_prefill_matches_oracle(q4k, E, H, F, T, K):
    c = _make(E, H, F, T, K, seed=E + H + F + T + K + 7)
    y, err = _gpu(q4k, c)
    assert err == 0
    tokens = list(range(T))
    yref, bound = _bound(c, c["ids"], c["wts"], tokens)
    _check(y[tokens], yref, bound, f"moe prefill E{E} H{H} F{F} T{T} k{K}")


def test_moe_prefill_one_expert_spans_several_slots(q4k):
    # 1100 tokens all routed to expert 2: slots of 256 pairs (four) and one of 76
    c = _make(4, 256, 512, 1100, 1, seed=90)
    ids = torch.full((1100, 1), 2, dtype=torch.int32)
    wts = torch.ones((1100, 1), dtype=torch.float32)
    y, err = _gpu(q4k, c, ids, wts)
    assert err == 0
    tokens = [0, 1, 255, 256, 257, 767, 768, 1023, 1024, 1099]
    yref, bound = _bound(c, ids, wts, tokens)
    _check(y[tokens], yref, bound, "one expert, three slots")


def test_moe_prefill_bad_ids_and_agreement_with_decode(q4k):
    # ids outside [0, E) are skipped and flagged; on 16 tokens the prefill
    # result agrees with the decode path within the sum of both bounds
    c = _make(8, 512, 512, 16, 3, seed=91)
    ids = c["ids"].clone()
    ids[2, 1] = 8
    ids[5, 0] = -1
    y, err = _gpu(q4k, c, ids=ids)
    assert err == 2  # Q4K_DEVERR_BAD_EXPERT
    keep = torch.ones_like(c["wts"])
    keep[2, 1] = 0
    keep[5, 0] = 0
    tokens = list(range(16))
    yref, bound = _bound(c, ids.clamp(0, 7), c["wts"] * keep, tokens)
    _check(y, yref, bound, "bad ids")
    yd = q4k.q4k_moe_gemv(c["wg"].to(DEV), c["wu"].to(DEV), c["wd"].to(DEV), c["stride"], c["E"],
                          c["H"], c["F"], c["x"].to(DEV), c["ids"].to(DEV), c["wts"].to(DEV))
    yp = q4k.q4k_moe_prefill(c["wg"].to(DEV), c["wu"].to(DEV), c["wd"].to(DEV), c["stride"], c["E"],
                             c["H"], c["F"], c["x"].to(DEV), c["ids"].to(DEV), c["wts"].to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    _, b2 = _bound(c, c["ids"], c["wts"], tokens)
    assert np.all(np.abs(yd.cpu().numpy() - yp.cpu().numpy()) <= 2 * b2 + 1e-30)


def test_moe_prefill_deterministic(q4k):
    c = _make(16, 512, 512, 200, 4, seed=92)
    a, _ = _gpu(q4k, c)
    b, _ = _gpu(q4k, c)
    assert np.array_equal(a, b)


def test_moe_prefill_235b_class_sampled_tokens(q4k):
    # 128 experts, hidden 4096, expert ffn 1536, 512 prefill tokens, top-8 Zipf(1.1)
    E, H, F, T, K = 128, 4096, 1536, 512, 8
    c = _make(E, H, F, T, K, seed=93, device=DEV)
    y, err = _gpu(q4k, c)
    assert err == 0
    tokens = [0, 255, 511]
    yref, bound = _bound(c, c["ids"], c["wts"], tokens)
    _check(y[tokens], yref, bound, "235B-class prefill")


def test_moe_prefill_most_experts_and_slots_per_token(q4k):
    # 2048 experts (the largest count), top-16 (the largest), 64 tokens
    E, H, F, T, K = 2048, 256, 256, 64, 16
    c = _make(E, H, F, T, K, seed=94)
    y, err = _gpu(q4k, c)
    assert err == 0
    tokens = [0, 31, 63]
    yref, bound = _bound(c, c["ids"], c["wts"], tokens)
    _check(y[tokens], yref, bound, "2048 experts top-16")


def test_moe_prefill_graph_replay_matches_eager(q4k):
    # the seven launches captured in one CUDA graph and replayed: the result
    # equals the eager call's (the path is deterministic)
    c = _make(16, 512, 512, 120, 4, seed=95)
    E, H, F = c["E"], c["H"], c["F"]
    T, K = c["ids"].shape
    args = [c[k].to(DEV) for k in ("wg", "wu", "wd")]
    x, ids, wts = c["x"].to(DEV), c["ids"].to(DEV), c["wts"].to(DEV)
    ws = torch.empty(q4k.q4k_moe_prefill_workspace_size(E, T, K, H, F), dtype=torch.uint8, device=DEV)
    eager = q4k.q4k_moe_prefill(*args, c["stride"], E, H, F, x, ids, wts, workspace=ws).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream(device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        q4k.q4k_moe_prefill(*args, c["stride"], E, H, F, x, ids, wts, out=out, workspace=ws, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            q4k.q4k_moe_prefill(*args, c["stride"], E, H, F, x, ids, wts, out=out, workspace=ws,
                                stream=s)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    assert torch.equal(out, eager)
