"""q4k_moe_gemv (routed-expert decode FFN) on the GPU against the oracle.

Bound: the fp32-path tolerance 2e-3 * sum|w||x| of every matmul stage,
propagated through SiLU(g)*u (|silu'| <= 1.1), the down projection and the
route-weighted sum:
  dh_k  = 1.1 dg_k |u_k| + |silu(g_k)| du_k + 1.1 dg_k du_k + 2^-15 |h_k|
  |dy|  <= sum_j |r_j| (2e-3 |Wd| |h| + 1.002 |Wd| dh)
with dg = 2e-3 |Wg||x|, du = 2e-3 |Wu||x| (the 2^-15 term covers h entering
the down MMA as two bf16 parts).
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


def _make(E, H, F, T, K, seed, quants="uniform", sigma=1.0):
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=seed, quants=quants).reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=seed + 1, quants=quants).reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=seed + 2, quants=quants).reshape(-1)
    x = synth.bf16_normal((T, H), seed=seed + 3, sigma=sigma)
    ids, wts = synth.zipf_routing(T, E, K, seed=seed + 4)
    return dict(wg=wg, wu=wu, wd=wd, stride=stride, E=E, H=H, F=F, x=x, ids=ids, wts=wts)


def _gpu(q4k, c, ids=None, wts=None, flags=0):
    ids = c["ids"] if ids is None else ids
    wts = c["wts"] if wts is None else wts
    y = q4k.q4k_moe_gemv_ex(c["wg"].to(DEV), c["wu"].to(DEV), c["wd"].to(DEV), c["stride"],
                            c["E"], c["H"], c["F"], c["x"].to(DEV), ids.to(DEV), wts.to(DEV),
                            flags=flags)
    torch.cuda.synchronize()
    err = q4k.q4k_get_device_error()
    return y.cpu().numpy().astype(np.float64), err


def _bound(c, ids, wts, tokens, weighted_down=False):
    """Reference y and the propagated error bound for the listed tokens (the
    same bound for both orders: |r| |Wd| |h| = |Wd| |r h|)."""
    E, H, F, s = c["E"], c["H"], c["F"], c["stride"]
    wg, wu, wd = (c[k].numpy() for k in ("wg", "wu", "wd"))
    xb = xbits(c["x"])
    xf = c["x"].to(torch.float64).numpy()
    ids_n = ids.numpy()
    wts_n = wts.numpy().astype(np.float64)
    yref = oracle.moe(wg, wu, wd, s, E, H, F, xb[tokens], ids_n[tokens],
                      wts_n[tokens].astype(np.float32), weighted_down=weighted_down)
    bound = np.zeros((len(tokens), H))
    for ti, t in enumerate(tokens):
        for j in range(ids_n.shape[1]):
            e = int(ids_n[t, j])
            if e < 0 or e >= E:
                continue
            ge, ue, de = (m[e * s:(e + 1) * s] for m in (wg, wu, wd))
            g = oracle.gemv_f64(ge, F, H, xf[t])[0]
            u = oracle.gemv_f64(ue, F, H, xf[t])[0]
            dg = 2e-3 * oracle.gemv_f64(ge, F, H, np.abs(xf[t]), use_abs=True)[0]
            du = 2e-3 * oracle.gemv_f64(ue, F, H, np.abs(xf[t]), use_abs=True)[0]
            sg = g / (1.0 + np.exp(-np.clip(g, -700.0, 700.0)))
            h = sg * u
            dh = 1.1 * dg * np.abs(u) + np.abs(sg) * du + 1.1 * dg * du + 2.0 ** -15 * np.abs(h)
            awd_h = oracle.gemv_f64(de, H, F, np.abs(h), use_abs=True)[0]
            awd_dh = oracle.gemv_f64(de, H, F, dh, use_abs=True)[0]
            bound[ti] += abs(wts_n[t, j]) * (2e-3 * awd_h + 1.002 * awd_dh)
    return yref, bound


def _check(y, yref, bound, what):
    err = np.abs(y - yref)
    bad = ~(err <= bound + 1e-30)
    assert not bad.any(), f"{what}: {bad.sum()} outside, worst {np.max(err - bound)}"


@pytest.mark.parametrize("E,H,F,T,K", [(8, 256, 256, 1, 1), (8, 512, 512, 3, 2), (16, 1024, 512, 16, 8),
                                       (32, 512, 768, 9, 4)])
@pytest.mark.parametrize("weighted_down", [False, True])
def test_moe_matches_oracle(q4k, E, H, F, T, K, weighted_down):
    c = _make(E, H, F, T, K, seed=E + H + F + T + K)
    y, err = _gpu(q4k, c, flags=int(weighted_down))
    assert err == 0
    tokens = list(range(T))
    yref, bound = _bound(c, c["ids"], c["wts"], tokens, weighted_down)
    _check(y[tokens], yref, bound, f"moe E{E} H{H} F{F} T{T} k{K} wd{int(weighted_down)}")


def test_moe_one_expert_for_all_tokens_spans_slots(q4k):
    # 20 tokens all routed (top-1) to expert 3: more pairs than one work slot holds
    c = _make(6, 512, 256, 20, 1, seed=5)
    ids = torch.full((20, 1), 3, dtype=torch.int32)
    wts = torch.ones((20, 1), dtype=torch.float32)
    y, err = _gpu(q4k, c, ids, wts)
    assert err == 0
    yref, bound = _bound(c, ids, wts, list(range(20)))
    _check(y, yref, bound, "single expert")


@pytest.mark.parametrize("weighted_down", [False, True])
def test_moe_every_slot_width(q4k, weighted_down):
    # expert e (e = 0..7) gets exactly e + 1 pairs: slots of 1 to 8 pairs in one
    # step, so every contraction width of the expert kernel runs (gate/up 1..8
    # columns, down 2..16)
    E, T, K = 8, 12, 3
    c = _make(E, 512, 512, T, K, seed=41)
    order = [e for e in range(E) for _ in range(e + 1)]  # 36 = T * K pairs
    # slot k of token t is pair k * T + t: an expert spans at most 8 < T
    # consecutive pairs, so no token meets one expert twice
    ids = torch.tensor(order, dtype=torch.int32).view(K, T).t().contiguous()
    y, err = _gpu(q4k, c, ids, c["wts"], flags=int(weighted_down))
    assert err == 0
    yref, bound = _bound(c, ids, c["wts"], list(range(T)), weighted_down)
    _check(y, yref, bound, f"slot widths wd{int(weighted_down)}")


def test_moe_duplicate_ids_and_bad_ids(q4k):
    c = _make(8, 512, 256, 4, 3, seed=7)
    ids = c["ids"].clone()
    ids[0, 1] = ids[0, 0]          # the same expert twice for one token
    ids[1, 2] = 8                  # out of range: skipped, flagged
    ids[2, 0] = -5
    y, err = _gpu(q4k, c, ids, c["wts"])
    assert err == 2                # Q4K_DEVERR_BAD_EXPERT
    yref, bound = _bound(c, ids, c["wts"], list(range(4)))
    _check(y, yref, bound, "dup/bad ids")


def test_moe_relabel_invariance_and_determinism(q4k):
    c = _make(8, 512, 256, 5, 2, seed=9)
    y1, _ = _gpu(q4k, c)
    y1b, _ = _gpu(q4k, c)
    assert np.array_equal(y1, y1b)
    perm = np.array([3, 7, 0, 1, 6, 2, 5, 4])   # new slot p holds old expert perm[p]
    inv = torch.from_numpy(np.argsort(perm).astype(np.int32))
    s = c["stride"]

    def permute(w):
        wn = w.numpy()
        return torch.from_numpy(np.concatenate([wn[perm[p] * s:(perm[p] + 1) * s] for p in range(8)]))

    c2 = dict(c, wg=permute(c["wg"]), wu=permute(c["wu"]), wd=permute(c["wd"]))
    y2, _ = _gpu(q4k, c2, inv[c["ids"].long()], c["wts"])
    assert np.array_equal(y1, y2)      # same pairs, same per-column arithmetic


@pytest.mark.parametrize("weighted_down", [False, True])
def test_moe_235b_class_sampled_tokens(q4k, weighted_down):
    # 128 experts, hidden 4096, expert ffn 1536, 16 decode tokens, top-8 Zipf(1.1)
    E, H, F, T, K = 128, 4096, 1536, 16, 8
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=41, device=DEV).reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=42, device=DEV).reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=43, device=DEV).reshape(-1)
    x = synth.bf16_normal((T, H), seed=44)
    ids, wts = synth.zipf_routing(T, E, K, seed=45)
    y = q4k.q4k_moe_gemv_ex(wg, wu, wd, stride, E, H, F, x.to(DEV), ids.to(DEV), wts.to(DEV),
                            flags=int(weighted_down))
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    tokens = [0, 7, 15]
    used = sorted({int(e) for t in tokens for e in ids[t].tolist()})
    # oracle on the experts these tokens use (copied to the host)
    c = dict(wg=wg.cpu(), wu=wu.cpu(), wd=wd.cpu(), stride=stride, E=E, H=H, F=F, x=x)
    yref, bound = _bound(c, ids, wts, tokens, weighted_down)
    _check(y.cpu().numpy().astype(np.float64)[tokens], yref, bound, "235B-class")
    assert len(used) > 1


def _gpu_stages(q4k, c, ids, wts, flags=0):
    """Run with an explicit workspace and read back the per-pair stages."""
    E, H, F = c["E"], c["H"], c["F"]
    T, K = ids.shape
    ws = torch.zeros(q4k.q4k_moe_workspace_size(E, T, K, H, F), dtype=torch.uint8, device=DEV)
    y = q4k.q4k_moe_gemv_ex(c["wg"].to(DEV), c["wu"].to(DEV), c["wd"].to(DEV), c["stride"], E, H,
                            F, c["x"].to(DEV), ids.to(DEV), wts.to(DEV), flags=flags,
                            workspace=ws)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    v = q4k.q4k_moe_workspace_views(E, T, K, H, F)
    P = T * K
    tj = ws[v["tj_pair"]:v["tj_pair"] + 4 * P].view(torch.int32).cpu().numpy()
    st = {}
    for name, width in (("g", F), ("u", F), ("h", F), ("p", H)):
        st[name] = ws[v[name]:v[name] + 4 * P * width].view(torch.float32).view(P, width).cpu().numpy()
    return y.cpu().numpy().astype(np.float64), tj, st


@pytest.mark.parametrize("weighted_down", [False, True])
@pytest.mark.parametrize("sigma", [1.0, 0.01])
@pytest.mark.parametrize("E,H,F,T,K", [(16, 1024, 512, 16, 8), (8, 512, 768, 5, 3)])
def test_moe_stagewise(q4k, E, H, F, T, K, sigma, weighted_down):
    # every stage against the oracle on its own: g and u within the GEMV bound,
    # h = silu(g) u of the GPU's own g and u, the down projection fed the GPU's
    # own h (times the route weight r in the weighted-down order), and y = the
    # sum of the GPU's own down outputs (weighted by r in the plain order).
    # sigma 0.01 keeps |g| small: SiLU's curved region.
    c = _make(E, H, F, T, K, seed=E + H + T + int(1000 * sigma), sigma=sigma)
    ids, wts = c["ids"], c["wts"]
    y, tj, st = _gpu_stages(q4k, c, ids, wts, flags=int(weighted_down))
    s = c["stride"]
    wg, wu, wd = (c[k].numpy() for k in ("wg", "wu", "wd"))
    xb = xbits(c["x"])
    _, (g_ref, u_ref, h_ref) = oracle.moe(wg, wu, wd, s, E, H, F, xb, ids.numpy(), wts.numpy(),
                                           return_stages=True)
    xf = c["x"].to(torch.float64).numpy()
    gmax = 0.0
    for t in range(T):
        yt = np.zeros(H)
        for j in range(K):
            q, e = t * K + j, int(ids[t, j])
            pos = int(tj[q])
            assert pos >= 0
            ge, ue, de = (m[e * s:(e + 1) * s] for m in (wg, wu, wd))
            sg = oracle.gemv_f64(ge, F, H, np.abs(xf[t]), use_abs=True)[0]
            su = oracle.gemv_f64(ue, F, H, np.abs(xf[t]), use_abs=True)[0]
            g, u, h = (st[k][pos].astype(np.float64) for k in ("g", "u", "h"))
            assert np.all(np.abs(g - g_ref[q]) <= 2e-3 * sg), f"g t{t} j{j}"
            assert np.all(np.abs(u - u_ref[q]) <= 2e-3 * su), f"u t{t} j{j}"
            hh = g / (1.0 + np.exp(-np.clip(g, -700, 700))) * u
            assert np.all(np.abs(h - hh) <= 2.0 ** -18 * np.abs(hh) + 1e-30), f"h t{t} j{j}"
            r = float(wts[t, j])
            hd = r * h if weighted_down else h     # r h is rounded once to fp32: 2^-24
            pd = oracle.gemv_f64(de, H, F, hd)[0]
            sd = oracle.gemv_f64(de, H, F, np.abs(hd), use_abs=True)[0]
            p = st["p"][pos].astype(np.float64)
            assert np.all(np.abs(p - pd) <= (2e-3 + 2.0 ** -16 + 2.0 ** -24) * sd), f"down t{t} j{j}"
            yt += p if weighted_down else r * p
            gmax = max(gmax, float(np.abs(g).max()))
        bound = 2.0 ** -20 * sum((1.0 if weighted_down else abs(float(wts[t, j])))
                                 * np.abs(st["p"][int(tj[t * K + j])]) for j in range(K))
        assert np.all(np.abs(y[t] - yt) <= bound + 1e-30), f"combine t{t}"
    if sigma < 0.1:
        assert gmax < 8.0          # the curved region of SiLU is what was tested



def test_moe_graph_replay_matches_eager_and_oracle(q4k):
    # route + persistent expert kernel captured in a CUDA graph and replayed
    # three times (the route kernel clears the work counters on every replay):
    # the output equals the eager call's and stays within the oracle bound
    c = _make(32, 1024, 512, 16, 8, seed=77)
    E, H, F = c["E"], c["H"], c["F"]
    T, K = c["ids"].shape
    wg, wu, wd = (c[k].to(DEV) for k in ("wg", "wu", "wd"))
    x, ids, wts = c["x"].to(DEV), c["ids"].to(DEV), c["wts"].to(DEV)
    ws = torch.empty(q4k.q4k_moe_workspace_size(E, T, K, H, F), dtype=torch.uint8, device=DEV)
    eager = q4k.q4k_moe_gemv(wg, wu, wd, c["stride"], E, H, F, x, ids, wts, workspace=ws).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream(device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        q4k.q4k_moe_gemv(wg, wu, wd, c["stride"], E, H, F, x, ids, wts, out=out, workspace=ws,
                         stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            q4k.q4k_moe_gemv(wg, wu, wd, c["stride"], E, H, F, x, ids, wts, out=out, workspace=ws,
                             stream=s)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    assert torch.equal(out, eager)
    tokens = list(range(T))
    yref, bound = _bound(c, c["ids"], c["wts"], tokens)
    _check(out.cpu().numpy().astype(np.float64), yref, bound, "moe graph replay")
