"""Benchmark of the Q4_K projection path on one GB300.

Default workload (the headline): a 27B-class dense decoder layer at batch 1 --
Q4_K projections QKV 5120->10240, O 8192->5120, gate and up 5120->17408, down
17408->5120 -- repeated over 64 layers of distinct random weights (13.0 GB of
Q4_K weights), all 320 projections back to back on one stream.  One step is one
pass over the 64 layers.  Metric: achieved HBM GB/s (algorithmic bytes: every
weight byte once, plus x and y).  Weights are far larger than L2, so nothing is
served from cache between steps.

Other configurations of the path (decode batch 4/16 on the same layers, the
4096x4096 single GEMV over a rotating pool, the 512-token prefill GEMM and the
routed-MoE decode) are measured in the same run and reported under "configs".

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--skip-extra]
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

HIDDEN = 5120
LAYER_SHAPES = [("qkv", 10240, 5120), ("o", 5120, 8192), ("gate", 17408, 5120),
                ("up", 17408, 5120), ("down", 5120, 17408)]
N_LAYERS = 64
SEED_C1 = 1001
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


@contextlib.contextmanager
def nvtx(name):
    """An NVTX range around one configuration (visible to profilers)."""
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


def q4k_bytes(n, k):
    return n * (k // 256) * 144


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[key] = float(v)
            if "hbm_gbs" in out:
                out["source"] = "measured"
                return out
        except Exception:
            pass
    out = dict(FALLBACK)
    out["source"] = "fallback"
    return out


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ workloads

class Layers:
    """64 layers of distinct Q4_K weights for the five projections, on the GPU."""

    def __init__(self, dev, n_layers=N_LAYERS, seed=SEED_C1):
        self.mats = []
        for layer in range(n_layers):
            for pi, (name, n, k) in enumerate(LAYER_SHAPES):
                w = synth.q4k_weight(n, k, seed=synth.derive_seed(seed, "w", layer, pi),
                                     quants="normal", device=dev)
                self.mats.append((name, n, k, w))

    def algorithmic_bytes(self, batch):
        return sum(q4k_bytes(n, k) + batch * k * 2 + batch * n * 4 for _, n, k, _ in self.mats)


def make_inputs(layers, batch, dev, seed):
    xs, ys = [], []
    for i, (_, n, k, _) in enumerate(layers.mats):
        xs.append(synth.bf16_normal((batch, k), seed=synth.derive_seed(seed, "x", batch, i),
                                    device=dev))
        ys.append(torch.empty((batch, n), dtype=torch.float32, device=dev))
    return xs, ys


def time_graph(fn, steps, warmup, stream):
    """Capture fn into a CUDA graph; time `steps` replays with CUDA events."""
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    per = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            g.replay()
            e.record(stream)
            per.append((s, e))
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    per_ms = [s.elapsed_time(e) for s, e in per]
    return total_ms / steps, per_ms, g


def bench_decode(q4k, layers, batch, steps, warmup, dev, stream, sampler=None, overlap=True):
    """One pass = the 320 projections as one q4k_gemv_seq call (at batch 1 one
    persistent launch that streams all 13 GB of weights back to back; at batch
    4/16 one launch per projection), captured in a CUDA graph.  With `overlap`
    a launch may start streaming its (static) weights while the previous one
    finishes (Q4K_FLAG_OVERLAP_WEIGHTS).  After timing, sampled rows of the last
    replay are checked against the oracle."""
    xs, ys = make_inputs(layers, batch, dev, seed=SEED_C1 + batch)
    flags = q4k.Q4K_FLAG_OVERLAP_WEIGHTS if overlap else 0
    ops = q4k.gemv_ops([(w, n, k, x, y) for (name, n, k, w), x, y in zip(layers.mats, xs, ys)])

    def step():
        q4k.q4k_gemv_seq(ops, batch, flags, stream=stream)

    if sampler is not None:
        with sampler:
            ms, per, g = time_graph(step, steps, warmup, stream)
    else:
        ms, per, g = time_graph(step, steps, warmup, stream)
    del g
    nbytes = layers.algorithmic_bytes(batch)
    launches = -(-len(layers.mats) // q4k.Q4K_SEQ_MATRICES_PER_LAUNCH)
    return {"ms_per_step": ms, "ms_min": min(per), "gbs": nbytes / (ms * 1e-3) / 1e9,
            "bytes_per_step": nbytes, "launches_per_step": launches,
            "verified": verify_decode(layers, xs, ys)}


def verify_decode(layers, xs, ys, n_ops=5, rows=24, tol=2e-3):
    """Sampled rows of sampled projections against the oracle, within the
    fp32-path bound 2e-3 sum |w||x|; returns the worst error / bound ratio
    (raises if any element is outside)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(2027)
    worst = 0.0
    picks = rng.choice(len(layers.mats), min(n_ops, len(layers.mats)), replace=False)
    for i in sorted(int(p) for p in picks):
        name, n, k, w = layers.mats[i]
        ri = np.unique(np.concatenate([rng.choice(n, rows, replace=False), [0, n - 1]]))
        rt = torch.from_numpy(ri).to(w.device)
        xb = xs[i].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        yref, sref = oracle.gemv(w[rt].cpu().numpy(), len(ri), k, xb)
        got = ys[i][:, rt].cpu().numpy().astype(np.float64)
        err = np.abs(got - yref)
        if not np.all(err <= tol * sref):
            raise AssertionError(f"bench result check failed: op {i} ({name})")
        worst = max(worst, float(np.max(err / (tol * sref))))
    return round(worst, 4)


def bench_decode_e2e(q4k, layers, batch, steps, warmup, dev, stream, groups=4):
    """Same pass through the public API with host buffers, launched eagerly (no
    graph).  Every step copies all projections' x from pinned host memory to the
    device and reads all y back; the layers run in `groups` groups, each with one
    q4k_gemv_seq call (programmatic dependent launch between its projections).
    The copies run on a second stream, ordered by events: group g starts once
    its x has landed, and its y is copied back while group g+1 computes."""
    kx = [k for _, _, k, _ in layers.mats]
    ny = [n for _, n, _, _ in layers.mats]
    host_x = torch.empty(batch * sum(kx), dtype=torch.bfloat16).pin_memory()
    host_y = torch.empty(batch * sum(ny), dtype=torch.float32).pin_memory()
    off = 0
    for i, k in enumerate(kx):
        x = synth.bf16_normal((batch, k), seed=synth.derive_seed(SEED_C1, "xe", i))
        host_x[off:off + batch * k] = x.reshape(-1)
        off += batch * k
    dev_x = torch.empty_like(host_x, device=dev)
    dev_y = torch.empty_like(host_y, device=dev)
    nmat = len(layers.mats)
    bounds = [nmat * g // groups for g in range(groups + 1)]
    ops, xr, yr = [], [], []
    ox = oy = 0
    for g in range(groups):
        tup = []
        x0, y0 = ox, oy
        for (name, n, k, w) in layers.mats[bounds[g]:bounds[g + 1]]:
            x = dev_x[ox:ox + batch * k].view(batch, k)
            y = dev_y[oy:oy + batch * n].view(batch, n)
            tup.append((w, n, k, x, y))
            ox += batch * k
            oy += batch * n
        ops.append(q4k.gemv_ops(tup))
        xr.append((x0, ox))
        yr.append((y0, oy))
    h2d = host_x.numel() * 2
    d2h = host_y.numel() * 4
    copy = torch.cuda.Stream(device=dev)
    landed = [torch.cuda.Event() for _ in range(groups)]
    done = [torch.cuda.Event() for _ in range(groups)]

    def step():
        with torch.cuda.stream(copy):
            for g in range(groups):
                a, b = xr[g]
                dev_x[a:b].copy_(host_x[a:b], non_blocking=True)
                landed[g].record(copy)
        for g in range(groups):
            stream.wait_event(landed[g])
            q4k.q4k_gemv_seq(ops[g], batch, q4k.Q4K_FLAG_OVERLAP_WEIGHTS, stream=stream)
            done[g].record(stream)
            copy.wait_event(done[g])
            with torch.cuda.stream(copy):
                a, b = yr[g]
                host_y[a:b].copy_(dev_y[a:b], non_blocking=True)

    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    copy.synchronize()
    stream.synchronize()
    sec = (time.perf_counter() - t0) / steps
    nbytes = layers.algorithmic_bytes(batch)
    return {"value": round(nbytes / sec / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 4)}


def bench_c0_pool(q4k, steps, warmup, dev, stream):
    """4096x4096 GEMV at batch 1 over a pool of distinct matrices (pool >> L2,
    so every matrix streams its weights from HBM), run as one q4k_gemv_seq call;
    also the time of one q4k_gemv call on one matrix (latency, L2-cold)."""
    n = k = 4096
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool = max(32, int(4 * l2 // q4k_bytes(n, k)) + 1)
    ws = [synth.q4k_weight(n, k, seed=synth.derive_seed(1000, "w", i), device=dev)
          for i in range(pool)]
    x = synth.bf16_normal((1, k), seed=1000, device=dev)
    ys = [torch.empty((1, n), device=dev) for _ in range(pool)]

    ops = q4k.gemv_ops([(w, n, k, x, y) for w, y in zip(ws, ys)])

    def step():  # the pool as one sequence: one persistent launch streams every matrix
        q4k.q4k_gemv_seq(ops, 1, q4k.Q4K_FLAG_OVERLAP_WEIGHTS, stream=stream)

    ms, per, g = time_graph(step, steps, warmup, stream)
    del g
    nbytes = pool * (q4k_bytes(n, k) + k * 2 + n * 4)

    def single():  # one matrix per call, a different one each call (graph of the pool)
        for w, y in zip(ws, ys):
            q4k.q4k_gemv_ex(w, n, k, x, q4k.Q4K_FLAG_OVERLAP_WEIGHTS, out=y, stream=stream)

    ms1, _, g1 = time_graph(single, max(3, steps // 2), 2, stream)
    del g1
    return {"pool": pool, "us_per_gemv": ms * 1e3 / pool, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "us_per_single_call": ms1 * 1e3 / pool}


def bench_glu(q4k, dev, stream, steps, warmup, n_layers=N_LAYERS, batch=1):
    """Fused gate/up (F1) on the 27B-class FFN: 64 layers of a 5120 -> 17408
    gate/up pair (6.4 GB), each as one fused op of one q4k_gemv_seq call,
    against the same matrices as two plain projections per layer."""
    n, k = 17408, 5120
    wg = [synth.q4k_weight(n, k, seed=synth.derive_seed(1006, "g", i), quants="normal", device=dev)
          for i in range(n_layers)]
    wu = [synth.q4k_weight(n, k, seed=synth.derive_seed(1006, "u", i), quants="normal", device=dev)
          for i in range(n_layers)]
    x = [synth.bf16_normal((batch, k), seed=synth.derive_seed(1006, "x", i), sigma=0.02, device=dev)
         for i in range(n_layers)]
    h = [torch.empty((batch, n), device=dev) for _ in range(n_layers)]
    g2 = [torch.empty((batch, n), device=dev) for _ in range(2 * n_layers)]
    fused = q4k.gemv_ops([(wg[i], n, k, x[i], h[i], wu[i]) for i in range(n_layers)])
    plain = q4k.gemv_ops([(m, n, k, x[i // 2], g2[i]) for i, m in
                          enumerate(v for pair in zip(wg, wu) for v in pair)])
    flags = q4k.Q4K_FLAG_OVERLAP_WEIGHTS
    ms_f, _, gf = time_graph(lambda: q4k.q4k_gemv_seq(fused, batch, flags, stream=stream),
                             steps, warmup, stream)
    del gf
    ms_p, _, gp = time_graph(lambda: q4k.q4k_gemv_seq(plain, batch, flags, stream=stream),
                             steps, warmup, stream)
    del gp
    nbytes = n_layers * (2 * q4k_bytes(n, k) + batch * (k * 2 + n * 4))
    return {"batch": batch, "ms_fused": round(ms_f, 4), "gbs_fused": round(nbytes / (ms_f * 1e-3) / 1e9, 1),
            "frac_of_8tbs_fused": round(nbytes / (ms_f * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "ms_two_projections": round(ms_p, 4),
            "speedup_vs_two_projections": round(ms_p / ms_f, 3)}


def bench_dequant(q4k, dev, stream, reps=20):
    """q4k_dequant of the 17408 x 5120 gate matrix (50 MB of Q4_K) to fp32 and
    bf16: GB/s over the bytes read and written."""
    n, k = 17408, 5120
    w = synth.q4k_weight(n, k, seed=1007, quants="normal", device=dev)
    out = {}
    for name, dt, ob in (("fp32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        o = torch.empty((n, k), dtype=dt, device=dev)
        ms, _, g = time_graph(lambda: q4k.q4k_dequant(w, n, k, out=o, stream=stream), reps, 3, stream)
        del g
        nbytes = q4k_bytes(n, k) + n * k * ob
        out[name] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return out


# ------------------------------------------------------------------ CPU baseline

def cpu_baseline(layers, budget_s=12.0):
    """The oracle as it stands, timed on the host cores, on a bounded sample of
    the headline workload: the same weights and activations (copied to the
    host), whole projections in pass order until about budget_s of oracle time
    (copies are not timed)."""
    import oracle
    oracle.build()
    elapsed, done_bytes, nproj = 0.0, 0, 0
    for i, (name, n, k, w) in enumerate(layers.mats):
        if elapsed >= budget_s:
            break
        wh = w.cpu().numpy()
        x = synth.bf16_normal((1, k), seed=synth.derive_seed(SEED_C1 + 1, "x", 1, i))
        xb = x.view(torch.int16).numpy().view(np.uint16)
        t = time.perf_counter()
        oracle.gemv(wh, n, k, xb)
        elapsed += time.perf_counter() - t
        done_bytes += q4k_bytes(n, k) + k * 2 + n * 4
        nproj += 1
    return {"value": round(done_bytes / elapsed / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle GEMV, batch 1, the first {nproj} projections of the pass "
                      f"({done_bytes / 1e9:.2f} GB of Q4_K weights), {elapsed:.1f} s of oracle time"}


def cpu_table(budget_s: float = 6.0) -> dict:
    """The oracle on the host cores, single-threaded and with every core, for
    each configuration, on bounded samples (whole projections or rows of them,
    stated per entry); no GPU involved.  Units: GB/s of Q4_K weights streamed
    (GEMV, MoE) or GFLOP/s (prefill GEMM)."""
    import oracle
    oracle.build()
    ncores = oracle.num_threads()
    out = {"cores_all": ncores}

    def timed(fn, min_s=0.5):
        reps, t0 = 0, time.perf_counter()
        while True:
            fn()
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_s or reps >= 50:
                return el / reps

    def both(name, fn, amount, unit, sample):
        res = {"unit": unit, "sample": sample}
        for label, th in (("1_core", 1), ("all_cores", ncores)):
            oracle.set_num_threads(th)
            sec = timed(fn)
            res[label] = round(amount / sec / 1e9, 4)
        oracle.set_num_threads(ncores)
        out[name] = res

    def xbits(x):
        return x.view(torch.int16).numpy().view(np.uint16)

    w0 = synth.q4k_weight(1024, 4096, seed=synth.derive_seed(1000, "cpu")).numpy()
    x0 = xbits(synth.bf16_normal((1, 4096), seed=1000))
    both("c0_gemv_4096_b1", lambda: oracle.gemv(w0, 1024, 4096, x0), 1024 * 16 * 144, "GB/s",
         "1024 of the 4096 rows of a 4096 x 4096 matrix")
    rows = 512
    lay = [(n, k, synth.q4k_weight(rows, k, seed=synth.derive_seed(SEED_C1, "cpu", i), quants="normal").numpy())
           for i, (_, n, k) in enumerate(LAYER_SHAPES)]
    for b in (1, 4, 16):
        xs = [xbits(synth.bf16_normal((b, k), seed=synth.derive_seed(SEED_C1, "cpux", b, i)))
              for i, (_, k, _) in enumerate(lay)]
        nbytes = sum(q4k_bytes(rows, k) for _, k, _ in lay)
        both(f"c{1 if b == 1 else 2}_27b_layer_b{b}",
             lambda xs=xs: [oracle.gemv(w, rows, k, x) for (_, k, w), x in zip(lay, xs)], nbytes,
             "GB/s", f"the first {rows} rows of each of the 5 projections of one layer, batch {b}")
    m = 16
    wg = synth.q4k_weight(256, 5120, seed=synth.derive_seed(1003, "cpu"), quants="normal").numpy()
    xg = xbits(synth.bf16_normal((m, 5120), seed=1003, sigma=0.5))
    both("c3_prefill_gate", lambda: oracle.gemv(wg, 256, 5120, xg), 2.0 * m * 256 * 5120, "GFLOP/s",
         f"{m} tokens x 256 rows of the 512-token gate projection")
    E, H, F, T, K = 16, 4096, 1536, 4, 8
    stride = F * (H // 256) * 144
    mg = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1004, "cg")).numpy().reshape(-1)
    mu = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1004, "cu")).numpy().reshape(-1)
    md = synth.q4k_weight(E * H, F, seed=synth.derive_seed(1004, "cd")).numpy().reshape(-1)
    mx = xbits(synth.bf16_normal((T, H), seed=1004))
    ids, wts = synth.zipf_routing(T, E, K, seed=1005)
    both("c4_moe_235b", lambda: oracle.moe(mg, mu, md, stride, E, H, F, mx, ids.numpy(), wts.numpy()),
         T * K * 3 * q4k_bytes(F, H), "GB/s",
         f"{T} tokens, top-{K} of {E} experts (128-expert shapes), bytes counted per (token, slot)")
    return out


def bench_prefill(q4k, dev, stream, reps=20):
    """512-token prefill: gate (5120 -> 17408) and down (17408 -> 5120), each
    timed on its own (events around `reps` launches; weights 50 MB each, X
    5-18 MB, so L2 holds them across launches -- the GEMM is tensor-bound)."""
    out = {}
    m = 512
    for name, n, k in (("gate", 17408, 5120), ("down", 5120, 17408)):
        w = synth.q4k_weight(n, k, seed=synth.derive_seed(1003, "w", name), quants="normal", device=dev)
        x = synth.bf16_normal((m, k), seed=synth.derive_seed(1003, "x", name), sigma=0.5, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                q4k.q4k_gemm(w, n, k, x, out=y, stream=stream)
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for _ in range(reps):
                q4k.q4k_gemm(w, n, k, x, out=y, stream=stream)
            e.record(stream)
        torch.cuda.synchronize()
        us = s.elapsed_time(e) * 1e3 / reps
        flop = 2.0 * m * n * k
        out[name] = {"us": round(us, 2), "tflops": round(flop / us / 1e6, 1)}
        # the same projection with the fused RMSNorm prologue (rinv kernel + GEMM
        # with gamma in the dequant and rinv in the epilogue)
        gamma = torch.rand(k, generator=torch.Generator().manual_seed(synth.derive_seed(1003, "g", name)))
        gamma = (gamma + 0.5).to(dev)
        rinv = torch.empty(m, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                q4k.q4k_gemm_rmsnorm(w, n, k, x, gamma, 1e-6, out=y, rinv=rinv, stream=stream)
            s.record(stream)
            for _ in range(reps):
                q4k.q4k_gemm_rmsnorm(w, n, k, x, gamma, 1e-6, out=y, rinv=rinv, stream=stream)
            e.record(stream)
        torch.cuda.synchronize()
        us_n = s.elapsed_time(e) * 1e3 / reps
        out[name + "_rmsnorm"] = {"us": round(us_n, 2), "tflops": round(flop / us_n / 1e6, 1),
                                  "vs_plain": round(us / us_n, 3)}
    return out


def bench_moe(q4k, dev, stream, reps=20):
    """235B-A22B-class routed MoE decode: 128 experts, hidden 4096, expert ffn
    1536, 16 tokens, top-8 Zipf(1.1).  Touched bytes = the distinct experts'
    gate/up/down weights + x + y; the 1.36 GB expert pool exceeds L2."""
    E, H, F, T, K = 128, 4096, 1536, 16, 8
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1004, "g"), device=dev).reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1004, "u"), device=dev).reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=synth.derive_seed(1004, "d"), device=dev).reshape(-1)
    x = synth.bf16_normal((T, H), seed=synth.derive_seed(1004, "x"), device=dev)
    ids, wts = synth.zipf_routing(T, E, K, seed=1005)
    distinct = len(set(ids.reshape(-1).tolist()))
    ids_d, wts_d = ids.to(dev), wts.to(dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = torch.empty(q4k.q4k_moe_workspace_size(E, T, K, H, F), dtype=torch.uint8, device=dev)

    def step():
        q4k.q4k_moe_gemv(wg, wu, wd, stride, E, H, F, x, ids_d, wts_d, out=y, workspace=ws,
                         stream=stream)

    ms, per, g = time_graph(step, reps, 3, stream)
    del g
    nbytes = distinct * 3 * q4k_bytes(F, H) + T * H * 2 + T * H * 4
    return {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_8tbs": round(nbytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "distinct_experts": distinct, "bytes": nbytes}


def bench_moe_prefill(q4k, dev, stream, reps=10):
    """235B-A22B-class routed MoE prefill: 128 experts, hidden 4096, expert ffn
    1536, 512 tokens, top-8 Zipf(1.1) (4096 pairs): route, gather, grouped
    tcgen05 GEMMs for gate/up/down, SiLU, weighted sum.  Useful flop = 2 x pairs
    x 3 x ffn x hidden; touched bytes = the distinct experts' weights + x + y."""
    E, H, F, T, K = 128, 4096, 1536, 512, 8
    stride = F * (H // 256) * 144
    wg = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1006, "g"), device=dev).reshape(-1)
    wu = synth.q4k_weight(E * F, H, seed=synth.derive_seed(1006, "u"), device=dev).reshape(-1)
    wd = synth.q4k_weight(E * H, F, seed=synth.derive_seed(1006, "d"), device=dev).reshape(-1)
    x = synth.bf16_normal((T, H), seed=synth.derive_seed(1006, "x"), device=dev)
    ids, wts = synth.zipf_routing(T, E, K, seed=1007)
    distinct = len(set(ids.reshape(-1).tolist()))
    ids_d, wts_d = ids.to(dev), wts.to(dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = torch.empty(q4k.q4k_moe_prefill_workspace_size(E, T, K, H, F), dtype=torch.uint8,
                     device=dev)

    def step():
        q4k.q4k_moe_prefill(wg, wu, wd, stride, E, H, F, x, ids_d, wts_d, out=y, workspace=ws,
                            stream=stream)

    ms, per, g = time_graph(step, reps, 3, stream)
    del g
    flop = 2.0 * T * K * 3 * F * H
    nbytes = distinct * 3 * q4k_bytes(F, H) + T * H * 2 + T * H * 4
    return {"us": round(ms * 1e3, 2), "tflops": round(flop / (ms * 1e-3) / 1e12, 1),
            "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "distinct_experts": distinct,
            "pairs": T * K}


def bench_kquant(q4k, dev, stream, reps=10):
    """Batch-1 decode projection in the other k-quant formats on the 27B-class
    down shape (5120 x 17408): a pool of 8 matrices per format (more than L2
    for every format) multiplied in turn, as one q4k_kq_gemv call each and as
    one q4k_kq_gemv_seq call over the pool, and at batch 4 as one call each;
    bytes = weights + x + y."""
    n, k, pool = 5120, 17408, 8
    out = {}
    names = {2: "q2_K", 3: "q3_K", 5: "Q5_K", 6: "Q6_K"}
    for fmt, name in names.items():
        ws = [synth.kq_weight(fmt, n, k, seed=synth.derive_seed(1008, name, i), device=dev)
              for i in range(pool)]
        x = synth.bf16_normal((1, k), seed=synth.derive_seed(1008, "x"), device=dev)
        ys = [torch.empty((1, n), dtype=torch.float32, device=dev) for _ in range(pool)]

        def step():
            for w, y in zip(ws, ys):
                q4k.q4k_kq_gemv(fmt, w, n, k, x, out=y, stream=stream)

        ms, per, g = time_graph(step, reps, 3, stream)
        del g
        ops = q4k.gemv_ops([(w, n, k, x, y) for w, y in zip(ws, ys)])
        ms_seq, _, g = time_graph(lambda: q4k.q4k_kq_gemv_seq(fmt, ops, 1, q4k.Q4K_FLAG_OVERLAP_WEIGHTS,
                                                                stream=stream), reps, 3, stream)
        del g
        nbytes = pool * (ws[0].numel() + 2 * k + 4 * n)
        gbs = nbytes / (ms * 1e-3) / 1e9
        # batch 4: Q5_K on the tensor cores, the others on the fp32 kernel
        x4 = synth.bf16_normal((4, k), seed=synth.derive_seed(1008, "x4"), device=dev)
        y4 = [torch.empty((4, n), dtype=torch.float32, device=dev) for _ in range(pool)]
        ms4, _, g = time_graph(lambda: [q4k.q4k_kq_gemv(fmt, w, n, k, x4, out=y, stream=stream)
                                        for w, y in zip(ws, y4)], reps, 3, stream)
        del g
        nbytes4 = pool * (ws[0].numel() + 4 * (2 * k + 4 * n))
        out[name] = {"us_per_gemv": round(ms * 1e3 / pool, 2), "gbs": round(gbs, 1),
                     "gbs_b4": round(nbytes4 / (ms4 * 1e-3) / 1e9, 1),
                     "us_per_gemv_seq": round(ms_seq * 1e3 / pool, 2),
                     "gbs_seq": round(nbytes / (ms_seq * 1e-3) / 1e9, 1),
                     "bytes_per_weight": round(ws[0].numel() / (n * k), 4)}
        del ws
        torch.cuda.empty_cache()
    return out


KERNEL_SOURCES = ("q4k_stream.cu", "q4k_device.cuh", "q4k_internal.h")


def kernel_fingerprint(read=None) -> str:
    """sha256 (16 hex digits) of the batch-1 stream kernel's sources with comments and
    whitespace removed: it changes when the compiled kernel can, not when a
    comment does.  `read(name)` returns a source's text (default: the tree)."""
    import hashlib
    import re
    if read is None:
        base = os.path.join(ROOT, "bit_block_quantized_q4_gb300", "csrc")
        read = lambda name: open(os.path.join(base, name)).read()  # noqa: E731
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        text = re.sub(r"/\*.*?\*/", " ", read(name), flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(pass_bytes: float):
    """DRAM traffic of one launch of the batch-1 stream kernel over the decode
    pass, from the committed ncu summary (profiles/gemv_stream_b1_27b_layer.md):
    the captured launch is one 27B-class layer (the full 64-layer pass is too
    large to capture), so its dram bytes are scaled to the pass by algorithmic
    bytes.  None when the kernel's sources have changed since the capture."""
    path = os.path.join(ROOT, "profiles", "gemv_stream_b1_27b_layer.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_fingerprint_16") != kernel_fingerprint():
        return None
    try:
        per_launch = float(vals["dram_bytes_per_launch"])
        captured = float(vals["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None
    return round(per_launch * pass_bytes / captured)


# ------------------------------------------------------------------ main

def run_case(case):
    """One small instance of a kernel, for ncu captures (no timing): one 27B-class
    layer of batch-1 projections (203 MB of weights) or two layers of batch-4
    and batch-16 projections (two layers are enough 64-row tiles for the
    persistent batch-16 launch), the 512-token gate and
    down prefill GEMMs (plain or with the RMSNorm prologue), one routed-MoE decode
    or prefill step, or one batch-1 projection in each other k-quant format."""
    import bit_block_quantized_q4_gb300 as q4k
    from bit_block_quantized_q4_gb300 import build as qb
    qb.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if case in ("gemv_layer", "gemv_layer_batched"):
        # one (batched: two) layer's projections as one q4k_gemv_seq call (at
        # batch 1 one launch of the stream kernel over 203 MB of weights)
        layers = Layers(dev, n_layers=1 if case == "gemv_layer" else 2)
        for batch in ((1,) if case == "gemv_layer" else (4, 16)):
            xs, ys = make_inputs(layers, batch, dev, seed=SEED_C1 + batch)
            ops = q4k.gemv_ops([(w, n, k, x, y) for (name, n, k, w), x, y in zip(layers.mats, xs, ys)])
            torch.cuda.synchronize()
            q4k.q4k_gemv_seq(ops, batch)
    elif case in ("gemm_prefill", "gemm_prefill_rmsnorm"):
        m = 512
        for name, n, k in (("gate", 17408, 5120), ("down", 5120, 17408)):
            w = synth.q4k_weight(n, k, seed=synth.derive_seed(1003, "w", name), quants="normal",
                                 device=dev)
            x = synth.bf16_normal((m, k), seed=synth.derive_seed(1003, "x", name), sigma=0.5,
                                  device=dev)
            torch.cuda.synchronize()
            if case == "gemm_prefill":
                q4k.q4k_gemm(w, n, k, x)
            else:
                gamma = torch.full((k,), 1.25, dtype=torch.float32, device=dev)
                q4k.q4k_gemm_rmsnorm(w, n, k, x, gamma, 1e-6)
    elif case == "kquant":
        for fmt in (2, 3, 5, 6):  # one batch-1 projection per format, 27B down shape
            n, k = 5120, 17408
            w = synth.kq_weight(fmt, n, k, seed=synth.derive_seed(1008, "case", fmt), device=dev)
            x = synth.bf16_normal((1, k), seed=synth.derive_seed(1008, "x"), device=dev)
            torch.cuda.synchronize()
            q4k.q4k_kq_gemv(fmt, w, n, k, x)
    elif case == "moe_prefill":
        bench_moe_prefill(q4k, dev, torch.cuda.Stream(device=dev), reps=1)
    else:
        bench_moe(q4k, dev, torch.cuda.Stream(device=dev), reps=1)
    torch.cuda.synchronize()
    assert q4k.q4k_get_device_error() == 0
    print(f"case {case} ok")


def max_over_ranks(value: float, world: int) -> float:
    """The largest of the ranks' values (every rank gets it); the value itself
    when there is one rank.  Works on the gloo (CPU tensor) and nccl (device
    tensor) backends."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_gbs(bytes_per_rank_step: float, ms_max: float, world: int) -> float:
    """Whole-job GB/s of `world` replicas that each move `bytes_per_rank_step`
    per step, timed by the slowest rank."""
    return bytes_per_rank_step * world / (ms_max * 1e-3) / 1e9


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, on the host cores, on a
    bounded sample of the headline workload per step."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    per_step = []
    nbytes = 0
    samples = []
    # 1024 rows of each projection (23.6 MB of Q4_K per step): enough rows for
    # the oracle's threads to stay busy, a few ms per step on the host cores.
    for pi, (name, n, k) in enumerate(LAYER_SHAPES):
        nrows = 1024
        w = synth.q4k_weight(nrows, k, seed=synth.derive_seed(SEED_C1, "w", 0, pi),
                             quants="normal").numpy()
        x = synth.bf16_normal((1, k), seed=synth.derive_seed(SEED_C1, "x", 1, pi))
        samples.append((w, nrows, k, x.view(torch.int16).numpy().view(np.uint16)))
        nbytes += q4k_bytes(nrows, k) + k * 2 + nrows * 4
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        for w, nrows, k, xb in samples:
            oracle.gemv(w, nrows, k, xb)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            per_step.append(dt)
    sec = sum(per_step) / len(per_step)
    value = nbytes / sec / 1e9
    line = {"metric": "Q4_K GEMV achieved HBM GB/s (27B-class dense layer, batch 1)",
            "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "27b_dense_layer_b1 (oracle sample: first 1024 rows of each "
                                   "projection of layer 0 per step)", "batch": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "first 1024 rows of each of the 5 projections of layer 0"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-extra", action="store_true", help="headline workload only")
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--cpu-table", action="store_true",
                    help="time the oracle on the host cores for every configuration, then exit")
    ap.add_argument("--case", default=None, choices=["gemv_layer", "gemv_layer_batched", "gemm_prefill", "gemm_prefill_rmsnorm", "moe",
                             "moe_prefill", "kquant"],
                    help="run one small instance of a kernel for a profiler, then exit")
    args = ap.parse_args()
    if args.cpu_table:
        print(json.dumps(cpu_table()), flush=True)
        return
    if args.case:
        run_case(args.case)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import bit_block_quantized_q4_gb300 as q4k
    from bit_block_quantized_q4_gb300 import build as qb
    if rank == 0:
        qb.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)

    layers = Layers(dev, n_layers=args.layers)
    sampler = ClockSampler(local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with nvtx("decode_b1 pass (timed)"):
        head = bench_decode(q4k, layers, 1, args.steps, args.warmup, dev, stream, sampler)
    ms = max_over_ranks(head["ms_per_step"], world)
    assert q4k.q4k_get_device_error(stream) == 0
    pk = peaks()
    nbytes = head["bytes_per_step"]
    achieved = nbytes / (ms * 1e-3) / 1e9  # per GPU, by the slowest rank
    total_value = replicas_gbs(nbytes, ms, world)
    launches = head["launches_per_step"]

    # one launch per step: its CUDA-event duration is the kernel's own
    kernel_ms = head["ms_per_step"] / head["launches_per_step"]
    with nvtx("decode_b1 pass e2e"):
        e2e = bench_decode_e2e(q4k, layers, 1, max(3, args.steps // 2), 2, dev, stream)
    e2e["ms_per_step"] = round(max_over_ranks(e2e["ms_per_step"], world), 4)
    e2e["value"] = round(replicas_gbs(layers.algorithmic_bytes(1), e2e["ms_per_step"], world), 2)

    cpu = cpu_baseline(layers) if rank == 0 else None
    extra = {}
    with nvtx("decode_b1 pass, plain launches"):
        r = bench_decode(q4k, layers, 1, max(5, args.steps // 2), 3, dev, stream, overlap=False)
    extra["decode_b1_no_overlap"] = {"gbs": round(r["gbs"], 1),
                                     "frac_of_8tbs": round(r["gbs"] / NOMINAL_HBM_GBS, 4),
                                     "ms_per_step": round(r["ms_per_step"], 4)}
    if not args.skip_extra:
        for b in (4, 16):
            with nvtx(f"decode_b{b} pass"):
                r = bench_decode(q4k, layers, b, max(5, args.steps // 2), 3, dev, stream)
            extra[f"decode_b{b}"] = {"gbs": round(r["gbs"], 1),
                                     "frac_of_8tbs": round(r["gbs"] / NOMINAL_HBM_GBS, 4),
                                     "ms_per_step": round(r["ms_per_step"], 4),
                                     "verified_worst_err_over_bound": r["verified"]}
        del layers
        torch.cuda.empty_cache()
        with nvtx("gemv 4096x4096 pool"):
            r = bench_c0_pool(q4k, max(5, args.steps // 2), 3, dev, stream)
        extra["gemv_4096_b1_pool"] = {"gbs": round(r["gbs"], 1),
                                      "frac_of_8tbs": round(r["gbs"] / NOMINAL_HBM_GBS, 4),
                                      "us_per_gemv": round(r["us_per_gemv"], 3), "pool": r["pool"],
                                      "us_per_single_call": round(r["us_per_single_call"], 3)}
        torch.cuda.empty_cache()
        with nvtx("fused gate/up"):
            extra["glu_27b_gate_up_b1"] = bench_glu(q4k, dev, stream, max(5, args.steps // 2), 3)
        torch.cuda.empty_cache()
        with nvtx("dequant"):
            extra["dequant_17408x5120"] = bench_dequant(q4k, dev, stream)
        torch.cuda.empty_cache()
        if world == 1:
            # the prefill GEMM's cluster multicast of X is for one-GPU runs only:
            # replica runs on several GPUs leave it out
            with nvtx("prefill 512"):
                pf = bench_prefill(q4k, dev, stream)
            for nm, v in pf.items():
                v["frac_of_measured_bf16"] = round(v["tflops"] / pk["bf16_tflops"], 4)
                v["frac_of_sustained_bf16"] = round(v["tflops"] / pk["bf16_tflops_sustained"], 4)
                v["l2"] = "warm: the same 50 MB W and X relaunched back to back"
            extra["prefill_512"] = pf
            torch.cuda.empty_cache()
        with nvtx("moe 235b t16"):
            extra["moe_235b_a22b_t16"] = bench_moe(q4k, dev, stream)
        torch.cuda.empty_cache()
        with nvtx("k-quant gemv"):
            kq = bench_kquant(q4k, dev, stream)
        for v in kq.values():
            v["frac_of_measured_hbm"] = round(v["gbs"] / pk["hbm_gbs"], 4)
            v["frac_of_measured_hbm_seq"] = round(v["gbs_seq"] / pk["hbm_gbs"], 4)
        extra["kquant_gemv_b1_down_5120x17408"] = kq
        torch.cuda.empty_cache()
        if world == 1:
            with nvtx("moe prefill 235b t512"):
                mp = bench_moe_prefill(q4k, dev, stream)
            mp["frac_of_measured_bf16"] = round(mp["tflops"] / pk["bf16_tflops"], 4)
            mp["frac_of_measured_hbm"] = round(mp["gbs"] / pk["hbm_gbs"], 4)
            extra["moe_prefill_235b_a22b_t512"] = mp
    clocks = sampler.summary()

    if rank == 0:
        line = {
            "metric": "Q4_K GEMV achieved HBM GB/s (27B-class dense layer, batch 1)",
            "value": round(total_value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Q4_K fields; x ~ N(0,1) bf16)",
            "config": {"workload": "27b_dense_layer_b1: 64 layers x {qkv 5120->10240, o 8192->5120, "
                                   "gate/up 5120->17408, down 17408->5120}, batch 1",
                       "batch": 1, "layers": args.layers, "weights_bytes": sum(
                           q4k_bytes(n, k) for _, n, k in LAYER_SHAPES) * args.layers,
                       "l2": "weights (13 GB) far exceed L2; no flush needed",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / launches / (kernel_ms * 1e-3) / 1e9, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(nbytes / launches / (kernel_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                         "traffic": profiled_traffic(nbytes / launches), "peak_source": pk["source"],
                         "algorithmic_bytes_per_launch": round(nbytes / launches),
                         "kernel": "gemv_stream_kernel (q4k_gemv_seq, batch 1: the 320 projections "
                                   "as %d persistent launches of %d)" % (launches, -(-320 // launches)),
                         "note": "CUDA events around each graph replay of the pass's launches; "
                                 "peak = measured copy bandwidth (read + write)"},
            "verified_worst_err_over_bound": head["verified"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "configs": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
