// q4k_moe.cu -- routed mixture-of-experts FFN for decode tokens with Q4_K
// experts ("Layer Package Repository Spec", section "Policy Resolution": a
// routed-FFN decode layer is the routed gate/up/down expert matmuls (96% of its
// time), a fused SwiGLU, and the route-weighted sum).
//
// Two launches on the caller's stream:
//   1. route    one CTA groups the T*k (token, slot) pairs by expert (counting
//               sort; experts ordered by id, at most 8 pairs per work slot, so a
//               heavily used expert spans several slots), validates ids (an id
//               out of range is skipped and flagged in the device error word)
//               and clears the work counters of launch 2.
//   2. experts  one persistent kernel, every CTA resident.  CTAs pull work items
//               in order from a counter: first the gate/up items (work slot,
//               64 rows of ffn), then the down items (work slot, 64 rows of
//               hidden).  A gate/up item streams the expert's gate and up rows
//               once (TMA) and contracts them with all of the slot's tokens on
//               the tensor cores (MMA columns = tokens); it writes g, u and
//               h = silu(g) * u in fp32, and h as two bf16 columns per pair,
//               h_hi = bf16(h) and h_lo = bf16(h - h_hi) (16 significant bits
//               together), in MMA fragment order.  With the weighted-down
//               order (Q4K_MOE_WEIGHTED_DOWN) the bf16 columns carry r * h,
//               r the pair's route weight, and the final sum below takes the
//               down outputs unweighted.  A down item waits (bounded)
//               until every gate/up item of its slot is done, streams the
//               expert's down rows and writes p = Wd h per pair.  The CTA that
//               completes the last down item of a 64-row group of hidden adds
//               y[t] = sum_j w[t, j] * p[t, j] over the slots j = 0..k-1 of
//               every token, in that order.
// Items are claimed in order and every CTA is resident, so a down item only
// waits on gate/up items already held by running CTAs.  Results do not depend
// on which CTA runs which item (columns of an MMA are independent; the sums
// are in fixed order).
#include <algorithm>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

namespace {

constexpr int kRows = 16;                    // rows per CTA (one MMA m-tile)
constexpr int kTile = kRows * kBlockBytes;   // 2304 bytes per super-block stage
#ifndef Q4K_MOE_STAGES  // ring stages per warp stream
#define Q4K_MOE_STAGES 2
#endif
constexpr int kStagesMoe = Q4K_MOE_STAGES;
constexpr int kMoeWarps = 4;                 // warps (weight streams) per expert CTA
constexpr int kMaxExperts = 2048;
#ifndef Q4K_MOE_SLOT_PAIRS  // pairs per work slot at most
#define Q4K_MOE_SLOT_PAIRS 8
#endif
constexpr int kSlotPairs = Q4K_MOE_SLOT_PAIRS;

// Workspace layout (all offsets 256-byte aligned).
// Ring of a warp stream: kStagesMoe stages of kStageStride bytes (a gate and
// an up tile per stage; a down stage uses the first half), then the stage
// barriers; TMA destinations must be 128-byte aligned, so the region is
// rounded up.
constexpr int kStageStride = 2 * kTile;
// After the ring and its barriers: the permuted x (or h) of the two columns of
// a small slot (expert_body_pair) and 64 zero bytes.
constexpr int kPermStrideMoe = 20;                     // words per sub-block (16 used)
constexpr int kPermWordsMoe = 8 * kPermStrideMoe + 4;  // one column; +4 staggers the banks
constexpr int kOffPermMoe = (kStagesMoe * kStageStride + 8 * kStagesMoe + 15) / 16 * 16;
constexpr int kOffZeroMoe = kOffPermMoe + 2 * kPermWordsMoe * 4;
constexpr int kWarpBytes = (kOffZeroMoe + 64 + 127) / 128 * 128;
constexpr int kMetaAbort = 2;  // workspace meta word: a wait timed out, stop taking items
constexpr int kGuTilesPerItem = 4;  // 16-row tiles of ffn per gate/up item (one per warp)
// 16-row tiles of hidden per down item (one per warp): each CTA's last item is
// a down item, so a small one keeps the step's tail short (measured on 128
// experts, 16 tokens, top-8: 8 tiles 2.36 TB/s, 4 tiles 2.50, 16 tiles 2.02)
constexpr int kDnTilesPerItem = 4;

struct MoeLayout {
  size_t meta, counters, slot_expert, slot_start, pair_token, pair_q, tj_pair, g, u, h, h_hi, h_lo, p,
      total;
  int n_counters;
  static int max_slots(int E, int P) { return std::min(E, P) + (P + kSlotPairs - 1) / kSlotPairs; }
  static int dn_groups(int64_t H) { return (int)((H + 16 * kDnTilesPerItem - 1) / (16 * kDnTilesPerItem)); }
  MoeLayout(int E, int P, int64_t H, int64_t F) {
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t S = (size_t)max_slots(E, P);
    // work counters: [0] next item, [1 .. 1+S) gate/up items done per slot,
    // [1+S ..) down items done per 64-row group of hidden
    n_counters = 1 + (int)S + dn_groups(H);
    size_t o = 0;
    meta = o;        o = al(o + 16 * sizeof(int));
    counters = o;    o = al(o + (size_t)n_counters * sizeof(int));
    slot_expert = o; o = al(o + S * sizeof(int));
    slot_start = o;  o = al(o + (S + 1) * sizeof(int));
    pair_token = o;  o = al(o + (size_t)P * sizeof(int));
    pair_q = o;      o = al(o + (size_t)P * sizeof(int));
    tj_pair = o;     o = al(o + (size_t)P * sizeof(int));
    g = o;           o = al(o + (size_t)P * F * sizeof(float));
    u = o;           o = al(o + (size_t)P * F * sizeof(float));
    h = o;           o = al(o + (size_t)P * F * sizeof(float));
    h_hi = o;        o = al(o + (size_t)P * F * 2);
    h_lo = o;        o = al(o + (size_t)P * F * 2);
    p = o;           o = al(o + (size_t)P * H * sizeof(float));
    total = o;
  }
};

struct MoeArgs {
  const __nv_bfloat16 *x;
  int64_t ldx;
  const int32_t *ids;
  const float *wts;
  float *y;
  int64_t ldy;
  int n_experts, n_tokens, top_k;
  int hidden, ffn;
  int *meta, *slot_expert, *slot_start, *pair_token, *pair_q, *tj_pair;
  int weighted_down;  // route weight applied to h before the down projection
  int *counters;
  int n_counters, max_slots;
  int slot_pairs;  // pairs per work slot at most (the route kernel's slot size)
  float *g, *u, *h, *p;
  __nv_bfloat16 *h_hi, *h_lo;
  unsigned *err;
};

// ---------------------------------------------------------------- 1. route
__global__ void __launch_bounds__(1024) moe_route_kernel(const MoeArgs a) {
  // Each of the four kernels is launched as a programmatic dependent of the
  // kernel before it and waits for it before touching global memory, so only
  // the launch latency overlaps.
  grid_dependency_wait();
  grid_launch_dependents();
  __shared__ int cnt[kMaxExperts];
  __shared__ int fill[kMaxExperts];
  __shared__ int start[kMaxExperts + 1];
  __shared__ int slot_of[kMaxExperts];
  __shared__ int wsum[32], wact[32];
  const int E = a.n_experts, P = a.n_tokens * a.top_k;
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < a.n_counters; i += nt) a.counters[i] = 0;
  for (int e = tid; e < E; e += nt) cnt[e] = fill[e] = 0;
  __syncthreads();
  for (int q = tid; q < P; q += nt) {
    const int e = a.ids[q];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      a.tj_pair[q] = -1;
      set_device_error(a.err, kDevErrBadExpert);
    }
  }
  __syncthreads();
  // Exclusive scans over experts of the pair counts and of the active flags:
  // thread tid owns the contiguous chunk [tid*per, (tid+1)*per).
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int s = 0, act = 0;
  for (int e = e0; e < e1; ++e) {
    s += cnt[e];
    act += (cnt[e] + a.slot_pairs - 1) / a.slot_pairs;
  }
  int incl_s = s, incl_a = act;
  const int lane = tid & 31, wid = tid >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const int vs = __shfl_up_sync(0xffffffffu, incl_s, o);
    const int va = __shfl_up_sync(0xffffffffu, incl_a, o);
    if (lane >= o) {
      incl_s += vs;
      incl_a += va;
    }
  }
  if (lane == 31) {
    wsum[wid] = incl_s;
    wact[wid] = incl_a;
  }
  __syncthreads();
  if (wid == 0) {
    const int nw = (nt + 31) / 32;
    int vs = lane < nw ? wsum[lane] : 0, va = lane < nw ? wact[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int us = __shfl_up_sync(0xffffffffu, vs, o);
      const int ua = __shfl_up_sync(0xffffffffu, va, o);
      if (lane >= o) {
        vs += us;
        va += ua;
      }
    }
    if (lane < nw) {
      wsum[lane] = vs;
      wact[lane] = va;
    }
  }
  __syncthreads();
  int run_s = (incl_s - s) + (wid ? wsum[wid - 1] : 0);
  int run_a = (incl_a - act) + (wid ? wact[wid - 1] : 0);
  for (int e = e0; e < e1; ++e) {
    start[e] = run_s;
    slot_of[e] = run_a;
    run_s += cnt[e];
    run_a += (cnt[e] + a.slot_pairs - 1) / a.slot_pairs;
  }
  if (tid == nt - 1) {
    a.meta[0] = run_a;  // work slots in use
    a.meta[1] = run_s;  // valid pairs
    a.meta[kMetaAbort] = 0;
  }
  __syncthreads();
  for (int e = tid; e < E; e += nt) {
    for (int q = 0; q * a.slot_pairs < cnt[e]; ++q) {
      a.slot_expert[slot_of[e] + q] = e;
      a.slot_start[slot_of[e] + q] = start[e] + q * a.slot_pairs;
      a.slot_start[slot_of[e] + q + 1] = min(start[e] + (q + 1) * a.slot_pairs, start[e] + cnt[e]);
    }
  }
  for (int q = tid; q < P; q += nt) {
    const int e = a.ids[q];
    if (e >= 0 && e < E) {
      const int pos = start[e] + atomicAdd(&fill[e], 1);
      a.tj_pair[q] = pos;
      a.pair_token[pos] = q / a.top_k;
      a.pair_q[pos] = q;
    }
  }
}

// ---------------------------------------------------------------- expert contraction
// A warp stream takes 16-row m-tiles of one slot's expert, each over the full
// K; its ring of weight stages and its x fragments run ahead continuously
// across those tiles, and each tile's result is written straight from the
// accumulators.  MMA
// columns are the slot's pairs:
//   gate/up (DOWN = false): column c = x row of the c-th pair's token;
//   down    (DOWN = true):  column 2i = h_hi, column 2i+1 = h_lo of pair i.
// Thread t's k-slots (2t, 2t+1) carry positions (o, o+2) and (2t+8, 2t+9)
// positions (o+1, o+3) of a sub-block, o = 8t + 4s for step s = 0/1: quant
// bytes 8t .. 8t+7 of the sub-block's 32-byte chunk.
// One warp's tiles of a slot with at most 8 NT MMA columns: tiles sid, sid +
// nsid, ... below tile_end.  The warp's ring (kStagesMoe stages of
// kStageStride bytes at `ring`, barriers `bars`, initialised once per kernel)
// carries on from ring iteration it0, which is advanced past this call's
// iterations.  Returns false after a timed-out wait (its copies in flight
// were given a bounded time to land; the ring must not be used again).
template <int NT, bool DOWN>
__device__ __forceinline__ bool expert_body(const CUtensorMap *map0p, const CUtensorMap *map1p,
                                            const MoeArgs &a, int nsb, int rows_total,
                                            uint8_t *ring, uint64_t *bars, uint32_t &it0,
                                            int slot, int sid, int nsid, int tile_end) {
  const CUtensorMap &map0 = *map0p, &map1 = *map1p;
  constexpr int NM = DOWN ? 1 : 2;  // weight matrices per stage (gate and up)
  constexpr int kStageBytes = NM * kTile;
  const int expert = a.slot_expert[slot];
  const int pstart = a.slot_start[slot];
  const int np = a.slot_start[slot + 1] - pstart;  // pairs of this slot (<= kSlotPairs)
  const int ncols = DOWN ? 2 * np : np;

  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int ntiles = min((rows_total + kRows - 1) / kRows, tile_end);
  const int ntl = sid < ntiles ? (ntiles - sid + nsid - 1) / nsid : 0;  // tiles of this warp
  const int total = ntl * nsb;                                          // ring iterations
  const uint32_t base = it0;
  const uint64_t policy = l2_evict_first_policy();
  // Ring iteration q = super-block q % nsb of this warp's tile q / nsb; it
  // uses stage (base + q) % kStagesMoe.
  auto issue = [&](int q) {
    const int j = q / nsb, u = q - j * nsb;
    const int row0 = (sid + j * nsid) * kRows;
    const uint32_t stage = (base + (uint32_t)q) % kStagesMoe;
    mbar_arrive_expect_tx(&bars[stage], kStageBytes);
    uint8_t *dst = ring + stage * kStageStride;
    tma_load_3d_hint(dst, &map0, &bars[stage], u * (kBlockBytes / 8), row0, expert, policy);
    if (NM == 2)
      tma_load_3d_hint(dst + kTile, &map1, &bars[stage], u * (kBlockBytes / 8), row0, expert,
                       policy);
  };
  if (lane == 0)
    for (int q = 0; q < kStagesMoe && q < total; ++q) issue(q);

  // bf16 source of this lane's column nt*8 + g (rows of K values).
  const __nv_bfloat16 *src[NT];
  bool cval[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = nt * 8 + g;
    cval[nt] = c < ncols;
    const int cc = cval[nt] ? c : 0;
    if (DOWN)
      src[nt] = ((cc & 1) ? a.h_lo : a.h_hi) + (size_t)(pstart + (cc >> 1)) * a.ffn;
    else
      src[nt] = a.x + (int64_t)a.pair_token[pstart + cc] * a.ldx;
  }
  // x (or h) fragments of CJ sub-blocks for this lane's columns, loaded one
  // chunk ahead of their use so the L2 latency stays off the MMA path.  They
  // depend only on the super-block, not on the row tile.
  constexpr int CJ = NT <= 2 ? 4 : 2;  // sub-blocks per chunk
  constexpr int NCH = 8 / CJ;          // chunks per super-block (even)
  auto load_x = [&](uint4(&dst)[CJ][NT], int q, int ch) {
    const int u = q % nsb;
#pragma unroll
    for (int jj = 0; jj < CJ; ++jj)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int64_t off = (int64_t)u * kQK + 32 * (ch * CJ + jj) + 8 * t;
        // h (down) is written by this kernel's gate/up items: read it through
        // L2, not the read-only path; x is the caller's and read-only
        const uint4 *ptr = reinterpret_cast<const uint4 *>(src[nt] + off);
        dst[jj][nt] = (cval[nt] && q < total) ? (DOWN ? __ldcg(ptr) : __ldg(ptr))
                                              : make_uint4(0, 0, 0, 0);
      }
  };
  uint4 xbuf[2][CJ][NT];
  load_x(xbuf[0], 0, 0);

  bool ok = true;
  for (int j = 0; j < ntl; ++j) {
    const int row0 = (sid + j * nsid) * kRows;
    float yacc[NM][NT][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        yacc[mi][nt][0] = yacc[mi][nt][1] = yacc[mi][nt][2] = yacc[mi][nt][3] = 0.f;
    for (int u = 0; u < nsb && ok; ++u) {
      const int q = j * nsb + u;
      const uint32_t gq = base + (uint32_t)q;
      const uint32_t stage = gq % kStagesMoe;
      if (!mbar_wait(&bars[stage], (gq / kStagesMoe) & 1u, a.err)) {
        ok = false;
        if (lane == 0) {
          atomicExch(&a.meta[kMetaAbort], 1);  // every CTA stops taking items
          // let this warp's copies in flight land (bounded)
          const uint64_t t0 = global_ns();
          for (int r = q; r < min(q + kStagesMoe, total); ++r) {
            const uint32_t gr = base + (uint32_t)r;
            while (!mbar_try_wait(&bars[gr % kStagesMoe], (gr / kStagesMoe) & 1u, 1000u))
              if (global_ns() - t0 > kWaitLimitNs) break;
          }
        }
        break;
      }
      const uint8_t *st = ring + stage * kStageStride;
      uint4 hdr[NM][2];
      uint2 qw[NM][2][4];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t *rp = st + mi * kTile + (g + 8 * r) * kBlockBytes;
          hdr[mi][r] = *reinterpret_cast<const uint4 *>(rp);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            qw[mi][r][c] = *reinterpret_cast<const uint2 *>(rp + kQsOffset + 32 * c + 8 * t);
        }
      __syncwarp();
      if (lane == 0 && q + kStagesMoe < total) issue(q + kStagesMoe);
      // Offset forms (offset_form) of sub-blocks 2t, 2t+1 (e = 0, 1) of rows
      // g, g+8 (r = 0, 1); the other lanes of the quad fetch them by shuffle.
      // The bf16 subtrahends of both rows travel packed in one word per e.
      float dsv[NM][2][2], eev[NM][2][2];
      uint32_t subp[NM][2];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi) {
        uint32_t sc2[2], m2[2];
#pragma unroll
        for (int r = 0; r < 2; ++r)
          scales_pair(hdr[mi][r].y, hdr[mi][r].z, hdr[mi][r].w, t, &sc2[r], &m2[r]);
        // rows g, g+8 as the two lanes of the packed fp32 operations
        float2 d2, nd23, dmin2, pdm23;
        scale_pairs(hdr[mi][0].x, hdr[mi][1].x, d2, nd23, dmin2, pdm23);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float2 ds2, ee2;
          offset_form_rows2_packed<16>(d2, nd23, dmin2, pdm23, byte_magic(sc2[0], e),
                                       byte_magic(sc2[1], e), byte_magic_neg(m2[0], e),
                                       byte_magic_neg(m2[1], e), ds2, ee2, subp[mi][e]);
          dsv[mi][0][e] = ds2.x;
          dsv[mi][1][e] = ds2.y;
          eev[mi][0][e] = ee2.x;
          eev[mi][1][e] = ee2.y;
        }
      }
      auto sub_block = [&](int jb, const uint4(&xv)[NT]) {
        const int c = jb >> 1;
        const bool hi = jb & 1;
        // B fragments: (x[o], x[o+2]) and (x[o+1], x[o+3]).  h of the down
        // projection is stored in that order already; x needs a byte permute.
        uint32_t b0[NT][2], b1[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 v = xv[nt];
          if (DOWN) {
            b0[nt][0] = v.x;
            b1[nt][0] = v.y;
            b0[nt][1] = v.z;
            b1[nt][1] = v.w;
          } else {
            b0[nt][0] = __byte_perm(v.x, v.y, 0x5410);
            b1[nt][0] = __byte_perm(v.x, v.y, 0x7632);
            b0[nt][1] = __byte_perm(v.z, v.w, 0x5410);
            b1[nt][1] = __byte_perm(v.z, v.w, 0x7632);
          }
        }
        // X_j of every column by two MMAs with A = 1 everywhere (every row
        // holds it, so column 2t+e is xsum[nt][e]).
        float xsum[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16_zc(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[nt][0], b1[nt][0]);
          mma_bf16(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[nt][1], b1[nt][1]);
        }
        // Offset forms of sub-block jb for rows g, g+8 live in lane (g, jb/2).
        const int srcl = (lane & ~3) | (jb >> 1);
#pragma unroll
        for (int mi = 0; mi < NM; ++mi) {
          const uint32_t sp = __shfl_sync(0xffffffffu, hi ? subp[mi][1] : subp[mi][0], srcl);
          const uint32_t sg = __byte_perm(sp, 0u, 0x1010u), sg8 = __byte_perm(sp, 0u, 0x3232u);
          float acc[NT][4];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint32_t w0 = s ? qw[mi][0][c].y : qw[mi][0][c].x;
            const uint32_t w1 = s ? qw[mi][1][c].y : qw[mi][1][c].x;
            const uint32_t a0 = sub_bf16x2(hi ? nib_hi(w0) : nib_lo(w0), sg);
            const uint32_t a1 = sub_bf16x2(hi ? nib_hi(w1) : nib_lo(w1), sg8);
            const uint32_t a2 = sub_bf16x2(hi ? nib_hi(w0 >> 8) : nib_lo(w0 >> 8), sg);
            const uint32_t a3 = sub_bf16x2(hi ? nib_hi(w1 >> 8) : nib_lo(w1 >> 8), sg8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (s == 0)
                mma_bf16_zc(acc[nt], a0, a1, a2, a3, b0[nt][0], b1[nt][0]);
              else
                mma_bf16(acc[nt], a0, a1, a2, a3, b0[nt][1], b1[nt][1]);
            }
          }
          // acc = sum (q - c) x over the sub-block: add ds * acc + e * X_j.
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float ds = __shfl_sync(0xffffffffu, hi ? dsv[mi][r][1] : dsv[mi][r][0], srcl);
            const float ee = __shfl_sync(0xffffffffu, hi ? eev[mi][r][1] : eev[mi][r][0], srcl);
            // columns 2t, 2t+1 share ds and e: one packed fma each (each lane
            // of a pair rounds as fmaf)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float2 yv = make_float2(yacc[mi][nt][2 * r], yacc[mi][nt][2 * r + 1]);
              yv = __ffma2_rn(make_float2(ds, ds), make_float2(acc[nt][2 * r], acc[nt][2 * r + 1]), yv);
              yv = __ffma2_rn(make_float2(ee, ee), make_float2(xsum[nt][0], xsum[nt][1]), yv);
              yacc[mi][nt][2 * r] = yv.x;
              yacc[mi][nt][2 * r + 1] = yv.y;
            }
          }
        }
      };
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        if (ch + 1 < NCH)
          load_x(xbuf[(ch + 1) & 1], q, ch + 1);
        else
          load_x(xbuf[0], q + 1, 0);
#pragma unroll
        for (int jj = 0; jj < CJ; ++jj) sub_block(ch * CJ + jj, xbuf[ch & 1][jj]);
      }
    }
    // This tile's outputs: thread (g, t) holds rows g, g+8 and columns
    // nt*8 + 2t + e.  After a timed-out wait the warp's remaining rows read NaN.
    const float nan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int grow = row0 + g + 8 * r;
        if (grow >= rows_total) continue;
        if (DOWN) {
          const int pr = nt * 4 + t;  // columns 2pr (h_hi) and 2pr+1 (h_lo)
          if (pr < np)
            a.p[(size_t)(pstart + pr) * a.hidden + grow] =
                ok ? yacc[0][nt][2 * r] + yacc[0][nt][2 * r + 1] : nan;
        } else {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pr = nt * 8 + 2 * t + e;
            if (pr >= np) continue;
            const float gg = yacc[0][nt][2 * r + e], uu = yacc[NM - 1][nt][2 * r + e];
            const float hv = ok ? gg / (1.f + __expf(-gg)) * uu : nan;
            // the down projection's input: h, or r h in the weighted-down order
            const float hd = a.weighted_down ? hv * a.wts[a.pair_q[pstart + pr]] : hv;
            const __nv_bfloat16 hh = __float2bfloat16_rn(hd);
            const __nv_bfloat16 hl = __float2bfloat16_rn(hd - __bfloat162float(hh));
            // h_hi / h_lo in B-fragment order: positions 1 and 2 of each group
            // of four swapped, so that 32-bit words hold (h[o], h[o+2]) and
            // (h[o+1], h[o+3]).
            const int pos = (grow & ~3) | ((grow & 1) << 1) | ((grow >> 1) & 1);
            a.g[(size_t)(pstart + pr) * a.ffn + grow] = ok ? gg : nan;
            a.u[(size_t)(pstart + pr) * a.ffn + grow] = ok ? uu : nan;
            a.h[(size_t)(pstart + pr) * a.ffn + grow] = hv;
            a.h_hi[(size_t)(pstart + pr) * a.ffn + pos] = hh;
            a.h_lo[(size_t)(pstart + pr) * a.ffn + pos] = hl;
          }
        }
      }
  }
  it0 = base + (uint32_t)total;
  return ok;
}

// A slot whose MMA columns fit one pair (gate/up: at most 2 pairs; down: one
// pair, its h_hi and h_lo columns) takes the contraction of the batch-1..4
// decode stream kernel instead: thread t's k-slots carry sub-block 2t (low
// nibbles, the "E" MMAs) or 2t+1 (high nibbles, "O") of rows g, g+8, and MMA
// column 2s + c holds column c's x (or h) only in the k-slots of thread s.
// So each thread ends with the sums of its own sub-blocks for both columns and
// applies the offset forms it decoded itself: no shuffles, 16 MMAs per
// super-block and matrix, and the scale epilogue once per super-block.
// X_j of each column: two MMAs with A = 1 per super-block.  The B fragments
// come from a per-warp permuted copy of the super-block's x (h is stored in
// that order already).  Same ring, item and result conventions as expert_body.
template <bool DOWN>
__device__ __forceinline__ bool expert_body_pair(const CUtensorMap *map0p, const CUtensorMap *map1p,
                                                 const MoeArgs &a, int nsb, int rows_total,
                                                 uint8_t *ring, uint64_t *bars, uint32_t &it0,
                                                 int slot, int sid, int nsid, int tile_end) {
  const CUtensorMap &map0 = *map0p, &map1 = *map1p;
  constexpr int NM = DOWN ? 1 : 2;  // weight matrices per stage (gate and up)
  constexpr int kStageBytes = NM * kTile;
  const int expert = a.slot_expert[slot];
  const int pstart = a.slot_start[slot];
  const int np = a.slot_start[slot + 1] - pstart;  // pairs of this slot
  const int ncols = DOWN ? 2 * np : np;             // 1 or 2

  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int ntiles = min((rows_total + kRows - 1) / kRows, tile_end);
  const int ntl = sid < ntiles ? (ntiles - sid + nsid - 1) / nsid : 0;  // tiles of this warp
  const int total = ntl * nsb;                                          // ring iterations
  const uint32_t base = it0;
  const uint64_t policy = l2_evict_first_policy();
  uint32_t *perm = reinterpret_cast<uint32_t *>(ring + kOffPermMoe);
  const uint32_t *zeros = reinterpret_cast<const uint32_t *>(ring + kOffZeroMoe);
  auto issue = [&](int q) {
    const int j = q / nsb, u = q - j * nsb;
    const int row0 = (sid + j * nsid) * kRows;
    const uint32_t stage = (base + (uint32_t)q) % kStagesMoe;
    mbar_arrive_expect_tx(&bars[stage], kStageBytes);
    uint8_t *dst = ring + stage * kStageStride;
    tma_load_3d_hint(dst, &map0, &bars[stage], u * (kBlockBytes / 8), row0, expert, policy);
    if (NM == 2)
      tma_load_3d_hint(dst + kTile, &map1, &bars[stage], u * (kBlockBytes / 8), row0, expert,
                       policy);
  };
  if (lane == 0)
    for (int q = 0; q < kStagesMoe && q < total; ++q) issue(q);

  // Column c's source rows: gate/up the x row of pair c's token, down h_hi
  // (c = 0) and h_lo (c = 1) of the pair.
  const __nv_bfloat16 *src[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int cc = c < ncols ? c : 0;
    if (DOWN)
      src[c] = (cc ? a.h_lo : a.h_hi) + (size_t)pstart * a.ffn;
    else
      src[c] = a.x + (int64_t)a.pair_token[pstart + cc] * a.ldx;
  }
  // This lane's 16 bytes of super-block q of each column: values 8t .. 8t+7
  // of sub-block g (of h: the same values, permuted within groups of four),
  // loaded one super-block ahead of their use.
  auto load_raw = [&](uint4(&dst)[2], int q) {
    const int u = q % nsb;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 *ptr = reinterpret_cast<const uint4 *>(src[c] + (int64_t)u * kQK + 32 * g + 8 * t);
      // h is written by this kernel's gate/up items: read it through L2
      dst[c] = (c < ncols && q < total) ? (DOWN ? __ldcg(ptr) : __ldg(ptr)) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 raw[2];
  load_raw(raw, 0);

  // Scale/min decode of sub-blocks 2t, 2t+1 of rows g, g+8 (see the stream
  // kernel): psel gathers bytes k0, k0+1 of rows g (bytes 0, 1) and g+8 (2, 3).
  const bool upper = t >= 2;
  const uint32_t k0 = 2 * (t & 1);
  const uint32_t psel = k0 | ((k0 + 1) << 4) | ((k0 + 4) << 8) | ((k0 + 5) << 12);
  const uint32_t mlo4 = upper ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
  const uint32_t mhi4 = upper ? 0x30303030u : 0u;
  // B fragments: lane (g, t) is column g; when t == g / 2 its k-slots carry
  // column g & 1 (sub-block 2t in the E MMAs, 2t+1 in the O MMAs).
  const int col = g & 1;
  const int bofs = (t == (g >> 1) && col < ncols) ? col * kPermWordsMoe + 2 * t * kPermStrideMoe : -1;
  const uint32_t *pe = bofs >= 0 ? perm + bofs : zeros;
  const uint32_t *po = bofs >= 0 ? perm + bofs + kPermStrideMoe : zeros;
  uint32_t magic;
  asm volatile("mov.b32 %0, %1;\n" : "=r"(magic) : "n"(kBf16Magic));

  bool ok = true;
  for (int j = 0; j < ntl; ++j) {
    const int row0 = (sid + j * nsid) * kRows;
    float yacc[NM][2][2];  // [matrix][row g, g+8][column], over sub-blocks 2t, 2t+1
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
      yacc[mi][0][0] = yacc[mi][0][1] = yacc[mi][1][0] = yacc[mi][1][1] = 0.f;
    for (int u = 0; u < nsb && ok; ++u) {
      const int q = j * nsb + u;
      const uint32_t gq = base + (uint32_t)q;
      const uint32_t stage = gq % kStagesMoe;
      if (!mbar_wait(&bars[stage], (gq / kStagesMoe) & 1u, a.err)) {
        ok = false;
        if (lane == 0) {
          atomicExch(&a.meta[kMetaAbort], 1);  // every CTA stops taking items
          // let this warp's copies in flight land (bounded)
          const uint64_t t0 = global_ns();
          for (int r = q; r < min(q + kStagesMoe, total); ++r) {
            const uint32_t gr = base + (uint32_t)r;
            while (!mbar_try_wait(&bars[gr % kStagesMoe], (gr / kStagesMoe) & 1u, 1000u))
              if (global_ns() - t0 > kWaitLimitNs) break;
          }
        }
        break;
      }
      const uint8_t *st = ring + stage * kStageStride;
      __syncwarp();  // the previous super-block's B-fragment reads are done
      // X_j of the eight sub-blocks of each column (A = 1; lane (g, t) holds
      // eight values of sub-block g, the B fragment of column g), and the
      // permuted copy: word 2G of a sub-block holds (x[4G], x[4G+2]), word
      // 2G+1 (x[4G+1], x[4G+3]).
      float xs[2][4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 v = raw[c];
        mma_bf16_zc(xs[c], kBf16One, kBf16One, kBf16One, kBf16One, v.x, v.y);
        mma_bf16(xs[c], kBf16One, kBf16One, kBf16One, kBf16One, v.z, v.w);
        uint4 pm = v;
        if (!DOWN) {
          pm.x = __byte_perm(v.x, v.y, 0x5410u);
          pm.y = __byte_perm(v.x, v.y, 0x7632u);
          pm.z = __byte_perm(v.z, v.w, 0x5410u);
          pm.w = __byte_perm(v.z, v.w, 0x7632u);
        }
        reinterpret_cast<uint4 *>(perm + c * kPermWordsMoe + g * kPermStrideMoe)[t] = pm;
      }
      uint4 hdr[NM][2], qa[NM][2][2];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t *rp = st + mi * kTile + (g + 8 * r) * kBlockBytes;
          hdr[mi][r] = *reinterpret_cast<const uint4 *>(rp);
          qa[mi][r][0] = *reinterpret_cast<const uint4 *>(rp + kQsOffset + 32 * t);
          qa[mi][r][1] = *reinterpret_cast<const uint4 *>(rp + kQsOffset + 32 * t + 16);
        }
      __syncwarp();  // permuted copy visible; the stage's reads are done
      if (lane == 0 && q + kStagesMoe < total) issue(q + kStagesMoe);
      load_raw(raw, q + 1);

      float ds[NM][2][2], ee[NM][2][2];
      uint32_t sub[NM][2][2];
#pragma unroll
      for (int mi = 0; mi < NM; ++mi) {
        const uint4 h0 = hdr[mi][0], h1 = hdr[mi][1];
        const uint32_t py = __byte_perm(h0.y, h1.y, psel);
        const uint32_t pz = __byte_perm(h0.z, h1.z, psel);
        const uint32_t pw4 = __byte_perm(h0.w, h1.w, psel);
        const uint32_t sc4 = ((upper ? pw4 : py) & mlo4) | ((py >> 2) & mhi4);
        const uint32_t m4 = ((upper ? (pw4 >> 4) : pz) & mlo4) | ((pz >> 2) & mhi4);
        // rows g, g+8 as the two lanes of the packed fp32 operations
        float2 d2, nd23, dmin2, pdm23;
        scale_pairs(h0.x, h1.x, d2, nd23, dmin2, pdm23);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float2 ds2, ee2;
          offset_form_rows2<16>(d2, nd23, dmin2, pdm23, byte_magic(sc4, e), byte_magic(sc4, 2 + e),
                                byte_magic_neg(m4, e), byte_magic_neg(m4, 2 + e), ds2, ee2,
                                sub[mi][0][e], sub[mi][1][e]);
          ds[mi][0][e] = ds2.x;
          ds[mi][1][e] = ds2.y;
          ee[mi][0][e] = ee2.x;
          ee[mi][1][e] = ee2.y;
        }
      }
      // accE[mi] column 2t + c = sum (q - c_j) x over sub-block 2t of column c
      // (rows g: [c], g+8: [2 + c]); accO likewise for 2t+1.
      float accE[NM][4], accO[NM][4];
#pragma unroll
      for (int G2 = 0; G2 < 4; ++G2) {
        const uint4 be = reinterpret_cast<const uint4 *>(pe)[G2];  // the zero block is 4 uint4
        const uint4 bo = reinterpret_cast<const uint4 *>(po)[G2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int G = 2 * G2 + h;
          const uint32_t be0 = h ? be.z : be.x, be1 = h ? be.w : be.y;
          const uint32_t bo0 = h ? bo.z : bo.x, bo1 = h ? bo.w : bo.y;
#pragma unroll
          for (int mi = 0; mi < NM; ++mi) {
            const uint4 qv0 = qa[mi][0][G >> 2], qv1 = qa[mi][1][G >> 2];
            const uint32_t w0 = (G & 3) == 0 ? qv0.x : (G & 3) == 1 ? qv0.y : (G & 3) == 2 ? qv0.z : qv0.w;
            const uint32_t w1 = (G & 3) == 0 ? qv1.x : (G & 3) == 1 ? qv1.y : (G & 3) == 2 ? qv1.z : qv1.w;
            // low nibbles: sub-block 2t, positions (4G, 4G+2) and (4G+1, 4G+3)
            const uint32_t a0 = sub_bf16x2(lop_nib(w0, magic), sub[mi][0][0]);
            const uint32_t a1 = sub_bf16x2(lop_nib(w1, magic), sub[mi][1][0]);
            const uint32_t a2 = sub_bf16x2(lop_nib(w0 >> 8, magic), sub[mi][0][0]);
            const uint32_t a3 = sub_bf16x2(lop_nib(w1 >> 8, magic), sub[mi][1][0]);
            // high nibbles: sub-block 2t+1
            const uint32_t c0 = sub_bf16x2(lop_nib(w0 >> 4, magic), sub[mi][0][1]);
            const uint32_t c1 = sub_bf16x2(lop_nib(w1 >> 4, magic), sub[mi][1][1]);
            const uint32_t c2 = sub_bf16x2(lop_nib(w0 >> 12, magic), sub[mi][0][1]);
            const uint32_t c3 = sub_bf16x2(lop_nib(w1 >> 12, magic), sub[mi][1][1]);
            if (G == 0) {
              mma_bf16_zc(accE[mi], a0, a1, a2, a3, be0, be1);
              mma_bf16_zc(accO[mi], c0, c1, c2, c3, bo0, bo1);
            } else {
              mma_bf16(accE[mi], a0, a1, a2, a3, be0, be1);
              mma_bf16(accO[mi], c0, c1, c2, c3, bo0, bo1);
            }
          }
        }
      }
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v = yacc[mi][r][c];
            v = fmaf(ds[mi][r][0], accE[mi][2 * r + c], v);
            v = fmaf(ee[mi][r][0], xs[c][0], v);
            v = fmaf(ds[mi][r][1], accO[mi][2 * r + c], v);
            v = fmaf(ee[mi][r][1], xs[c][1], v);
            yacc[mi][r][c] = v;
          }
    }
    // Rows: add the quad's sub-block pairs (t = 0..3), then lanes t == 0
    // write rows g, g+8.  After a timed-out wait the warp's remaining rows
    // read NaN.
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float v = yacc[mi][r][c];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          yacc[mi][r][c] = v;
        }
    const float nan = __int_as_float(0x7fc00000);
    if (t == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int grow = row0 + g + 8 * r;
        if (grow >= rows_total) continue;
        if (DOWN) {
          a.p[(size_t)pstart * a.hidden + grow] = ok ? yacc[0][r][0] + yacc[0][r][1] : nan;
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (c >= np) continue;
            const float gg = yacc[0][r][c], uu = yacc[NM - 1][r][c];
            const float hv = ok ? gg / (1.f + __expf(-gg)) * uu : nan;
            // the down projection's input: h, or r h in the weighted-down order
            const float hd = a.weighted_down ? hv * a.wts[a.pair_q[pstart + c]] : hv;
            const __nv_bfloat16 hh = __float2bfloat16_rn(hd);
            const __nv_bfloat16 hl = __float2bfloat16_rn(hd - __bfloat162float(hh));
            // h_hi / h_lo in B-fragment order (positions 1 and 2 of each group
            // of four swapped)
            const int pos = (grow & ~3) | ((grow & 1) << 1) | ((grow >> 1) & 1);
            a.g[(size_t)(pstart + c) * a.ffn + grow] = ok ? gg : nan;
            a.u[(size_t)(pstart + c) * a.ffn + grow] = ok ? uu : nan;
            a.h[(size_t)(pstart + c) * a.ffn + grow] = hv;
            a.h_hi[(size_t)(pstart + c) * a.ffn + pos] = hh;
            a.h_lo[(size_t)(pstart + c) * a.ffn + pos] = hl;
          }
        }
      }
    }
  }
  it0 = base + (uint32_t)total;
  return ok;
}

// One slot's share of an item: the MMA width follows the slot's pair count
// (8 columns when its pairs fit, else 16 or 32, NTMAX n-tiles of 8 at most),
// so a slot with few pairs does no work for empty columns.  Warp w of the CTA
// takes the item's tiles t0 + w, t0 + w + 4, ... below t0 + per_item.
template <int NTMAX, bool DOWN>
__device__ __forceinline__ bool slot_item(const CUtensorMap *m0, const CUtensorMap *m1,
                                          const MoeArgs &a, int nsb, int rows, uint8_t *ring,
                                          uint64_t *bars, uint32_t &it, int slot, int t0,
                                          int per_item) {
  const int np = a.slot_start[slot + 1] - a.slot_start[slot];
  const int ncols = DOWN ? 2 * np : np;
  const int nt = ncols <= 8 ? 1 : ncols <= 16 ? 2 : 4;  // n-tiles this slot needs
  const int sid = t0 + (int)(threadIdx.x >> 5);
  if (ncols <= 2)
    return expert_body_pair<DOWN>(m0, m1, a, nsb, rows, ring, bars, it, slot, sid, kMoeWarps,
                                  t0 + per_item);
  if (nt == 1 || NTMAX == 1)
    return expert_body<1, DOWN>(m0, m1, a, nsb, rows, ring, bars, it, slot, sid, kMoeWarps,
                                t0 + per_item);
  if (nt == 2 || NTMAX == 2)
    return expert_body<(NTMAX >= 2 ? 2 : 1), DOWN>(m0, m1, a, nsb, rows, ring, bars, it, slot, sid,
                                                   kMoeWarps, t0 + per_item);
  return expert_body<NTMAX, DOWN>(m0, m1, a, nsb, rows, ring, bars, it, slot, sid, kMoeWarps,
                                  t0 + per_item);
}

__device__ __forceinline__ int load_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *count reaches target (acquire: the writes made before
// the matching releases are visible afterwards).  Returns false at once when
// another CTA has raised the abort word; after the wall-clock limit it sets
// the timeout bit of the device error word, raises the abort word and
// returns false.
__device__ __forceinline__ bool wait_count(const int *count, int target, int *abort_word,
                                           unsigned *err) {
  const uint64_t t0 = global_ns();
  for (;;) {
    if (load_acquire(count) >= target) return true;
    if (load_acquire(abort_word) != 0) return false;
    if (global_ns() - t0 > kWaitLimitNs) break;
    __nanosleep(256);
  }
  set_device_error(err, kDevErrTimeout);
  atomicExch(abort_word, 1);
  return false;
}

// ---------------------------------------------------------------- 2. experts
template <int NTGU, int NTDN>
__global__ void __launch_bounds__(kMoeWarps * 32) moe_persistent_kernel(
    const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mu,
    const __grid_constant__ CUtensorMap md, const MoeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_item[2], s_last, s_fail;
  // Each warp's ring and barriers, set up once: items only carry the ring
  // iteration count on, so no barrier is ever initialised twice and no copy
  // lands in memory that held a barrier.
  const int lane = threadIdx.x & 31;
  uint8_t *ring = smem + (threadIdx.x >> 5) * kWarpBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kStagesMoe * kStageStride);
  if (lane == 0) {
    prefetch_tmap(&mg);
    prefetch_tmap(&mu);
    prefetch_tmap(&md);
    for (int s = 0; s < kStagesMoe; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  if (lane < 16) reinterpret_cast<uint32_t *>(ring + kOffZeroMoe)[lane] = 0u;
  if (threadIdx.x == 0) s_fail = 0;
  __syncthreads();
  uint32_t it = 0;  // this warp's ring iterations so far
  grid_dependency_wait();
  grid_launch_dependents();
  const int S = a.meta[0];  // work slots in use
  const int nsb_gu = a.hidden / kQK, nsb_dn = a.ffn / kQK;
  const int gu_tiles = (a.ffn + kRows - 1) / kRows, dn_tiles = (a.hidden + kRows - 1) / kRows;
  const int gu_groups = (gu_tiles + kGuTilesPerItem - 1) / kGuTilesPerItem;
  const int dn_groups = (dn_tiles + kDnTilesPerItem - 1) / kDnTilesPerItem;
  const int n_gu = S * gu_groups, n_items = n_gu + S * dn_groups;
  int *next = a.counters, *slot_done = a.counters + 1, *grp_done = a.counters + 1 + a.max_slots;
  int *abort_word = a.meta + kMetaAbort;
  for (int par = 0;; par ^= 1) {
    // after a timed-out wait anywhere, no CTA takes another item; the claim
    // alternates between two words, so the item's own barriers separate each
    // word's reads from its next write
    if (threadIdx.x == 0) s_item[par] = load_acquire(abort_word) ? n_items : atomicAdd(next, 1);
    __syncthreads();
    const int item = s_item[par];
    if (item >= n_items) break;
    if (item < n_gu) {
      const int slot = item / gu_groups, grp = item - slot * gu_groups;
      if (!slot_item<NTGU, false>(&mg, &mu, a, nsb_gu, a.ffn, ring, bars, it, slot,
                                  grp * kGuTilesPerItem, kGuTilesPerItem))
        s_fail = 1;
      // Every thread's g, u, h writes come before the barrier; thread 0's
      // GPU-scope fence after it is cumulative over them (a release of the
      // whole CTA's writes), so one fence per item, not one per thread.
      __syncthreads();
      if (s_fail) break;
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&slot_done[slot], 1);
      }
    } else {
      const int j = item - n_gu, slot = j / dn_groups, grp = j - slot * dn_groups;
      if (threadIdx.x == 0 && !wait_count(&slot_done[slot], gu_groups, abort_word, a.err))
        s_fail = 1;
      __syncthreads();
      if (s_fail) break;
      if (!slot_item<NTDN, true>(&md, &md, a, nsb_dn, a.hidden, ring, bars, it, slot,
                                 grp * kDnTilesPerItem, kDnTilesPerItem))
        s_fail = 1;
      __syncthreads();  // every thread's down outputs precede thread 0's release
      if (s_fail) break;
      if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&grp_done[grp], 1) == S - 1;
        __threadfence();  // the last one acquires every other CTA's outputs
      }
      __syncthreads();
      if (s_last) {
        // Every slot's down outputs of this group of hidden rows are in: the
        // route-weighted sum over each token's slots, in slot order.
        const int r0 = grp * kDnTilesPerItem * kRows;
        const int r1 = min(a.hidden, r0 + kDnTilesPerItem * kRows);
        for (int idx = threadIdx.x; idx < (r1 - r0) * a.n_tokens; idx += blockDim.x) {
          const int t = idx / (r1 - r0), i = r0 + idx - t * (r1 - r0);
          float acc = 0.f;
          for (int k = 0; k < a.top_k; ++k) {
            const int q = t * a.top_k + k;
            const int pos = a.tj_pair[q];
            if (pos < 0) continue;
            const float pv = __ldcg(&a.p[(size_t)pos * a.hidden + i]);
            acc = a.weighted_down ? acc + pv : fmaf(a.wts[q], pv, acc);
          }
          a.y[(int64_t)t * a.ldy + i] = acc;
        }
      }
    }
  }
}

std::once_flag g_moe_attr[kMaxDevices];  // cudaFuncSetAttribute acts on the current device

// Launch as a programmatic dependent of the previous kernel on the stream.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kExpertSmem = kMoeWarps * kWarpBytes;  // shared memory of the persistent kernel

int g_moe_occ[kMaxDevices][2];

void moe_attributes(int dev) {
  cudaFuncSetAttribute(moe_persistent_kernel<1, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kExpertSmem);
  cudaFuncSetAttribute(moe_persistent_kernel<2, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kExpertSmem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_moe_occ[dev][0], moe_persistent_kernel<1, 2>,
                                                kMoeWarps * 32, kExpertSmem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_moe_occ[dev][1], moe_persistent_kernel<2, 4>,
                                                kMoeWarps * 32, kExpertSmem);
}

CUresult expert_map(CUtensorMap *map, const void *base, int64_t rows, int64_t k, int64_t stride,
                    int n_experts) {
  const int64_t nsb = k / kQK;
  const uint64_t dims[3] = {(uint64_t)nsb * (kBlockBytes / 8), (uint64_t)rows, (uint64_t)n_experts};
  const uint64_t strides[2] = {(uint64_t)nsb * kBlockBytes, (uint64_t)stride};
  const uint32_t box[3] = {(uint32_t)(kBlockBytes / 8), (uint32_t)kRows, 1u};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(base), dims,
                      strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

size_t moe_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                          int64_t ffn) {
  return MoeLayout(n_experts, n_tokens * top_k, hidden, ffn).total;
}

void moe_workspace_views(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                         int64_t ffn, uint64_t out[5]) {
  const MoeLayout L(n_experts, n_tokens * top_k, hidden, ffn);
  out[0] = L.tj_pair;
  out[1] = L.g;
  out[2] = L.u;
  out[3] = L.h;
  out[4] = L.p;
}

cudaError_t launch_moe(const void *w_gate, const void *w_up, const void *w_down,
                       int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                       const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                       const float *wts, int32_t top_k, float *y, int64_t ldy, void *workspace,
                       bool weighted_down, cudaStream_t stream) {
  if (n_experts > kMaxExperts) return cudaErrorInvalidValue;
  std::call_once(g_moe_attr[device_facts()->device], moe_attributes, device_facts()->device);
  const int P = n_tokens * top_k;
  const MoeLayout L(n_experts, P, hidden, ffn);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  MoeArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.ldx = ldx;
  a.ids = ids;
  a.wts = wts;
  a.y = y;
  a.ldy = ldy;
  a.n_experts = n_experts;
  a.n_tokens = n_tokens;
  a.top_k = top_k;
  a.hidden = (int)hidden;
  a.ffn = (int)ffn;
  a.meta = reinterpret_cast<int *>(ws + L.meta);
  a.counters = reinterpret_cast<int *>(ws + L.counters);
  a.n_counters = L.n_counters;
  a.max_slots = MoeLayout::max_slots(n_experts, P);
  a.slot_pairs = kSlotPairs;
  a.slot_expert = reinterpret_cast<int *>(ws + L.slot_expert);
  a.slot_start = reinterpret_cast<int *>(ws + L.slot_start);
  a.pair_token = reinterpret_cast<int *>(ws + L.pair_token);
  a.pair_q = reinterpret_cast<int *>(ws + L.pair_q);
  a.weighted_down = weighted_down ? 1 : 0;
  a.tj_pair = reinterpret_cast<int *>(ws + L.tj_pair);
  a.g = reinterpret_cast<float *>(ws + L.g);
  a.u = reinterpret_cast<float *>(ws + L.u);
  a.h = reinterpret_cast<float *>(ws + L.h);
  a.h_hi = reinterpret_cast<__nv_bfloat16 *>(ws + L.h_hi);
  a.h_lo = reinterpret_cast<__nv_bfloat16 *>(ws + L.h_lo);
  a.p = reinterpret_cast<float *>(ws + L.p);
  a.err = device_error_word();

  CUtensorMap mg, mu, md;
  if (expert_map(&mg, w_gate, ffn, hidden, expert_stride, n_experts) != CUDA_SUCCESS ||
      expert_map(&mu, w_up, ffn, hidden, expert_stride, n_experts) != CUDA_SUCCESS ||
      expert_map(&md, w_down, hidden, ffn, expert_stride, n_experts) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  cudaError_t e = launch_pdl(moe_route_kernel, dim3(1), 1024, 0, stream, a);
  if (e != cudaSuccess) return e;
  // The widest slot decides the instantiation: 8-column slots fit the <1, 2>
  // kernel (gate/up one column per pair, down two), wider ones the <2, 4>.
  // With 8-pair slots (the default) every call takes the <1, 2> kernel: it
  // holds 3 CTAs per SM against 2, which outweighs reading an expert with more
  // than 8 tokens once per 8 of them.
  const int cap = std::min(P, kSlotPairs);  // pairs per slot at most
  const int wide = cap > 8 ? 1 : 0;
  const DeviceFacts *f = device_facts();
  const int occ = g_moe_occ[f->device][wide];
  if (occ <= 0) return cudaErrorInvalidConfiguration;
  // every CTA resident; no more CTAs than there can be items
  const int S_max = MoeLayout::max_slots(n_experts, P);
  const long items = (long)S_max * (((ffn + kRows - 1) / kRows + kGuTilesPerItem - 1) / kGuTilesPerItem +
                                    MoeLayout::dn_groups(hidden));
  const int grid = (int)std::min<long>((long)occ * f->sm_count, items);
  e = wide ? launch_pdl(moe_persistent_kernel<2, 4>, dim3((unsigned)grid), kMoeWarps * 32,
                        (size_t)kExpertSmem, stream, mg, mu, md, a)
           : launch_pdl(moe_persistent_kernel<1, 2>, dim3((unsigned)grid), kMoeWarps * 32,
                        (size_t)kExpertSmem, stream, mg, mu, md, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4k

// ---------------------------------------------------------------------------
// Routed-MoE prefill (token blocks; "Layer Package Repository Spec", section
// "Policy Resolution": routed gate/up/down expert matmuls, fused SwiGLU,
// route-weighted sum).  The expert matmuls are grouped tcgen05 GEMMs over
// expert-sorted token rows: every active expert's weights are dequantized once
// per block of up to 256 of its (token, slot) pairs.  Seven launches on the
// caller's stream, each a programmatic dependent of the one before:
//   1. route    as for decode, with work slots of up to 256 pairs
//   2. gather   Xs[pos] = x[token of pair pos]          (bf16 rows, expert-sorted)
//   3. gate     G = Xs Wg_e^T, slot by slot             (grouped GEMM, bf16 out)
//   4. up       U = Xs Wu_e^T                           (grouped GEMM, bf16 out)
//   5. silu     H = bf16(silu(G) U), fp32 arithmetic
//   6. down     Pd = H Wd_e^T                           (grouped GEMM, bf16 out)
//   7. combine  y[t] = sum_j w[t, j] Pd[pos(t, j)]      (fp32, slots in order j)
namespace q4k {

namespace {

constexpr int kPrefillSlot = 256;  // pairs per work slot: the grouped GEMM's token tile

struct PrefillLayout {
  size_t meta, slot_expert, slot_start, pair_token, pair_q, tj_pair, xs, g, u, h, p, total;
  int max_slots;
  PrefillLayout(int E, int P, int64_t H, int64_t F) {
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    max_slots = std::min(E, P) + (P + kPrefillSlot - 1) / kPrefillSlot;
    const size_t S = (size_t)max_slots;
    size_t o = 0;
    meta = o;        o = al(o + 16 * sizeof(int));
    slot_expert = o; o = al(o + S * sizeof(int));
    slot_start = o;  o = al(o + (S + 1) * sizeof(int));
    pair_token = o;  o = al(o + (size_t)P * sizeof(int));
    pair_q = o;      o = al(o + (size_t)P * sizeof(int));
    tj_pair = o;     o = al(o + (size_t)P * sizeof(int));
    xs = o;          o = al(o + (size_t)P * H * 2);
    g = o;           o = al(o + (size_t)P * F * 2);
    u = o;           o = al(o + (size_t)P * F * 2);
    h = o;           o = al(o + (size_t)P * F * 2);
    p = o;           o = al(o + (size_t)P * H * 2);
    total = o;
  }
};

// One CTA per pair position: copies the pair's token row of x.
__global__ void __launch_bounds__(256) moe_gather_kernel(const MoeArgs a, __nv_bfloat16 *xs) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int pos = blockIdx.x;
  if (pos >= a.meta[1]) return;  // pairs with a valid expert id
  const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)a.pair_token[pos] * a.ldx);
  uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)pos * a.hidden);
  for (int i = threadIdx.x; i < a.hidden / 8; i += blockDim.x) dst[i] = src[i];
}

// H = bf16(silu(G) * U) over the valid pairs' rows, 8 values per thread step.
__global__ void __launch_bounds__(256) moe_silu_kernel(const int *meta, const __nv_bfloat16 *g,
                                                       const __nv_bfloat16 *u, __nv_bfloat16 *h,
                                                       int64_t ffn) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t total = (int64_t)meta[1] * ffn / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 gv = reinterpret_cast<const uint4 *>(g)[i];
    const uint4 uv = reinterpret_cast<const uint4 *>(u)[i];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t hw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = __uint_as_float(gw[e] << 16), g1 = __uint_as_float(gw[e] & 0xFFFF0000u);
      const float u0 = __uint_as_float(uw[e] << 16), u1 = __uint_as_float(uw[e] & 0xFFFF0000u);
      const __nv_bfloat162 hv = __floats2bfloat162_rn(g0 / (1.f + __expf(-g0)) * u0,
                                                      g1 / (1.f + __expf(-g1)) * u1);
      hw[e] = *reinterpret_cast<const uint32_t *>(&hv);
    }
    reinterpret_cast<uint4 *>(h)[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  }
}

// y[t, i] = sum_j w[t, j] Pd[pos(t, j), i] in slot order j (skipped ids add nothing).
__global__ void __launch_bounds__(256) moe_prefill_combine_kernel(const MoeArgs a,
                                                                  const __nv_bfloat16 *pd) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.hidden) return;
  float acc = 0.f;
  for (int j = 0; j < a.top_k; ++j) {
    const int q = t * a.top_k + j;
    const int pos = a.tj_pair[q];
    if (pos < 0) continue;
    acc = fmaf(a.wts[q], __bfloat162float(pd[(size_t)pos * a.hidden + i]), acc);
  }
  a.y[(int64_t)t * a.ldy + i] = acc;
}

}  // namespace

size_t moe_prefill_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k,
                                  int64_t hidden, int64_t ffn) {
  return PrefillLayout(n_experts, n_tokens * top_k, hidden, ffn).total;
}

cudaError_t launch_moe_prefill(const void *w_gate, const void *w_up, const void *w_down,
                               int64_t expert_stride, int32_t n_experts, int64_t hidden,
                               int64_t ffn, const void *x, int32_t n_tokens, int64_t ldx,
                               const int32_t *ids, const float *wts, int32_t top_k, float *y,
                               int64_t ldy, void *workspace, cudaStream_t stream) {
  if (n_experts > kMaxExperts) return cudaErrorInvalidValue;
  const int P = n_tokens * top_k;
  const PrefillLayout L(n_experts, P, hidden, ffn);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  MoeArgs a = {};
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.ldx = ldx;
  a.ids = ids;
  a.wts = wts;
  a.y = y;
  a.ldy = ldy;
  a.n_experts = n_experts;
  a.n_tokens = n_tokens;
  a.top_k = top_k;
  a.hidden = (int)hidden;
  a.ffn = (int)ffn;
  a.meta = reinterpret_cast<int *>(ws + L.meta);
  a.slot_expert = reinterpret_cast<int *>(ws + L.slot_expert);
  a.slot_start = reinterpret_cast<int *>(ws + L.slot_start);
  a.pair_token = reinterpret_cast<int *>(ws + L.pair_token);
  a.pair_q = reinterpret_cast<int *>(ws + L.pair_q);
  a.tj_pair = reinterpret_cast<int *>(ws + L.tj_pair);
  a.counters = nullptr;
  a.n_counters = 0;
  a.max_slots = L.max_slots;
  a.slot_pairs = kPrefillSlot;
  a.err = device_error_word();
  auto *xs = reinterpret_cast<__nv_bfloat16 *>(ws + L.xs);
  auto *g = reinterpret_cast<__nv_bfloat16 *>(ws + L.g);
  auto *u = reinterpret_cast<__nv_bfloat16 *>(ws + L.u);
  auto *h = reinterpret_cast<__nv_bfloat16 *>(ws + L.h);
  auto *pd = reinterpret_cast<__nv_bfloat16 *>(ws + L.p);
  const DeviceFacts *f = device_facts();

  cudaError_t e = launch_pdl(moe_route_kernel, dim3(1), 1024, 0, stream, a);
  if (e == cudaSuccess) e = launch_pdl(moe_gather_kernel, dim3((unsigned)P), 256, 0, stream, a, xs);
  if (e == cudaSuccess)
    e = launch_gemm_grouped(w_gate, expert_stride, n_experts, ffn, hidden, xs, P, hidden, g, ffn,
                            a.slot_expert, a.slot_start, a.meta, L.max_slots, stream);
  if (e == cudaSuccess)
    e = launch_gemm_grouped(w_up, expert_stride, n_experts, ffn, hidden, xs, P, hidden, u, ffn,
                            a.slot_expert, a.slot_start, a.meta, L.max_slots, stream);
  if (e == cudaSuccess)
    e = launch_pdl(moe_silu_kernel, dim3((unsigned)(8 * f->sm_count)), 256, 0, stream,
                   (const int *)a.meta, (const __nv_bfloat16 *)g, (const __nv_bfloat16 *)u, h,
                   ffn);
  if (e == cudaSuccess)
    e = launch_gemm_grouped(w_down, expert_stride, n_experts, hidden, ffn, h, P, ffn, pd, hidden,
                            a.slot_expert, a.slot_start, a.meta, L.max_slots, stream);
  if (e == cudaSuccess)
    e = launch_pdl(moe_prefill_combine_kernel,
                   dim3((unsigned)((hidden + 255) / 256), (unsigned)n_tokens), 256, 0, stream, a,
                   (const __nv_bfloat16 *)pd);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4k

// ---------------------------------------------------------------------------
// Allocation-free variant.  Its workspace is a file-scope device array of a
// fixed size, so a caller that cannot call cudaMalloc gets a working MoE call
// without handing in memory.  Every GPU that loads the library holds this array
// until the process exits.  All calls on a device share it: it keeps the last
// call's contents, every byte a call reads is first written by that same call
// (nothing needs clearing), and calls that overlap on the GPU race on it.
namespace q4k {

__device__ __align__(256) uint8_t g_moe_scratch[kMoeScratchBytes];

namespace {

void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Host code may not use g_moe_scratch as an address (it names a host-side
// stand-in); the device address is looked up with the device current, on the
// first call made on it.  Only a successful look-up is kept: after a failure
// the next call tries again.
cudaError_t scratch_address(int dev, void **out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_moe_scratch(const void *w_gate, const void *w_up, const void *w_down,
                               int64_t expert_stride, int32_t n_experts, int64_t hidden,
                               int64_t ffn, const void *x, int32_t n_tokens, int64_t ldx,
                               const int32_t *ids, const float *wts, int32_t top_k, float *y,
                               int64_t ldy, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void *scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) return e;
  return launch_moe(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn, x, n_tokens, ldx,
                    ids, wts, top_k, y, ldy, scratch, false, stream);
}

}  // namespace q4k
