// q4k_moe.cu -- routed mixture-of-experts FFN for decode tokens with Q4_K
// experts ("Layer Package Repository Spec", section "Policy Resolution": a
// routed-FFN decode layer is the routed gate/up/down expert matmuls (96% of its
// time), a fused SwiGLU, and the route-weighted sum).
//
// Four launches on the caller's stream:
//   1. route    one CTA groups the T*k (token, slot) pairs by expert (counting
//               sort; experts ordered by id, at most 16 pairs per work slot, so a
//               heavily used expert spans several slots), validates ids (an id
//               out of range is skipped and flagged in the device error word).
//   2. gate/up  per work slot, warp streams of 16-row tiles of ffn: the
//               expert's gate and up rows are streamed once (TMA) and contracted
//               with all of the slot's tokens on the tensor cores (MMA columns =
//               tokens); the epilogue writes h = silu(g) * u in fp32 and as two
//               bf16 columns per pair, h_hi = bf16(h) and h_lo = bf16(h - h_hi)
//               (together 16 significant bits), stored in MMA fragment order.
//   3. down     per work slot, warp streams of 16-row tiles of hidden, full K
//               (ffn) per tile; MMA columns = (h_hi, h_lo) of each pair; the
//               epilogue writes p = Wd h per pair.
//   4. combine  y[t] = sum_j w[t, j] * p[t, j] in slot order j = 0..k-1.
// Grids are sized for the worst case; CTAs whose slot is not in use exit at
// once.  Results do not depend on the order of pairs inside a group (columns of
// an MMA are independent).
#include <algorithm>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

namespace {

constexpr int kRows = 16;                    // rows per CTA (one MMA m-tile)
constexpr int kTile = kRows * kBlockBytes;   // 2304 bytes per super-block stage
constexpr int kStagesMoe = 4;
constexpr int kMoeWarps = 4;                 // warps (weight streams) per expert CTA
constexpr int kMaxExperts = 2048;
constexpr int kSlotPairs = 16;               // pairs per work slot

// Workspace layout (all offsets 256-byte aligned).
struct MoeLayout {
  size_t meta, slot_expert, slot_start, pair_token, tj_pair, g, u, h, h_hi, h_lo, p, total;
  static int max_slots(int E, int P) { return std::min(E, P) + (P + kSlotPairs - 1) / kSlotPairs; }
  MoeLayout(int E, int P, int64_t H, int64_t F) {
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t S = (size_t)max_slots(E, P);
    size_t o = 0;
    meta = o;        o = al(o + 16 * sizeof(int));
    slot_expert = o; o = al(o + S * sizeof(int));
    slot_start = o;  o = al(o + (S + 1) * sizeof(int));
    pair_token = o;  o = al(o + (size_t)P * sizeof(int));
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
  int *meta, *slot_expert, *slot_start, *pair_token, *tj_pair;
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
    act += (cnt[e] + kSlotPairs - 1) / kSlotPairs;
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
    run_a += (cnt[e] + kSlotPairs - 1) / kSlotPairs;
  }
  if (tid == nt - 1) {
    a.meta[0] = run_a;  // work slots in use
    a.meta[1] = run_s;  // valid pairs
  }
  __syncthreads();
  for (int e = tid; e < E; e += nt) {
    for (int q = 0; q * kSlotPairs < cnt[e]; ++q) {
      a.slot_expert[slot_of[e] + q] = e;
      a.slot_start[slot_of[e] + q] = start[e] + q * kSlotPairs;
      a.slot_start[slot_of[e] + q + 1] = min(start[e] + (q + 1) * kSlotPairs, start[e] + cnt[e]);
    }
  }
  for (int q = tid; q < P; q += nt) {
    const int e = a.ids[q];
    if (e >= 0 && e < E) {
      const int pos = start[e] + atomicAdd(&fill[e], 1);
      a.tj_pair[q] = pos;
      a.pair_token[pos] = q / a.top_k;
    }
  }
}

// ---------------------------------------------------------------- 2./3. experts
// One CTA = kMoeWarps warps of work slot blockIdx.y.  Warp stream
// s = blockIdx.x * kMoeWarps + warp takes the slot's 16-row m-tiles s, s + S,
// s + 2S, ... (S = gridDim.x * kMoeWarps), each over the full K; its ring of
// weight stages and its x fragments run ahead continuously across those tiles,
// and each tile's result is written straight from the accumulators.  MMA
// columns are the slot's pairs:
//   gate/up (DOWN = false): column c = x row of the c-th pair's token;
//   down    (DOWN = true):  column 2i = h_hi, column 2i+1 = h_lo of pair i.
// Thread t's k-slots (2t, 2t+1) carry positions (o, o+2) and (2t+8, 2t+9)
// positions (o+1, o+3) of a sub-block, o = 8t + 4s for step s = 0/1: quant
// bytes 8t .. 8t+7 of the sub-block's 32-byte chunk.
// One CTA's work for a slot with at most 8 NT MMA columns.
template <int NT, bool DOWN>
__device__ __forceinline__ void expert_body(const CUtensorMap *map0p, const CUtensorMap *map1p,
                                            const MoeArgs &a, int nsb, int rows_total,
                                            uint8_t *smem, int slot, int ctas) {
  const CUtensorMap &map0 = *map0p, &map1 = *map1p;
  constexpr int NM = DOWN ? 1 : 2;  // weight matrices per stage (gate and up)
  constexpr int kStageBytes = NM * kTile;
  // TMA destinations must be 128-byte aligned: round each warp's region up.
  constexpr int kWarpBytes = (kStagesMoe * kStageBytes + 64 + 127) / 128 * 128;
  const int expert = a.slot_expert[slot];
  const int pstart = a.slot_start[slot];
  const int np = a.slot_start[slot + 1] - pstart;  // pairs of this slot (<= 16)
  const int ncols = DOWN ? 2 * np : np;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ntiles = (rows_total + kRows - 1) / kRows;
  const int sid = blockIdx.x * kMoeWarps + warp, nsid = ctas * kMoeWarps;
  const int ntl = sid < ntiles ? (ntiles - sid + nsid - 1) / nsid : 0;  // tiles of this warp
  const int total = ntl * nsb;                                          // ring iterations
  uint8_t *ring = smem + warp * kWarpBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kStagesMoe * kStageBytes);

  if (lane == 0) {
    prefetch_tmap(&map0);
    if (NM == 2) prefetch_tmap(&map1);
    for (int s = 0; s < kStagesMoe; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  // Ring iteration q = super-block q % nsb of this warp's tile q / nsb.
  auto issue = [&](int q) {
    const int j = q / nsb, u = q - j * nsb;
    const int row0 = (sid + j * nsid) * kRows;
    const int stage = q % kStagesMoe;
    mbar_arrive_expect_tx(&bars[stage], kStageBytes);
    uint8_t *dst = ring + stage * kStageBytes;
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
        dst[jj][nt] = (cval[nt] && q < total)
                          ? __ldg(reinterpret_cast<const uint4 *>(src[nt] + off))
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
      const int stage = q % kStagesMoe;
      if (!mbar_wait(&bars[stage], (uint32_t)((q / kStagesMoe) & 1), a.err)) {
        ok = false;
        if (lane == 0) {  // let this warp's copies in flight land (bounded)
          const uint64_t t0 = global_ns();
          for (int r = q; r < min(q + kStagesMoe, total); ++r)
            while (!mbar_try_wait(&bars[r % kStagesMoe], (uint32_t)((r / kStagesMoe) & 1), 1000u))
              if (global_ns() - t0 > kWaitLimitNs) break;
        }
        break;
      }
      const uint8_t *st = ring + stage * kStageBytes;
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
        uint32_t sub[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t sc2, m2;
          scales_pair(hdr[mi][r].y, hdr[mi][r].z, hdr[mi][r].w, t, &sc2, &m2);
          const float d = half_lo_to_float(hdr[mi][r].x), dmin = half_hi_to_float(hdr[mi][r].x);
          const float nd23 = d * -8388608.f, ndm23 = dmin * -8388608.f;
#pragma unroll
          for (int e = 0; e < 2; ++e)
            offset_form(d, nd23, dmin, ndm23, byte_magic(sc2, e), byte_magic(m2, e),
                        dsv[mi][r][e], eev[mi][r][e], sub[r][e]);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) subp[mi][e] = __byte_perm(sub[0][e], sub[1][e], 0x5410u);
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
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float &yv = yacc[mi][nt][2 * r + e];
                yv = fmaf(ds, acc[nt][2 * r + e], yv);
                yv = fmaf(ee, xsum[nt][e], yv);
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
            const __nv_bfloat16 hh = __float2bfloat16_rn(hv);
            const __nv_bfloat16 hl = __float2bfloat16_rn(hv - __bfloat162float(hh));
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
}

// The MMA width follows the slot: 8 columns when its pairs fit, else 16 or 32
// (NTMAX n-tiles of 8 at most), so a slot with few pairs does no work for
// empty columns.  A slot with nt n-tiles gets nt times the warp streams (each
// with 1/nt of the row tiles), so every stream does about the same work; the
// grid is sized for the widest class (one tile per stream at NTMAX) and the
// CTAs a slot does not need exit.  The choice is uniform per CTA.
template <int NTMAX, bool DOWN>
__global__ void __launch_bounds__(kMoeWarps * 32) moe_expert_kernel(
    const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
    const MoeArgs a, int nsb, int rows_total) {
  extern __shared__ __align__(128) uint8_t smem[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int slot = blockIdx.y;
  if (slot >= a.meta[0]) return;  // slot not in use
  const int np = a.slot_start[slot + 1] - a.slot_start[slot];
  const int ncols = DOWN ? 2 * np : np;
  const int nt = ncols <= 8 ? 1 : ncols <= 16 ? 2 : 4;  // n-tiles this slot needs
  const int ctas = (int)gridDim.x * min(nt, NTMAX) / NTMAX;  // CTAs of this slot
  if ((int)blockIdx.x >= ctas) return;
  if (nt == 1 || NTMAX == 1)
    expert_body<1, DOWN>(&map0, &map1, a, nsb, rows_total, smem, slot, ctas);
  else if (nt == 2 || NTMAX == 2)
    expert_body<(NTMAX >= 2 ? 2 : 1), DOWN>(&map0, &map1, a, nsb, rows_total, smem, slot, ctas);
  else
    expert_body<NTMAX, DOWN>(&map0, &map1, a, nsb, rows_total, smem, slot, ctas);
}

// ---------------------------------------------------------------- 4. combine
__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.hidden) return;
  float acc = 0.f;
  for (int j = 0; j < a.top_k; ++j) {
    const int q = t * a.top_k + j;
    const int pos = a.tj_pair[q];
    if (pos >= 0) acc = fmaf(a.wts[q], a.p[(size_t)pos * a.hidden + i], acc);
  }
  a.y[(int64_t)t * a.ldy + i] = acc;
}

std::once_flag g_moe_attr[kMaxDevices];  // cudaFuncSetAttribute acts on the current device

// Launch as a programmatic dependent of the previous kernel on the stream.
template <typename K, typename... Args>
void launch_pdl(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t stream, Args... args) {
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
  cudaLaunchKernelEx(&cfg, kernel, args...);
}
#ifndef Q4K_MOE_GU_TILES  // gate/up: m-tiles per warp stream
#define Q4K_MOE_GU_TILES 2
#endif
#ifndef Q4K_MOE_DN_TILES  // down: m-tiles per warp stream
#define Q4K_MOE_DN_TILES 4
#endif
constexpr int kGuTiles = Q4K_MOE_GU_TILES;
constexpr int kDnTiles = Q4K_MOE_DN_TILES;

template <int NT, bool DOWN>
constexpr int expert_smem() {
  return kMoeWarps * ((kStagesMoe * (DOWN ? 1 : 2) * kTile + 64 + 127) / 128 * 128);
}

template <int NT, bool DOWN>
void allow() {
  cudaFuncSetAttribute(moe_expert_kernel<NT, DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       expert_smem<NT, DOWN>());
}

void moe_attributes() {
  allow<1, false>();
  allow<2, false>();
  allow<1, true>();
  allow<2, true>();
  allow<4, true>();
}

// tiles_per_warp: row tiles per warp stream of an 8-column slot; a slot with
// nt n-tiles has nt times the streams.  The grid holds NT times the streams
// of an 8-column slot, rounded to a multiple of NT CTAs.
template <int NT, bool DOWN>
void launch_expert(int rows, int tiles_per_warp, int max_slots, const CUtensorMap &m0,
                   const CUtensorMap &m1, const MoeArgs &a, int nsb, cudaStream_t stream) {
  const int ntiles = (rows + kRows - 1) / kRows;
  const int per_cta = kMoeWarps * tiles_per_warp;
  const int base = (ntiles + per_cta - 1) / per_cta;  // CTAs of an 8-column slot
  dim3 grid((unsigned)(base * NT), (unsigned)max_slots);
  launch_pdl(moe_expert_kernel<NT, DOWN>, grid, kMoeWarps * 32, (size_t)expert_smem<NT, DOWN>(),
             stream, m0, m1, a, nsb, rows);
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
                       cudaStream_t stream) {
  if (n_experts > kMaxExperts) return cudaErrorInvalidValue;
  std::call_once(g_moe_attr[device_facts()->device], moe_attributes);
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
  a.slot_expert = reinterpret_cast<int *>(ws + L.slot_expert);
  a.slot_start = reinterpret_cast<int *>(ws + L.slot_start);
  a.pair_token = reinterpret_cast<int *>(ws + L.pair_token);
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

  launch_pdl(moe_route_kernel, dim3(1), 1024, 0, stream, a);
  const int max_slots = MoeLayout::max_slots(n_experts, P);
  const int cap = std::min(P, kSlotPairs);  // pairs per slot at most
  {  // gate/up: K = hidden, one column per pair
    const int nsb = (int)(hidden / kQK);
    if (cap <= 8)
      launch_expert<1, false>((int)ffn, kGuTiles, max_slots, mg, mu, a, nsb, stream);
    else
      launch_expert<2, false>((int)ffn, kGuTiles, max_slots, mg, mu, a, nsb, stream);
  }
  {  // down: K = ffn, two columns per pair
    const int nsb = (int)(ffn / kQK);
    if (2 * cap <= 8)
      launch_expert<1, true>((int)hidden, kDnTiles, max_slots, md, md, a, nsb, stream);
    else if (2 * cap <= 16)
      launch_expert<2, true>((int)hidden, kDnTiles, max_slots, md, md, a, nsb, stream);
    else
      launch_expert<4, true>((int)hidden, kDnTiles, max_slots, md, md, a, nsb, stream);
  }
  {
    dim3 grid((unsigned)((hidden + 255) / 256), (unsigned)n_tokens);
    launch_pdl(moe_combine_kernel, grid, 256, 0, stream, a);
  }
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
                    ids, wts, top_k, y, ldy, scratch, stream);
}

}  // namespace q4k
