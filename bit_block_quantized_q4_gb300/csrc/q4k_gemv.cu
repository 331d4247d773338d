// q4k_gemv.cu -- batched decode projection Y[b] = W X[b] for batch 2..16 with W
// in Q4_K, and the fused gate/up projection H[b] = silu(Wg X[b]) * (Wu X[b])
// at the same batch sizes ("spec: specialized model runtimes", sections
// "Architecture" (T0 GEMM) and "Development sequence" (decode throughput);
// batched decode steps: "PRD: Performant Concurrent Distributed GGUF Runtime",
// DGR-012; merged gate/up: "Layer Package Repository Spec", section "Policy
// Resolution").  Batch 1 runs in q4k_stream.cu.
//
// The weights are streamed from HBM exactly once and contracted with all batch
// rows.  Each warp owns 16*MT output rows and a contiguous slice of
// super-blocks; a private ring of shared-memory stages is filled by TMA (one
// 2-D box = 16*MT rows x one 144-byte super-block, per weight matrix).  The
// contraction runs on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32
// accumulate) with the MMA columns = batch rows (one or two n-tiles of 8) and
// every sub-block its own two-step accumulation.  Sub-block j of a row is
// taken in offset form (offset_form): the A operand is the exact small integer
// q - c in bf16, and per (row, sub-block, column) the epilogue adds
// ds * sum (q - c) x + e * X_j, X_j the column's sum of x over the sub-block
// (two MMAs with A = 1).  Each lane decodes the offset forms of sub-blocks 2t,
// 2t+1 of its rows g, g+8; the other lanes of its quad fetch them by shuffle.
// The x fragments are loaded from L2 half a super-block ahead of their use.
//
// Split-K: the warps of a CTA take consecutive super-block slices of the same
// rows; partial sums meet in shared memory and are added in warp order, so the
// result is deterministic.  Grids are sized so that every CTA is resident at
// once (one wave) whenever the shape allows.  With programmatic dependent
// launch (Q4K_FLAG_OVERLAP_WEIGHTS) the first weight stages are requested
// before the wait for the previous kernel; x only after it.
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <unordered_map>

#include "q4k_device.cuh"
#include "q4k_internal.h"

// Tuning knobs (compile time).
#ifndef Q4K_GEMV_STAGES
#define Q4K_GEMV_STAGES 4
#endif
#ifndef Q4K_GEMV_PROMO  // L2 promotion of the weight tensor map: 0 none, 1 128 B, 2 256 B
#define Q4K_GEMV_PROMO 2
#endif
#ifndef Q4K_GEMV_EVICT_FIRST  // L2 evict-first hint on weight loads
#define Q4K_GEMV_EVICT_FIRST 1
#endif
#ifndef Q4K_GEMV_INFLIGHT_KB  // planner: weight bytes in flight per SM worth having, at most
#define Q4K_GEMV_INFLIGHT_KB 96
#endif
#ifndef Q4K_GEMV_BN_MT2_COST  // per-row cost of an MT = 2 warp relative to MT = 1
#define Q4K_GEMV_BN_MT2_COST 0.8
#endif
#ifndef Q4K_GEMV_FORCE_MT
#define Q4K_GEMV_FORCE_MT 0
#endif

namespace q4k {

namespace {

constexpr int kRowsPerTile = 16;
constexpr int kTileBytes = kRowsPerTile * kBlockBytes;  // 2304, a multiple of 128
constexpr int kStages = Q4K_GEMV_STAGES;

struct GemvArgs {
  const __nv_bfloat16 *x;
  float *y;
  int64_t ldx, ldy;
  int n;           // rows
  int nsb;         // super-blocks per row
  int ks;          // super-blocks per warp
  int batch;
  int warp_bytes;  // shared bytes per warp region
  unsigned *err;   // device error word
};

// W is viewed as a 2-D array of 8-byte elements, [n rows][nsb * 18]; one box
// covers one super-block (144 contiguous bytes) of 16*MT rows.
__device__ __forceinline__ void load_tile(void *dst, const CUtensorMap *map, uint64_t *bar, int sb,
                                          int row0, uint64_t policy) {
#if Q4K_GEMV_EVICT_FIRST
  tma_load_2d_hint(dst, map, bar, sb * (kBlockBytes / 8), row0, policy);
#else
  (void)policy;
  tma_load_2d(dst, map, bar, sb * (kBlockBytes / 8), row0);
#endif
}

// After a timed-out wait: give the ring iterations it .. end-1 still in
// flight the same bounded time to land before the CTA exits.
__device__ __noinline__ void drain_bn(uint64_t *bars, int stages, int it, int end) {
  const uint64_t t0 = global_ns();
  for (int j = it; j < end; ++j)
    while (!mbar_try_wait(&bars[j % stages], (j / stages) & 1, 1000u))
      if (global_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

// MMA columns = batch rows (NT n-tiles of 8).  Sub-block j = 2c+hi, step s:
// thread t's k-slots (2t, 2t+1) carry positions (o, o+2) and (2t+8, 2t+9)
// positions (o+1, o+3), o = 8t + 4s, i.e. quant bytes 8t .. 8t+7 of chunk c.
// NM = 2: a stage holds the gate tile then the up tile of the same rows and
// the result is silu(gate) * up.
template <int MT, int NT, int NM, int STAGES>
__global__ void __launch_bounds__(256) gemv_bn_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const __grid_constant__ CUtensorMap umap,
                                                      const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kStageBytes = NM * MT * kTileBytes;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * (MT * kRowsPerTile);
  const int sb0 = warp * a.ks;
  const int nsteps = max(0, min(a.nsb, sb0 + a.ks) - sb0);
  constexpr int kCols = NT * 8;

  uint8_t *ring = smem + (size_t)warp * a.warp_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + STAGES * kStageBytes);
  float *red = reinterpret_cast<float *>(smem + (size_t)nwarps * a.warp_bytes);

  if (lane == 0) {
    prefetch_tmap(&wmap);
    if (NM == 2) prefetch_tmap(&umap);
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int s, int sb) {
    mbar_arrive_expect_tx(&bars[s], kStageBytes);
    uint8_t *dst = ring + s * kStageBytes;
    load_tile(dst, &wmap, &bars[s], sb, row0, policy);
    if (NM == 2) load_tile(dst + MT * kTileBytes, &umap, &bars[s], sb, row0, policy);
  };
  if (lane == 0)
    for (int s = 0; s < STAGES && s < nsteps; ++s) issue(s, sb0 + s);
  grid_dependency_wait();
  grid_launch_dependents();
  // x rows of this lane's batch columns (g and g+8); rows past the batch read
  // zeros.
  const uint4 *xrow[NT];
  bool xval[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int b = nt * 8 + g;
    xval[nt] = b < a.batch;
    xrow[nt] = reinterpret_cast<const uint4 *>(a.x + (int64_t)(xval[nt] ? b : 0) * a.ldx);
  }

  float yacc[NM][MT][NT][4];
#pragma unroll
  for (int mi = 0; mi < NM; ++mi)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        yacc[mi][mt][nt][0] = yacc[mi][mt][nt][1] = yacc[mi][mt][nt][2] = yacc[mi][mt][nt][3] = 0.f;

  // x of half a super-block (sub-blocks 4h .. 4h+3) for this lane's batch
  // columns, loaded one half ahead of its use (L2 latency off the MMA path).
  auto load_x_half = [&](uint4(&dst)[4][NT], int i, int h) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        dst[jj][nt] = (xval[nt] && i < nsteps)
                          ? __ldg(xrow[nt] + ((int64_t)(sb0 + i) * kQK + 32 * (4 * h + jj) + 8 * t) / 8)
                          : make_uint4(0, 0, 0, 0);
  };
  uint4 xA[4][NT], xB[4][NT];
  load_x_half(xA, 0, 0);

  bool ok = true;
  for (int i = 0; i < nsteps; ++i) {
    const int stage = i % STAGES;
    const int sb = sb0 + i;
    if (!mbar_wait(&bars[stage], (uint32_t)((i / STAGES) & 1), a.err)) {
      ok = false;
      if (lane == 0) drain_bn(bars, STAGES, i, min(i + STAGES, nsteps));
      break;
    }
    const uint8_t *st = ring + stage * kStageBytes;
    uint4 hdr[NM][MT][2];
    uint2 qw[NM][MT][2][4];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t *rp = st + ((mi * MT + mt) * kRowsPerTile + g + 8 * r) * kBlockBytes;
          hdr[mi][mt][r] = *reinterpret_cast<const uint4 *>(rp);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            qw[mi][mt][r][c] = *reinterpret_cast<const uint2 *>(rp + kQsOffset + 32 * c + 8 * t);
        }
    __syncwarp();
    if (lane == 0 && i + STAGES < nsteps) issue(stage, sb + STAGES);
    load_x_half(xB, i, 1);
    // Offset forms of sub-blocks 2t, 2t+1 (e = 0, 1) of rows g, g+8 (r = 0, 1);
    // the bf16 subtrahends of both rows travel packed in one word per e.
    float dsv[NM][MT][2][2], eev[NM][MT][2][2];
    uint32_t subp[NM][MT][2];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t sc2[2], m2[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint4 h = hdr[mi][mt][r];
          scales_pair(h.y, h.z, h.w, t, &sc2[r], &m2[r]);
        }
        // rows g, g+8 as the two lanes of the packed fp32 operations
        float2 d2, nd23, dmin2, pdm23;
        scale_pairs(hdr[mi][mt][0].x, hdr[mi][mt][1].x, d2, nd23, dmin2, pdm23);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float2 ds2, ee2;
          offset_form_rows2_packed<16>(d2, nd23, dmin2, pdm23, byte_magic(sc2[0], e),
                                       byte_magic(sc2[1], e), byte_magic_neg(m2[0], e),
                                       byte_magic_neg(m2[1], e), ds2, ee2, subp[mi][mt][e]);
          dsv[mi][mt][0][e] = ds2.x;
          dsv[mi][mt][1][e] = ds2.y;
          eev[mi][mt][0][e] = ee2.x;
          eev[mi][mt][1][e] = ee2.y;
        }
      }
    auto sub_block = [&](int j, const uint4(&xv)[NT]) {
      const int c = j >> 1;
      const bool hi = j & 1;
      uint32_t b0[2][NT], b1[2][NT];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t lo = s ? xv[nt].z : xv[nt].x;
          const uint32_t hi2 = s ? xv[nt].w : xv[nt].y;
          b0[s][nt] = __byte_perm(lo, hi2, 0x5410);
          b1[s][nt] = __byte_perm(lo, hi2, 0x7632);
        }
      // X_j of every column (A = 1 everywhere: every row holds it, so column
      // 2t+e is xsum[nt][e]).
      float xsum[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_zc(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[0][nt], b1[0][nt]);
        mma_bf16(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[1][nt], b1[1][nt]);
      }
      // Offset forms of sub-block j for rows g, g+8 live in lane (g, j/2).
      const int src = (lane & ~3) | (j >> 1);
#pragma unroll
      for (int mi = 0; mi < NM; ++mi)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t sp = __shfl_sync(0xffffffffu, hi ? subp[mi][mt][1] : subp[mi][mt][0], src);
          const uint32_t sg = __byte_perm(sp, 0u, 0x1010u), sg8 = __byte_perm(sp, 0u, 0x3232u);
          float acc[NT][4];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint32_t w0 = s ? qw[mi][mt][0][c].y : qw[mi][mt][0][c].x;
            const uint32_t w1 = s ? qw[mi][mt][1][c].y : qw[mi][mt][1][c].x;
            const uint32_t a0 = sub_bf16x2(hi ? nib_hi(w0) : nib_lo(w0), sg);
            const uint32_t a1 = sub_bf16x2(hi ? nib_hi(w1) : nib_lo(w1), sg8);
            const uint32_t a2 = sub_bf16x2(hi ? nib_hi(w0 >> 8) : nib_lo(w0 >> 8), sg);
            const uint32_t a3 = sub_bf16x2(hi ? nib_hi(w1 >> 8) : nib_lo(w1 >> 8), sg8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (s == 0)
                mma_bf16_zc(acc[nt], a0, a1, a2, a3, b0[0][nt], b1[0][nt]);
              else
                mma_bf16(acc[nt], a0, a1, a2, a3, b0[1][nt], b1[1][nt]);
            }
          }
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float ds = __shfl_sync(0xffffffffu, hi ? dsv[mi][mt][r][1] : dsv[mi][mt][r][0], src);
            const float ee = __shfl_sync(0xffffffffu, hi ? eev[mi][mt][r][1] : eev[mi][mt][r][0], src);
            // columns 2t, 2t+1 share ds and e: one packed fma each (each lane
            // of a pair rounds as fmaf)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float2 yv = make_float2(yacc[mi][mt][nt][2 * r], yacc[mi][mt][nt][2 * r + 1]);
              yv = __ffma2_rn(make_float2(ds, ds), make_float2(acc[nt][2 * r], acc[nt][2 * r + 1]), yv);
              yv = __ffma2_rn(make_float2(ee, ee), make_float2(xsum[nt][0], xsum[nt][1]), yv);
              yacc[mi][mt][nt][2 * r] = yv.x;
              yacc[mi][mt][nt][2 * r + 1] = yv.y;
            }
          }
        }
    };
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sub_block(jj, xA[jj]);
    load_x_half(xA, i + 1, 0);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sub_block(4 + jj, xB[jj]);
  }

  // Across warps: red[warp][matrix][row][col].
  const int tile_rows = MT * kRowsPerTile;
#pragma unroll
  for (int mi = 0; mi < NM; ++mi)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = mt * kRowsPerTile + g + 8 * (e >> 1);
          const int col = nt * 8 + 2 * t + (e & 1);
          red[((warp * NM + mi) * tile_rows + row) * kCols + col] = yacc[mi][mt][nt][e];
        }
  __syncwarp();
  if (!ok && lane == 0) red[(warp * NM * tile_rows) * kCols] = __int_as_float(0x7fc00000);
  __syncthreads();
  for (int idx = threadIdx.x; idx < tile_rows * kCols; idx += blockDim.x) {
    const int row = idx / kCols, col = idx % kCols;
    float s0 = 0.f, s1 = 0.f;
    for (int w = 0; w < nwarps; ++w) {
      s0 += red[((w * NM) * tile_rows + row) * kCols + col];
      if (NM == 2) s1 += red[((w * NM + 1) * tile_rows + row) * kCols + col];
    }
    const int grow = row0 + row;
    if (grow < a.n && col < a.batch) a.y[(int64_t)col * a.ldy + grow] = NM == 2 ? silu_mul(s0, s1) : s0;
  }
}

// ---------------------------------------------------------------- launch
struct Plan {
  int mt = 1, wk = 1, ks = 1, warp_bytes = 0, smem = 0, grid = 0;
  double score = -1e30;
};

int warp_bytes_bn(int mt, int nm) {
  int b = kStages * nm * mt * kTileBytes + kStages * 8;
  return (b + 127) / 128 * 128;
}

template <typename K>
int occupancy(K kernel, int threads, int smem) {
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess)
    return 0;
  return blocks;
}

// 8 columns: choose how K is split across the warps of a CTA so that every CTA
// is resident at once (one wave); among those plans prefer more weight bytes
// in flight per SM (latency hiding), then an even split.
template <typename K>
Plan plan_for(K kernel, int mt, int nm, int n, int nsb, int cols, const DeviceFacts *f) {
  Plan best;
  const int tile_rows = mt * kRowsPerTile;
  const int grid = (n + tile_rows - 1) / tile_rows;
  for (int wk = 1; wk <= 8; ++wk) {
    int ks = (nsb + wk - 1) / wk;
    if ((nsb + ks - 1) / ks != wk) continue;  // no empty warps
    if (ks < 2 && nsb >= 2) continue;
    const int wb = warp_bytes_bn(mt, nm);
    const int smem = wk * wb + wk * nm * tile_rows * cols * 4;
    if (smem > f->max_smem_optin) continue;
    const int occ = occupancy(kernel, wk * 32, smem);
    if (occ <= 0) continue;
    const int slots = occ * f->sm_count;
    const int waves = (grid + slots - 1) / slots;
    const int per_sm = std::min(occ, (grid + f->sm_count - 1) / f->sm_count);
    const int warps_sm = per_sm * wk;
    const double inflight_kb = warps_sm * (kStages - 1) * nm * mt * kTileBytes / 1024.0;
    const double balance = (double)nsb / (double)(ks * wk);  // 1.0 = even split
    const double score = -1000.0 * waves + std::min(inflight_kb, (double)Q4K_GEMV_INFLIGHT_KB) / 8.0 +
                         0.5 * std::min(warps_sm, 24) + 6.0 * balance + (mt == 2 ? 1.0 : 0.0);
    if (score > best.score) {
      best.score = score;
      best.mt = mt;
      best.wk = wk;
      best.ks = ks;
      best.warp_bytes = wb;
      best.smem = smem;
      best.grid = grid;
    }
  }
  return best;
}

// 16 columns: every CTA resident at once; among those plans take the smallest
// load of the busiest SM: ceil(CTAs / SMs) x warps per CTA x super-blocks per
// warp x rows per warp (an MT = 2 warp shares its x fragments between its two
// row tiles, taken as 0.8 of MT = 1's cost per row), plus a penalty for fewer
// than 8 resident warps per SM.
template <typename K>
Plan plan_bn(K kernel, int mt, int nm, int n, int nsb, int cols, const DeviceFacts *f) {
  Plan best;
  const int tile_rows = mt * kRowsPerTile;
  const int tiles = (n + tile_rows - 1) / tile_rows;
  for (int wk = 1; wk <= 8; ++wk) {
    const int ks = (nsb + wk - 1) / wk;
    if ((nsb + ks - 1) / ks != wk) continue;  // every warp gets super-blocks
    const int wb = warp_bytes_bn(mt, nm);
    const int smem = wk * wb + wk * nm * tile_rows * cols * 4;
    if (smem > f->max_smem_optin) continue;
    const int occ = occupancy(kernel, wk * 32, smem);
    if (occ <= 0) continue;
    if (tiles > occ * f->sm_count) continue;  // one wave
    const long per_sm = (tiles + f->sm_count - 1) / f->sm_count;
    const long warps_sm = per_sm * wk;
    double load = (double)per_sm * wk * ks * mt * nm * (mt == 2 ? Q4K_GEMV_BN_MT2_COST : 1.0);
    if (warps_sm < 8) load *= 1.0 + 0.08 * (8 - warps_sm);
    if (-load > best.score) {
      best.score = -load;
      best.mt = mt;
      best.wk = wk;
      best.ks = ks;
      best.warp_bytes = wb;
      best.smem = smem;
      best.grid = tiles;
    }
  }
  if (best.grid == 0) {  // more tiles than one wave holds: the plan with the most in flight
    Plan p = plan_for(kernel, mt, nm, n, nsb, cols, f);
    if (p.grid) return p;
  }
  return best;
}

std::once_flag g_attr_once[kMaxDevices];  // cudaFuncSetAttribute acts on the current device

using GemvKernel = void (*)(CUtensorMap, CUtensorMap, GemvArgs);

template <int MT, int NT, int NM>
constexpr GemvKernel bn_kernel() {
  return gemv_bn_kernel<MT, NT, NM, kStages>;
}

void set_attributes(const DeviceFacts *f) {
  const GemvKernel ks[] = {bn_kernel<1, 1, 1>(), bn_kernel<1, 2, 1>(), bn_kernel<2, 1, 1>(),
                           bn_kernel<2, 2, 1>(), bn_kernel<1, 1, 2>(), bn_kernel<1, 2, 2>()};
  for (GemvKernel k : ks)
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, f->max_smem_optin);
}

GemvKernel bn_select(int mt, int nt, int nm) {
  if (nm == 2) return nt == 1 ? bn_kernel<1, 1, 2>() : bn_kernel<1, 2, 2>();
  if (mt == 2) return nt == 1 ? bn_kernel<2, 1, 1>() : bn_kernel<2, 2, 1>();
  return nt == 1 ? bn_kernel<1, 1, 1>() : bn_kernel<1, 2, 1>();
}

// Plans depend only on (device, N, K, column tiles, matrices), so they are kept
// per process.  Bounded: the cache is cleared when it reaches kMaxPlans entries.
struct PlanKey {
  int dev, n, nsb, cls;
  bool operator==(const PlanKey &o) const {
    return dev == o.dev && n == o.n && nsb == o.nsb && cls == o.cls;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey &k) const {
    uint64_t h = (uint64_t)(uint32_t)k.n * 0x9E3779B97F4A7C15ull;
    h ^= ((uint64_t)(uint32_t)k.nsb << 20) ^ ((uint64_t)k.dev << 52) ^ ((uint64_t)k.cls << 44);
    return (size_t)(h ^ (h >> 29));
  }
};
constexpr size_t kMaxPlans = 4096;
std::mutex g_plan_mu;
std::unordered_map<PlanKey, Plan, PlanKeyHash> g_plans;

template <typename F>
Plan cached_plan(const PlanKey &key, F compute) {
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) return it->second;
  }
  const Plan p = compute();
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (g_plans.size() >= kMaxPlans) g_plans.clear();
  g_plans.emplace(key, p);
  return p;
}

}  // namespace

cudaError_t launch_gemv(const void *w, const void *w_up, int64_t n, int64_t k, const void *x,
                        int64_t batch, int64_t ldx, float *y, int64_t ldy, bool overlap,
                        cudaStream_t stream) {
  const DeviceFacts *f = device_facts();
  std::call_once(g_attr_once[f->device], set_attributes, f);
  const int nsb = (int)(k / kQK);
  const int nm = w_up ? 2 : 1;
  const int nt = batch <= 8 ? 1 : 2;

  // W viewed as [n rows][nsb super-blocks][144 bytes]; one box = 16*mt rows
  // of one super-block.
  auto encode = [&](CUtensorMap *map, const void *base, int mt) {
    const uint64_t dims[2] = {(uint64_t)nsb * (kBlockBytes / 8), (uint64_t)n};
    const uint64_t strides[1] = {(uint64_t)nsb * kBlockBytes};
    const uint32_t box[2] = {(uint32_t)(kBlockBytes / 8), (uint32_t)(mt * kRowsPerTile)};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims,
                        strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                        Q4K_GEMV_PROMO == 0   ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                        : Q4K_GEMV_PROMO == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                              : CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  };

  const Plan p = cached_plan(PlanKey{f->device, (int)n, nsb, 4 * nm + nt}, [&] {
    Plan best;
    for (int mt = 1; mt <= (nm == 2 ? 1 : 2); ++mt) {  // the gate/up kernel keeps 16-row tiles
      if (Q4K_GEMV_FORCE_MT && mt != Q4K_GEMV_FORCE_MT && nm == 1) continue;
      // Measured on the 64-layer pass: the busiest-SM load objective wins at
      // 16 columns, the in-flight score at 8.
      const Plan q = nt == 2 ? plan_bn(bn_select(mt, nt, nm), mt, nm, (int)n, nsb, nt * 8, f)
                             : plan_for(bn_select(mt, nt, nm), mt, nm, (int)n, nsb, nt * 8, f);
      if (q.grid && q.score > best.score) best = q;
    }
    return best;
  });
  if (p.grid == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap wmap, umap;
  if (encode(&wmap, w, p.mt) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (nm == 2) {
    if (encode(&umap, w_up, p.mt) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    umap = wmap;
  }
  GemvArgs args = {};
  args.x = static_cast<const __nv_bfloat16 *>(x);
  args.y = y;
  args.ldx = ldx;
  args.ldy = ldy;
  args.n = (int)n;
  args.nsb = nsb;
  args.batch = (int)batch;
  args.err = device_error_word();
  args.ks = p.ks;
  args.warp_bytes = p.warp_bytes;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)(p.wk * 32), 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, bn_select(p.mt, nt, nm), wmap, umap, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4k
