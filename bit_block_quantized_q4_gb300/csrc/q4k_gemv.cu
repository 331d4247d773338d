// q4k_gemv.cu -- decode projection Y[b] = W X[b] for batch 1..16 with W in
// Q4_K ("spec: specialized model runtimes", sections "Architecture" (T0 GEMM,
// quant/dequant) and "Development sequence" (decode throughput); batched decode
// steps: "PRD: Performant Concurrent Distributed GGUF Runtime", DGR-012).
//
// The weights are streamed from HBM exactly once.  Each warp owns 16*MT output
// rows and a contiguous slice of super-blocks; a private ring of shared-memory
// stages is filled by TMA (one 2-D box = 16*MT rows x S 144-byte super-blocks
// per stage).  The contraction runs on the tensor cores (mma.sync m16n8k16,
// fp32 accumulate) in the factored form
//     sum_i (d sc_j q_i - dmin m_j) x_i = d sc_j S_j - dmin m_j X_j,
// S_j = sum_i q_i x_i, X_j = sum_i x_i over sub-block j, with the scales
// applied in fp32 once per (row, sub-block, batch column).
//
// Batch 1 (fp16 operands): each warp copies its x slice into shared memory with
// one bulk copy and converts it in place, per 256-value super-block, to fp16
// scaled by a power of two 2^s (largest magnitude in [2^14, 2^15): exact for
// every value within 2^28 of that maximum), plus -1024 X_j from two MMAs with a
// constant A operand; the weight MMAs start their accumulators there.  A quant
// becomes the fp16 value 1024+q (low nibble) or 1024+16q (high nibble) with
// one LOP3.  The eight MMA columns carry the eight sub-blocks of a super-block
// (column j of B holds x only in the k-slots that carry sub-block j), so one
// super-block needs 16 MMAs per 16 rows and each thread ends with exactly the
// (row, sub-block) sums whose scales it decodes itself; each super-block's
// contribution is multiplied by 2^-s before it joins the row sum.
// Batch 2..16 (bf16 operands): a quant becomes the bf16 value 128+q (exact);
// the MMA columns carry the batch rows (one or two n-tiles of 8); every
// sub-block is its own 2-step accumulation, -128 X_j comes from the same MMA
// path with a constant A = -128 (so an all-zero sub-block cancels exactly; with
// one column tile it seeds the weight MMAs), and the scales are shared within a
// thread quad by shuffles.  The x fragments are
// loaded from L2 half a super-block ahead of their use.
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
#include <vector>

#include "q4k_device.cuh"
#include "q4k_internal.h"

// Tuning knobs (compile time).
#ifndef Q4K_GEMV_STAGES
#define Q4K_GEMV_STAGES 4
#endif
#ifndef Q4K_GEMV_PROMO  // L2 promotion of the weight tensor map: 0 none, 1 128 B, 2 256 B
#define Q4K_GEMV_PROMO 2
#endif
#ifndef Q4K_GEMV_PRE_STAGES  // batch 1: weight stages issued before x and the dependency wait
#define Q4K_GEMV_PRE_STAGES 2
#endif
#ifndef Q4K_GEMV_EVICT_FIRST  // L2 evict-first hint on weight loads
#define Q4K_GEMV_EVICT_FIRST 1
#endif

namespace q4k {

namespace {

constexpr int kRowsPerTile = 16;
constexpr int kTileBytes = kRowsPerTile * kBlockBytes;  // 2304, a multiple of 128

struct GemvArgs {
  const uint8_t *w;      // weights (row-major super-blocks)
  int64_t row_bytes;     // bytes per weight row
  const __nv_bfloat16 *x;
  float *y;
  int64_t ldx, ldy;
  int n;        // rows
  int nsb;      // super-blocks per row
  int ks;       // super-blocks per warp
  int batch;
  int warp_bytes;  // shared bytes per warp region
  unsigned *err;   // device error word
  int pre;         // batch 1: weight stages issued before the dependency wait
};

// W is viewed as a 2-D array of 8-byte elements, [n rows][nsb * 18]; one box
// covers S super-blocks (S * 144 contiguous bytes) of 16*MT rows.
__device__ __forceinline__ void load_tile(void *dst, const CUtensorMap *map, uint64_t *bar, int sb,
                                          int row0, uint64_t policy) {
#if Q4K_GEMV_EVICT_FIRST
  tma_load_2d_hint(dst, map, bar, sb * (kBlockBytes / 8), row0, policy);
#else
  (void)policy;
  tma_load_2d(dst, map, bar, sb * (kBlockBytes / 8), row0);
#endif
}

// Count rounded up to a multiple of 4 (keeps what follows an fp32 array of
// that many entries on a 16-byte boundary).
__host__ __device__ __forceinline__ int pad4(int n) { return (n + 3) & ~3; }

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Lane constants of the batch-1 scale/min decode (sub-blocks 2t, 2t+1).
struct B1Lane {
  bool upper;     // t >= 2: sub-blocks 4..7
  uint32_t psel;  // PRMT selector gathering bytes k0, k0+1 of rows g and g+8
  uint32_t mlo4, mhi4;
};

__device__ __forceinline__ B1Lane b1_lane(int t) {
  B1Lane l;
  l.upper = t >= 2;
  const uint32_t k0 = 2 * (t & 1);  // byte of sub-block 2t within its word
  l.psel = k0 | ((k0 + 1) << 4) | ((k0 + 4) << 8) | ((k0 + 5) << 12);
  l.mlo4 = l.upper ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
  l.mhi4 = l.upper ? 0x30303030u : 0u;
  return l;
}

// One super-block of 16*MT rows for batch 1: hdr/qa hold the two rows (g, g+8)
// of each m-tile (header; quant chunk t), pe/po the B fragments of the even /
// odd steps, xq = (-1024 X_{2t}, -1024 X_{2t+1}, the same again) from the scaled
// sub-block sums X_j, us = 2^-s of the super-block.  Adds the super-block's
// contribution to yacc[mt] = (row g, row g+8).
template <int MT>
__device__ __forceinline__ void b1_super_block(const uint4 (&hdr)[MT][2], const uint4 (&qa)[MT][2][2],
                                               const uint32_t *pe, const uint32_t *po,
                                               const float4 xq, float us, const B1Lane &lc,
                                               uint32_t magic, float2 (&yacc)[MT]) {
  const bool upper = lc.upper;
  const uint32_t psel = lc.psel, mlo4 = lc.mlo4, mhi4 = lc.mhi4;
  // Two accumulator sets: even steps add only to column 2t (accE[0], [2]),
  // odd steps only to column 2t+1 (accO[1], [3]), so splitting them halves
  // the dependent MMA chain at no cost.  Both start at xq, so that column 2t
  // of accE ends at sum (1024 + q) x - 1024 X_{2t} = sum q x and column 2t+1
  // of accO at sum (1024 + 16 q) x - 1024 X_{2t+1} = 16 sum q x.
  float accE[MT][4], accO[MT][4];
#pragma unroll
  for (int G2 = 0; G2 < 4; ++G2) {
    const uint4 be = reinterpret_cast<const uint4 *>(pe)[G2];  // words 4G2 .. 4G2+3
    const uint4 bo = reinterpret_cast<const uint4 *>(po)[G2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int G = 2 * G2 + h;  // quant word of the chunk
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t w0 = word_of(qa[mt][0][G >> 2], G & 3);
        const uint32_t w1 = word_of(qa[mt][1][G >> 2], G & 3);
        const uint32_t w0s = w0 >> 8, w1s = w1 >> 8;
        // low nibbles, 1024+q: sub-block 2t
        const uint32_t be0 = h ? be.z : be.x, be1 = h ? be.w : be.y;
        if (G == 0)
          mma_f16_c(accE[mt], xq, lop_nib(w0, magic), lop_nib(w1, magic), lop_nib(w0s, magic),
                    lop_nib(w1s, magic), be0, be1);
        else
          mma_f16(accE[mt], lop_nib(w0, magic), lop_nib(w1, magic), lop_nib(w0s, magic),
                  lop_nib(w1s, magic), be0, be1);
        // high nibbles, 1024+16q: sub-block 2t+1
        const uint32_t bo0 = h ? bo.z : bo.x, bo1 = h ? bo.w : bo.y;
        if (G == 0)
          mma_f16_c(accO[mt], xq, lop_nib_hi16(w0, magic), lop_nib_hi16(w1, magic),
                    lop_nib_hi16(w0s, magic), lop_nib_hi16(w1s, magic), bo0, bo1);
        else
          mma_f16(accO[mt], lop_nib_hi16(w0, magic), lop_nib_hi16(w1, magic),
                  lop_nib_hi16(w0s, magic), lop_nib_hi16(w1s, magic), bo0, bo1);
      }
    }
  }
  // Apply the scales: the scale/min bytes of both rows are gathered into one
  // word each with PRMT, and each byte b becomes a float by placing it under
  // the exponent of 2^23 (b exactly) or of 2^19 (b / 16 exactly, which also
  // undoes the 16 of the high nibbles) and subtracting that power of two.
  // xq carries -1024 X, so the mins meet dmin / 1024.
  constexpr uint32_t kExp = 0x4B490000u;  // byte 7: 2^23, byte 6: 2^19
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const uint4 h0 = hdr[mt][0], h1 = hdr[mt][1];
    const uint32_t py = __byte_perm(h0.y, h1.y, psel);  // s[k0], s[k0+1] of g, g+8
    const uint32_t pz = __byte_perm(h0.z, h1.z, psel);  // s[k0+4], s[k0+5]
    const uint32_t pw = __byte_perm(h0.w, h1.w, psel);  // s[k0+8], s[k0+9]
    // lanes t < 2: sc = s[j] & 63, m = s[j+4] & 63; lanes t >= 2:
    // sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4
    const uint32_t sc4 = ((upper ? pw : py) & mlo4) | ((py >> 2) & mhi4);
    const uint32_t m4 = ((upper ? (pw >> 4) : pz) & mlo4) | ((pz >> 2) & mhi4);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t h = r ? h1.x : h0.x;
      const float d = half_lo_to_float(h), dmn = half_hi_to_float(h) * (1.f / 1024.f);
      const float sca = __uint_as_float(__byte_perm(sc4, kExp, 0x7440u + 2 * r)) - 8388608.f;
      const float scb = __uint_as_float(__byte_perm(sc4, kExp, 0x6441u + 2 * r)) - 524288.f;
      const float ma = __uint_as_float(__byte_perm(m4, kExp, 0x7440u + 2 * r)) - 8388608.f;
      const float mb = __uint_as_float(__byte_perm(m4, kExp, 0x7441u + 2 * r)) - 8388608.f;
      const float uu = fmaf(scb, accO[mt][2 * r + 1], sca * accE[mt][2 * r]);
      const float vv = fmaf(mb, xq.y, ma * xq.x);
      float &yv = r ? yacc[mt].y : yacc[mt].x;
      yv = fmaf(us, fmaf(dmn, vv, d * uu), yv);  // back from the 2^s scaled units
    }
  }
}

// Stage super-blocks first .. first+count-1 (count <= C) of a warp's x slice
// for batch 1.  For each super-block i: an fp16 copy of its 256 values scaled by 2^s_i, with s_i chosen
// so that the super-block's largest magnitude lands in [2^14, 2^15) (the scaled
// value is exact for every entry within 2^28 of that maximum), permuted so that
// word 2G of a sub-block holds (x[4G], x[4G+2]) and word 2G+1 (x[4G+1],
// x[4G+3]); xq[4 i + t] = (-1024 X_{2t}, -1024 X_{2t+1}, the same again), X_j
// the sum of scaled sub-block j; unscale[i] = 2^-s_i.
// Lane l handles values 8l .. 8l+7 of each super-block, i.e. lane (g, t) holds
// a quarter of sub-block g -- exactly the B fragment of column g of an
// m16n8k16 MMA, so two MMAs with every A entry -1024 produce -1024 X_n in
// column n of every row, and lane (g, t) ends with the quad it needs.  The
// loads of the chunk are all issued before any of them is used.
// On entry xperm holds the raw bf16 slice (one bulk copy); each lane rewrites
// only the 16 bytes it read.
template <int C>
__device__ __forceinline__ void b1_stage_chunk(int first, int count, uint32_t *xperm, float4 *xq,
                                               float *unscale, int lane) {
  const uint4 *xs = reinterpret_cast<const uint4 *>(xperm);
  constexpr uint32_t kNeg1024 = 0xE400E400u;  // fp16 -1024 in both halves
  uint4 u[C];
  uint32_t mx[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    u[j] = (j < count) ? xs[(first + j) * 32 + lane] : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < C; ++j) {  // largest |x| as bf16 bits (sign cleared, 16-bit lanes)
    const uint4 v = u[j];
    const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    mx[j] = max(m & 0xFFFFu, m >> 16);
  }
#pragma unroll
  for (int j = 0; j < C; ++j) mx[j] = __reduce_max_sync(0xffffffffu, mx[j]);
  float4 c[C];
  int sh2[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    const uint4 v = u[j];
    const int emax = mx[j] ? (int)(mx[j] >> 7) - 127 : 0;  // exponent of the largest |x|
    sh2[j] = min(126, max(-126, 14 - emax));
    const float scale = __int_as_float((127 + sh2[j]) << 23);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
    const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z));
    const float2 f3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.w));
    const __half2 h02 = __floats2half2_rn(f0.x * scale, f1.x * scale);  // x0, x2
    const __half2 h13 = __floats2half2_rn(f0.y * scale, f1.y * scale);  // x1, x3
    const __half2 h46 = __floats2half2_rn(f2.x * scale, f3.x * scale);  // x4, x6
    const __half2 h57 = __floats2half2_rn(f2.y * scale, f3.y * scale);  // x5, x7
    u[j].x = *reinterpret_cast<const uint32_t *>(&h02);
    u[j].y = *reinterpret_cast<const uint32_t *>(&h13);
    u[j].z = *reinterpret_cast<const uint32_t *>(&h46);
    u[j].w = *reinterpret_cast<const uint32_t *>(&h57);
    float acc[4];
    mma_f16_zc(acc, kNeg1024, kNeg1024, kNeg1024, kNeg1024, u[j].x, u[j].y);
    mma_f16(acc, kNeg1024, kNeg1024, kNeg1024, kNeg1024, u[j].z, u[j].w);
    c[j] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
#pragma unroll
  for (int j = 0; j < C; ++j) {
    if (j < count) {
      reinterpret_cast<uint4 *>(xperm)[(first + j) * 32 + lane] = u[j];
      if (lane < 4) xq[(first + j) * 4 + lane] = c[j];  // g = 0: t = lane
      if (lane == 0) unscale[first + j] = __int_as_float((127 - sh2[j]) << 23);
    }
  }
  __syncwarp();
}

// Batch 1 epilogue: quad reduction (sub-blocks 2t, 2t+1 -> the row), then the
// split-K partials of the CTA's warps in warp order, store y.
template <int MT>
__device__ __forceinline__ void b1_finish(const float2 (&yacc)[MT], bool ok,
                                          float *red, int row0, const GemvArgs &a) {
  constexpr int kRows = MT * kRowsPerTile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float v = r ? yacc[mt].y : yacc[mt].x;
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (t == 0) red[warp * kRows + mt * kRowsPerTile + g + 8 * r] = v;
    }
  }
  __syncwarp();
  if (!ok && lane == 0) red[warp * kRows] = __int_as_float(0x7fc00000);
  __syncthreads();
  if (threadIdx.x < kRows) {
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) sum += red[w * kRows + threadIdx.x];
    const int row = row0 + (int)threadIdx.x;
    if (row < a.n) a.y[row] = sum;
  }
}

// After a timed-out wait: give the copies a warp may still have in flight (the
// x slice when xbar is given, then ring iterations it .. end-1 of a ring of
// `stages` slots) the same bounded time to land before the CTA exits and its
// shared memory is handed to another CTA.
__device__ __noinline__ void b1_drain_ring(uint64_t *bars, int stages, int it, int end,
                                           uint64_t *xbar) {
  const uint64_t t0 = global_ns();
  auto landed = [&](uint64_t *b, uint32_t parity) {
    while (!mbar_try_wait(b, parity, 1000u))
      if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
  };
  if (xbar != nullptr && !landed(xbar, 0)) return;
  for (int j = it; j < end; ++j)
    if (!landed(&bars[j % stages], (j / stages) & 1)) return;
}

// ---------------------------------------------------------------- batch 1
// MMA mapping (per super-block, 16 steps s = 2G + e, G = 0..7):
//   thread (g, t) owns quant chunk t of rows g and g+8; word G of the chunk
//   holds positions 4G..4G+3 of sub-blocks 2t (low nibbles) and 2t+1 (high).
//   Step e = 0 feeds the low nibbles, e = 1 the high ones: k-slots (2t, 2t+1)
//   carry positions (4G, 4G+2) and k-slots (2t+8, 2t+9) positions
//   (4G+1, 4G+3) of sub-block 2t+e.
//   MMA column n is sub-block n: lane (g, t) feeds x of sub-block g in both
//   b0 and b1 when g = 2t + e, zeros otherwise, so accumulator column n sums
//   exactly sub-block n and thread t ends with sub-blocks 2t, 2t+1 of its rows.
// Shared memory per warp: STAGES weight tiles (16*MT rows x S super-blocks,
// row stride S*144 bytes) | x of the warp's slice, word 2G of a sub-block
// holding (x[4G], x[4G+2]) and word 2G+1 (x[4G+1], x[4G+3]) | per super-block
// four quads (-1024 X_{2t}, -1024 X_{2t+1}, the same again), t = 0..3 | 2^-s_i of
// each super-block (padded to 16 bytes) | 64 zero bytes | STAGES + 1 mbarriers
// (the ring, x).
template <int MT, int S, int STAGES>
__global__ void __launch_bounds__(256) gemv_b1_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const GemvArgs a) {
  constexpr int kStageBytes = MT * S * kTileBytes;
  constexpr int kRowBytes = S * kBlockBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * (MT * kRowsPerTile);
  const int sb0 = warp * a.ks;
  const int nsteps = max(0, min(a.nsb, sb0 + a.ks) - sb0);  // super-blocks of this warp
  const int nstages = (nsteps + S - 1) / S;

  uint8_t *wreg = smem + (size_t)warp * a.warp_bytes;
  uint8_t *ring = wreg;
  uint32_t *xperm = reinterpret_cast<uint32_t *>(wreg + STAGES * kStageBytes);  // ks*128 words
  float4 *xq = reinterpret_cast<float4 *>(xperm + a.ks * 128);                   // ks*4 quads
  float *xuns = reinterpret_cast<float *>(xq + a.ks * 4);  // ks floats, padded to 16 bytes
  uint32_t *xzero = reinterpret_cast<uint32_t *>(xuns + pad4(a.ks));            // 16 words
  uint64_t *bars = reinterpret_cast<uint64_t *>(xzero + 16);  // STAGES ring + 1 for x
  float *red = reinterpret_cast<float *>(smem + (size_t)nwarps * a.warp_bytes);

  if (lane == 0) {
    prefetch_tmap(&wmap);
    for (int s = 0; s <= STAGES; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  // Copy order on the warp's TMA queue: a.pre weight stages (they do not depend
  // on earlier kernels, so with programmatic dependent launch they go out before
  // the dependency wait), then the x slice, then the rest of the ring.  x is small and read by every CTA, and a
  // copy queued behind a full ring of weights waits for that ring to drain
  // from DRAM; this order keeps x near the head.
  const int kPre = min(a.pre, STAGES);  // 0 unless launched with programmatic dependence
  if (lane == 0) {
    for (int s = 0; s < kPre && s < nstages; ++s) {
      mbar_arrive_expect_tx(&bars[s], kStageBytes);
      load_tile(ring + s * kStageBytes, &wmap, &bars[s], sb0 + s * S, row0, policy);
    }
  }
  grid_dependency_wait();
  if (lane == 0 && nsteps > 0) {
    mbar_arrive_expect_tx(&bars[STAGES], nsteps * kQK * 2);
    bulk_load(xperm, a.x + (int64_t)sb0 * kQK, nsteps * kQK * 2, &bars[STAGES]);
  }
  if (lane == 0) {
    for (int s = kPre; s < STAGES && s < nstages; ++s) {
      mbar_arrive_expect_tx(&bars[s], kStageBytes);
      load_tile(ring + s * kStageBytes, &wmap, &bars[s], sb0 + s * S, row0, policy);
    }
  }
  grid_launch_dependents();
  bool ok = nsteps == 0 || mbar_wait(&bars[STAGES], 0, a.err);
  // The whole slice is converted before the main loop, in chunks of 8
  // super-blocks and a last chunk of the smallest size in {1, 2, 4, 8} that
  // covers the rest: a chunk's slots all do the full work, and a chunk of 8
  // for 2 super-blocks made the 4096 x 4096 projection 9% slower.  (Converting
  // a chunk one step ahead inside the main loop instead measured 1-3% slower
  // on the 27B-class shapes.)
  if (ok) {
    int b = 0;
    for (; nsteps - b > 8; b += 8) b1_stage_chunk<8>(b, 8, xperm, xq, xuns, lane);
    const int rest = nsteps - b;
    if (rest > 4)
      b1_stage_chunk<8>(b, rest, xperm, xq, xuns, lane);
    else if (rest > 2)
      b1_stage_chunk<4>(b, rest, xperm, xq, xuns, lane);
    else if (rest == 2)
      b1_stage_chunk<2>(b, rest, xperm, xq, xuns, lane);
    else if (rest == 1)
      b1_stage_chunk<1>(b, rest, xperm, xq, xuns, lane);
    if (lane < 16) xzero[lane] = 0u;
    __syncwarp();
  } else if (lane == 0) {
    b1_drain_ring(bars, STAGES, 0, min(STAGES, nstages), &bars[STAGES]);
  }

  // B fragments: lane (g, t) with t == g/2 carries sub-block g on the steps of
  // parity g & 1 (pointer pe for even steps, po for odd steps); all other
  // (lane, step) combinations read zeros.
  const bool own = (t == (g >> 1));
  const bool own_e = own && !(g & 1), own_o = own && (g & 1);
  const uint32_t *pe = own_e ? xperm + g * 16 : xzero;
  const uint32_t *po = own_o ? xperm + g * 16 : xzero;
  const int adv_e = own_e ? 128 : 0, adv_o = own_o ? 128 : 0;

  // Scale/min decode of sub-blocks 2t, 2t+1, branch-free: lanes t < 2 read the
  // low six bits of s[j], s[j+4]; lanes t >= 2 combine a nibble of s[j+4] with
  // the top two bits of s[j-4] (scales) or s[j] (mins).
  const B1Lane lc = b1_lane(t);

  float2 yacc[MT];  // rows (g, g+8)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) yacc[mt] = make_float2(0.f, 0.f);
  // The magic constant lives in a register so each nibble op is one LOP3.
  uint32_t magic;
  asm volatile("mov.b32 %0, %1;\n" : "=r"(magic) : "n"(kF16Magic));

  uint32_t phase = 0;
  const float4 *pq = xq + t;
  for (int base = 0; base < nstages && ok; base += STAGES, phase ^= 1u) {
#pragma unroll
    for (int stage = 0; stage < STAGES; ++stage) {
      const int it = base + stage;
      if (it >= nstages) break;
      if (!mbar_wait(&bars[stage], phase, a.err)) {
        ok = false;
        if (lane == 0) b1_drain_ring(bars, STAGES, it, min(it + STAGES, nstages), nullptr);
        break;
      }
      uint8_t *st = ring + stage * kStageBytes;
      const int cnt = min(S, nsteps - it * S);
#pragma unroll
      for (int u = 0; u < S; ++u) {
        if (u >= cnt) break;
        const int i = it * S + u;  // super-block index within the slice
        uint4 hdr[MT][2], qa[MT][2][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint8_t *rp =
                st + (mt * kRowsPerTile + g + 8 * r) * kRowBytes + u * kBlockBytes;
            hdr[mt][r] = *reinterpret_cast<const uint4 *>(rp);
            qa[mt][r][0] = *reinterpret_cast<const uint4 *>(rp + kQsOffset + 32 * t);
            qa[mt][r][1] = *reinterpret_cast<const uint4 *>(rp + kQsOffset + 32 * t + 16);
          }
        }
        if (u == cnt - 1) {  // stage fully read: refill it
          __syncwarp();
          if (lane == 0 && it + STAGES < nstages) {
            mbar_arrive_expect_tx(&bars[stage], kStageBytes);
            load_tile(st, &wmap, &bars[stage], sb0 + (it + STAGES) * S, row0, policy);
          }
        }

        b1_super_block<MT>(hdr, qa, pe, po, pq[4 * i], xuns[i], lc, magic, yacc);
        pe += adv_e;
        po += adv_o;
      }
    }
  }

  b1_finish<MT>(yacc, ok, red, row0, a);
}

// ---------------------------------------------------------------- batch 2..16
// MMA columns = batch rows (NT n-tiles of 8).  Sub-block j = 2c+hi, step s:
// thread t's k-slots (2t, 2t+1) carry positions (o, o+2) and (2t+8, 2t+9)
// positions (o+1, o+3), o = 8t + 4s, i.e. quant bytes 8t .. 8t+7 of chunk c.
template <int MT, int NT, int STAGES>
__global__ void __launch_bounds__(256) gemv_bn_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * (MT * kRowsPerTile);
  const int sb0 = warp * a.ks;
  const int nsteps = max(0, min(a.nsb, sb0 + a.ks) - sb0);
  constexpr int kCols = NT * 8;

  uint8_t *ring = smem + (size_t)warp * a.warp_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + STAGES * MT * kTileBytes);
  float *red = reinterpret_cast<float *>(smem + (size_t)nwarps * a.warp_bytes);

  if (lane == 0) {
    prefetch_tmap(&wmap);
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  if (lane == 0) {
    for (int s = 0; s < STAGES && s < nsteps; ++s) {
      mbar_arrive_expect_tx(&bars[s], MT * kTileBytes);
      load_tile(ring + s * MT * kTileBytes, &wmap, &bars[s], sb0 + s, row0, policy);
    }
  }
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

  float yacc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) yacc[mt][nt][0] = yacc[mt][nt][1] = yacc[mt][nt][2] = yacc[mt][nt][3] = 0.f;

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
      if (lane == 0) b1_drain_ring(bars, STAGES, i, min(i + STAGES, nsteps), nullptr);
      break;
    }
    const uint8_t *st = ring + stage * MT * kTileBytes;
    uint4 hdr[MT][2];
    uint2 qw[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint8_t *rp = st + (mt * kRowsPerTile + g + 8 * r) * kBlockBytes;
        hdr[mt][r] = *reinterpret_cast<const uint4 *>(rp);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          qw[mt][r][c] = *reinterpret_cast<const uint2 *>(rp + kQsOffset + 32 * c + 8 * t);
      }
    __syncwarp();
    if (lane == 0 && i + STAGES < nsteps) {
      mbar_arrive_expect_tx(&bars[stage], MT * kTileBytes);
      load_tile(ring + stage * MT * kTileBytes, &wmap, &bars[stage], sb + STAGES, row0, policy);
    }
    load_x_half(xB, i, 1);
    // This lane decodes sub-blocks 2t, 2t+1 of rows g, g+8 (per m-tile).
    float dsA[MT][2], dsB[MT][2], dmA[MT][2], dmB[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t sc2, m2;
        scales_pair(hdr[mt][r].y, hdr[mt][r].z, hdr[mt][r].w, t, &sc2, &m2);
        const float d = half_lo_to_float(hdr[mt][r].x), dmin = half_hi_to_float(hdr[mt][r].x);
        dsA[mt][r] = d * (float)(sc2 & 0xFFu);
        dsB[mt][r] = d * (float)(sc2 >> 8);
        dmA[mt][r] = dmin * (float)(m2 & 0xFFu) * (1.f / 128.f);
        dmB[mt][r] = dmin * (float)(m2 >> 8) * (1.f / 128.f);
      }
    auto sub_block_seeded = [&](int j, const uint4(&xv)[NT]) {
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
      // -128 X_j of every column by MMAs with A = -128 everywhere (every row
      // holds it, so column 2t+e is cneg[nt][e]); the weight MMAs start there,
      // so acc = sum (128 + q) x - 128 X_j = sum q x.
      float cneg[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_zc(cneg[nt], kBf16Neg128, kBf16Neg128, kBf16Neg128, kBf16Neg128, b0[0][nt], b1[0][nt]);
        mma_bf16(cneg[nt], kBf16Neg128, kBf16Neg128, kBf16Neg128, kBf16Neg128, b0[1][nt], b1[1][nt]);
      }
      float acc[MT][NT][4];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t w0 = s ? qw[mt][0][c].y : qw[mt][0][c].x;
          const uint32_t w1 = s ? qw[mt][1][c].y : qw[mt][1][c].x;
          const uint32_t a0 = hi ? nib_hi(w0) : nib_lo(w0);
          const uint32_t a1 = hi ? nib_hi(w1) : nib_lo(w1);
          const uint32_t a2 = hi ? nib_hi(w0 >> 8) : nib_lo(w0 >> 8);
          const uint32_t a3 = hi ? nib_hi(w1 >> 8) : nib_lo(w1 >> 8);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (s == 0)
              mma_bf16_c(acc[mt][nt], cneg[nt], a0, a1, a2, a3, b0[0][nt], b1[0][nt]);
            else
              mma_bf16(acc[mt][nt], a0, a1, a2, a3, b0[1][nt], b1[1][nt]);
          }
        }
      }
      // Scales of sub-block j for rows g, g+8 live in lane (g, j/2); dm
      // carries the 1/128 of cneg and meets it with the sign folded in.
      const int src = (lane & ~3) | (j >> 1);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float ds = __shfl_sync(0xffffffffu, hi ? dsB[mt][r] : dsA[mt][r], src);
          const float dm = __shfl_sync(0xffffffffu, hi ? dmB[mt][r] : dmA[mt][r], src);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float &yv = yacc[mt][nt][2 * r + e];
              yv = fmaf(ds, acc[mt][nt][2 * r + e], yv);
              yv = fmaf(dm, cneg[nt][e], yv);
            }
          }
        }
      }
    };
    auto sub_block_plain = [&](int j, const uint4(&xv)[NT]) {
      const int c = j >> 1;
      const bool hi = j & 1;
      float acc[MT][NT][4];
      float c128[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        c128[nt][0] = c128[nt][1] = c128[nt][2] = c128[nt][3] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t lo = s ? xv[nt].z : xv[nt].x;
          const uint32_t hi2 = s ? xv[nt].w : xv[nt].y;
          b0[nt] = __byte_perm(lo, hi2, 0x5410);
          b1[nt] = __byte_perm(lo, hi2, 0x7632);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t w0 = s ? qw[mt][0][c].y : qw[mt][0][c].x;
          const uint32_t w1 = s ? qw[mt][1][c].y : qw[mt][1][c].x;
          const uint32_t a0 = hi ? nib_hi(w0) : nib_lo(w0);
          const uint32_t a1 = hi ? nib_hi(w1) : nib_lo(w1);
          const uint32_t a2 = hi ? nib_hi(w0 >> 8) : nib_lo(w0 >> 8);
          const uint32_t a3 = hi ? nib_hi(w1 >> 8) : nib_lo(w1 >> 8);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[mt][nt], a0, a1, a2, a3, b0[nt], b1[nt]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16(c128[nt], kBf16Magic, kBf16Magic, kBf16Magic, kBf16Magic, b0[nt], b1[nt]);
      }
      // Scales of sub-block j for rows g, g+8 live in lane (g, j/2).
      const int src = (lane & ~3) | (j >> 1);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float ds = __shfl_sync(0xffffffffu, hi ? dsB[mt][r] : dsA[mt][r], src);
          const float dm = __shfl_sync(0xffffffffu, hi ? dmB[mt][r] : dmA[mt][r], src);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float cv = acc[mt][nt][2 * r + e];
              const float c1 = c128[nt][e];
              yacc[mt][nt][2 * r + e] = fmaf(ds, cv - c1, yacc[mt][nt][2 * r + e]);
              yacc[mt][nt][2 * r + e] = fmaf(-dm, c1, yacc[mt][nt][2 * r + e]);
            }
          }
        }
      }
    };
    // One column tile: the weight MMAs start at -128 X_j (seeded).  Two: the
    // column sums run beside the weight MMAs instead, which measured faster
    // there (the seeded chain is one MMA pair deeper and holds more registers).
    auto sub_block = [&](int j, const uint4(&xv)[NT]) {
      if constexpr (NT == 1)
        sub_block_seeded(j, xv);
      else
        sub_block_plain(j, xv);
    };
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sub_block(jj, xA[jj]);
    load_x_half(xA, i + 1, 0);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sub_block(4 + jj, xB[jj]);
  }

  // Across warps: red[warp][row][col].
  const int tile_rows = MT * kRowsPerTile;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = mt * kRowsPerTile + g + 8 * (e >> 1);
        const int col = nt * 8 + 2 * t + (e & 1);
        red[(warp * tile_rows + row) * kCols + col] = yacc[mt][nt][e];
      }
  __syncwarp();
  if (!ok && lane == 0) red[(warp * tile_rows) * kCols] = __int_as_float(0x7fc00000);
  __syncthreads();
  for (int idx = threadIdx.x; idx < tile_rows * kCols; idx += blockDim.x) {
    const int row = idx / kCols, col = idx % kCols;
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += red[(w * tile_rows + row) * kCols + col];
    const int grow = row0 + row;
    if (grow < a.n && col < a.batch) a.y[(int64_t)col * a.ldy + grow] = s;
  }
}

// ---------------------------------------------------------------- launch
constexpr int kStages = Q4K_GEMV_STAGES;  // batch 2..16 (one super-block per stage)
// Stages for batch 1 with S super-blocks per stage.
#ifndef Q4K_GEMV_B1_STAGES_S1  // batch-1 ring depth (stages) for S = 1, 2, 4 super-blocks a stage
#define Q4K_GEMV_B1_STAGES_S1 4
#endif
#ifndef Q4K_GEMV_B1_STAGES_S2
#define Q4K_GEMV_B1_STAGES_S2 3
#endif
#ifndef Q4K_GEMV_B1_STAGES_S4
#define Q4K_GEMV_B1_STAGES_S4 2
#endif
#ifndef Q4K_GEMV_INFLIGHT_KB  // planner: weight bytes in flight per SM worth having, at most
#define Q4K_GEMV_INFLIGHT_KB 96
#endif
#ifndef Q4K_GEMV_BN_MT2_COST  // batch 2..16: per-row cost of an MT = 2 warp relative to MT = 1
#define Q4K_GEMV_BN_MT2_COST 0.8
#endif
#ifndef Q4K_GEMV_LOG_PLAN  // 1: print each batch-1 plan to stderr (tuning aid)
#define Q4K_GEMV_LOG_PLAN 0
#endif
template <int S> struct B1Stages {
  static constexpr int value =
      S == 1 ? Q4K_GEMV_B1_STAGES_S1 : (S == 2 ? Q4K_GEMV_B1_STAGES_S2 : Q4K_GEMV_B1_STAGES_S4);
};

#ifndef Q4K_GEMV_FORCE_S  // 0: choose per shape
#define Q4K_GEMV_FORCE_S 0
#endif
#ifndef Q4K_GEMV_FORCE_MT
#define Q4K_GEMV_FORCE_MT 0
#endif

struct Plan {
  int mt = 1, s = 1, wk = 1, ks = 1, warp_bytes = 0, smem = 0, grid = 0;
  double score = -1e30;
};

int warp_bytes_b1(int mt, int s, int stages, int ks) {
  int b = stages * mt * s * kTileBytes + ks * (512 + 64) + 4 * pad4(ks) + 64 + (stages + 1) * 8;
  return (b + 127) / 128 * 128;
}
int warp_bytes_bn(int mt) {
  int b = kStages * mt * kTileBytes + kStages * 8;
  return (b + 127) / 128 * 128;
}

template <typename K>
int occupancy(K kernel, int threads, int smem) {
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess)
    return 0;
  return blocks;
}

// Choose how the K dimension is split across the warps of a CTA.  Every CTA
// should be resident at once (one wave); among those plans, prefer more weight
// bytes in flight per SM (latency hiding), then an even split.
template <typename K>
Plan plan_for(K kernel, bool b1, int mt, int s, int stages, int n, int nsb, int cols,
              const DeviceFacts *f) {
  Plan best;
  const int tile_rows = mt * kRowsPerTile;
  const int grid = (n + tile_rows - 1) / tile_rows;
  for (int wk = 1; wk <= 8; ++wk) {
    int ks = (nsb + wk - 1) / wk;
    ks = (ks + s - 1) / s * s;
    if ((nsb + ks - 1) / ks != wk) continue;  // no empty warps
    if (ks < 2 * s && nsb >= 2 * s) continue;
    const int wb = b1 ? warp_bytes_b1(mt, s, stages, ks) : warp_bytes_bn(mt);
    const int smem = wk * wb + wk * tile_rows * cols * 4;
    if (smem > f->max_smem_optin) continue;
    const int occ = occupancy(kernel, wk * 32, smem);
    if (occ <= 0) continue;
    const int slots = occ * f->sm_count;
    const int waves = (grid + slots - 1) / slots;
    const int per_sm = std::min(occ, (grid + f->sm_count - 1) / f->sm_count);
    const int warps_sm = per_sm * wk;
    // stages == 0: register-streamed kernel, about 1.5 super-blocks in flight
    const double inflight_kb =
        warps_sm * (stages ? stages - 1 : 1.5) * mt * s * kTileBytes / 1024.0;
    const double balance = (double)nsb / (double)(ks * wk);  // 1.0 = even split
    const double score = -1000.0 * waves + std::min(inflight_kb, (double)Q4K_GEMV_INFLIGHT_KB) / 8.0 +
                         0.5 * std::min(warps_sm, 24) + 6.0 * balance + (mt == 2 ? 1.0 : 0.0);
    if (score > best.score) {
      best.score = score;
      best.mt = mt;
      best.s = s;
      best.wk = wk;
      best.ks = ks;
      best.warp_bytes = wb;
      best.smem = smem;
      best.grid = grid;
    }
  }
  return best;
}

std::once_flag g_attr_once[kMaxDevices];  // cudaFuncSetAttribute acts on the current device

// Batch-1 plan.  A row tile's K is split over the wk warps of its CTA.  Every
// CTA must be resident at once; among those plans take the smallest load of
// the busiest SM: ceil(CTAs / SMs) x warps per CTA x super-blocks per warp x
// rows per warp x the per-row cost of the tile height (an MT = 2 warp spends
// 0.72 of an MT = 1 warp's instructions per row: 269 vs 373 per 16-row tile,
// measured when the weight was fitted; a forced-plan sweep of the current
// kernel still favours these choices except for qkv, where one tile per warp
// ran 7% faster and o 16% slower), plus a penalty for fewer than 8 resident warps per SM (too little
// to hide latency).  (Splitting a tile's K further over a cluster of CTAs, with
// the partials summed through distributed shared memory, balanced the SMs
// better on paper but measured slower at every cluster size.)
// Batch 2..16: the same load objective; an MT = 2 warp shares its x
// fragments between its two row tiles (taken as 0.8 of MT = 1's cost per row).
template <typename K>
Plan plan_bn(K kernel, int mt, int stages, int n, int nsb, int cols, const DeviceFacts *f) {
  Plan best;
  const int tile_rows = mt * kRowsPerTile;
  const int tiles = (n + tile_rows - 1) / tile_rows;
  for (int wk = 1; wk <= 8; ++wk) {
    const int ks = (nsb + wk - 1) / wk;
    if ((nsb + ks - 1) / ks != wk) continue;  // every warp gets super-blocks
    const int wb = warp_bytes_bn(mt);
    const int smem = wk * wb + wk * tile_rows * cols * 4;
    if (smem > f->max_smem_optin) continue;
    const int occ = occupancy(kernel, wk * 32, smem);
    if (occ <= 0) continue;
    if (tiles > occ * f->sm_count) continue;  // one wave
    const long per_sm = (tiles + f->sm_count - 1) / f->sm_count;
    const long warps_sm = per_sm * wk;
    double load = (double)per_sm * wk * ks * mt * (mt == 2 ? Q4K_GEMV_BN_MT2_COST : 1.0);
    if (warps_sm < 8) load *= 1.0 + 0.08 * (8 - warps_sm);
    if (-load > best.score) {
      best.score = -load;
      best.mt = mt;
      best.s = 1;
      best.wk = wk;
      best.ks = ks;
      best.warp_bytes = wb;
      best.smem = smem;
      best.grid = tiles;
    }
  }
  return best;
}

template <typename K>
Plan plan_b1(K kernel, int mt, int s, int stages, int n, int nsb, const DeviceFacts *f) {
  Plan best;
  const int tile_rows = mt * kRowsPerTile;
  const int tiles = (n + tile_rows - 1) / tile_rows;
  for (int wk = 1; wk <= 8; ++wk) {
    int ks = (nsb + wk - 1) / wk;
    ks = (ks + s - 1) / s * s;
    if ((nsb + ks - 1) / ks != wk) continue;  // every warp gets super-blocks
    if (ks < 2 * s && nsb >= 2 * s) continue;
    const int wb = warp_bytes_b1(mt, s, stages, ks);
    const int smem = wk * wb + wk * tile_rows * 4;
    if (smem > f->max_smem_optin) continue;
    const int occ = occupancy(kernel, wk * 32, smem);
    if (occ <= 0) continue;
    if (tiles > occ * f->sm_count) continue;  // one wave
    const long per_sm = (tiles + f->sm_count - 1) / f->sm_count;
    const long warps_sm = per_sm * wk;
    double load = (double)per_sm * wk * ks * mt * (mt == 2 ? 0.72 : 1.0);
    if (warps_sm < 8) load *= 1.0 + 0.08 * (8 - warps_sm);
    if (-load > best.score) {
      best.score = -load;
      best.mt = mt;
      best.s = s;
      best.wk = wk;
      best.ks = ks;
      best.warp_bytes = wb;
      best.smem = smem;
      best.grid = tiles;
    }
  }
  return best;
}

template <typename K>
void allow_smem(K kernel, const DeviceFacts *f) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, f->max_smem_optin);
}

template <int MT, int S>
constexpr auto b1_kernel() {
  return gemv_b1_kernel<MT, S, B1Stages<S>::value>;
}

void set_attributes(const DeviceFacts *f) {
  allow_smem(b1_kernel<1, 1>(), f);
  allow_smem(b1_kernel<1, 2>(), f);
  allow_smem(b1_kernel<1, 4>(), f);
  allow_smem(b1_kernel<2, 1>(), f);
  allow_smem(b1_kernel<2, 2>(), f);
  allow_smem(gemv_bn_kernel<1, 1, kStages>, f);
  allow_smem(gemv_bn_kernel<1, 2, kStages>, f);
  allow_smem(gemv_bn_kernel<2, 1, kStages>, f);
  allow_smem(gemv_bn_kernel<2, 2, kStages>, f);
}

using GemvKernel = void (*)(CUtensorMap, GemvArgs);

GemvKernel b1_select(int mt, int s) {
  if (mt == 2) return s == 2 ? b1_kernel<2, 2>() : b1_kernel<2, 1>();
  return s == 4 ? b1_kernel<1, 4>() : s == 2 ? b1_kernel<1, 2>() : b1_kernel<1, 1>();
}

}  // namespace

template <typename K, typename... Args>
cudaError_t launch(K kernel, const Plan &p, bool pdl, cudaStream_t stream, Args... kargs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)(p.wk * 32), 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, kargs...);
}

namespace {
// Plans depend only on (device, N, K, batch class); computing one takes a few
// dozen occupancy queries, so they are kept per process.  Bounded: the cache is
// cleared when it reaches kMaxPlans entries.
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

cudaError_t launch_gemv(const void *w, int64_t n, int64_t k, const void *x, int64_t batch,
                        int64_t ldx, float *y, int64_t ldy, bool overlap, cudaStream_t stream) {
  const DeviceFacts *f = device_facts();
  std::call_once(g_attr_once[f->device], set_attributes, f);
  const int nsb = (int)(k / kQK);

  // W viewed as [n rows][nsb super-blocks][144 bytes]; one box = 16*mt rows
  // of one super-block.
  CUtensorMap map;
  auto encode = [&](int mt, int s) {
    const uint64_t dims[2] = {(uint64_t)nsb * (kBlockBytes / 8), (uint64_t)n};
    const uint64_t strides[1] = {(uint64_t)nsb * kBlockBytes};
    const uint32_t box[2] = {(uint32_t)(s * (kBlockBytes / 8)), (uint32_t)(mt * kRowsPerTile)};
    return encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(w), dims,
                        strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                        Q4K_GEMV_PROMO == 0   ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                        : Q4K_GEMV_PROMO == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                              : CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  };

  GemvArgs args = {};
  args.w = static_cast<const uint8_t *>(w);
  args.row_bytes = (int64_t)nsb * kBlockBytes;
  args.x = static_cast<const __nv_bfloat16 *>(x);
  args.y = y;
  args.ldx = ldx;
  args.ldy = ldy;
  args.n = (int)n;
  args.nsb = nsb;
  args.batch = (int)batch;
  args.err = device_error_word();

  if (batch == 1) {
    const Plan p = cached_plan(PlanKey{f->device, (int)n, nsb, 1}, [&] {
      Plan best;
      const int cand[5][2] = {{1, 1}, {1, 2}, {1, 4}, {2, 1}, {2, 2}};
      for (const auto &c : cand) {
        if (Q4K_GEMV_FORCE_MT && c[0] != Q4K_GEMV_FORCE_MT) continue;
        if (Q4K_GEMV_FORCE_S && c[1] != Q4K_GEMV_FORCE_S) continue;
        const int stages = c[1] == 1 ? B1Stages<1>::value : c[1] == 2 ? B1Stages<2>::value
                                                                       : B1Stages<4>::value;
        const Plan q = plan_b1(b1_select(c[0], c[1]), c[0], c[1], stages, (int)n, nsb, f);
        if (q.grid && q.score > best.score) best = q;
      }
      return best;
    });
    if (p.grid == 0) return cudaErrorInvalidConfiguration;
    GemvKernel kern = b1_select(p.mt, p.s);
    args.pre = overlap ? Q4K_GEMV_PRE_STAGES : 0;
    static int logged = 0;
    if (Q4K_GEMV_LOG_PLAN && logged < 64 && ++logged)
      fprintf(stderr, "q4k_gemv plan n=%lld k=%lld: mt=%d s=%d warps=%d ks=%d smem=%d grid=%d\n",
              (long long)n, (long long)k, p.mt, p.s, p.wk, p.ks, p.smem, p.grid);
    if (encode(p.mt, p.s) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    args.ks = p.ks;
    args.warp_bytes = p.warp_bytes;
    cudaError_t e = launch(kern, p, overlap, stream, map, args);
    if (e != cudaSuccess) return e;
  } else {
    const int nt = batch <= 8 ? 1 : 2;
    auto bn_select = [&](int mt) {
      return (mt == 2) ? (nt == 1 ? gemv_bn_kernel<2, 1, kStages> : gemv_bn_kernel<2, 2, kStages>)
                       : (nt == 1 ? gemv_bn_kernel<1, 1, kStages> : gemv_bn_kernel<1, 2, kStages>);
    };
    const Plan p = cached_plan(PlanKey{f->device, (int)n, nsb, 1 + nt}, [&] {
      Plan best;
      for (int mt = 1; mt <= 2; ++mt) {  // the tile height is part of the plan, as at batch 1
        if (Q4K_GEMV_FORCE_MT && mt != Q4K_GEMV_FORCE_MT) continue;
        // Measured on the 64-layer pass: the busiest-SM load objective wins at
        // 16 columns (B = 16: 1356 -> 1503 GB/s), the older score at 8 (B = 4:
        // 1951 vs 1543 GB/s).
        const Plan q = nt == 2 ? plan_bn(bn_select(mt), mt, kStages, (int)n, nsb, nt * 8, f)
                               : plan_for(bn_select(mt), false, mt, 1, kStages, (int)n, nsb, nt * 8, f);
        if (q.grid && q.score > best.score) best = q;
      }
      return best;
    });
    if (p.grid == 0) return cudaErrorInvalidConfiguration;
    const int mt = p.mt;
    auto kern = bn_select(mt);
    if (Q4K_GEMV_LOG_PLAN)
      fprintf(stderr, "q4k_gemv batched plan n=%lld k=%lld b=%lld: mt=%d warps=%d ks=%d smem=%d grid=%d\n",
              (long long)n, (long long)k, (long long)batch, mt, p.wk, p.ks, p.smem, p.grid);
    if (encode(mt, 1) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    args.ks = p.ks;
    args.warp_bytes = p.warp_bytes;
    cudaError_t e = launch(kern, p, overlap, stream, map, args);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace q4k
