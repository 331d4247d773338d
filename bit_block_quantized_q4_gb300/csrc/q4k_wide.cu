// q4k_wide.cu -- decode projections Y[b] = W X[b] with W in Q4_K for batch
// 5..16, any number of them in one persistent launch ("PRD: Performant
// Concurrent Distributed GGUF Runtime", DGR-012: batched decode steps; "spec:
// specialized model runtimes", section "Architecture": the T0 GEMM), and the
// fused gate/up projection H[b] = silu(Wg X[b]) * (Wu X[b]) ("Layer Package
// Repository Spec", section "Policy Resolution": merged gate/up).
//
// Work: a tile is 64 weight rows of one op over the op's whole K (a gate/up
// op's tile is its gate rows, then the same up rows).  The tiles of all ops of
// a launch form one list; each CTA takes a contiguous run of it, balanced by
// weight bytes, so a sequence of projections streams its weights back to back.
//
// The four warps of a CTA consume the same stages in lockstep: a stage is SB
// super-blocks of the tile's 64 rows (one TMA tile) plus the x of those
// super-blocks for the 8*NT batch rows (one bulk copy per super-block and
// batch row), completing on the slot's mbarrier and released by a CTA
// barrier.  So the x of a super-block is read from L2 once per 64 rows and the
// warps hold no x in registers between super-blocks.  Warp w contracts rows
// 16w .. 16w+15.  (With 16-byte cp.async chunks copied by every thread, the
// chunk addresses and predicates cost each thread about a hundred integer
// instructions per stage.)
//
// Contraction (mma.sync m16n8k16 bf16 -> fp32), as in the per-op batched
// kernel: the MMA columns are the batch rows (NT n-tiles of 8); sub-block j of
// a row is taken in offset form (offset_form) and accumulated by two MMAs on
// the exact small integers q - c; per (row, sub-block, column) the thread adds
// ds * acc + e * X_j, X_j the column's sum of x over the sub-block (two MMAs
// with A = 1).  Lane (g, t) decodes the offset forms of sub-blocks 2t, 2t+1 of
// its rows g, g+8; the other lanes of its quad fetch them by shuffle.  Every
// sum is taken in a fixed order: the result does not depend on timing.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "q4k.h"
#include "q4k_device.cuh"
#include "q4k_internal.h"

// Super-blocks per stage and ring stages, batch 5..8 (NT1) and 9..16 (NT2);
// measured on the 64-layer pass with TMA stages: two stages of one
// super-block 2.73 / 2.67 / 2.00 TB/s at batch 5 / 8 / 16, against 2.70 /
// 2.64 / 1.96 with three stages, 2.71 / 2.64 / 1.75 with four, 2.75 / 2.67 /
// 1.96 with two of two super-blocks.
#ifndef Q4K_WIDE_SB_NT1
#define Q4K_WIDE_SB_NT1 1
#endif
#ifndef Q4K_WIDE_STAGES_NT1
#define Q4K_WIDE_STAGES_NT1 2
#endif
#ifndef Q4K_WIDE_SB_NT2
#define Q4K_WIDE_SB_NT2 1
#endif
#ifndef Q4K_WIDE_STAGES_NT2
#define Q4K_WIDE_STAGES_NT2 2
#endif
// Resident CTAs per SM the register budget is sized for, batch 5..8 and
// 9..16 (measured on the 64-layer pass: 6 CTAs at batch 5 / 8 2.78 / 2.73
// TB/s against 2.74 / 2.67 at 4 and 2.53 / 2.44 at 3; batch 16 2.00 at 4,
// 1.97 at 5, 1.99 at 6, 1.81 at 3).
#ifndef Q4K_WIDE_MINB_NT1
#define Q4K_WIDE_MINB_NT1 6
#endif
#ifndef Q4K_WIDE_MINB_NT2
#define Q4K_WIDE_MINB_NT2 4
#endif
#ifndef Q4K_WIDE_PRE  // weight stages requested before the dependency wait (PDL)
#define Q4K_WIDE_PRE 2
#endif

namespace q4k {

namespace {

constexpr int kWideWarps = 4;
constexpr int kWideThreads = kWideWarps * 32;
constexpr int kWideRows = 16 * kWideWarps;  // rows per tile
// weight matrices (tensor maps) and ops per launch: with a 128-byte map per
// matrix the kernel parameter table stays under 32 KB
constexpr int kWideMaxOps = Q4K_SEQ_MATRICES_PER_LAUNCH;
// x rows in a stage: 512 bytes of a super-block plus 64 bytes, so that the
// 16-byte fragment reads of 8 batch rows by a quarter warp hit distinct banks.
constexpr int kXRowBytes = 576;

template <int NT>
struct WideCfg {
  static constexpr int kNB = 8 * NT;  // batch rows the kernel carries
  static constexpr int kSB = NT == 1 ? Q4K_WIDE_SB_NT1 : Q4K_WIDE_SB_NT2;
  static constexpr int kStages = NT == 1 ? Q4K_WIDE_STAGES_NT1 : Q4K_WIDE_STAGES_NT2;
  // a row's slot in a stage: its kSB super-blocks, padded by 16 bytes when kSB
  // is even so that rows fall on different banks
  static constexpr int kRowBytes = kSB * kBlockBytes + (kSB % 2 == 0 ? 16 : 0);
  static constexpr int kWBytes = kWideRows * kRowBytes;
  static constexpr int kXBytes = kSB * kNB * kXRowBytes;  // [super-block][batch row][576]
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kOffBar = kStages * kStageBytes;  // the ring's mbarriers
  static constexpr int kSmem = kOffBar + 8 * kStages;
  static_assert(kWBytes % 128 == 0 && kStageBytes % 128 == 0 && kRowBytes % 16 == 0,
                "TMA destinations 128-byte aligned, tile rows whole 16-byte units");
};

struct WideOp {
  const uint8_t *w;   // weights; the gate matrix of a gate/up op
  const uint8_t *w2;  // up matrix of a gate/up op, nullptr for a plain projection
  const __nv_bfloat16 *x;
  float *y;
  long long byte0;    // weight bytes of the ops before this one
  int n, nsb, ntiles, parts;
  int ldx, ldy;       // batch-row strides of x and y (elements)
  int map;            // index of the weight matrix's tensor map (the up matrix's is map + 1)
};

template <int NOPS>
struct WideParams {
  CUtensorMap map[NOPS == 1 ? 2 : NOPS];  // 2-D maps over the weight matrices (first: aligned)
  WideOp op[NOPS];
  unsigned *err;  // device error word (a timed-out wait on a stage)
  int nops;
  int batch;
  int pre;    // weight stages requested before the dependency wait
  int nctas;  // CTAs of the grid (tile runs)
  long long total;
};
static_assert(sizeof(WideParams<kWideMaxOps>) <= 32764, "kernel parameters are limited to 32764 bytes");

// Stage walk: super-blocks sb .. sb+SB-1 of part `part` of tile `tile` of op
// `op`, over the CTA's run of tiles [tiles starting in bytes lo .. hi).
struct WPos {
  int op, tile, part, sb;
  bool valid;
};

template <int NOPS>
__device__ __forceinline__ long long wide_tile_start(const WideParams<NOPS> &p, int op, int tile) {
  const WideOp &o = p.op[op];
  return o.byte0 + (long long)tile * kWideRows * o.nsb * kBlockBytes * o.parts;
}

// First tile of a run: the first tile that starts at or after byte lo.
template <int NOPS>
__device__ __forceinline__ void wide_first(const WideParams<NOPS> &p, long long lo, long long hi,
                                           WPos &s) {
  int a = 0, b = p.nops - 1;
  while (a < b) {
    const int m = (a + b + 1) >> 1;
    if (p.op[m].byte0 <= lo) a = m; else b = m - 1;
  }
  s.op = a;
  const WideOp &o = p.op[a];
  const long long cost = (long long)kWideRows * o.nsb * kBlockBytes * o.parts;
  s.tile = lo <= o.byte0 ? 0 : (int)((lo - o.byte0 + cost - 1) / cost);
  if (s.tile >= o.ntiles) {
    ++s.op;
    s.tile = 0;
  }
  s.part = 0;
  s.sb = 0;
  s.valid = s.op < p.nops && wide_tile_start(p, s.op, s.tile) < hi;
}

template <int SB, int NOPS>
__device__ __forceinline__ void wide_next(const WideParams<NOPS> &p, long long hi, WPos &s) {
  const WideOp &o = p.op[s.op];
  if ((s.sb += SB) < o.nsb) return;
  s.sb = 0;
  if (++s.part < o.parts) return;
  s.part = 0;
  if (++s.tile >= o.ntiles) {
    ++s.op;
    s.tile = 0;
  }
  s.valid = s.op < p.nops && wide_tile_start(p, s.op, s.tile) < hi;
}

__device__ __forceinline__ float silu_mul_w(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

template <int NT, int NOPS>
__global__ void __launch_bounds__(kWideThreads, NT == 1 ? Q4K_WIDE_MINB_NT1 : Q4K_WIDE_MINB_NT2)
    gemv_wide_kernel(const __grid_constant__ WideParams<NOPS> p) {
  using C = WideCfg<NT>;
  constexpr int SB = C::kSB, ST = C::kStages, NB = C::kNB;
  static_assert(ST >= 2, "the ring needs two stages");
  static_assert((SB * NB) % kWideWarps == 0, "x rows per warp");
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const long long lo = p.total * blockIdx.x / p.nctas, hi = p.total * (blockIdx.x + 1) / p.nctas;
  const int batch = p.batch;

  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);  // one mbarrier per ring slot
  // x rows past the batch stay zero in every slot (the copies below fill
  // rows b < batch only), so the consumer needs no test per column
  for (int idx = tid; idx < ST * SB * NB * (kQK * 2 / 16); idx += kWideThreads) {
    const int c16 = idx % (kQK * 2 / 16), rowi = idx / (kQK * 2 / 16);  // rowi = (slot, u, b)
    const int b = rowi % NB, su = rowi / NB;
    if (b >= batch)
      *reinterpret_cast<uint4 *>(smem + (su / SB) * C::kStageBytes + C::kWBytes +
                                 ((su % SB) * NB + b) * kXRowBytes + 16 * c16) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) {
    for (int st = 0; st < ST; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- producer (warp 0): a stage is one TMA tile of the weight matrix (64
  // rows by the row slot's bytes; rows past the matrix read as zeros) and one
  // bulk copy of 512 bytes of x per (super-block, batch row), both completing
  // on the slot's mbarrier, which thread 0 arms with the stage's bytes.
  auto issue_w = [&](int slot, const WPos &s) {
    if (tid == 0) {
      const uint64_t pol = l2_evict_first_policy();  // weights are read once
      const WideOp &o = p.op[s.op];
      const int cnt = min(SB, o.nsb - s.sb);
      mbar_arrive_expect_tx(&full[slot], (uint32_t)(C::kWBytes + batch * cnt * kQK * 2));
      tma_load_2d_hint(smem + slot * C::kStageBytes, &p.map[o.map + s.part], &full[slot],
                       s.sb * (kBlockBytes / 8), s.tile * kWideRows, pol);
    }
  };
  auto issue_x = [&](int slot, const WPos &s) {
    const WideOp &o = p.op[s.op];
    const int cnt = min(SB, o.nsb - s.sb);
    const int u = lane / NB, b = lane % NB;  // lane = (super-block u, batch row b)
    if (warp == 0 && lane < SB * NB && u < cnt && b < batch)
      bulk_load(smem + slot * C::kStageBytes + C::kWBytes + lane * kXRowBytes,
                o.x + (size_t)b * o.ldx + (size_t)(s.sb + u) * kQK, (uint32_t)(kQK * 2), &full[slot]);
  };
  // After its copies of a stage have landed, a thread puts its own x chunks in
  // B-fragment order in place: 16 bytes hold values 8l .. 8l+7 of a sub-block
  // and become (x0, x2), (x1, x3), (x4, x6), (x5, x7) -- the pairs the nibble
  // operands meet -- so no warp permutes x again.
  auto permute_x = [&](int slot, int cnt) {
    uint8_t *dst = smem + slot * C::kStageBytes + C::kWBytes + lane * 16;
#pragma unroll
    for (int m = 0; m < SB * NB / kWideWarps; ++m) {
      const int idx = warp + kWideWarps * m;
      if (idx / NB < cnt) {
        uint4 *q = reinterpret_cast<uint4 *>(dst + idx * kXRowBytes);
        const uint4 v = *q;
        uint4 pm;
        pm.x = __byte_perm(v.x, v.y, 0x5410u);
        pm.y = __byte_perm(v.x, v.y, 0x7632u);
        pm.z = __byte_perm(v.z, v.w, 0x5410u);
        pm.w = __byte_perm(v.z, v.w, 0x7632u);
        *q = pm;
      }
    }
  };

  // Ring: stage i lives in slot i % ST, ST - 1 stages ahead of the consumer.
  // With programmatic dependent launch the first weight stages go out before
  // the wait for the previous kernel, their x after it.
  WPos pp;
  wide_first(p, lo, hi, pp);
  int npre = 0;
  {
    WPos q = pp;
    for (; npre < p.pre && npre < ST - 1 && q.valid; ++npre) {
      issue_w(npre, q);
      wide_next<SB>(p, hi, q);
    }
  }
  grid_dependency_wait();
  int inflight = 0;  // stages requested and not yet consumed
  for (int s = 0; s < ST - 1; ++s) {
    if (pp.valid) {
      if (s >= npre) issue_w(s, pp);
      issue_x(s, pp);
      wide_next<SB>(p, hi, pp);
      ++inflight;
    }
  }
  grid_launch_dependents();

  // ---- consumer
  const int wrow = warp * 16;  // this warp's rows of the tile
  WPos cs;
  wide_first(p, lo, hi, cs);
  int slot = 0;
  uint32_t phase = 0;  // parity of the slot's next phase (flips when slot wraps)
  float yacc[NT][4], ygate[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) yacc[nt][e] = ygate[nt][e] = 0.f;
  while (cs.valid) {
    const WideOp &o = p.op[cs.op];
    const int cnt = min(SB, o.nsb - cs.sb);
    const int tile = cs.tile, part = cs.part;
    const bool last_of_part = cs.sb + SB >= o.nsb;
    const bool landed = mbar_wait(&full[slot], phase, p.err);  // the stage's copies
    permute_x(slot, cnt);
    fence_proxy_async_smem();  // the in-place x writes come before a later TMA refill of the slot
    // every thread's permuted x is visible, and the previous stage is consumed;
    // after a timed-out wait the CTA lets its copies in flight land and stops
    if (__syncthreads_or(!landed)) {
      if (tid == 0) drain_ring(full, ST, slot, phase, inflight);
      __syncthreads();
      break;
    }
    --inflight;
    {
      const int rs = slot == 0 ? ST - 1 : slot - 1;  // the slot the previous stage used
      if (pp.valid) {
        issue_w(rs, pp);
        issue_x(rs, pp);
        wide_next<SB>(p, hi, pp);
        ++inflight;
      }
    }
    const uint8_t *wst = smem + slot * C::kStageBytes;
    const uint8_t *xst = wst + C::kWBytes;
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      if (u >= cnt) break;
      // Super-block u of this stage for rows wrow + g, wrow + g + 8.
      uint4 hdr[2];
      uint2 qw[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint8_t *rp = wst + (wrow + g + 8 * r) * C::kRowBytes + u * kBlockBytes;
        hdr[r] = *reinterpret_cast<const uint4 *>(rp);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          qw[r][c] = *reinterpret_cast<const uint2 *>(rp + kQsOffset + 32 * c + 8 * t);
      }
      // Offset forms of sub-blocks 2t, 2t+1 (e = 0, 1) of rows g, g+8 (r);
      // the bf16 subtrahends of both rows travel packed in one word per e.
      float dsv[2][2], eev[2][2];
      uint32_t subp[2];
      {
        uint32_t sc2[2], m2[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) scales_pair(hdr[r].y, hdr[r].z, hdr[r].w, t, &sc2[r], &m2[r]);
        // rows g, g+8 as the two lanes of the packed fp32 operations
        float2 d2, nd23, dmin2, pdm23;
        scale_pairs(hdr[0].x, hdr[1].x, d2, nd23, dmin2, pdm23);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float2 ds2, ee2;
          offset_form_rows2_packed<16>(d2, nd23, dmin2, pdm23, byte_magic(sc2[0], e),
                                       byte_magic(sc2[1], e), byte_magic_neg(m2[0], e),
                                       byte_magic_neg(m2[1], e), ds2, ee2, subp[e]);
          dsv[0][e] = ds2.x;
          dsv[1][e] = ds2.y;
          eev[0][e] = ee2.x;
          eev[1][e] = ee2.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = j >> 1;
        const bool hi = j & 1;
        // B fragments of sub-block j: this lane's 16 bytes (values 8t .. 8t+7,
        // permuted) of batch row nt*8 + g: (x[o], x[o+2]) and (x[o+1], x[o+3]).
        uint32_t b0[2][NT], b1[2][NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 v = *reinterpret_cast<const uint4 *>(
              xst + (u * NB + nt * 8 + g) * kXRowBytes + 64 * j + 16 * t);
          b0[0][nt] = v.x;
          b1[0][nt] = v.y;
          b0[1][nt] = v.z;
          b1[1][nt] = v.w;
        }
        // X_j of every column (A = 1: column 2t+e is xsum[nt][e]).
        float xsum[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16_zc(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[0][nt], b1[0][nt]);
          mma_bf16(xsum[nt], kBf16One, kBf16One, kBf16One, kBf16One, b0[1][nt], b1[1][nt]);
        }
        // Offset forms of sub-block j for rows g, g+8 live in lane (g, j/2).
        const int srcl = (lane & ~3) | (j >> 1);
        const uint32_t sp = __shfl_sync(0xffffffffu, hi ? subp[1] : subp[0], srcl);
        const uint32_t sg = __byte_perm(sp, 0u, 0x1010u), sg8 = __byte_perm(sp, 0u, 0x3232u);
        float acc[NT][4];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint32_t w0 = s ? qw[0][c].y : qw[0][c].x;
          const uint32_t w1 = s ? qw[1][c].y : qw[1][c].x;
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
          const float ds = __shfl_sync(0xffffffffu, hi ? dsv[r][1] : dsv[r][0], srcl);
          const float ee = __shfl_sync(0xffffffffu, hi ? eev[r][1] : eev[r][0], srcl);
          // columns 2t, 2t+1 share ds and e: one packed fma each (each lane
          // of a pair rounds as fmaf)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float2 yv = make_float2(yacc[nt][2 * r], yacc[nt][2 * r + 1]);
            yv = __ffma2_rn(make_float2(ds, ds), make_float2(acc[nt][2 * r], acc[nt][2 * r + 1]), yv);
            yv = __ffma2_rn(make_float2(ee, ee), make_float2(xsum[nt][0], xsum[nt][1]), yv);
            yacc[nt][2 * r] = yv.x;
            yacc[nt][2 * r + 1] = yv.y;
          }
        }
      }
    }
    if (++slot == ST) {
      slot = 0;
      phase ^= 1u;
    }
    wide_next<SB>(p, hi, cs);
    if (last_of_part) {
      if (o.parts == 2 && part == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) ygate[nt][e] = yacc[nt][e];
      } else {
        // This warp's rows g, g+8 and columns nt*8 + 2t + (e & 1).
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = tile * kWideRows + wrow + g + 8 * (e >> 1);
            const int col = nt * 8 + 2 * t + (e & 1);
            if (row < o.n && col < batch)
              o.y[(size_t)col * o.ldy + row] =
                  o.parts == 2 ? silu_mul_w(ygate[nt][e], yacc[nt][e]) : yacc[nt][e];
          }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) yacc[nt][e] = 0.f;
    }
  }
  // Every stage requested was consumed (or, after a timed-out wait, given the
  // bounded time to land); nothing is left in flight.
}

// ---------------------------------------------------------------- host side

std::once_flag g_wide_attr[kMaxDevices];
int g_wide_occ[kMaxDevices][2][2];  // resident CTAs per SM: [NT - 1][op table small/large]

template <int NT, int NOPS>
int wide_setup() {
  cudaFuncSetAttribute(gemv_wide_kernel<NT, NOPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       WideCfg<NT>::kSmem);
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemv_wide_kernel<NT, NOPS>,
                                                    kWideThreads, WideCfg<NT>::kSmem) != cudaSuccess)
    return 0;
  return blocks;
}

void wide_attributes(int dev) {
  g_wide_occ[dev][0][0] = wide_setup<1, 1>();
  g_wide_occ[dev][0][1] = wide_setup<1, kWideMaxOps>();
  g_wide_occ[dev][1][0] = wide_setup<2, 1>();
  g_wide_occ[dev][1][1] = wide_setup<2, kWideMaxOps>();
}

template <int NT, int NOPS>
cudaError_t wide_chunk(const StreamOpDesc *ops, int count, int batch, int grid, bool overlap,
                       cudaStream_t stream) {
  WideParams<NOPS> prm;
  memset(&prm, 0, sizeof prm);
  long long total = 0;
  int nops = 0, nmaps = 0;
  constexpr int kMapCap = (int)(sizeof prm.map / sizeof prm.map[0]);
  // the matrix as a 2-D array of 8-byte words, one row per weight row; a tile
  // is the row slot's words of 64 rows
  auto weight_map = [&](const uint8_t *w, int n, int nsb) -> cudaError_t {
    if (nmaps >= kMapCap) return cudaErrorInvalidValue;
    const uint64_t dims[2] = {(uint64_t)nsb * (kBlockBytes / 8), (uint64_t)n};
    const uint64_t strides[1] = {(uint64_t)nsb * kBlockBytes};
    const uint32_t box[2] = {(uint32_t)(WideCfg<NT>::kRowBytes / 8), (uint32_t)kWideRows};
    const CUresult r = encode_tiled(&prm.map[nmaps++], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2,
                                    const_cast<uint8_t *>(w), dims, strides, box,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
  };
  for (int i = 0; i < count; ++i) {
    const StreamOpDesc &d = ops[i];
    if (d.n <= 0) continue;
    WideOp &o = prm.op[nops++];
    o.w = static_cast<const uint8_t *>(d.w);
    o.w2 = static_cast<const uint8_t *>(d.w_up);
    o.x = static_cast<const __nv_bfloat16 *>(d.x);
    o.y = d.y;
    o.n = (int)d.n;
    o.nsb = (int)(d.k / kQK);
    o.ntiles = (int)((d.n + kWideRows - 1) / kWideRows);
    o.parts = d.w_up ? 2 : 1;
    o.ldx = (int)d.ldx;
    o.ldy = (int)d.ldy;
    o.byte0 = total;
    o.map = nmaps;
    cudaError_t e = weight_map(o.w, o.n, o.nsb);
    if (e == cudaSuccess && o.w2) e = weight_map(o.w2, o.n, o.nsb);
    if (e != cudaSuccess) return e;
    total += (long long)d.n * o.nsb * kBlockBytes * o.parts;
  }
  if (nops == 0) return cudaSuccess;
  prm.err = device_error_word();
  prm.nops = nops;
  prm.batch = batch;
  prm.pre = overlap ? Q4K_WIDE_PRE : 0;
  prm.nctas = grid;
  prm.total = total;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kWideThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)WideCfg<NT>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_wide_kernel<NT, NOPS>, prm);
}

// Ops [i, j) of a launch chunk: ops with rows holding at most `per` weight
// matrices (a fused gate/up op holds two).
int64_t wide_chunk_end(const StreamOpDesc *ops, int64_t count, int64_t i, long long per,
                       long long *tiles) {
  int64_t j = i, used = 0, maps = 0;
  *tiles = 0;
  while (j < count) {
    if (ops[j].n > 0) {
      const int need = ops[j].w_up ? 2 : 1;
      if (used > 0 && maps + need > per) break;
      maps += need;
      ++used;
      *tiles += (ops[j].n + kWideRows - 1) / kWideRows;
    }
    ++j;
  }
  return j;
}

}  // namespace

int wide_min_batch() { return 5; }

bool wide_worth_it(const StreamOpDesc *ops, int64_t count, int batch) {
  if (batch < wide_min_batch() || batch > 16) return false;
  const DeviceFacts *f = device_facts();
  std::call_once(g_wide_attr[f->device], wide_attributes, f->device);
  const int occ = g_wide_occ[f->device][batch <= 8 ? 0 : 1][1];
  if (occ <= 0) return false;
  long long tiles = 0;
  for (int64_t i = 0; i < count; ++i)
    if (ops[i].n > 0) tiles += (ops[i].n + kWideRows - 1) / kWideRows;
  // at least two tiles per resident CTA: fewer leave SMs idle or the ring
  // fill exposed, where the per-op kernel's split of K does better
  return tiles >= 2LL * occ * f->sm_count;
}

cudaError_t launch_wide(const StreamOpDesc *ops, int64_t count, int batch, bool overlap,
                        cudaStream_t stream) {
  if (batch < 1 || batch > 16) return cudaErrorInvalidValue;
  const DeviceFacts *f = device_facts();
  std::call_once(g_wide_attr[f->device], wide_attributes, f->device);
  const int ntv = batch <= 8 ? 0 : 1;
  // Launches: as few as the kWideMaxOps weight matrices per launch allow, each
  // taking about the same number of matrices.
  long long mats = 0;
  for (int64_t i = 0; i < count; ++i)
    if (ops[i].n > 0) mats += ops[i].w_up ? 2 : 1;
  const long long nlaunch = (mats + kWideMaxOps - 1) / kWideMaxOps;
  const long long per = nlaunch > 0 ? (mats + nlaunch - 1) / nlaunch : kWideMaxOps;
  int64_t i = 0;
  while (i < count) {
    long long tiles = 0;
    const int64_t j = wide_chunk_end(ops, count, i, per, &tiles);
    if (tiles > 0) {
      const bool single = j - i == 1;
      const int occ = g_wide_occ[f->device][ntv][single ? 0 : 1];
      if (occ <= 0) return cudaErrorInvalidConfiguration;
      const int grid = (int)std::min<long long>((long long)occ * f->sm_count, tiles);
      const int n = (int)(j - i);
      cudaError_t e;
      if (ntv == 0)
        e = single ? wide_chunk<1, 1>(ops + i, n, batch, grid, overlap, stream)
                   : wide_chunk<1, kWideMaxOps>(ops + i, n, batch, grid, overlap, stream);
      else
        e = single ? wide_chunk<2, 1>(ops + i, n, batch, grid, overlap, stream)
                   : wide_chunk<2, kWideMaxOps>(ops + i, n, batch, grid, overlap, stream);
      if (e != cudaSuccess) return e;
    }
    i = j;
  }
  return cudaGetLastError();
}

}  // namespace q4k
