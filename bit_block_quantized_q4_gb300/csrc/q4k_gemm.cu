// q4k_gemm.cu -- prefill projection Y = X W^T with W in Q4_K ("spec:
// specialized model runtimes", section "Feasibility gate": one quantized GEMM;
// prefill throughput is a reported metric in "PRD: Performant Concurrent
// Distributed GGUF Runtime", DGR-001).
//
// One CTA computes a 512-token x BN-weight-row output tile (BN = 128, or 112
// when that spreads a narrow projection over more SMs), so every weight is
// dequantized exactly once per 512 tokens.  Warp roles:
//   warp 0      TMA producer of X k-blocks (512 x 64 bf16, 128-byte swizzle),
//               optionally multicast across a cluster of CTAs that share X
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer: four
//               128 x BN x 16 MMAs per 16-wide k step (one per 128-token
//               sub-tile) accumulate in fp32 in tensor memory
//   warp 2      TMA producer of raw Q4_K super-blocks (BN rows x 144 bytes)
//   warps 4..7  dequantize: thread = weight row; each 64-wide k-block is one
//               32-byte quant chunk of a super-block (low nibbles: sub-block
//               2c, high nibbles: 2c+1).  The weight is fma(d sc, q, -dmin m)
//               in fp32 (the exact value rounded once), rounded to nearest-even
//               bf16 and written in the 128-byte-swizzled K-major layout the MMA
//               reads.  After the last k-block they drain TMEM (one lane
//               quarter each), round to bf16 and store Y.
// Stages are chained by mbarriers; every wait is bounded and reports a
// timeout through the device error word instead of hanging.
#include <algorithm>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

namespace {

#ifndef Q4K_GEMM_DQ_WARPS  // dequantizing warps per CTA: 4 (a thread per weight row) or 8 (two; measured slower)
#define Q4K_GEMM_DQ_WARPS 4
#endif
constexpr int kBK = 64;  // k per block = one 128-byte swizzle panel (X stage and weight stage)

// Shared-memory plan of one CTA: SUB 128-token sub-tiles of X per stage, BN
// weight rows (dequantized bf16 stage + raw Q4_K stage), barriers, TMEM slot.
template <int BN, int SUB, int DQ>
struct GemmSmem {
  static constexpr int kTokens = 128 * SUB;
  static constexpr int kDqWarps = DQ;                      // dequantizing warps
  static constexpr int kRowSpan = BN > 128 ? BN : 128;     // weight rows one pass of them covers
  static constexpr int kPerRow = 32 * DQ / kRowSpan;       // threads per weight row (1 or 2)
  static constexpr int kThreads = 128 + 32 * kDqWarps;
  static constexpr int kXSubBytes = 128 * kBK * 2;
  static constexpr int kXStageBytes = SUB * kXSubBytes;
  static constexpr int kXStages = 2;
  static constexpr int kBStages = SUB == 4 ? 3 : 2;
  static constexpr int kRawStages = 2;
  static constexpr int kBStageBytes = BN * kBK * 2;
  static constexpr int kRawBytes = BN * kBlockBytes;
  static constexpr int kX = 0;
  static constexpr int kB = kX + kXStages * kXStageBytes;
  static constexpr int kRaw = kB + kBStages * kBStageBytes;
  static constexpr int kBars = kRaw + kRawStages * kRawBytes;
  // barriers: xfull, xempty, bfull, bempty, rfull, rempty, acc
  static constexpr int kNumBars = 2 * kXStages + 2 * kBStages + 2 * kRawStages + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct GemmArgs {
  __nv_bfloat16 *y;
  int64_t ldy;
  int m, n, k;
  unsigned *err;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Stores 16 fp32 accumulator values of row m, columns n .. n+15, as bf16.
__device__ __forceinline__ void store_y16(const GemmArgs &a, int m, int n, const float (&v)[16]) {
  if (m >= a.m || n >= a.n) return;
  __nv_bfloat16 *yrow = a.y + (int64_t)m * a.ldy;
  uint4 o0, o1;
  o0.x = pack_bf16(v[0], v[1]);
  o0.y = pack_bf16(v[2], v[3]);
  o0.z = pack_bf16(v[4], v[5]);
  o0.w = pack_bf16(v[6], v[7]);
  o1.x = pack_bf16(v[8], v[9]);
  o1.y = pack_bf16(v[10], v[11]);
  o1.z = pack_bf16(v[12], v[13]);
  o1.w = pack_bf16(v[14], v[15]);
  if (n + 16 <= a.n) {
    *reinterpret_cast<uint4 *>(yrow + n) = o0;
    *reinterpret_cast<uint4 *>(yrow + n + 8) = o1;
  } else {
    const uint32_t w[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
    for (int e = 0; e < 16 && n + e < a.n; ++e)
      yrow[n + e] = __ushort_as_bfloat16((unsigned short)(w[e >> 1] >> (16 * (e & 1))));
  }
}

// A cluster is CS x KS CTAs, rank = n + CS z.  The CS CTAs with the same z
// take consecutive BN-row weight tiles over the same K range and share X (TMA
// multicast).  The KS CTAs with the same n split K: CTA z contracts
// super-blocks [z nsb / KS, (z+1) nsb / KS) into its own TMEM, and the partial
// tiles are summed through distributed shared memory (below).
template <int BN, int SUB, int DQ, int CS, int KS>
__global__ void __launch_bounds__(GemmSmem<BN, SUB, DQ>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const GemmArgs a) {
  using L = GemmSmem<BN, SUB, DQ>;
  static_assert(L::kPerRow == 1 || L::kPerRow == 2, "one or two threads per weight row");
  static_assert(BN % 16 == 0 && BN <= 256 && SUB * BN <= 512, "MMA shape / TMEM columns");
  static_assert(BN / 16 * 128 * 64 <= L::kBars, "split-K exchange buffer");
  constexpr int kXStages = L::kXStages, kBStages = L::kBStages, kRawStages = L::kRawStages;
  constexpr int kDqWarps = L::kDqWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
  uint64_t *xfull = bars;
  uint64_t *xempty = xfull + kXStages;
  uint64_t *bfull = xempty + kXStages;
  uint64_t *bempty = bfull + kBStages;
  uint64_t *rfull = bempty + kBStages;
  uint64_t *rempty = rfull + kRawStages;
  uint64_t *accfull = rempty + kRawStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * L::kTokens;
  const uint32_t crank = (CS * KS > 1) ? cluster_ctarank() : 0u;
  const uint32_t rank = crank % CS;   // position among the CTAs sharing X
  const uint32_t krank = crank / CS;  // K range of this CTA
  // This CTA's super-blocks [sb_lo, sb_lo + nsb); every loop below runs over
  // indices relative to the range (k-block kb covers k = 64 (kb_lo + kb) ..).
  const int nsb_all = a.k / kQK;
  const int sb_lo = (int)((int64_t)krank * nsb_all / KS);
  const int nsb = (int)((int64_t)(krank + 1) * nsb_all / KS) - sb_lo;
  const int nkb = nsb * (kQK / kBK);
  const int kb_lo = sb_lo * (kQK / kBK);
  const uint16_t kMask = (uint16_t)(((1u << CS) - 1u) << (krank * CS));  // X sharers

  if (threadIdx.x == 0) {
    prefetch_tmap(&xmap);
    prefetch_tmap(&wmap);
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], CS);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&bfull[s], kDqWarps);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&rfull[s], 1);
      mbar_init(&rempty[s], kDqWarps);
    }
    mbar_init(accfull, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (CS * KS > 1) cluster_sync();  // peers' barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  bool acc_ready = false;  // dequant warps: the accumulator tile is complete

  if (warp == 0) {
    // ---------------------------------------------------------- X producer
    if (lane == 0) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kXStages;
        const uint32_t ph = (uint32_t)((kb / kXStages) & 1);
        if (!mbar_wait(&xempty[s], ph ^ 1u, a.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&xfull[s], L::kXStageBytes);
        uint8_t *dst = smem + L::kX + s * L::kXStageBytes;
        const int kx = (kb_lo + kb) * kBK;
        for (int sub = (int)rank; sub < SUB; sub += CS) {
          if (CS > 1)
            tma_load_2d_mc(dst + sub * L::kXSubBytes, &xmap, &xfull[s], kx, m0 + 128 * sub, kMask);
          else
            tma_load_2d(dst + sub * L::kXSubBytes, &xmap, &xfull[s], kx, m0 + 128 * sub);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
      const uint32_t xbase = smem_u32(smem + L::kX);
      const uint32_t bbase = smem_u32(smem + L::kB);
      for (int kb = 0; kb < nkb; ++kb) {
        const int xs = kb % kXStages, bs = kb % kBStages;
        if (!mbar_wait(&xfull[xs], (uint32_t)((kb / kXStages) & 1), a.err)) { ok = false; break; }
        if (!mbar_wait(&bfull[bs], (uint32_t)((kb / kBStages) & 1), a.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16) {
          const uint64_t bdesc = sdesc_sw128(bbase + bs * L::kBStageBytes + k16 * 32, 1024);
#pragma unroll
          for (int sub = 0; sub < SUB; ++sub) {
            const uint64_t adesc =
                sdesc_sw128(xbase + xs * L::kXStageBytes + sub * L::kXSubBytes + k16 * 32, 1024);
            tc_mma_f16(tmem + sub * BN, adesc, bdesc, idesc, (kb | k16) != 0);
          }
        }
        tc_commit(&bempty[bs]);
        if (CS > 1)
          tc_commit_mc(&xempty[xs], kMask);
        else
          tc_commit(&xempty[xs]);
      }
      tc_commit(accfull);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- raw W producer
    if (lane == 0) {
      for (int sb = 0; sb < nsb; ++sb) {
        const int s = sb % kRawStages;
        const uint32_t ph = (uint32_t)((sb / kRawStages) & 1);
        if (!mbar_wait(&rempty[s], ph ^ 1u, a.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&rfull[s], L::kRawBytes);
        tma_load_3d(smem + L::kRaw + s * L::kRawBytes, &wmap, &rfull[s], 0, sb_lo + sb, n0);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- dequantize
    const int dq = threadIdx.x - 128;
    const int row = dq % L::kRowSpan;   // weight row within the tile
    const int part = dq / L::kRowSpan;  // which chunks of a k block this thread writes
    const bool live = row < BN;         // threads past BN only keep the barrier protocol
    const int r8 = row & 7;
    uint8_t *brow0 = smem + L::kB + (live ? row >> 3 : 0) * 1024 + r8 * 128;
    for (int sb = 0; sb < nsb && ok; ++sb) {
      const int rs = sb % kRawStages;
      if (!mbar_wait(&rfull[rs], (uint32_t)((sb / kRawStages) & 1), a.err)) { ok = false; break; }
      const uint8_t *raw = smem + L::kRaw + rs * L::kRawBytes + (live ? row : 0) * kBlockBytes;
      const uint4 h = *reinterpret_cast<const uint4 *>(raw);
      uint32_t sc_lo, sc_hi, m_lo, m_hi;
      scales_all(h.y, h.z, h.w, &sc_lo, &sc_hi, &m_lo, &m_hi);
      const float d = half_lo_to_float(h.x), dmin = half_hi_to_float(h.x);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kb = sb * 4 + c;
        const int bs = kb % kBStages;
        const uint4 q0 = *reinterpret_cast<const uint4 *>(raw + kQsOffset + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4 *>(raw + kQsOffset + 32 * c + 16);
        if (c == 3) {  // raw stage fully read
          __syncwarp();
          if (lane == 0) mbar_arrive(&rempty[rs]);
        }
        // scales of sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)
        const uint32_t scw = (c < 2) ? sc_lo : sc_hi, mw = (c < 2) ? m_lo : m_hi;
        const int b0 = (2 * c) & 3;
        const float ds0 = d * (float)((scw >> (8 * b0)) & 0xFFu);
        const float ds1 = d * (float)((scw >> (8 * b0 + 8)) & 0xFFu);
        const float dm0 = dmin * (float)((mw >> (8 * b0)) & 0xFFu);
        const float dm1 = dmin * (float)((mw >> (8 * b0 + 8)) & 0xFFu);
        if (!mbar_wait(&bempty[bs], (uint32_t)(((kb / kBStages) & 1) ^ 1), a.err)) {
          ok = false;
          break;
        }
        uint8_t *brow = brow0 + bs * L::kBStageBytes;
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int jj = 0; jj < 8 / L::kPerRow; ++jj) {  // 16-byte chunk j holds k = 8j .. 8j+7
          const int j = part * (8 / L::kPerRow) + jj;
          const int hi = j >> 2;                        // chunks 4..7: high nibbles
          const uint32_t wa = words[2 * (j & 3)], wb = words[2 * (j & 3) + 1];
          const uint32_t ma = (hi ? (wa >> 4) : wa) & 0x0F0F0F0Fu;
          const uint32_t mb = (hi ? (wb >> 4) : wb) & 0x0F0F0F0Fu;
          const float ds = hi ? ds1 : ds0, dm = hi ? dm1 : dm0;
          float q[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // 0x4B00000q is 2^23 + q exactly
            q[e] = __uint_as_float(__byte_perm(ma, 0x4B000000u, 0x7540u + e)) - 8388608.f;
            q[4 + e] = __uint_as_float(__byte_perm(mb, 0x4B000000u, 0x7540u + e)) - 8388608.f;
          }
          uint4 o;
          o.x = pack_bf16(fmaf(ds, q[0], -dm), fmaf(ds, q[1], -dm));
          o.y = pack_bf16(fmaf(ds, q[2], -dm), fmaf(ds, q[3], -dm));
          o.z = pack_bf16(fmaf(ds, q[4], -dm), fmaf(ds, q[5], -dm));
          o.w = pack_bf16(fmaf(ds, q[6], -dm), fmaf(ds, q[7], -dm));
          if (live) *reinterpret_cast<uint4 *>(brow + ((j ^ r8) << 4)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bfull[bs]);
      }
    }
    acc_ready = ok && mbar_wait(accfull, 0u, a.err);
  }

  // ------------------------------------------------------------ epilogue
  // Dequant warp w drains TMEM lane quarter w % 4 (tokens 32 (w % 4) ..) and
  // its share h = (w - 4) / 4 of the 16-column chunks.
  const bool epi = warp >= 4;
  const int q = warp & 3;
  const int row = 32 * q + lane;  // token within a sub-tile
  constexpr int kPerQuarter = (BN / 16 + DQ / 4 - 1) / (DQ / 4);  // chunks per warp of a quarter
  const int c_lo = epi ? ((warp - 4) >> 2) * kPerQuarter : 0;     // first 16-column chunk
  const int c_hi = epi ? min(BN / 16, c_lo + kPerQuarter) : 0;    // end of this warp's chunks
  if (epi && acc_ready) tc_fence_after();
  if constexpr (KS == 1) {
    if (epi && acc_ready) {
      for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(sub * BN + 16 * c), r);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
          store_y16(a, m0 + 128 * sub + row, n0 + 16 * c, v);
        }
      }
    }
  } else {
    // Split-K sum, one round per 128-token sub-tile.  Every CTA copies its
    // partials of the chunks it does not own from TMEM into its own shared
    // memory (idle now: all copies and MMAs are done); after a cluster barrier
    // each CTA takes the chunks c with c % KS == its K rank, adds the KS
    // partials in K-rank order (its own from TMEM, the others from the peers'
    // shared memory) and stores Y; a second barrier frees the buffers.  Every
    // thread of every CTA passes both barriers of each round, whatever happened
    // before.  Layout: 16 columns of a row are four 16-byte units, unit u stored
    // at slot u ^ ((row >> 1) & 3) so that eight consecutive rows hit eight
    // different bank groups.
    float4 *buf = reinterpret_cast<float4 *>(smem);  // [chunk][row][4]
    const int swz = (row >> 1) & 3;
    auto unit = [&](int c, int u) { return (c * 128 + row) * 4 + (u ^ swz); };
    for (int sub = 0; sub < SUB; ++sub) {
      if (epi && acc_ready) {
#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          if (c % KS == (int)krank) continue;  // kept in TMEM, read there below
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(sub * BN + 16 * c), r);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 4; ++u)
            buf[unit(c, u)] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                          __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
        }
      }
      cluster_sync();
      if (epi && acc_ready) {
#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          if (c % KS != (int)krank) continue;
          float4 pv[KS][4];
#pragma unroll
          for (int z = 0; z < KS; ++z)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (z != (int)krank)
                pv[z][u] = ld_peer_v4(peer_smem(smem_u32(&buf[unit(c, u)]), rank + CS * (uint32_t)z));
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(sub * BN + 16 * c), r);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int z = 0; z < KS; ++z) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool mine = z == (int)krank;
              const float t0 = mine ? __uint_as_float(r[4 * u]) : pv[z][u].x;
              const float t1 = mine ? __uint_as_float(r[4 * u + 1]) : pv[z][u].y;
              const float t2 = mine ? __uint_as_float(r[4 * u + 2]) : pv[z][u].z;
              const float t3 = mine ? __uint_as_float(r[4 * u + 3]) : pv[z][u].w;
              v[4 * u] = z ? v[4 * u] + t0 : t0;
              v[4 * u + 1] = z ? v[4 * u + 1] + t1 : t1;
              v[4 * u + 2] = z ? v[4 * u + 2] + t2 : t2;
              v[4 * u + 3] = z ? v[4 * u + 3] + t3 : t3;
            }
          }
          store_y16(a, m0 + 128 * sub + row, n0 + 16 * c, v);
        }
      }
      cluster_sync();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CS * KS > 1) cluster_sync();  // no peer may still multicast into this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

std::once_flag g_gemm_attr;

constexpr int kDQ = Q4K_GEMM_DQ_WARPS;

template <int BN, int SUB, int CS, int KS>
void gemm_allow() {
  cudaFuncSetAttribute(gemm_kernel<BN, SUB, kDQ, CS, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem<BN, SUB, kDQ>::kAlloc);
}

template <int BN, int SUB>
void gemm_allow_all() {
  gemm_allow<BN, SUB, 1, 1>();
  gemm_allow<BN, SUB, 2, 1>();
  gemm_allow<BN, SUB, 1, 2>();
  gemm_allow<BN, SUB, 1, 3>();
  gemm_allow<BN, SUB, 1, 4>();
  gemm_allow<BN, SUB, 2, 2>();
  gemm_allow<BN, SUB, 2, 3>();
  gemm_allow<BN, SUB, 2, 4>();
}

void gemm_attributes() {
  gemm_allow_all<128, 4>();
  gemm_allow_all<112, 4>();
}

template <int BN, int SUB>
cudaError_t gemm_go(cudaLaunchConfig_t &cfg, int cs, int ks, const CUtensorMap &xmap,
                    const CUtensorMap &wmap, const GemmArgs &args) {
  cfg.dynamicSmemBytes = GemmSmem<BN, SUB, kDQ>::kAlloc;
  cfg.blockDim = dim3((unsigned)GemmSmem<BN, SUB, kDQ>::kThreads, 1, 1);
  auto go = [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, xmap, wmap, args); };
  if (cs == 2) {
    if (ks == 4) return go(gemm_kernel<BN, SUB, kDQ, 2, 4>);
    if (ks == 3) return go(gemm_kernel<BN, SUB, kDQ, 2, 3>);
    if (ks == 2) return go(gemm_kernel<BN, SUB, kDQ, 2, 2>);
    return go(gemm_kernel<BN, SUB, kDQ, 2, 1>);
  }
  if (ks == 4) return go(gemm_kernel<BN, SUB, kDQ, 1, 4>);
  if (ks == 3) return go(gemm_kernel<BN, SUB, kDQ, 1, 3>);
  if (ks == 2) return go(gemm_kernel<BN, SUB, kDQ, 1, 2>);
  return go(gemm_kernel<BN, SUB, kDQ, 1, 1>);
}

}  // namespace

#ifndef Q4K_GEMM_CLUSTER
#define Q4K_GEMM_CLUSTER 2
#endif
#ifndef Q4K_GEMM_SPLITK  // split K across a cluster when the output tiles cannot fill the SMs
#define Q4K_GEMM_SPLITK 1
#endif
#ifndef Q4K_GEMM_SHAPE  // 0: choose the tile per call; 128 or 112: force that weight-tile width
#define Q4K_GEMM_SHAPE 0
#endif

cudaError_t launch_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                        void *y, int64_t ldy, cudaStream_t stream) {
  std::call_once(g_gemm_attr, gemm_attributes);
  const int nsb = (int)(k / kQK);
  CUtensorMap xmap, wmap;
  {
    const uint64_t dims[2] = {(uint64_t)k, (uint64_t)m};
    const uint64_t strides[1] = {(uint64_t)ldx * 2};
    const uint32_t box[2] = {(uint32_t)kBK, 128u};
    if (encode_tiled(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  GemmArgs args;
  args.y = static_cast<__nv_bfloat16 *>(y);
  args.ldy = ldy;
  args.m = (int)m;
  args.n = (int)n;
  args.k = (int)k;
  args.err = device_error_word();

  // Tile shape, K split and X sharing.  Candidates: 512 tokens x 128 or 112
  // weight rows (112 spreads a narrow projection over more SMs).  K is split
  // across a cluster when the output tiles cannot fill the SMs.  Estimated time =
  // waves x k-blocks per CTA x the larger of the X feed (SUB x 16 KB at ~64 GB/s
  // per SM, measured) and the MMA time (~12.7 TFLOP/s per SM).  A 256 x 256 tile
  // (half the X bytes per flop, weights dequantized once per 256 tokens) was
  // measured slower on both 512-token projections and is not offered.
  const int sms = device_facts()->sm_count;
  struct Shape { int bn, sub; };
  const Shape shapes[2] = {{128, 4}, {112, 4}};
  int bn = 128, cs = 1, ks = 1, ntiles = 0, mtiles = 0;
  double best = -1;
  for (const Shape &c : shapes) {
    if (Q4K_GEMM_SHAPE && c.bn != Q4K_GEMM_SHAPE) continue;
    const int mt = (int)((m + 128 * c.sub - 1) / (128 * c.sub));
    int nt = (int)((n + c.bn - 1) / c.bn);
    int kk = 1;
    if (Q4K_GEMM_SPLITK) {
      kk = std::max(1, std::min(4, sms / std::max(1, nt * mt)));
      while (kk > 1 && nsb < 2 * kk) --kk;
    }
    int cc = Q4K_GEMM_CLUSTER > 1 ? 2 : 1;
    while (cc > 1 && (nt < 2 * cc || cc * kk > 8)) cc >>= 1;
    nt = (nt + cc - 1) / cc * cc;
    const long ctas = (long)nt * mt * kk;
    const double t_kb = std::max(c.sub * 16384.0 / 64.0, 2.0 * 128 * c.sub * c.bn * kBK / 12.7e3);
    const double est = (double)((ctas + sms - 1) / sms) * ((nsb + kk - 1) / kk) * 4 * t_kb;
    if (best < 0 || est < best) {
      best = est;
      bn = c.bn;
      cs = cc;
      ks = kk;
      ntiles = nt;
      mtiles = mt;
    }
  }
  {
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)nsb, (uint64_t)n};
    const uint64_t strides[2] = {(uint64_t)kBlockBytes, (uint64_t)nsb * kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, 1u, (uint32_t)bn};
    if (encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(w), dims, strides,
                     box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ntiles, (unsigned)mtiles, (unsigned)ks);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ks;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bn == 112) return gemm_go<112, 4>(cfg, cs, ks, xmap, wmap, args);
  return gemm_go<128, 4>(cfg, cs, ks, xmap, wmap, args);
}

}  // namespace q4k
