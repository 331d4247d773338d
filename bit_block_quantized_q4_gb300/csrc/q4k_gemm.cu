// q4k_gemm.cu -- prefill projection Y = X W^T with W in Q4_K ("spec:
// specialized model runtimes", section "Feasibility gate": one quantized GEMM;
// prefill throughput is a reported metric in "PRD: Performant Concurrent
// Distributed GGUF Runtime", DGR-001).
//
// One CTA computes a 512-token x BN-weight-row output tile, so every weight is
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

#ifndef Q4K_GEMM_XK  // k width of an X stage: 64 (128-byte swizzle) or 32 (64-byte swizzle)
#define Q4K_GEMM_XK 64
#endif
constexpr int kSub = 4;                 // 128-token sub-tiles per CTA
constexpr int kTokens = 128 * kSub;     // tokens per CTA
constexpr int kBK = 64;                 // k per weight block = one 128-byte swizzle panel
constexpr int kXK = Q4K_GEMM_XK;        // k per X stage (one swizzle panel of X)
constexpr int kXPanels = kBK / kXK;     // X stages per weight block
constexpr int kXSubBytes = 128 * kXK * 2;        // one 128-token sub-tile of an X stage
constexpr int kXStageBytes = kSub * kXSubBytes;  // 32768 or 65536
constexpr int kXStages = 131072 / kXStageBytes;  // 128 KB of X in flight either way
constexpr int kBStages = 3;
constexpr int kRawStages = 2;
constexpr int kThreads = 256;

template <int BN>
struct GemmSmem {
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

// Address of the same shared-memory byte in CTA `rank` of the cluster, and a
// 32-bit load from there.
__device__ __forceinline__ uint32_t peer_smem(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

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
// take consecutive 128-row weight tiles over the same K range and share X
// (TMA multicast).  The KS CTAs with the same n split K: CTA z contracts
// super-blocks [z nsb / KS, (z+1) nsb / KS) into its own TMEM, and the partial
// tiles meet through distributed shared memory in the z = 0 CTA, which adds
// them in z order and stores Y.
template <int BN, int CS, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const GemmArgs a) {
  static_assert(2 * BN * 128 * 4 <= kXStages * kXStageBytes, "split-K exchange buffer");
  static_assert(BN % 16 == 0, "16-column epilogue chunks");
  using L = GemmSmem<BN>;
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
  const int m0 = blockIdx.y * kTokens;
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
      mbar_init(&bfull[s], 4);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&rfull[s], 1);
      mbar_init(&rempty[s], 4);
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
      for (int xp = 0; xp < nkb * kXPanels; ++xp) {
        const int s = xp % kXStages;
        const uint32_t ph = (uint32_t)((xp / kXStages) & 1);
        if (!mbar_wait(&xempty[s], ph ^ 1u, a.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&xfull[s], kXStageBytes);
        uint8_t *dst = smem + L::kX + s * kXStageBytes;
        const int kx = kb_lo * kBK + xp * kXK;
        for (int sub = (int)rank; sub < kSub; sub += CS) {
          if (CS > 1)
            tma_load_2d_mc(dst + sub * kXSubBytes, &xmap, &xfull[s], kx, m0 + 128 * sub, kMask);
          else
            tma_load_2d(dst + sub * kXSubBytes, &xmap, &xfull[s], kx, m0 + 128 * sub);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
      const uint32_t xbase = smem_u32(smem + L::kX);
      const uint32_t bbase = smem_u32(smem + L::kB);
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int bs = kb % kBStages;
        if (!mbar_wait(&bfull[bs], (uint32_t)((kb / kBStages) & 1), a.err)) { ok = false; break; }
        for (int h = 0; h < kXPanels; ++h) {
          const int xp = kb * kXPanels + h, xs = xp % kXStages;
          if (!mbar_wait(&xfull[xs], (uint32_t)((xp / kXStages) & 1), a.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k16 = 0; k16 < kXK / 16; ++k16) {
            const uint64_t bdesc =
                sdesc_sw128(bbase + bs * L::kBStageBytes + (h * (kXK / 16) + k16) * 32, 1024);
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              const uint32_t xa = xbase + xs * kXStageBytes + sub * kXSubBytes + k16 * 32;
              const uint64_t adesc = kXK == 64 ? sdesc_sw128(xa, 1024) : sdesc_sw64(xa, 512);
              tc_mma_f16(tmem + sub * BN, adesc, bdesc, idesc, (kb | h | k16) != 0);
            }
          }
          if (CS > 1)
            tc_commit_mc(&xempty[xs], kMask);
          else
            tc_commit(&xempty[xs]);
        }
        if (!ok) break;
        tc_commit(&bempty[bs]);
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
    const int row = threadIdx.x - 128;  // weight row within the tile
    const int r8 = row & 7;
    uint8_t *brow0 = smem + L::kB + (row >> 3) * 1024 + r8 * 128;
    for (int sb = 0; sb < nsb && ok; ++sb) {
      const int rs = sb % kRawStages;
      if (!mbar_wait(&rfull[rs], (uint32_t)((sb / kRawStages) & 1), a.err)) { ok = false; break; }
      const uint8_t *raw = smem + L::kRaw + rs * L::kRawBytes + row * kBlockBytes;
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
        for (int j = 0; j < 8; ++j) {     // 16-byte chunk j holds k = 8j .. 8j+7
          const int hi = j >> 2;          // chunks 4..7: high nibbles
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
          *reinterpret_cast<uint4 *>(brow + ((j ^ r8) << 4)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bfull[bs]);
      }
    }
    // ---------------------------------------------------------- epilogue
    acc_ready = ok && mbar_wait(accfull, 0u, a.err);
    if (KS == 1 && acc_ready) {
      tc_fence_after();
      const int q = warp & 3;  // TMEM lane quarter of this warp
      for (int sub = 0; sub < kSub; ++sub) {
        const int m = m0 + 128 * sub + 32 * q + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(sub * BN + c0), r);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
          store_y16(a, m, n0 + c0, v);
        }
      }
    }
  }

  if constexpr (KS > 1) {
    // ---------------------------------------------------------- split-K sum
    // Two rounds of two 128-token sub-tiles.  Every CTA copies its partials
    // from TMEM into its own X stage area (idle now); after a cluster barrier
    // each CTA takes the 16-column chunks i with i % KS == its K rank, adds the
    // KS partials of those in K-rank order (its own from TMEM, the others from
    // the peers' shared memory) and stores Y; a second barrier frees the
    // buffers.  Every thread of every CTA passes both barriers of each round,
    // whatever happened before.  Layout: 16 columns of a row are four 16-byte
    // units, unit u stored at slot u ^ ((row >> 1) & 3) so that eight
    // consecutive rows hit eight different bank groups.
    float4 *buf = reinterpret_cast<float4 *>(smem + L::kX);  // [s2][c0/16][row][4]
    const bool epi = warp >= 4;
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const int swz = (row >> 1) & 3;
    constexpr int kChunks = 2 * (BN / 16);  // 16-column chunks per round
    auto unit = [&](int idx, int u) { return (idx * 128 + row) * 4 + (u ^ swz); };
    if (epi && acc_ready) tc_fence_after();
    for (int p = 0; p < kSub / 2; ++p) {
      if (epi && acc_ready) {
#pragma unroll 1
        for (int idx = 0; idx < kChunks; ++idx) {
          if (idx % KS == (int)krank) continue;  // kept in TMEM, read there below
          const int s2 = idx / (BN / 16), c0 = (idx % (BN / 16)) * 16;
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((2 * p + s2) * BN + c0), r);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 4; ++u)
            buf[unit(idx, u)] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                            __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
        }
      }
      cluster_sync();
      if (epi && acc_ready) {
#pragma unroll 1
        for (int idx = (int)krank; idx < kChunks; idx += KS) {
          const int s2 = idx / (BN / 16), c0 = (idx % (BN / 16)) * 16;
          float4 pv[KS][4];
#pragma unroll
          for (int z = 0; z < KS; ++z)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (z != (int)krank)
                pv[z][u] = ld_peer_v4(peer_smem(smem_u32(&buf[unit(idx, u)]), rank + CS * (uint32_t)z));
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((2 * p + s2) * BN + c0), r);
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
          store_y16(a, m0 + 128 * (2 * p + s2) + row, n0 + c0, v);
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

constexpr int kBN = 128;

std::once_flag g_gemm_attr;

template <int CS, int KS>
void gemm_allow() {
  cudaFuncSetAttribute(gemm_kernel<kBN, CS, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem<kBN>::kAlloc);
  if (CS * KS > 8)
    cudaFuncSetAttribute(gemm_kernel<kBN, CS, KS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

void gemm_attributes() {
  gemm_allow<1, 1>();
  gemm_allow<2, 1>();
  gemm_allow<4, 1>();
  gemm_allow<1, 2>();
  gemm_allow<1, 3>();
  gemm_allow<1, 4>();
  gemm_allow<2, 2>();
  gemm_allow<2, 3>();
  gemm_allow<2, 4>();
}

}  // namespace

#ifndef Q4K_GEMM_CLUSTER
#define Q4K_GEMM_CLUSTER 2
#endif
#ifndef Q4K_GEMM_SPLITK  // split K across a cluster when the output tiles cannot fill the SMs
#define Q4K_GEMM_SPLITK 1
#endif

cudaError_t launch_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                        void *y, int64_t ldy, cudaStream_t stream) {
  std::call_once(g_gemm_attr, gemm_attributes);
  const int nsb = (int)(k / kQK);
  CUtensorMap xmap, wmap;
  {
    const uint64_t dims[2] = {(uint64_t)k, (uint64_t)m};
    const uint64_t strides[1] = {(uint64_t)ldx * 2};
    const uint32_t box[2] = {(uint32_t)kXK, 128u};
    if (encode_tiled(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims,
                     strides, box,
                     kXK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)nsb, (uint64_t)n};
    const uint64_t strides[2] = {(uint64_t)kBlockBytes, (uint64_t)nsb * kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, 1u, (uint32_t)kBN};
    if (encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(w), dims, strides,
                     box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  GemmArgs args;
  args.y = static_cast<__nv_bfloat16 *>(y);
  args.ldy = ldy;
  args.m = (int)m;
  args.n = (int)n;
  args.k = (int)k;
  args.err = device_error_word();

  int ntiles = (int)((n + kBN - 1) / kBN);
  const int mtiles = (int)((m + kTokens - 1) / kTokens);
  // Too few output tiles to fill the SMs (a wide-K projection such as the
  // 17408 -> 5120 down projection): split K across a cluster instead.
  int ks = 1;
  if (Q4K_GEMM_SPLITK) {
    ks = std::max(1, std::min(4, device_facts()->sm_count / std::max(1, ntiles * mtiles)));
    while (ks > 1 && nsb < 2 * ks) --ks;
  }
  int cs = Q4K_GEMM_CLUSTER;
  while (cs > 1 && (ntiles < 2 * cs || cs * ks > 8)) cs >>= 1;
  ntiles = (ntiles + cs - 1) / cs * cs;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ntiles, (unsigned)mtiles, (unsigned)ks);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = GemmSmem<kBN>::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ks;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto go = [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, xmap, wmap, args); };
  if (cs == 2) {
    if (ks == 4) return go(gemm_kernel<kBN, 2, 4>);
    if (ks == 3) return go(gemm_kernel<kBN, 2, 3>);
    if (ks == 2) return go(gemm_kernel<kBN, 2, 2>);
    return go(gemm_kernel<kBN, 2, 1>);
  }
  if (cs == 4) return go(gemm_kernel<kBN, 4, 1>);
  if (ks == 4) return go(gemm_kernel<kBN, 1, 4>);
  if (ks == 3) return go(gemm_kernel<kBN, 1, 3>);
  if (ks == 2) return go(gemm_kernel<kBN, 1, 2>);
  return go(gemm_kernel<kBN, 1, 1>);
}

}  // namespace q4k
