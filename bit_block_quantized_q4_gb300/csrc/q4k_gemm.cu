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

constexpr int kSub = 4;                 // 128-token sub-tiles per CTA
constexpr int kTokens = 128 * kSub;     // tokens per CTA
constexpr int kBK = 64;                 // k per block = one 128-byte swizzle panel
constexpr int kXStageBytes = kTokens * kBK * 2;  // 65536
constexpr int kXStages = 2;
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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int BN, int CS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const GemmArgs a) {
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
  const int nkb = a.k / kBK;
  const int nsb = a.k / kQK;
  const uint32_t rank = (CS > 1) ? cluster_ctarank() : 0u;
  constexpr uint16_t kMask = (uint16_t)((1u << CS) - 1u);

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
  if (CS > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------- X producer
    if (lane == 0) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kXStages;
        const uint32_t ph = (uint32_t)((kb / kXStages) & 1);
        if (!mbar_wait(&xempty[s], ph ^ 1u, a.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&xfull[s], kXStageBytes);
        uint8_t *dst = smem + L::kX + s * kXStageBytes;
        for (int sub = (int)rank; sub < kSub; sub += CS) {
          if (CS > 1)
            tma_load_2d_mc(dst + sub * (128 * 128), &xmap, &xfull[s], kb * kBK, m0 + 128 * sub,
                           kMask);
          else
            tma_load_2d(dst + sub * (128 * 128), &xmap, &xfull[s], kb * kBK, m0 + 128 * sub);
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
          for (int sub = 0; sub < kSub; ++sub) {
            const uint64_t adesc =
                sdesc_sw128(xbase + xs * kXStageBytes + sub * (128 * 128) + k16 * 32, 1024);
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
        tma_load_3d(smem + L::kRaw + s * L::kRawBytes, &wmap, &rfull[s], 0, sb, n0);
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
    if (ok && mbar_wait(accfull, 0u, a.err)) {
      tc_fence_after();
      const int q = warp & 3;  // TMEM lane quarter of this warp
      for (int sub = 0; sub < kSub; ++sub) {
        const int m = m0 + 128 * sub + 32 * q + lane;
        __nv_bfloat16 *yrow = a.y + (int64_t)m * a.ldy;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(sub * BN + c0), r);
          tmem_ld_wait();
          const int n = n0 + c0;
          if (m < a.m && n < a.n) {
            uint4 o0, o1;
            o0.x = pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1]));
            o0.y = pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3]));
            o0.z = pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5]));
            o0.w = pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7]));
            o1.x = pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9]));
            o1.y = pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11]));
            o1.z = pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13]));
            o1.w = pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15]));
            if (n + 16 <= a.n) {
              *reinterpret_cast<uint4 *>(yrow + n) = o0;
              *reinterpret_cast<uint4 *>(yrow + n + 8) = o1;
            } else {
              const uint32_t v[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
              for (int e = 0; e < 16 && n + e < a.n; ++e)
                yrow[n + e] = __ushort_as_bfloat16((unsigned short)(v[e >> 1] >> (16 * (e & 1))));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CS > 1) cluster_sync();  // no peer may still multicast into this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr int kBN = 128;

std::once_flag g_gemm_attr;

void gemm_attributes() {
  cudaFuncSetAttribute(gemm_kernel<kBN, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem<kBN>::kAlloc);
  cudaFuncSetAttribute(gemm_kernel<kBN, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem<kBN>::kAlloc);
  cudaFuncSetAttribute(gemm_kernel<kBN, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem<kBN>::kAlloc);
  cudaFuncSetAttribute(gemm_kernel<kBN, 2>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncSetAttribute(gemm_kernel<kBN, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

#ifndef Q4K_GEMM_CLUSTER
#define Q4K_GEMM_CLUSTER 2
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
  int cs = Q4K_GEMM_CLUSTER;
  while (cs > 1 && ntiles < 2 * cs) cs >>= 1;
  ntiles = (ntiles + cs - 1) / cs * cs;
  const int mtiles = (int)((m + kTokens - 1) / kTokens);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ntiles, (unsigned)mtiles, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = GemmSmem<kBN>::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cs == 4) return cudaLaunchKernelEx(&cfg, gemm_kernel<kBN, 4>, xmap, wmap, args);
  if (cs == 2) return cudaLaunchKernelEx(&cfg, gemm_kernel<kBN, 2>, xmap, wmap, args);
  return cudaLaunchKernelEx(&cfg, gemm_kernel<kBN, 1>, xmap, wmap, args);
}

}  // namespace q4k
