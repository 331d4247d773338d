// q4k_gemm.cu -- prefill projection Y = X W^T with W in Q4_K ("spec:
// specialized model runtimes", section "Feasibility gate": one quantized GEMM;
// prefill throughput is a reported metric in "PRD: Performant Concurrent
// Distributed GGUF Runtime", DGR-001).
//
// One CTA computes a 512-token x 128-weight-row output tile, so every weight
// is dequantized exactly once per 512 tokens.  The MMA is oriented with the
// weights as its A operand (M = 128 rows) and X as its B operand (N = 256
// tokens): per 16-wide k step two 128 x 256 x 16 MMAs read 4 KB of weights
// twice and 16 KB of X once from shared memory, where X as A would read the
// weights four times.  Shared-memory bandwidth, not the tensor pipe, is what
// bounds this kernel: the MMA operand reads, the X copies and the dequantized
// weight stores all go through it.  Warp roles:
//   warp 0      TMA producer of X k-blocks (512 x 64 bf16, 128-byte swizzle,
//               each 256-token half with its own barriers), optionally
//               multicast across a cluster of CTAs that share X
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer; the fp32
//               accumulator D[row][token] fills all 512 TMEM columns
//   warp 2      TMA producer of raw Q4_K super-blocks (128 rows x 144 bytes)
//   warps 4..7  dequantize: thread = weight row; each 64-wide k-block is one
//               32-byte quant chunk of a super-block (low nibbles: sub-block
//               2c, high nibbles: 2c+1).  The weight is fma(d sc, q, -dmin m)
//               in fp32 (the exact value rounded once), rounded to nearest-even
//               bf16 and written in the 128-byte-swizzled K-major layout the MMA
//               reads.
// After the last k-block all eight warps drain TMEM (warp w: lane quarter
// w % 4, half w / 4 of the columns) and round to bf16; the tile is staged as
// [token][row] in the idle shared memory and written as whole token rows.
// With split K the CTAs of a weight tile first push the partials of the column
// chunks they do not own into the owners' shared memory (below).
// With an RMSNorm prologue (q4k_gemm_rmsnorm) the normalised activations are
// never formed: Y[t, n] = rinv[t] sum_k (W[n, k] gamma[k]) X[t, k].  The
// dequantizing warps round fma(d sc, q, -dmin m) * gamma[k] to bf16 (gamma
// through the read-only path: every lane of a warp reads the same address),
// and the epilogue scales each token's accumulators by rinv[t], computed by
// rms_rinv_kernel (one CTA per token) while the main loop runs.
// Grouped (G = true; the expert matmuls of routed-MoE prefill): CTA (n-tile,
// slot) multiplies the tokens of one work slot -- rows [p0, p0 + np) of an
// expert-sorted X, np <= 256 -- by 128 rows of the slot's expert, whose Q4_K
// matrix is reached through a fourth (expert) dimension of the weight tensor
// map.  The slot table comes from the route kernel; a CTA whose slot is not in
// use does nothing.  The slot's 128-row sub-tiles that hold tokens are copied
// and multiplied with N = np rounded up to 16 (rows past the slot's end are
// computed and not stored).  With so few tokens per weight tile the latency of
// the X copies is what bounds the tile, so the X region holds four stages of
// 256 tokens instead of two of 512.  Output rows are the slot's rows of an
// expert-sorted Y.
// The kernel is launched as a programmatic dependent of the kernel before it
// and touches no global memory before that kernel has completed.
// Stages are chained by mbarriers; every wait is bounded and reports a
// timeout through the device error word instead of hanging; after a timeout
// the CTA writes no Y.
#include <algorithm>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

namespace {

constexpr int kBK = 64;        // k per block = one 128-byte swizzle panel (X stage and weight stage)
constexpr int kBN = 128;       // weight rows per CTA = the MMA's M
constexpr int kTokens = 512;   // tokens per CTA = two MMAs of N = 256
constexpr int kSub = kTokens / 128;  // 128-token sub-tiles (one X copy each)
constexpr int kDqWarps = 4;    // dequantizing warps, a thread per weight row
constexpr int kThreads = 128 + 32 * kDqWarps;

// Shared-memory plan of one CTA.
struct GemmSmem {
  static constexpr int kXSubBytes = 128 * kBK * 2;            // 16 KB
  static constexpr int kXStageBytes = kSub * kXSubBytes;      // 64 KB
  static constexpr int kXStages = 2;
  static constexpr int kXParts = 2;                           // 256-token halves per stage
  static constexpr int kXPartBytes = kXStageBytes / kXParts;  // 32 KB
  static constexpr int kBStages = 3;
  static constexpr int kRawStages = 2;
  static constexpr int kBStageBytes = kBN * kBK * 2;          // 16 KB
  static constexpr int kRawBytes = kBN * kBlockBytes;         // 18 KB
  static constexpr int kX = 0;
  static constexpr int kB = kX + kXStages * kXStageBytes;
  static constexpr int kRaw = kB + kBStages * kBStageBytes;
  static constexpr int kRinv = kRaw + kRawStages * kRawBytes;  // rinv of the tile's tokens
  static constexpr int kBars = kRinv + kTokens * 4;
  // barriers: xfull, xempty (per stage and half), bfull, bempty, rfull, rempty,
  // acc, split-K partials received
  // grouped tiles (at most 256 tokens) use the X region as 4 stages of one
  // 256-token half each: the same 4 pairs of X barriers
  static constexpr int kXStagesG = kXStages * kXParts;
  static constexpr int kNumBars = 4 * kXStages + 2 * kBStages + 2 * kRawStages + 2;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};
static_assert(GemmSmem::kAlloc <= 227 * 1024, "shared memory per CTA");
// Split-K: the 16-column chunks of the accumulator (8 per 128-token sub-tile)
// are dealt out to the K ranks, chunk c to rank c % KS.  A rank receives the
// other ranks' partials of its chunks into the stage memory below the barriers,
// one 8 KB block (128 rows x 64 bytes) per (sub-tile, owned chunk, sender).
__host__ __device__ constexpr int owned_max(int ks) { return (kBN / 16 + ks - 1) / ks; }
__host__ __device__ constexpr int recv_bytes(int ks) {
  return ks > 1 ? kSub * owned_max(ks) * (ks - 1) * 128 * 64 : 0;
}
static_assert(recv_bytes(2) <= GemmSmem::kBars && recv_bytes(3) <= GemmSmem::kBars &&
                  recv_bytes(4) <= GemmSmem::kBars,
              "split-K receive buffer");

struct GemmArgs {
  __nv_bfloat16 *y;
  int64_t ldy;
  int m, n, k;
  const float *gamma;  // RMSNorm weights (k), or null: no norm
  const float *rinv;   // per-token 1/rms (m), when gamma is set
  // grouped: the route kernel's slot table (meta[0] = slots in use)
  const int *slot_expert, *slot_start, *meta;
  unsigned *err;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Stores 16 fp32 accumulator values of weight row n, tokens m .. m+15, as bf16.
// Lanes 2i and 2i+1 hold adjacent rows: after one exchange the even lane writes
// the (row n, row n+1) pairs of tokens m, m+2, .. and the odd lane those of
// tokens m+1, m+3, .., four bytes per store.  Every lane of the warp calls it.
__device__ __forceinline__ void store_y16_rows(const GemmArgs &a, int m, int n, const float (&v)[16]) {
  const bool odd = (threadIdx.x & 1) != 0;
  const int nn = odd ? n - 1 : n;  // first row of the pair
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float got = __shfl_xor_sync(0xffffffffu, odd ? v[e] : v[e + 1], 1);
    const int mm = m + e + (odd ? 1 : 0);
    const float lo = odd ? got : v[e];
    const float hi = odd ? v[e + 1] : got;
    if (mm < a.m && nn < a.n) {
      __nv_bfloat16 *p = a.y + (int64_t)mm * a.ldy + nn;
      if (nn + 1 < a.n)
        *reinterpret_cast<uint32_t *>(p) = pack_bf16(lo, hi);
      else
        *p = __float2bfloat16_rn(lo);
    }
  }
}

// A cluster is CS x KS CTAs, rank = n + CS z.  The CS CTAs with the same z
// take consecutive 128-row weight tiles over the same K range and share X (TMA
// multicast).  The KS CTAs with the same n split K: CTA z contracts
// super-blocks [z nsb / KS, (z+1) nsb / KS) into its own TMEM, and the partial
// tiles are summed through distributed shared memory (below).
template <int CS, int KS, bool G = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const GemmArgs a) {
  static_assert(!G || (CS == 1 && KS == 1), "grouped tiles: one CTA per tile, no multicast");
  using L = GemmSmem;
  // X stages: 2 of 512 tokens (two 256-token halves), or, grouped, 4 of 256
  constexpr int kXStages = G ? L::kXStagesG : L::kXStages;
  constexpr int kXParts = G ? 1 : L::kXParts;
  constexpr int kXStride = G ? L::kXPartBytes : L::kXStageBytes;
  constexpr int kBStages = L::kBStages, kRawStages = L::kRawStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  auto raw_stage = [&](int s) -> uint8_t * { return smem + L::kRaw + s * L::kRawBytes; };
  auto b_stage = [&](int s) -> uint8_t * { return smem + L::kB + s * L::kBStageBytes; };
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
  uint64_t *xfull = bars;  // [stage * kXParts + half]
  uint64_t *xempty = xfull + kXStages * kXParts;
  uint64_t *bfull = xempty + kXStages * kXParts;
  uint64_t *bempty = bfull + kBStages;
  uint64_t *rfull = bempty + kBStages;
  uint64_t *rempty = rfull + kRawStages;
  uint64_t *accfull = rempty + kRawStages;
  uint64_t *redfull = accfull + 1;  // split-K: all peer partials of the owned chunks landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN;
  int m0 = G ? 0 : blockIdx.y * kTokens;
  const uint32_t crank = (CS * KS > 1) ? cluster_ctarank() : 0u;
  const uint32_t rank = crank % CS;   // position among the CTAs sharing X
  const uint32_t krank = crank / CS;  // K range of this CTA
  // This CTA's super-blocks [sb_lo, sb_lo + nsb); every loop below runs over
  // indices relative to the range (k-block kb covers k = 64 (kb_lo + kb) ..).
  const int nsb_all = a.k / kQK;
  const int sb_lo = (int)((int64_t)krank * nsb_all / KS);
  int nsb = (int)((int64_t)(krank + 1) * nsb_all / KS) - sb_lo;
  int nkb = nsb * (kQK / kBK);
  const int kb_lo = sb_lo * (kQK / kBK);
  int np = kTokens;  // tokens of this tile (grouped: of the slot)
  int expert = 0;
  const uint16_t kMask = (uint16_t)(((1u << CS) - 1u) << (krank * CS));  // X sharers

  if (threadIdx.x == 0) {
    prefetch_tmap(&xmap);
    prefetch_tmap(&wmap);
    for (int s = 0; s < kXStages * kXParts; ++s) {
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
    mbar_init(redfull, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // Every barrier below is reached by whole, reconverged warps: a warp whose
  // lanes arrive separately would be counted more than once.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (CS * KS > 1) cluster_sync();  // peers' barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  // Launched as a programmatic dependent of the previous kernel on the stream:
  // everything above overlaps its tail; no thread touches global memory before
  // that kernel has completed.  With the RMSNorm prologue the previous kernel
  // is rms_rinv_kernel, and this kernel cannot start before each of its CTAs
  // has waited for the kernel before it (the producer of X) and only then let
  // its dependents launch: X and W are complete here, and only rinv is waited
  // for (before the epilogue), so the main loop overlaps the rinv pass.
  if (!a.gamma) grid_dependency_wait();
  if constexpr (G) {
    // the slot table is the route kernel's output: read after the wait
    const int slot = blockIdx.y;
    if (slot < a.meta[0]) {
      m0 = a.slot_start[slot];
      // at most 256 (the route kernel's slot size): one 256-token X stage
      np = min(a.slot_start[slot + 1] - m0, 256);
      expert = a.slot_expert[slot];
    } else {
      np = 0;
    }
    if (np <= 0) nsb = nkb = 0;  // every role loop below is empty
  } else {
    np = min(kTokens, a.m - m0);
  }

  if (warp == 0) {
    // ---------------------------------------------------------- X producer
    if (lane == 0) {
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kXStages;
        const uint32_t ph = (uint32_t)((kb / kXStages) & 1);
        uint8_t *dst = smem + L::kX + s * kXStride;
        const int kx = (kb_lo + kb) * kBK;
        for (int h = 0; h < kXParts; ++h) {
          if (G && np <= 256 * h) break;  // no tokens in this half
          uint64_t *full = &xfull[s * kXParts + h];
          if (!mbar_wait(&xempty[s * kXParts + h], ph ^ 1u, a.err)) { ok = false; break; }
          // grouped: only the 128-row sub-tiles that hold tokens
          const int nsub = G ? min(2, (np - 256 * h + 127) / 128) : 2;
          mbar_arrive_expect_tx(full, (uint32_t)nsub * L::kXSubBytes);
          for (int sub = 2 * h + (int)rank; sub < 2 * h + nsub; sub += CS) {
            if (CS > 1)
              tma_load_2d_mc(dst + sub * L::kXSubBytes, &xmap, full, kx, m0 + 128 * sub, kMask);
            else
              tma_load_2d(dst + sub * L::kXSubBytes, &xmap, full, kx, m0 + 128 * sub);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // N = 256 per half; grouped: the half's tokens rounded up to 16
      const uint32_t idesc0 = G ? idesc_bf16_f32(kBN, min(256, (np + 15) / 16 * 16))
                                : idesc_bf16_f32(kBN, 256);
      const uint32_t idesc1 = G ? idesc_bf16_f32(kBN, max(16, min(256, (np - 256 + 15) / 16 * 16)))
                                : idesc_bf16_f32(kBN, 256);
      const uint32_t xbase = smem_u32(smem + L::kX);

      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int xs = kb % kXStages, bs = kb % kBStages;
        if (!mbar_wait(&bfull[bs], (uint32_t)((kb / kBStages) & 1), a.err)) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < kXParts; ++h) {
          if (G && np <= 256 * h) break;  // no tokens in this half
          const uint32_t idesc = h ? idesc1 : idesc0;
          if (!mbar_wait(&xfull[xs * kXParts + h], (uint32_t)((kb / kXStages) & 1), a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // D[row][token] += W[row][k] X[token][k] for the tokens of half h:
          // A = the 128 weight rows, B = sub-tiles 2h, 2h+1 (256 rows of 128
          // bytes, contiguous), accumulated in TMEM columns 256 h ...
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16) {
            const uint64_t wdesc = sdesc_sw128(smem_u32(b_stage(bs)) + k16 * 32, 1024);
            const uint64_t xdesc =
                sdesc_sw128(xbase + xs * kXStride + h * L::kXPartBytes + k16 * 32, 1024);
            tc_mma_f16(tmem + h * 256, wdesc, xdesc, idesc, (kb | k16) != 0);
          }
          if (CS > 1)
            tc_commit_mc(&xempty[xs * kXParts + h], kMask);
          else
            tc_commit(&xempty[xs * kXParts + h]);
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
        if (G)
          tma_load_4d(raw_stage(s), &wmap, &rfull[s], 0, sb_lo + sb, n0, expert);
        else
          tma_load_3d(raw_stage(s), &wmap, &rfull[s], 0, sb_lo + sb, n0);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- dequantize
    const int row = threadIdx.x - 128;  // weight row within the tile
    const int r8 = row & 7;
    const bool norm = a.gamma != nullptr;
    const int brow_off = (row >> 3) * 1024 + r8 * 128;
    for (int sb = 0; sb < nsb && ok; ++sb) {
      const int rs = sb % kRawStages;
      if (!mbar_wait(&rfull[rs], (uint32_t)((sb / kRawStages) & 1), a.err)) { ok = false; break; }
      const uint8_t *raw = raw_stage(rs) + row * kBlockBytes;
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
        uint8_t *brow = b_stage(bs) + brow_off;
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // 16-byte chunk j holds k = 8j .. 8j+7
          const int hi = j >> 2;       // chunks 4..7: high nibbles
          const uint32_t wa = words[2 * (j & 3)], wb = words[2 * (j & 3) + 1];
          const uint32_t ma = (hi ? (wa >> 4) : wa) & 0x0F0F0F0Fu;
          const uint32_t mb = (hi ? (wb >> 4) : wb) & 0x0F0F0F0Fu;
          const float ds = hi ? ds1 : ds0, dm = hi ? dm1 : dm0;
          // pairs of weights on the packed fp32 pipe (each lane of a pair
          // rounds exactly as the scalar operation): 0x4B00000q is 2^23 + q
          // exactly, so the subtraction gives q exactly; then fma(ds, q, -dm)
          const float2 m23 = make_float2(-8388608.f, -8388608.f);
          const float2 ds2 = make_float2(ds, ds), ndm2 = make_float2(-dm, -dm);
          float2 wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t src = e < 2 ? ma : mb;
            const float2 qq = __fadd2_rn(
                make_float2(__uint_as_float(__byte_perm(src, 0x4B000000u, 0x7540u + 2 * (e & 1))),
                            __uint_as_float(__byte_perm(src, 0x4B000000u, 0x7541u + 2 * (e & 1)))),
                m23);
            wv[e] = __ffma2_rn(ds2, qq, ndm2);
          }
          if (norm) {  // gamma of k = 64 c + 8 j .. + 7 (the same for every row)
            const float4 *gp = reinterpret_cast<const float4 *>(
                a.gamma + (size_t)(sb_lo + sb) * kQK + 64 * c + 8 * j);
            const float4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
            wv[0] = __fmul2_rn(wv[0], make_float2(g0.x, g0.y));
            wv[1] = __fmul2_rn(wv[1], make_float2(g0.z, g0.w));
            wv[2] = __fmul2_rn(wv[2], make_float2(g1.x, g1.y));
            wv[3] = __fmul2_rn(wv[3], make_float2(g1.z, g1.w));
          }
          uint4 o;
          o.x = pack_bf16(wv[0].x, wv[0].y);
          o.y = pack_bf16(wv[1].x, wv[1].y);
          o.z = pack_bf16(wv[2].x, wv[2].y);
          o.w = pack_bf16(wv[3].x, wv[3].y);
          *reinterpret_cast<uint4 *>(brow + ((j ^ r8) << 4)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bfull[bs]);
      }
    }
  }

  // ------------------------------------------------------------ epilogue
  // Warp w drains TMEM lane quarter w % 4 (weight rows 32 (w % 4) ..) and, of
  // each 128-token sub-tile, the 16-column chunks [4 (w / 4), 4 (w / 4) + 4).
  __syncwarp();
  ok = __all_sync(0xffffffffu, ok);  // a role loop that timed out ran on lane 0 only
  const bool acc_ready = ok && mbar_wait(accfull, 0u, a.err) && np > 0;
  grid_launch_dependents();  // the next kernel's CTAs may take this SM as soon as it is free
  const int q = warp & 3;
  const int row = 32 * q + lane;  // weight row within the tile
  const int c_lo = (warp >> 2) * 4, c_hi = c_lo + 4;
  const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
  if (acc_ready) tc_fence_after();
  // 1/rms of the tile's tokens, staged once (every role loop is done; the
  // region is used by nothing else)
  float *rinv_s = reinterpret_cast<float *>(smem + L::kRinv);
  if (a.gamma) {
    grid_dependency_wait();  // rms_rinv_kernel has completed: rinv is written
    for (int i = threadIdx.x; i < kTokens; i += kThreads)
      rinv_s[i] = (m0 + i < a.m) ? a.rinv[m0 + i] : 0.f;
    __syncthreads();
  }
  if constexpr (KS == 1) {
    // The bf16 tile is staged as [token][row] in shared memory (idle now: all
    // copies and MMAs are done) and then written as whole 256-byte token rows;
    // stores straight from the lanes (one weight row each) write 64 contiguous
    // bytes at a time and measured ~10x slower.
    __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(smem);  // [kTokens][kBN]
    if (acc_ready) {
#pragma unroll 1
      for (int sub = 0; sub < kSub && 128 * sub < np; ++sub) {
        // the warp's four 16-column chunks of the sub-tile: loads together, one wait
        uint32_t r[4][16];
#pragma unroll
        for (int ci = 0; ci < 4; ++ci)
          tmem_ld_x16(tq + (uint32_t)(sub * 128 + 16 * (c_lo + ci)), r[ci]);
        tmem_ld_wait();
        __nv_bfloat16 *col = stage + (128 * sub + 16 * c_lo) * kBN + row;
        const float *rv = rinv_s + 128 * sub + 16 * c_lo;
#pragma unroll
        for (int ci = 0; ci < 4; ++ci)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float v = __uint_as_float(r[ci][e]);
            col[(16 * ci + e) * kBN] = __float2bfloat16_rn(a.gamma ? v * rv[16 * ci + e] : v);
          }
      }
    }
    if (__syncthreads_and(acc_ready)) {
      const int seg = threadIdx.x & 15;  // 16-byte segment of a token row
      const int n = n0 + 8 * seg;
      for (int tok = threadIdx.x >> 4; tok < np; tok += kThreads / 16) {
        const uint4 v = *reinterpret_cast<const uint4 *>(stage + tok * kBN + 8 * seg);
        __nv_bfloat16 *dst = a.y + (int64_t)(m0 + tok) * a.ldy + n;
        if (n + 8 <= a.n) {
          *reinterpret_cast<uint4 *>(dst) = v;
        } else {
          const __nv_bfloat16 *e8 = reinterpret_cast<const __nv_bfloat16 *>(&v);
          for (int e = 0; e < 8 && n + e < a.n; ++e) dst[e] = e8[e];
        }
      }
    }
  } else {
    // Split-K sum.  After a cluster barrier (every CTA is done with its stage
    // memory), each CTA pushes its partials of the chunks it does not own
    // straight from TMEM into the owner's receive blocks (st.async, counted on
    // the owner's redfull barrier); the owner waits for all of them, adds the
    // KS partials in K-rank order (its own from TMEM) and stores Y.  Every
    // thread of every CTA passes the cluster barriers whatever happened before.
    // Block layout: 16 columns of a row are four 16-byte units, unit u stored at
    // slot u ^ ((row >> 1) & 3) so that eight consecutive rows hit eight
    // different bank groups.
    constexpr int kOwn = owned_max(KS);
    const int swz = (row >> 1) & 3;
    auto block_off = [&](int sub, int c, int sender_slot) {
      return (uint32_t)(((sub * kOwn + c / KS) * (KS - 1) + sender_slot) * (128 * 64));
    };
    auto unit_off = [&](int u) { return (uint32_t)((row * 4 + (u ^ swz)) * 16); };
    if (threadIdx.x == 0) {
      const int own = (kBN / 16 - (int)krank + KS - 1) / KS;  // chunks c with c % KS == krank
      mbar_arrive_expect_tx(redfull, (uint32_t)(kSub * own * (KS - 1) * 128 * 64));
    }
    cluster_sync();
    const uint32_t base = smem_u32(smem);
    if (acc_ready) {
      // per 128-token sub-tile: the TMEM loads of all of this warp's pushed
      // chunks first, one wait, then the pushes (the load latency is paid once
      // per sub-tile, not once per chunk)
#pragma unroll 1
      for (int sub = 0; sub < kSub; ++sub) {
        uint32_t r[4][16];
#pragma unroll
        for (int ci = 0; ci < 4; ++ci)
          if ((c_lo + ci) % KS != (int)krank)  // the same for every lane: a warp-wide load
            tmem_ld_x16(tq + (uint32_t)(sub * 128 + 16 * (c_lo + ci)), r[ci]);
        tmem_ld_wait();
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
          const int c = c_lo + ci;
          const int owner = c % KS;
          if (owner == (int)krank) continue;
          const uint32_t peer = rank + CS * (uint32_t)owner;
          const int slot = (int)krank < owner ? (int)krank : (int)krank - 1;
          const uint32_t dst = peer_smem(base + block_off(sub, c, slot), peer);
          const uint32_t bar = peer_smem(smem_u32(redfull), peer);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_async_v4(dst + unit_off(u),
                        make_float4(__uint_as_float(r[ci][4 * u]), __uint_as_float(r[ci][4 * u + 1]),
                                    __uint_as_float(r[ci][4 * u + 2]),
                                    __uint_as_float(r[ci][4 * u + 3])),
                        bar);
        }
      }
    }
    const bool got = mbar_wait(redfull, 0u, a.err);
    if (acc_ready && got) {
#pragma unroll 1
      for (int sub = 0; sub < kSub; ++sub) {
        uint32_t ro[4][16];  // this warp's owned chunks of the sub-tile, loaded together
#pragma unroll
        for (int ci = 0; ci < 4; ++ci)
          if ((c_lo + ci) % KS == (int)krank)
            tmem_ld_x16(tq + (uint32_t)(sub * 128 + 16 * (c_lo + ci)), ro[ci]);
        tmem_ld_wait();
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
          const int c = c_lo + ci;
          if (c % KS != (int)krank) continue;
          const uint32_t (&r)[16] = ro[ci];
          float v[16];
#pragma unroll
          for (int z = 0; z < KS; ++z) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float4 t;
              if (z == (int)krank) {
                t = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
              } else {
                const int slot = z < (int)krank ? z : z - 1;
                t = *reinterpret_cast<const float4 *>(smem + block_off(sub, c, slot) + unit_off(u));
              }
              v[4 * u] = z ? v[4 * u] + t.x : t.x;
              v[4 * u + 1] = z ? v[4 * u + 1] + t.y : t.y;
              v[4 * u + 2] = z ? v[4 * u + 2] + t.z : t.z;
              v[4 * u + 3] = z ? v[4 * u + 3] + t.w : t.w;
            }
          }
          if (a.gamma) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= rinv_s[128 * sub + 16 * c + e];
          }
          store_y16_rows(a, m0 + 128 * sub + 16 * c, n0 + row, v);
        }
      }
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

std::once_flag g_gemm_attr[kMaxDevices];  // cudaFuncSetAttribute acts on the current device

template <int CS, int KS, bool G = false>
void gemm_allow() {
  cudaFuncSetAttribute(gemm_kernel<CS, KS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemmSmem::kAlloc);
}

void gemm_attributes() {
  gemm_allow<1, 1>();
  gemm_allow<2, 1>();
  gemm_allow<1, 2>();
  gemm_allow<1, 3>();
  gemm_allow<1, 4>();
  gemm_allow<2, 2>();
  gemm_allow<2, 3>();
  gemm_allow<2, 4>();
  gemm_allow<1, 1, true>();
}

cudaError_t gemm_go(cudaLaunchConfig_t &cfg, int cs, int ks, const CUtensorMap &xmap,
                    const CUtensorMap &wmap, const GemmArgs &args) {
  cfg.dynamicSmemBytes = GemmSmem::kAlloc;
  cfg.blockDim = dim3((unsigned)kThreads, 1, 1);
  auto go = [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, xmap, wmap, args); };
  if (cs == 2) {
    if (ks == 4) return go(gemm_kernel<2, 4>);
    if (ks == 3) return go(gemm_kernel<2, 3>);
    if (ks == 2) return go(gemm_kernel<2, 2>);
    return go(gemm_kernel<2, 1>);
  }
  if (ks == 4) return go(gemm_kernel<1, 4>);
  if (ks == 3) return go(gemm_kernel<1, 3>);
  if (ks == 2) return go(gemm_kernel<1, 2>);
  return go(gemm_kernel<1, 1>);
}

#ifndef Q4K_GEMM_CLUSTER
#define Q4K_GEMM_CLUSTER 2
#endif
#ifndef Q4K_GEMM_SPLITK  // split K across a cluster when the output tiles cannot fill the SMs
#define Q4K_GEMM_SPLITK 1
#endif

// 1/rms of each token row of X: one CTA of 256 threads per token (the whole
// of X in flight at once), fp32 sum of squares in a fixed order (thread i
// takes the 16-byte pieces i, i + 256, ...; a butterfly within each warp; the
// eight warp sums added in warp order), rinv = 1 / sqrt(sum / k + eps) with
// IEEE division and square root.  Launched as a programmatic dependent of the
// kernel before it.
__global__ void __launch_bounds__(256) rms_rinv_kernel(const __nv_bfloat16 *x, int64_t ldx, int m,
                                                       int k, float eps, float *rinv) {
  __shared__ float part[8];
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4 *row = reinterpret_cast<const uint4 *>(x + (int64_t)t * ldx);
  float s = 0.f;
#pragma unroll 4
  for (int i = threadIdx.x; i < k / 8; i += 256) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
      s = fmaf(lo, lo, s);
      s = fmaf(hi, hi, s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) part[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = part[0];
#pragma unroll
    for (int w8 = 1; w8 < 8; ++w8) tot += part[w8];
    rinv[t] = 1.f / sqrtf(tot / (float)k + eps);
  }
}

}  // namespace

cudaError_t launch_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                        void *y, int64_t ldy, cudaStream_t stream) {
  return launch_gemm_rmsnorm(w, n, k, x, m, ldx, nullptr, 0.f, nullptr, y, ldy, stream);
}

cudaError_t launch_gemm_rmsnorm(const void *w, int64_t n, int64_t k, const void *x, int64_t m,
                                int64_t ldx, const float *gamma, float eps, float *rinv, void *y,
                                int64_t ldy, cudaStream_t stream) {
  std::call_once(g_gemm_attr[device_facts()->device], gemm_attributes);
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
  args.gamma = gamma;
  args.rinv = rinv;
  args.slot_expert = args.slot_start = args.meta = nullptr;
  args.err = device_error_word();

  // K is split across a cluster (up to 4 ways) when the output tiles cannot
  // fill the SMs; pairs of CTAs over the same K range share X by multicast.
  const int sms = device_facts()->sm_count;
  const int mt = (int)((m + kTokens - 1) / kTokens);
  int nt = (int)((n + kBN - 1) / kBN);
  int ks = 1;
  if (Q4K_GEMM_SPLITK) {
    ks = std::max(1, std::min(4, sms / std::max(1, nt * mt)));
    while (ks > 1 && nsb < 2 * ks) --ks;
  }
  int cs = Q4K_GEMM_CLUSTER > 1 ? 2 : 1;
  while (cs > 1 && (nt < 2 * cs || cs * ks > 8)) cs >>= 1;
  nt = (nt + cs - 1) / cs * cs;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nt, (unsigned)mt, (unsigned)ks);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ks;
  // Programmatic dependent launch is safe for any caller: the kernel waits for
  // the previous kernel before its first global access.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (gamma) {
    cudaLaunchConfig_t pre = {};
    pre.gridDim = dim3((unsigned)m, 1, 1);
    pre.blockDim = dim3(256, 1, 1);
    pre.stream = stream;
    pre.attrs = &attr[1];  // programmatic dependent of the kernel before it
    pre.numAttrs = 1;
    const cudaError_t e =
        cudaLaunchKernelEx(&pre, rms_rinv_kernel, static_cast<const __nv_bfloat16 *>(x), ldx,
                           (int)m, (int)k, eps, rinv);
    if (e != cudaSuccess) return e;
  }
  return gemm_go(cfg, cs, ks, xmap, wmap, args);
}

cudaError_t launch_gemm_grouped(const void *w, int64_t expert_stride, int n_experts, int64_t n,
                                int64_t k, const void *x, int64_t rows, int64_t ldx, void *y,
                                int64_t ldy, const int *slot_expert, const int *slot_start,
                                const int *meta, int max_slots, cudaStream_t stream) {
  std::call_once(g_gemm_attr[device_facts()->device], gemm_attributes);
  const int nsb = (int)(k / kQK);
  CUtensorMap xmap, wmap;
  {
    const uint64_t dims[2] = {(uint64_t)k, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)ldx * 2};
    const uint32_t box[2] = {(uint32_t)kBK, 128u};
    if (encode_tiled(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // (byte of the super-block, super-block, row, expert)
    const uint64_t dims[4] = {(uint64_t)kBlockBytes, (uint64_t)nsb, (uint64_t)n,
                              (uint64_t)n_experts};
    const uint64_t strides[3] = {(uint64_t)kBlockBytes, (uint64_t)nsb * kBlockBytes,
                                 (uint64_t)expert_stride};
    const uint32_t box[4] = {(uint32_t)kBlockBytes, 1u, (uint32_t)kBN, 1u};
    if (encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(w), dims, strides,
                     box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  GemmArgs args = {};
  args.y = static_cast<__nv_bfloat16 *>(y);
  args.ldy = ldy;
  args.m = (int)rows;
  args.n = (int)n;
  args.k = (int)k;
  args.slot_expert = slot_expert;
  args.slot_start = slot_start;
  args.meta = meta;
  args.err = device_error_word();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + kBN - 1) / kBN), (unsigned)max_slots, 1);
  cfg.blockDim = dim3((unsigned)kThreads, 1, 1);
  cfg.dynamicSmemBytes = GemmSmem::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<1, 1, true>, xmap, wmap, args);
}

}  // namespace q4k
