// q4k_dequant.cu -- Q4_K -> fp32 / bf16 expansion ("spec: specialized model
// runtimes", section "Architecture": the quant/dequant op of kernel tier T0).
//
// One warp per 144-byte super-block; lane i produces weights 8i .. 8i+7, which
// all sit in sub-block j = i/4 and come from the 8 quant bytes 8(i%4) .. +7 of
// chunk j/2 (low nibbles for even j, high nibbles for odd j).  The weight is
// fma(d*sc_j, q, -dmin*m_j): d*sc_j and dmin*m_j are exact in fp32 (at most 17
// significant bits), d*sc_j*q is exact (at most 21 bits), so the single rounding
// of the fma is the round-to-nearest-even of the exact weight.  bf16 output
// rounds that fp32 value to nearest even.  Streaming kernel: 144 B in, 1024 B
// (fp32) or 512 B (bf16) out per super-block, fully coalesced 16-byte accesses;
// each warp loads several super-blocks before converting them.
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

// The output is written once and not read back here: evict-first stores.
__device__ __forceinline__ void st_out(uint4 *p, uint4 v) { __stcs(p, v); }

// Super-blocks per warp per loop step, their loads issued together: measured
// best at 8 for fp32 output (5.4 against 4.3 TB/s at 1) and 2 for bf16 (4.7
// against 4.3; 8 fell to 3.2).
#ifndef Q4K_DQ_UNROLL_F32
#define Q4K_DQ_UNROLL_F32 8
#endif
#ifndef Q4K_DQ_UNROLL_BF16
#define Q4K_DQ_UNROLL_BF16 2
#endif
// Warps per CTA and the grid cap (CTAs per SM; CTAs beyond the resident ones
// run in later waves, and a CTA loops over further super-blocks only past the
// cap): measured on the 17408 x 5120 matrix, 4 warps and 128 per SM 5.67 /
// 5.06 TB/s (fp32 / bf16), against 5.40 / 4.70 at 8 warps and 16 per SM, 5.66
// / 4.98 at 4 warps and 64, 5.52 / 4.83 at 4 warps and 32.
#ifndef Q4K_DQ_CTAS_PER_SM
#define Q4K_DQ_CTAS_PER_SM 128
#endif
#ifndef Q4K_DQ_WARPS
#define Q4K_DQ_WARPS 4
#endif
template <int OUT_BF16>
__host__ __device__ constexpr int dq_unroll() { return OUT_BF16 ? Q4K_DQ_UNROLL_BF16 : Q4K_DQ_UNROLL_F32; }

template <int OUT_BF16>
__global__ void __launch_bounds__(Q4K_DQ_WARPS * 32) dequant_kernel(const uint8_t *__restrict__ w,
                                                      int64_t nblocks, void *__restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int j = lane >> 2;            // sub-block
  const int c = j >> 1;               // 32-byte quant chunk
  const int shift = (j & 1) * 4;      // low or high nibbles
  constexpr int U = dq_unroll<OUT_BF16>();
  for (int64_t b0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * U; b0 < nblocks;
       b0 += warps_total * U) {
    uint4 h[U];
    uint2 q8[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {  // the loads of all U blocks first
      const int64_t b = min(b0 + u, nblocks - 1);
      const uint8_t *blk = w + b * kBlockBytes;
      h[u] = __ldg(reinterpret_cast<const uint4 *>(blk));
      q8[u] = __ldg(reinterpret_cast<const uint2 *>(blk + kQsOffset + 32 * c + 8 * (lane & 3)));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t b = b0 + u;
      if (b >= nblocks) break;
      uint32_t sc_lo, sc_hi, m_lo, m_hi;
      scales_all(h[u].y, h[u].z, h[u].w, &sc_lo, &sc_hi, &m_lo, &m_hi);
      const uint32_t scw = (j < 4) ? sc_lo : sc_hi;
      const uint32_t mw = (j < 4) ? m_lo : m_hi;
      const uint32_t sc = (scw >> (8 * (j & 3))) & 0xFFu;
      const uint32_t mm = (mw >> (8 * (j & 3))) & 0xFFu;
      const float ds = half_lo_to_float(h[u].x) * (float)sc;   // exact
      const float dm = half_hi_to_float(h[u].x) * (float)mm;   // exact
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t word = e < 4 ? q8[u].x : q8[u].y;
        const uint32_t q = (word >> (8 * (e & 3) + shift)) & 15u;
        v[e] = fmaf(ds, (float)q, -dm);
      }
      if (OUT_BF16) {
        uint4 o;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[4], v[5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(v[6], v[7]);
        o.x = *reinterpret_cast<uint32_t *>(&p0);
        o.y = *reinterpret_cast<uint32_t *>(&p1);
        o.z = *reinterpret_cast<uint32_t *>(&p2);
        o.w = *reinterpret_cast<uint32_t *>(&p3);
        st_out(reinterpret_cast<uint4 *>(out) + (b * 32 + lane), o);
      } else {
        uint4 *o = reinterpret_cast<uint4 *>(out) + (b * 64 + lane * 2);
        st_out(o, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                             __float_as_uint(v[3])));
        st_out(o + 1, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]),
                                 __float_as_uint(v[7])));
      }
    }
  }
}

cudaError_t launch_dequant(const void *w, int64_t n, int64_t k, void *out, int out_dtype,
                           cudaStream_t stream) {
  const DeviceFacts *f = device_facts();
  const int64_t nblocks = n * (k / kQK);
  const int warps_per_cta = Q4K_DQ_WARPS;
  const int64_t per_cta = (int64_t)warps_per_cta * (out_dtype == 1 ? dq_unroll<1>() : dq_unroll<0>());
  int64_t grid = (nblocks + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)f->sm_count * Q4K_DQ_CTAS_PER_SM;
  if (grid > cap) grid = cap;
  if (out_dtype == 1) {
    dequant_kernel<1><<<(unsigned)grid, warps_per_cta * 32, 0, stream>>>(
        static_cast<const uint8_t *>(w), nblocks, out);
  } else {
    dequant_kernel<0><<<(unsigned)grid, warps_per_cta * 32, 0, stream>>>(
        static_cast<const uint8_t *>(w), nblocks, out);
  }
  return cudaGetLastError();
}

}  // namespace q4k
