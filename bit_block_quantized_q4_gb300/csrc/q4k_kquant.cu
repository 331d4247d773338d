// q4k_kquant.cu -- the other k-quant formats: q2_K, q3_K (the routed-down
// recipes of "Layer Package Repository Spec", section "Policy Resolution"),
// Q5_K and Q6_K (found in "_XL" mixes): dequantization and the decode
// projection Y = W X for batch 2..16 (batch 1 runs on the tensor cores in the
// stream kernel, q4k_stream.cu).
//
// Super-blocks of 256 weights (the GGUF k-quant layouts; field offsets below):
//   q2_K  84 B: sc[16] (scale | min << 4) @0, qs[64] @16, d @80, dmin @82;
//         16 sub-blocks of 16, w = d sc q - dmin m, q 2 bits.
//   q3_K 110 B: hmask[32] @0, qs[64] @32, scales[12] @96, d @108;
//         16 sub-blocks of 16, w = d (sc - 32) q, q = 2 bits - (mask bit ? 0 : 4).
//   Q5_K 176 B: d @0, dmin @2, scales[12] @4 (as Q4_K), qh[32] @16, qs[128] @48;
//         8 sub-blocks of 32, w = d sc q - dmin m, q = nibble + 16 high bit.
//   Q6_K 210 B: ql[128] @0, qh[64] @128, sc[16] (int8) @192, d @208;
//         16 sub-blocks of 16, w = d sc q, q = 6 bits - 32.
// Lane l of a warp takes weights 8l .. 8l+7 of a super-block: 8 consecutive
// quant bytes (plus 8 consecutive high-bit bytes) and one scale field.  Each
// weight is its exact value rounded once to fp32: q2_K and Q5_K by one fma of
// the exact products d sc and dmin m, q3_K and Q6_K exactly (at most 24
// significant bits), computed on the packed fp32 pipe in pairs.
//
// Dequantization: a warp per super-block, coalesced 32- or 16-byte stores.
// Projection: a warp per weight row.  The row's bytes go to shared memory by
// 16-byte cp.async copies (from the row start rounded down to 16 bytes; the
// matrix's last copy is cut at its end), double-buffered across the warp's
// rows; the lanes decode from there and contract with x in fp32.
#include <algorithm>
#include <mutex>

#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

namespace {

__host__ __device__ constexpr int kq_bytes(int f) {
  return f == 2 ? 84 : f == 3 ? 110 : f == 5 ? 176 : f == 6 ? 210 : 0;
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) {
  return *reinterpret_cast<const uint16_t *>(p);
}
// 8 bytes at a 2-byte-aligned address, as two little-endian words (two 4-byte
// loads when the address allows; the choice is the same for every lane of a
// warp, whose fields differ by multiples of 8 bytes).
__device__ __forceinline__ void ld8(const uint8_t *p, uint32_t &lo, uint32_t &hi) {
  if ((reinterpret_cast<uintptr_t>(p) & 3) == 0) {
    lo = *reinterpret_cast<const uint32_t *>(p);
    hi = *reinterpret_cast<const uint32_t *>(p + 4);
  } else {
    lo = ld_u16(p) | (ld_u16(p + 2) << 16);
    hi = ld_u16(p + 4) | (ld_u16(p + 6) << 16);
  }
}
__device__ __forceinline__ float half_at(const uint8_t *p) {
  return __half2float(__ushort_as_half((unsigned short)ld_u16(p)));
}
__device__ __forceinline__ uint32_t byte_at(const uint8_t *p, int i) {
  return (ld_u16(p + (i & ~1)) >> (8 * (i & 1))) & 0xFFu;
}
// The four bytes of v (each an integer u < 2^8) as floats u - bias, in pairs
// (bytes 0, 1) and (2, 3): 0x4B0000uu is 2^23 + u exactly, so the packed
// subtraction of 2^23 + bias is exact.
__device__ __forceinline__ void bytes_to_f2(uint32_t v, float bias, float2 &p01, float2 &p23) {
  const float2 m = make_float2(-8388608.f - bias, -8388608.f - bias);
  p01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7540u)),
                               __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7541u))), m);
  p23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7542u)),
                               __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7543u))), m);
}

// Weights 8l .. 8l+7 of the super-block at b (2-byte aligned), fp32, as pairs
// w[0] = (8l, 8l+1) .. w[3] = (8l+6, 8l+7).  The quants of four weights are
// taken a word at a time (one per byte), then: q2_K and Q5_K
// w = fma(d sc, q, -dmin m); q3_K and Q6_K w = (d sc) q, exact.
template <int F>
__device__ __forceinline__ void decode8(const uint8_t *b, int l, float2 (&w)[4]) {
  const int o = 8 * (l & 3);
  uint32_t u[2];  // the 8 quants, one per byte (unsigned), 4 per word
  float mul, add, bias;
  if constexpr (F == 2) {
    const int h = l >> 4, g = (l & 15) >> 2;
    uint32_t lo, hi;
    ld8(b + 16 + 32 * h + o, lo, hi);
    u[0] = (lo >> (2 * g)) & 0x03030303u;
    u[1] = (hi >> (2 * g)) & 0x03030303u;
    const uint32_t sm = byte_at(b, l >> 1);  // sub-block of 16: scale | min << 4
    mul = half_at(b + 80) * (float)(sm & 15u);
    add = -(half_at(b + 82) * (float)(sm >> 4));
    bias = 0.f;
  } else if constexpr (F == 3) {
    const int h = l >> 4, g = (l & 15) >> 2, j = l >> 1;
    uint32_t lo, hi, mlo, mhi;
    ld8(b + 32 + 32 * h + o, lo, hi);
    ld8(b + o, mlo, mhi);
    const int bit = 4 * h + g;
    u[0] = ((lo >> (2 * g)) & 0x03030303u) | (((mlo >> bit) & 0x01010101u) << 2);
    u[1] = ((hi >> (2 * g)) & 0x03030303u) | (((mhi >> bit) & 0x01010101u) << 2);
    const uint8_t *s = b + 96;
    const uint32_t low4 = j < 8 ? byte_at(s, j) & 15u : byte_at(s, j - 8) >> 4;
    const uint32_t hi2 = (byte_at(s, 8 + (j & 3)) >> (2 * (j >> 2))) & 3u;
    mul = half_at(b + 108) * (float)((int)(low4 | (hi2 << 4)) - 32);
    add = 0.f;
    bias = 4.f;  // q = u - 4 (u = 2 bits + 4 * mask bit)
  } else if constexpr (F == 5) {
    const int c = l >> 3, high = (l >> 2) & 1, j = l >> 2;
    uint32_t lo, hi, hlo, hhi;
    ld8(b + 48 + 32 * c + o, lo, hi);
    ld8(b + 16 + o, hlo, hhi);
    const int bit = 2 * c + high;
    u[0] = ((lo >> (4 * high)) & 0x0F0F0F0Fu) | (((hlo >> bit) & 0x01010101u) << 4);
    u[1] = ((hi >> (4 * high)) & 0x0F0F0F0Fu) | (((hhi >> bit) & 0x01010101u) << 4);
    const uint8_t *s = b + 4;
    uint32_t sc, m;
    if (j < 4) {
      sc = byte_at(s, j) & 63u;
      m = byte_at(s, j + 4) & 63u;
    } else {
      sc = (byte_at(s, j + 4) & 15u) | ((byte_at(s, j - 4) >> 6) << 4);
      m = (byte_at(s, j + 4) >> 4) | ((byte_at(s, j) >> 6) << 4);
    }
    mul = half_at(b) * (float)sc;
    add = -(half_at(b + 2) * (float)m);
    bias = 0.f;
  } else {  // F == 6
    const int h = l >> 4, v = (l & 15) >> 2;
    uint32_t lo, hi, hlo, hhi;
    ld8(b + 64 * h + o + 32 * (v & 1), lo, hi);
    ld8(b + 128 + 32 * h + o, hlo, hhi);
    const int sh = v < 2 ? 0 : 4;
    u[0] = ((lo >> sh) & 0x0F0F0F0Fu) | (((hlo >> (2 * v)) & 0x03030303u) << 4);
    u[1] = ((hi >> sh) & 0x0F0F0F0Fu) | (((hhi >> (2 * v)) & 0x03030303u) << 4);
    mul = half_at(b + 208) * (float)(int)(int8_t)byte_at(b + 192, l >> 1);
    add = 0.f;
    bias = 32.f;  // q = u - 32
  }
  const float2 mul2 = make_float2(mul, mul), add2 = make_float2(add, add);
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    float2 q01, q23;
    bytes_to_f2(u[hw], bias, q01, q23);
    if constexpr (F == 2 || F == 5) {
      w[2 * hw] = __ffma2_rn(mul2, q01, add2);
      w[2 * hw + 1] = __ffma2_rn(mul2, q23, add2);
    } else {
      w[2 * hw] = __fmul2_rn(mul2, q01);
      w[2 * hw + 1] = __fmul2_rn(mul2, q23);
    }
  }
}

// ------------------------------------------------------------ dequantization
template <int F, bool BF16>
__global__ void __launch_bounds__(256) kq_dequant_kernel(const uint8_t *w, int64_t nblocks,
                                                         void *out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t bi = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); bi < nblocks;
       bi += warps) {
    float2 v2[4];
    decode8<F>(w + bi * kq_bytes(F), lane, v2);
    const float v[8] = {v2[0].x, v2[0].y, v2[1].x, v2[1].y, v2[2].x, v2[2].y, v2[3].x, v2[3].y};
    const int64_t o = bi * 256 + 8 * lane;
    if (BF16) {
      uint4 pk;
      __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]),
                     c = __floats2bfloat162_rn(v[4], v[5]), d = __floats2bfloat162_rn(v[6], v[7]);
      pk.x = *reinterpret_cast<uint32_t *>(&a);
      pk.y = *reinterpret_cast<uint32_t *>(&b);
      pk.z = *reinterpret_cast<uint32_t *>(&c);
      pk.w = *reinterpret_cast<uint32_t *>(&d);
      *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + o) = pk;
    } else {
      float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(out) + o);
      p[0] = make_float4(v[0], v[1], v[2], v[3]);
      p[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// ------------------------------------------------------------ projection
constexpr int kKqWarps = 4;  // warps (row streams) per CTA

struct KqArgs {
  const uint8_t *w;
  int64_t total_bytes;  // of the whole matrix
  int n, nsb;           // rows, super-blocks per row
  const __nv_bfloat16 *x;
  int64_t ldx;
  int batch;
  float *y;
  int64_t ldy;
  int buf_bytes;  // per row buffer: row bytes + 16, rounded up to 16
};


// Copies row r's bytes [start, start + row bytes) from start rounded down to 16
// into buf; returns the offset of the row's first byte in buf.
template <int F>
__device__ __forceinline__ int stage_row(const KqArgs &a, int r, uint8_t *buf, int lane) {
  const int64_t row_bytes = (int64_t)a.nsb * kq_bytes(F);
  const int64_t start = (int64_t)r * row_bytes;
  const int64_t s0 = start & ~int64_t(15);
  const int64_t end = start + row_bytes;
  const int chunks = (int)((end - s0 + 15) >> 4);
  for (int c = lane; c < chunks; c += 32) {
    const int64_t src = s0 + 16 * (int64_t)c;
    const int64_t avail = a.total_bytes - src;  // the matrix's last copy is cut at its end
    cp_async16(buf + 16 * c, a.w + src, avail >= 16 ? 16 : (int)avail);
  }
  return (int)(start - s0);
}

template <int F, int NB>
__global__ void __launch_bounds__(kKqWarps * 32) kq_gemv_kernel(const KqArgs a) {
  extern __shared__ __align__(16) uint8_t kq_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *bufs = kq_smem + (size_t)warp * 2 * a.buf_bytes;
  const int nwarps = gridDim.x * kKqWarps;
  int r = blockIdx.x * kKqWarps + warp;
  if (r >= a.n) return;
  int cur = 0;
  int off = stage_row<F>(a, r, bufs, lane);
  cp_async_commit();
  for (; r < a.n; r += nwarps) {
    const int rn = r + nwarps;
    int off_n = 0;
    if (rn < a.n) off_n = stage_row<F>(a, rn, bufs + (cur ^ 1) * a.buf_bytes, lane);
    cp_async_commit();  // (an empty group when there is no next row)
    cp_async_wait<1>();  // this row's copies have landed
    __syncwarp();
    const uint8_t *row = bufs + cur * a.buf_bytes + off;
    float2 acc[NB];  // pairs of partial sums (even, odd weights), added at the end
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = make_float2(0.f, 0.f);
    // x of SBU super-blocks is loaded ahead of their decoding (it comes from L2)
    constexpr int SBU = NB <= 4 ? 4 : NB <= 8 ? 2 : 1;
    for (int sb0 = 0; sb0 < a.nsb; sb0 += SBU) {
      uint4 xv[SBU][NB];
#pragma unroll
      for (int u = 0; u < SBU; ++u)
#pragma unroll
        for (int b = 0; b < NB; ++b)
          xv[u][b] = (sb0 + u < a.nsb && b < a.batch)
                         ? __ldg(reinterpret_cast<const uint4 *>(a.x + b * a.ldx +
                                                                 256 * (sb0 + u) + 8 * lane))
                         : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < SBU; ++u) {
        if (sb0 + u >= a.nsb) break;
        float2 w[4];
        decode8<F>(row + (sb0 + u) * kq_bytes(F), lane, w);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const uint32_t xw[4] = {xv[u][b].x, xv[u][b].y, xv[u][b].z, xv[u][b].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[b] = __ffma2_rn(w[e], make_float2(__uint_as_float(xw[e] << 16),
                                                  __uint_as_float(xw[e] & 0xFFFF0000u)), acc[b]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float v = acc[b].x + acc[b].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && b < a.batch) a.y[b * a.ldy + r] = v;
    }
    __syncwarp();  // every lane is done with this buffer before it is refilled
    cur ^= 1;
    off = off_n;
  }
  cp_async_wait<0>();
}

std::once_flag g_kq_attr[kMaxDevices];

template <int F>
void kq_allow_format() {
  const int max_smem = 227 * 1024;
  cudaFuncSetAttribute(kq_gemv_kernel<F, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(kq_gemv_kernel<F, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(kq_gemv_kernel<F, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  cudaFuncSetAttribute(kq_gemv_kernel<F, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

void kq_attributes() {
  kq_allow_format<2>();
  kq_allow_format<3>();
  kq_allow_format<5>();
  kq_allow_format<6>();
}

// Resident CTAs per SM of one instantiation at one shared-memory size, looked
// up once per (device, format, batch class, size).
std::mutex g_kq_occ_mu;
struct KqOcc {
  int dev, fmt, nb;
  size_t smem;
  int occ;
};
KqOcc g_kq_occ[64];
int g_kq_occ_n = 0;

template <typename K>
int kq_occupancy(K kernel, int fmt, int nb, size_t smem) {
  const int dev = device_facts()->device;
  std::lock_guard<std::mutex> lk(g_kq_occ_mu);
  for (int i = 0; i < g_kq_occ_n; ++i)
    if (g_kq_occ[i].dev == dev && g_kq_occ[i].fmt == fmt && g_kq_occ[i].nb == nb &&
        g_kq_occ[i].smem == smem)
      return g_kq_occ[i].occ;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kKqWarps * 32, smem) !=
      cudaSuccess)
    occ = 1;
  occ = std::max(occ, 1);
  if (g_kq_occ_n < 64) g_kq_occ[g_kq_occ_n++] = KqOcc{dev, fmt, nb, smem, occ};
  return occ;
}

// Only resident CTAs: each warp then streams several rows, the next row's
// copies in flight while it contracts the current one.
template <int F, int NB>
cudaError_t launch_kq_gemv_nb(const KqArgs &a, size_t smem, cudaStream_t stream) {
  const int occ = kq_occupancy(kq_gemv_kernel<F, NB>, F, NB, smem);
  const int64_t need = ((int64_t)a.n + kKqWarps - 1) / kKqWarps;
  const int ctas = (int)std::min<int64_t>(need, (int64_t)occ * device_facts()->sm_count);
  kq_gemv_kernel<F, NB><<<(unsigned)ctas, kKqWarps * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int F>
cudaError_t launch_kq_gemv_f(const KqArgs &a, size_t smem, cudaStream_t stream) {
  if (a.batch <= 1) return launch_kq_gemv_nb<F, 1>(a, smem, stream);
  if (a.batch <= 4) return launch_kq_gemv_nb<F, 4>(a, smem, stream);
  if (a.batch <= 8) return launch_kq_gemv_nb<F, 8>(a, smem, stream);
  return launch_kq_gemv_nb<F, 16>(a, smem, stream);
}

template <int F>
cudaError_t launch_kq_dequant_f(const void *w, int64_t nblocks, void *out, int out_dtype,
                                cudaStream_t stream) {
  const int sms = device_facts()->sm_count;
  const int64_t ctas = std::min<int64_t>((nblocks + 7) / 8, 16 * sms);
  if (out_dtype == 1)
    kq_dequant_kernel<F, true><<<(unsigned)ctas, 256, 0, stream>>>(static_cast<const uint8_t *>(w),
                                                                   nblocks, out);
  else
    kq_dequant_kernel<F, false><<<(unsigned)ctas, 256, 0, stream>>>(static_cast<const uint8_t *>(w),
                                                                    nblocks, out);
  return cudaGetLastError();
}

}  // namespace

int kq_block_bytes(int format) { return kq_bytes(format); }

size_t kq_gemv_smem(int format, int64_t k) {
  const int64_t row = (k / kQK) * kq_bytes(format);
  const int64_t buf = (row + 16 + 15) / 16 * 16;
  return (size_t)(kKqWarps * 2 * buf);
}

cudaError_t launch_kq_dequant(int format, const void *w, int64_t n, int64_t k, void *out,
                              int out_dtype, cudaStream_t stream) {
  const int64_t nblocks = n * (k / kQK);
  switch (format) {
    case 2: return launch_kq_dequant_f<2>(w, nblocks, out, out_dtype, stream);
    case 3: return launch_kq_dequant_f<3>(w, nblocks, out, out_dtype, stream);
    case 5: return launch_kq_dequant_f<5>(w, nblocks, out, out_dtype, stream);
    case 6: return launch_kq_dequant_f<6>(w, nblocks, out, out_dtype, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_kq_gemv(int format, const void *w, int64_t n, int64_t k, const void *x,
                           int64_t batch, int64_t ldx, float *y, int64_t ldy,
                           cudaStream_t stream) {
  std::call_once(g_kq_attr[device_facts()->device], kq_attributes);
  KqArgs a;
  a.w = static_cast<const uint8_t *>(w);
  a.nsb = (int)(k / kQK);
  a.n = (int)n;
  a.total_bytes = n * a.nsb * (int64_t)kq_bytes(format);
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.ldx = ldx;
  a.batch = (int)batch;
  a.y = y;
  a.ldy = ldy;
  const size_t smem = kq_gemv_smem(format, k);
  a.buf_bytes = (int)(smem / (2 * kKqWarps));
  switch (format) {
    case 2: return launch_kq_gemv_f<2>(a, smem, stream);
    case 3: return launch_kq_gemv_f<3>(a, smem, stream);
    case 5: return launch_kq_gemv_f<5>(a, smem, stream);
    case 6: return launch_kq_gemv_f<6>(a, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace q4k
