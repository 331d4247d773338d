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
//   2. gate/up  one CTA per (slot, 16-row tile of ffn): the expert's gate and up
//               rows are streamed once (TMA) and contracted with all of the
//               slot's tokens on the tensor cores (MMA columns = tokens); the
//               epilogue writes h = silu(g) * u in fp32.
//   3. down     one CTA per (slot, 128-row tile of hidden): h of the slot's pairs
//               is staged once in shared memory as two bf16 columns per pair,
//               h_hi = bf16(h) and h_lo = bf16(h - h_hi) (together 16
//               significant bits), and each of the 8 warps streams 16 down rows.
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
constexpr int kMaxExperts = 2048;
constexpr int kSlotPairs = 16;               // pairs per work slot

// Workspace layout (all offsets 256-byte aligned).
struct MoeLayout {
  size_t meta, slot_expert, slot_start, pair_token, tj_pair, h, h_hi, h_lo, p, total;
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
  float *h, *p;
  __nv_bfloat16 *h_hi, *h_lo;
  unsigned *err;
};

// ---------------------------------------------------------------- 1. route
__global__ void __launch_bounds__(1024) moe_route_kernel(const MoeArgs a) {
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
// One CTA = (work slot blockIdx.y, 16*WM output rows from blockIdx.x).  Warp w
// takes m-tile w / WK and the (w % WK)-th super-block slice of K; slices of an
// m-tile meet in shared memory.  MMA columns are the slot's pairs:
//   gate/up (DOWN = false): column c = x row of the c-th pair's token;
//   down    (DOWN = true):  column 2i = h_hi, column 2i+1 = h_lo of pair i.
// Thread t's k-slots (2t, 2t+1) carry positions (o, o+2) and (2t+8, 2t+9)
// positions (o+1, o+3) of a sub-block, o = 8t + 4s for step s = 0/1: quant
// bytes 8t .. 8t+7 of the sub-block's 32-byte chunk.
template <int NT, bool DOWN, int WM, int WK>
__global__ void __launch_bounds__(WM * WK * 32) moe_expert_kernel(
    const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
    const MoeArgs a, int nsb, int ks, int rows_total) {
  constexpr int NM = DOWN ? 1 : 2;  // weight matrices per CTA (gate and up)
  constexpr int kCols = NT * 8;
  constexpr int kStageBytes = NM * kTile;
  // TMA destinations must be 128-byte aligned: round each warp's region up.
  constexpr int kWarpBytes = (kStagesMoe * kStageBytes + 64 + 127) / 128 * 128;
  extern __shared__ __align__(128) uint8_t smem[];
  const int slot = blockIdx.y;
  if (slot >= a.meta[0]) return;  // slot not in use (uniform per CTA)
  const int expert = a.slot_expert[slot];
  const int pstart = a.slot_start[slot];
  const int np = a.slot_start[slot + 1] - pstart;  // pairs of this slot (<= 16)
  const int ncols = DOWN ? 2 * np : np;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int mtile = warp / WK, kslice = warp % WK;
  const int row0 = blockIdx.x * (kRows * WM) + mtile * kRows;
  const int sb0 = kslice * ks;
  const int nsteps = max(0, min(nsb, sb0 + ks) - sb0);
  uint8_t *ring = smem + warp * kWarpBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kStagesMoe * kStageBytes);
  float *red = reinterpret_cast<float *>(smem + WM * WK * kWarpBytes);

  if (lane == 0) {
    prefetch_tmap(&map0);
    if (NM == 2) prefetch_tmap(&map1);
    for (int s = 0; s < kStagesMoe; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int stage, int sb) {
    mbar_arrive_expect_tx(&bars[stage], kStageBytes);
    uint8_t *dst = ring + stage * kStageBytes;
    tma_load_3d_hint(dst, &map0, &bars[stage], sb * (kBlockBytes / 8), row0, expert, policy);
    if (NM == 2)
      tma_load_3d_hint(dst + kTile, &map1, &bars[stage], sb * (kBlockBytes / 8), row0, expert,
                       policy);
  };
  if (lane == 0)
    for (int s = 0; s < kStagesMoe && s < nsteps; ++s) issue(s, sb0 + s);

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

  float yacc[NM][NT][4];
#pragma unroll
  for (int mi = 0; mi < NM; ++mi)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      yacc[mi][nt][0] = yacc[mi][nt][1] = yacc[mi][nt][2] = yacc[mi][nt][3] = 0.f;

  bool ok = true;
  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0; i < nsteps; ++i) {
    const int sb = sb0 + i;
    if (!mbar_wait(&bars[stage], phase, a.err)) {
      ok = false;
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
    if (lane == 0 && i + kStagesMoe < nsteps) issue(stage, sb + kStagesMoe);
    if (++stage == kStagesMoe) {
      stage = 0;
      phase ^= 1u;
    }
    // This lane decodes sub-blocks 2t, 2t+1 of rows g, g+8; the other lanes of
    // its quad fetch them by shuffle.
    float dsA[NM][2], dsB[NM][2], dmA[NM][2], dmB[NM][2];
#pragma unroll
    for (int mi = 0; mi < NM; ++mi)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t sc2, m2;
        scales_pair(hdr[mi][r].y, hdr[mi][r].z, hdr[mi][r].w, t, &sc2, &m2);
        const float d = half_lo_to_float(hdr[mi][r].x), dmin = half_hi_to_float(hdr[mi][r].x);
        dsA[mi][r] = d * (float)(sc2 & 0xFFu);
        dsB[mi][r] = d * (float)(sc2 >> 8);
        dmA[mi][r] = dmin * (float)(m2 & 0xFFu);
        dmB[mi][r] = dmin * (float)(m2 >> 8);
      }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = j >> 1;
      const bool hi = j & 1;
      uint32_t b0[NT][2], b1[NT][2];
      float xs[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int64_t off = (int64_t)sb * kQK + 32 * j + 8 * t;
        const uint4 v = cval[nt] ? __ldg(reinterpret_cast<const uint4 *>(src[nt] + off))
                                 : make_uint4(0, 0, 0, 0);
        b0[nt][0] = __byte_perm(v.x, v.y, 0x5410);
        b1[nt][0] = __byte_perm(v.x, v.y, 0x7632);
        b0[nt][1] = __byte_perm(v.z, v.w, 0x5410);
        b1[nt][1] = __byte_perm(v.z, v.w, 0x7632);
        const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        const float2 p2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z));
        const float2 p3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.w));
        xs[nt] = ((p0.x + p0.y) + (p1.x + p1.y)) + ((p2.x + p2.y) + (p3.x + p3.y));
      }
      // X_j of column nt*8+g is its quad's sum; accumulator column 2t+e needs the
      // sum of column 2t+e, held by the quad of lane 4(2t+e).
      float Xc[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float sum = xs[nt];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        Xc[nt][0] = __shfl_sync(0xffffffffu, sum, 4 * (2 * t));
        Xc[nt][1] = __shfl_sync(0xffffffffu, sum, 4 * (2 * t + 1));
      }
      const int srcl = (lane & ~3) | (j >> 1);
#pragma unroll
      for (int mi = 0; mi < NM; ++mi) {
        float acc[NT][4];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint32_t w0 = s ? qw[mi][0][c].y : qw[mi][0][c].x;
          const uint32_t w1 = s ? qw[mi][1][c].y : qw[mi][1][c].x;
          const uint32_t a0 = hi ? nib_hi(w0) : nib_lo(w0);
          const uint32_t a1 = hi ? nib_hi(w1) : nib_lo(w1);
          const uint32_t a2 = hi ? nib_hi(w0 >> 8) : nib_lo(w0 >> 8);
          const uint32_t a3 = hi ? nib_hi(w1 >> 8) : nib_lo(w1 >> 8);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (s == 0)
              mma_bf16_zc(acc[nt], a0, a1, a2, a3, b0[nt][0], b1[nt][0]);
            else
              mma_bf16(acc[nt], a0, a1, a2, a3, b0[nt][1], b1[nt][1]);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float ds = __shfl_sync(0xffffffffu, hi ? dsB[mi][r] : dsA[mi][r], srcl);
          const float dm = __shfl_sync(0xffffffffu, hi ? dmB[mi][r] : dmA[mi][r], srcl);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float X = Xc[nt][e];
              float &yv = yacc[mi][nt][2 * r + e];
              yv = fmaf(ds, fmaf(-128.f, X, acc[nt][2 * r + e]), yv);
              yv = fmaf(-dm, X, yv);
            }
        }
      }
    }
  }

  // Split-K partials of each m-tile: red[mi][warp][row][col].
#pragma unroll
  for (int mi = 0; mi < NM; ++mi)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = g + 8 * (e >> 1);
        const int col = nt * 8 + 2 * t + (e & 1);
        red[((mi * WM * WK + warp) * kRows + row) * kCols + col] = yacc[mi][nt][e];
      }
  __syncwarp();
  if (!ok && lane == 0) red[(warp * kRows) * kCols] = __int_as_float(0x7fc00000);
  __syncthreads();
  const int nout = DOWN ? np : ncols;  // outputs per row: pairs
  for (int idx = threadIdx.x; idx < WM * kRows * nout; idx += blockDim.x) {
    const int m = idx / (kRows * nout);
    const int row = (idx / nout) % kRows;
    const int pr = idx % nout;
    const int grow = blockIdx.x * (kRows * WM) + m * kRows + row;
    if (grow >= rows_total) continue;
    auto part = [&](int mi, int col) {
      float v = 0.f;
      for (int k = 0; k < WK; ++k) v += red[((mi * WM * WK + m * WK + k) * kRows + row) * kCols + col];
      return v;
    };
    if (DOWN) {
      a.p[(size_t)(pstart + pr) * a.hidden + grow] = part(0, 2 * pr) + part(0, 2 * pr + 1);
    } else {
      const float gg = part(0, pr), uu = part(1, pr);
      const float hv = gg / (1.f + __expf(-gg)) * uu;
      const __nv_bfloat16 hh = __float2bfloat16_rn(hv);
      const __nv_bfloat16 hl = __float2bfloat16_rn(hv - __bfloat162float(hh));
      a.h[(size_t)(pstart + pr) * a.ffn + grow] = hv;
      a.h_hi[(size_t)(pstart + pr) * a.ffn + grow] = hh;
      a.h_lo[(size_t)(pstart + pr) * a.ffn + grow] = hl;
    }
  }
}

// ---------------------------------------------------------------- 4. combine
__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeArgs a) {
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

std::once_flag g_moe_attr;
constexpr int kGuWK = 4;  // gate/up: 4 warps split K (hidden)
constexpr int kDnWM = 4;  // down: 4 m-tiles per CTA, full K (ffn) per warp

template <int NT, bool DOWN, int WM, int WK>
constexpr int expert_smem() {
  return WM * WK * ((kStagesMoe * (DOWN ? 1 : 2) * kTile + 64 + 127) / 128 * 128) +
         (DOWN ? 1 : 2) * WM * WK * kRows * NT * 8 * 4;
}

template <int NT, bool DOWN, int WM, int WK>
void allow() {
  cudaFuncSetAttribute(moe_expert_kernel<NT, DOWN, WM, WK>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, expert_smem<NT, DOWN, WM, WK>());
}

void moe_attributes() {
  allow<1, false, 1, kGuWK>();
  allow<2, false, 1, kGuWK>();
  allow<1, true, kDnWM, 1>();
  allow<2, true, kDnWM, 1>();
  allow<4, true, kDnWM, 1>();
}

template <int NT, bool DOWN, int WM, int WK>
void launch_expert(dim3 grid, const CUtensorMap &m0, const CUtensorMap &m1, const MoeArgs &a,
                   int nsb, int ks, int rows, cudaStream_t stream) {
  moe_expert_kernel<NT, DOWN, WM, WK><<<grid, WM * WK * 32, expert_smem<NT, DOWN, WM, WK>(),
                                       stream>>>(m0, m1, a, nsb, ks, rows);
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

cudaError_t launch_moe(const void *w_gate, const void *w_up, const void *w_down,
                       int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                       const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                       const float *wts, int32_t top_k, float *y, int64_t ldy, void *workspace,
                       cudaStream_t stream) {
  if (n_experts > kMaxExperts) return cudaErrorInvalidValue;
  std::call_once(g_moe_attr, moe_attributes);
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

  moe_route_kernel<<<1, 1024, 0, stream>>>(a);
  const int max_slots = MoeLayout::max_slots(n_experts, P);
  const int cap = std::min(P, kSlotPairs);  // pairs per slot at most
  {  // gate/up: K = hidden
    const int nsb = (int)(hidden / kQK);
    const int ks = (nsb + kGuWK - 1) / kGuWK;
    dim3 grid((unsigned)((ffn + kRows - 1) / kRows), (unsigned)max_slots);
    if (cap <= 8)
      launch_expert<1, false, 1, kGuWK>(grid, mg, mu, a, nsb, ks, (int)ffn, stream);
    else
      launch_expert<2, false, 1, kGuWK>(grid, mg, mu, a, nsb, ks, (int)ffn, stream);
  }
  {  // down: K = ffn, two columns per pair
    const int nsb = (int)(ffn / kQK);
    dim3 grid((unsigned)((hidden + kRows * kDnWM - 1) / (kRows * kDnWM)), (unsigned)max_slots);
    if (2 * cap <= 8)
      launch_expert<1, true, kDnWM, 1>(grid, md, md, a, nsb, nsb, (int)hidden, stream);
    else if (2 * cap <= 16)
      launch_expert<2, true, kDnWM, 1>(grid, md, md, a, nsb, nsb, (int)hidden, stream);
    else
      launch_expert<4, true, kDnWM, 1>(grid, md, md, a, nsb, nsb, (int)hidden, stream);
  }
  {
    dim3 grid((unsigned)((hidden + 255) / 256), (unsigned)n_tokens);
    moe_combine_kernel<<<grid, 256, 0, stream>>>(a);
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

void *g_scratch_ptr[64];
cudaError_t g_scratch_status[64];
std::once_flag g_scratch_once[64];

// Host code may not use g_moe_scratch as an address (it names a host-side
// stand-in); the device address is resolved once per device, with that device
// current, on the first call made on it.
void resolve_scratch(int dev) {
  void *p = nullptr;
  g_scratch_status[dev] = cudaGetSymbolAddress(&p, g_moe_scratch);
  g_scratch_ptr[dev] = (g_scratch_status[dev] == cudaSuccess) ? p : nullptr;
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
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], resolve_scratch, dev);
  if (g_scratch_ptr[dev] == nullptr) return g_scratch_status[dev];
  return launch_moe(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn, x, n_tokens, ldx,
                    ids, wts, top_k, y, ldy, g_scratch_ptr[dev], stream);
}

}  // namespace q4k
