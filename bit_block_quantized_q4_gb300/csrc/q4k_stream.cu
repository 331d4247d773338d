// q4k_stream.cu -- decode projections Y[b] = W X[b] with W in Q4_K for batch
// 1..4, any number of them in one persistent launch ("spec: specialized model
// runtimes", sections "Architecture" (T0 GEMM, quant/dequant) and "Development
// sequence" (decode throughput is the metric; graph-captured decode); small
// decode batches: "PRD: Performant Concurrent Distributed GGUF Runtime",
// DGR-012), and the fused gate/up projection H[b] = silu(Wg X[b]) * (Wu X[b])
// of a dense or shared-expert FFN ("Layer Package Repository Spec", section
// "Policy Resolution": merged shared gate/up).  The same kernel takes batch-1
// projections of the other k-quant formats (FMT = 2, 3, 5, 6: q2_K, q3_K,
// Q5_K, Q6_K; "Layer Package Repository Spec", sections "Policy Resolution"
// and "Repository Identity"), each with its own unpack of the super-block.
//
// Work: a tile is 16*MT weight rows of one op over the op's whole K (a GLU op's
// tile is its gate rows, then the same up rows).  The ops of a launch form one
// list of tiles in op order; each tile stream takes a contiguous run of it,
// balanced by weight bytes, so a sequence of projections streams its weights
// back to back with no launch boundary between them.  A stream is one warp
// (KP = 1), or KP warps that split each tile's super-blocks and add their
// partial sums in warp order through shared memory (for launches with too few
// tiles to occupy the GPU).
//
// Each warp owns a ring of shared-memory stages: SB super-blocks of each of its
// 16*MT rows plus the x of those super-blocks for each of the NB batch rows
// (512 bytes per super-block and row), copied by the warp's own lanes in
// 16-byte cp.async chunks, one cp.async group per stage.  The ring runs ahead
// across tile, part and op boundaries; with programmatic dependent launch the
// first weight stages are requested before the wait for the previous kernel, x
// only after it.  (There is no wait on another agent: a lane waits only for
// its own copies, cp.async.wait_group.)
//
// Contraction (tensor cores, mma.sync m16n8k16 bf16 -> fp32).  Sub-block j of a
// row is taken in offset form: w = ds (q - c) + e with c the integer nearest to
// dmin m_j / (d sc_j) (see offset_form), so the A operand is the exact small
// integer q - c in bf16 ((128 + q) from one LOP3, minus 128 + c) and x enters
// unconverted as bf16.  Thread t's k-slots carry sub-block 2t (low nibbles, the
// "E" MMAs) or 2t+1 (high nibbles, the "O" MMAs) of its rows g, g+8, and the
// eight MMA columns are (slot s, batch row b): column 2s + (b & 1) of the MMAs
// of batch-row pair b/2 holds x of row b only in the k-slots of thread s and
// zeros elsewhere.  So one super-block is 16 MMAs per 16 rows and batch-row
// pair, and thread (g, t) ends with exactly the (row, sub-block, batch row)
// sums of rows g, g+8, sub-blocks 2t, 2t+1 and both rows of each pair, whose
// scales it decodes itself: no shuffles and no per-sub-block epilogue outside
// the thread.  X_j = sum of x over sub-block j comes from two more MMAs per
// batch row with A = 1.  Per super-block the thread adds ds * S_j + e * X_j for
// its (row, sub-block, batch row) triples; at the end of a tile a quad shuffle
// adds the sub-blocks of a row.  Every sum is taken in a fixed order: the
// result does not depend on timing.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "q4k.h"
#include "q4k_device.cuh"
#include "q4k_internal.h"

#ifndef Q4K_STREAM_STAGES_MT1  // ring stages per warp, 16-row tiles
#define Q4K_STREAM_STAGES_MT1 2
#endif
#ifndef Q4K_STREAM_MINB_MT1  // resident CTAs per SM the register budget is sized for
#define Q4K_STREAM_MINB_MT1 4
#endif
#ifndef Q4K_STREAM_SB  // super-blocks per stage (SB * 144 bytes of each row)
#define Q4K_STREAM_SB 2
#endif
#ifndef Q4K_STREAM_SHIFT_MUL  // 1: nibble shifts as multiply-high (FMA pipe) instead of shifts (ALU)
#define Q4K_STREAM_SHIFT_MUL 0
#endif
#ifndef Q4K_STREAM_PRE  // weight stages requested before the dependency wait (PDL)
#define Q4K_STREAM_PRE 2
#endif
#ifndef Q4K_STREAM_FORCE_KP
#define Q4K_STREAM_FORCE_KP 0
#endif
// Batch rows 2 and 3..4 (NB = 2, 4): super-blocks per stage, ring stages and
// resident CTAs per SM the register budget is sized for (measured on the
// 64-layer pass: batch 2 best at two super-blocks and two stages, 3.87 TB/s
// against 3.72 at one and three; batch 4 at one and three, 2.89 against 2.69
// at two and two, where the smaller stages let a third CTA fit per SM).
#ifndef Q4K_STREAM_SB_NB2
#define Q4K_STREAM_SB_NB2 2
#endif
#ifndef Q4K_STREAM_STAGES_NB2
#define Q4K_STREAM_STAGES_NB2 2
#endif
#ifndef Q4K_STREAM_MINB_NB2
#define Q4K_STREAM_MINB_NB2 4
#endif
#ifndef Q4K_STREAM_SB_NB4
#define Q4K_STREAM_SB_NB4 1
#endif
#ifndef Q4K_STREAM_STAGES_NB4
#define Q4K_STREAM_STAGES_NB4 3
#endif
#ifndef Q4K_STREAM_MINB_NB4
#define Q4K_STREAM_MINB_NB4 3
#endif
// Q6_K at batch 1: super-blocks per stage and ring stages (its slot is
// refilled only after the super-block's contraction, which reads the quants
// from shared memory as it goes; measured on the 5120 x 17408 projection: one
// super-block and two stages 1.68 TB/s, three stages 1.65, four 1.62, two
// super-blocks 1.20).
#ifndef Q4K_STREAM_SB_Q6
#define Q4K_STREAM_SB_Q6 1
#endif
#ifndef Q4K_STREAM_STAGES_Q6
#define Q4K_STREAM_STAGES_Q6 2
#endif
// q3_K at batch 1: super-blocks per stage and ring stages (refilled after the
// contraction, as Q6_K).
#ifndef Q4K_STREAM_SB_Q3
#define Q4K_STREAM_SB_Q3 1
#endif
#ifndef Q4K_STREAM_STAGES_Q3
#define Q4K_STREAM_STAGES_Q3 2
#endif
// q2_K at batch 1: super-blocks per stage and ring stages.
#ifndef Q4K_STREAM_SB_Q2
#define Q4K_STREAM_SB_Q2 2
#endif
#ifndef Q4K_STREAM_STAGES_Q2
#define Q4K_STREAM_STAGES_Q2 2
#endif
// Q5_K at batch 1: super-blocks per stage and ring stages (measured on the
// 5120 x 17408 projection: one and two, 2.01 TB/s, against 1.83 at two and
// two, where the 368-byte row slots leave room for only 3 CTAs per SM).
#ifndef Q4K_STREAM_SB_Q5
#define Q4K_STREAM_SB_Q5 1
#endif
#ifndef Q4K_STREAM_STAGES_Q5
#define Q4K_STREAM_STAGES_Q5 2
#endif

namespace q4k {

namespace {

constexpr int kWarps = 4;              // warps per CTA
constexpr int kXBytes = kQK * 2;       // bf16 x of one super-block
constexpr int kPermStride = 20;        // words per sub-block in the permuted x (16 used)
// words of one batch row of one super-block in the permuted x: 4 more than the
// eight sub-blocks, so that the B-fragment reads of batch rows 2P and 2P+1
// fall on different banks
constexpr int kPermWords = 8 * kPermStride + 4;
// Q4_K weight matrices (tensor maps) and ops per launch: with a 128-byte map
// per matrix the kernel parameter table stays under 32 KB.
constexpr int kMaxOps = Q4K_SEQ_MATRICES_PER_LAUNCH;

struct StreamOp {
  const uint8_t *w;   // weights; the gate matrix of a GLU op
  const uint8_t *w2;  // up matrix of a GLU op, nullptr for a plain projection
  const __nv_bfloat16 *x;
  float *y;
  long long byte0;  // weight bytes of the ops before this one
  int n, nsb, ntiles, parts;
  int ldx, ldy;     // batch-row strides of x and y (elements)
  int map;          // Q4_K, Q5_K: index of the weight matrix's tensor map (the up matrix's is map + 1)
};

template <int NOPS>
struct StreamParams {
  // Q4_K, Q5_K: 2-D tensor maps over the weight matrices (unused by the other
  // formats); first, for their 64-byte alignment
  CUtensorMap map[NOPS == 1 ? 2 : NOPS];
  StreamOp op[NOPS];
  unsigned *err;  // device error word (a timed-out wait on a stage)
  int nops;
  int batch;     // batch rows (1 .. NB of the kernel)
  int kp;        // warps per tile stream (split of each tile's super-blocks)
  int pre;       // weight stages requested before the dependency wait
  int nstreams;  // tile streams in the grid
  long long total;
};
static_assert(sizeof(StreamParams<kMaxOps>) <= 32764, "kernel parameters are limited to 32764 bytes");

template <int MT, int NB, int FMT = 4>
struct StreamCfg {
  static_assert(FMT == 4 || MT == 1, "the other k-quants run with 16-row tiles");
  static constexpr int kRows = 16 * MT;
  // Super-block layout: Q4_K 144 bytes (quants at 16); Q5_K 176 bytes (the
  // fifth bits at 16, the low nibbles at 48) -- the first 16 bytes (d, dmin,
  // 12 scale bytes) are Q4_K's; q2_K 84 bytes (16 scale | min << 4 bytes,
  // 64 bytes of 2-bit quants at 16, d and dmin at 80); Q6_K 210 bytes (128
  // low-nibble bytes, 64 bytes of high bits at 128, 16 int8 scales at 192,
  // d at 208); q3_K 110 bytes (32 mask bytes, 64 bytes of 2-bit quants at 32,
  // 12 bytes of 6-bit scales at 96, d at 108).
  static constexpr int kBlock =
      FMT == 5 ? 176 : FMT == 2 ? 84 : FMT == 6 ? 210 : FMT == 3 ? 110 : kBlockBytes;
  static constexpr int kQs = FMT == 5 ? 48 : kQsOffset;
  // q2_K blocks are only 4-byte aligned, q3_K and Q6_K ones 2-byte aligned: a
  // stage copies a row's bytes from its start rounded down to 16 (at most 12
  // or 14 bytes early).
  static constexpr int kLead = FMT == 2 ? 12 : (FMT == 3 || FMT == 6) ? 14 : 0;
  static constexpr int kPairs = (NB + 1) / 2;      // MMA column groups (batch-row pairs)
  static constexpr int kSB = FMT == 5  ? Q4K_STREAM_SB_Q5
                             : FMT == 2 ? Q4K_STREAM_SB_Q2
                             : FMT == 6 ? Q4K_STREAM_SB_Q6
                             : FMT == 3 ? Q4K_STREAM_SB_Q3
                             : NB == 1 ? Q4K_STREAM_SB
                             : NB == 2 ? Q4K_STREAM_SB_NB2
                                       : Q4K_STREAM_SB_NB4;
  static constexpr int kStages = FMT == 5  ? Q4K_STREAM_STAGES_Q5
                                 : FMT == 2 ? Q4K_STREAM_STAGES_Q2
                                 : FMT == 6 ? Q4K_STREAM_STAGES_Q6
                                 : FMT == 3 ? Q4K_STREAM_STAGES_Q3
                                 : NB == 1 ? Q4K_STREAM_STAGES_MT1
                                 : NB == 2 ? Q4K_STREAM_STAGES_NB2
                                           : Q4K_STREAM_STAGES_NB4;
  static constexpr int kMinBlocks = NB == 1 ? Q4K_STREAM_MINB_MT1
                                            : NB == 2 ? Q4K_STREAM_MINB_NB2 : Q4K_STREAM_MINB_NB4;
  // 16-byte chunks a row's stage copy needs at most
  static constexpr int kChunks = (kLead + kSB * kBlock + 15) / 16;
  // a row's slot in a stage: its kSB super-blocks (and the lead), padded by 16
  // bytes when needed so that the 16*MT rows fall on different banks
  static constexpr int kRowBytes =
      (FMT == 2 || FMT == 3 || FMT == 6) ? 16 * kChunks + 16
                                         : kSB * kBlock + (kSB % 2 == 0 ? 16 : 0);
  static constexpr int kWBytes = kRows * kRowBytes;    // weight bytes of a stage
  static constexpr int kXStage = NB * kSB * kXBytes;   // x bytes of a stage: [batch row][sb]
  // permuted-x buffers: two at NB = 1 (written and read on alternate
  // super-blocks), one otherwise (a warp barrier separates the reads of one
  // super-block from the writes of the next)
  static constexpr int kPermBufs = NB == 1 ? 2 : 1;
  static constexpr int kPermBuf = NB * kPermWords;     // words of one buffer: [batch row][sub-block]
  // Q5_K: the super-block's fifth bits (32 bytes per row) are copied out of
  // the ring before the slot is refilled, into one of two buffers with rows
  // 48 bytes apart (the reads of 8 rows by a warp then hit distinct banks).
  static constexpr int kQhRow = 48;
  static constexpr int kQhBuf = FMT == 5 ? kRows * kQhRow : 0;
  // Q4_K and Q5_K stages are one TMA tile of the weight matrix (16*MT rows by
  // the row slot's bytes: with the 16-byte pad the tile reaches 16 bytes into
  // the next stage, or past the row's end, which reads as zeros) and one bulk
  // copy of x per batch row, both completing on the slot's mbarrier.  The
  // other formats (blocks not 16-byte aligned) copy 16-byte chunks with
  // cp.async.
  static constexpr bool kTma = FMT == 4 || FMT == 5;
  // warp region: ring weights | ring x | permuted-x buffers | 64 zero bytes |
  // fifth-bit buffers (Q5_K) | ring mbarriers (Q4_K)
  static constexpr int kOffX = kStages * kWBytes;
  static constexpr int kOffPerm = kOffX + kStages * kXStage;
  static constexpr int kOffZero = kOffPerm + kPermBufs * kPermBuf * 4;
  static constexpr int kOffQh = kOffZero + 64;
  static constexpr int kOffBar = (kOffQh + 2 * kQhBuf + 7) / 8 * 8;
  static constexpr int kWarpBytes = (kOffBar + (kTma ? 8 * kStages : 0) + 127) / 128 * 128;
  static_assert(!kTma || (kWBytes % 128 == 0 && kXStage % 128 == 0 && kRowBytes % 16 == 0),
                "TMA destinations 128-byte aligned, tile rows whole 16-byte units");
  static constexpr int kRedBytes = 2 * kWarps * 2 * NB * kRows * 4;  // split-K partials
  static constexpr int kSmem = kWarps * kWarpBytes + kRedBytes;
};

// Position of a warp's next stage: super-blocks sb .. sb+SB-1 (at most kb1 - sb
// of them) of part `part` of tile `tile` of op `op`; [kb0, kb1) is the warp's
// share of the op's super-blocks.  For the current (op, tile, part) it keeps
// this lane's weight row (nullptr when the tile has no row for the lane), the
// op's x and the bytes of one super-block of the tile, so that issuing a stage
// is a few instructions.
struct Pos {
  int op, tile, part, sb, kb0, kb1;
  bool valid;
  const uint8_t *src;   // the tile's first weight row (of this part's matrix)
  const __nv_bfloat16 *xsrc;
  int ldx;
  int nrows;            // weight rows of the tile
  long long rstride;    // bytes from one weight row to the next
  const uint8_t *wend;  // end of this part's weight matrix
  int map;              // Q4_K, Q5_K: tensor map of this part's matrix
};

template <int NOPS>
__device__ __forceinline__ long long tile_start(const StreamParams<NOPS> &p, int op, int tile,
                                                int rows) {
  const StreamOp &o = p.op[op];
  return o.byte0 + (long long)tile * rows * o.nsb * kBlockBytes * o.parts;
}

__device__ __forceinline__ void krange(int nsb, int kp, int KP, int &kb0, int &kb1) {
  const int ks = (nsb + KP - 1) / KP;
  kb0 = min(nsb, kp * ks);
  kb1 = min(nsb, kb0 + ks);
}

// First tile of a stream: the first tile that starts at or after byte lo.
template <int NOPS>
__device__ __forceinline__ void first_tile(const StreamParams<NOPS> &p, int rows, long long lo,
                                           long long hi, int &op, int &tile, bool &valid) {
  int a = 0, b = p.nops - 1;
  while (a < b) {
    const int m = (a + b + 1) >> 1;
    if (p.op[m].byte0 <= lo) a = m; else b = m - 1;
  }
  op = a;
  const StreamOp &o = p.op[op];
  const long long cost = (long long)rows * o.nsb * kBlockBytes * o.parts;
  tile = (int)((lo - o.byte0 + cost - 1) / cost);
  if (lo <= o.byte0) tile = 0;
  if (tile >= o.ntiles) {
    ++op;
    tile = 0;
  }
  valid = op < p.nops && tile_start(p, op, tile, rows) < hi;
}

template <int NOPS>
__device__ __forceinline__ void next_tile(const StreamParams<NOPS> &p, int rows, long long hi,
                                          int &op, int &tile, bool &valid) {
  if (++tile >= p.op[op].ntiles) {
    ++op;
    tile = 0;
  }
  valid = op < p.nops && tile_start(p, op, tile, rows) < hi;
}

// (The walk measures work in units of 144 bytes per super-block whatever the
// format: every op of a launch has the same format, so only the addresses
// below use the real block size BLK.)
template <int BLK, int NOPS>
__device__ __forceinline__ void pos_load(const StreamParams<NOPS> &p, int rows, Pos &s) {
  const StreamOp &o = p.op[s.op];
  const int row0 = s.tile * rows;
  s.nrows = min(rows, o.n - row0);
  s.rstride = (long long)o.nsb * BLK;
  const uint8_t *w = s.part ? o.w2 : o.w;
  s.src = w + (size_t)row0 * s.rstride;
  s.wend = w + (size_t)o.n * s.rstride;
  s.xsrc = o.x;
  s.ldx = o.ldx;
  s.map = o.map + s.part;
}

// Producer walk over the non-empty stages of a stream, for warp kp of KP:
// moves forward until the position names a stage (skips tiles whose share of
// super-blocks is empty for this warp) and loads the tile's sources.
template <int BLK, int NOPS>
__device__ __forceinline__ void pos_settle(const StreamParams<NOPS> &p, int rows, long long hi,
                                        int kp, Pos &s) {
  while (s.valid && s.sb >= s.kb1) {
    if (++s.part < p.op[s.op].parts) {
      s.sb = s.kb0;
      continue;
    }
    next_tile(p, rows, hi, s.op, s.tile, s.valid);
    if (!s.valid) break;
    s.part = 0;
    krange(p.op[s.op].nsb, kp, p.kp, s.kb0, s.kb1);
    s.sb = s.kb0;
  }
  if (s.valid) pos_load<BLK>(p, rows, s);
}

template <int SB, int BLK, int NOPS>
__device__ __forceinline__ void pos_next(const StreamParams<NOPS> &p, int rows, long long hi,
                                         int kp, Pos &s) {
  if ((s.sb += SB) < s.kb1) return;
  pos_settle<BLK>(p, rows, hi, kp, s);
}

// (x & 0x00030003) | magic_reg as one LOP3: the 2-bit quants in bytes 0 and 2
// of x as the bf16 pair (128 + q0, 128 + q2).
__device__ __forceinline__ uint32_t lop_q2(uint32_t x, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00030003, %2, 0xEA;\n" : "=r"(d) : "r"(x), "r"(magic_reg));
  return d;
}
// (x & 0x00040004) | magic_reg as one LOP3: bit 2 of both halves of x over
// the bf16 magic.
__device__ __forceinline__ uint32_t lop_bit2(uint32_t x, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00040004, %2, 0xEA;\n" : "=r"(d) : "r"(x), "r"(magic_reg));
  return d;
}
// (x & 0x00300030) | magic_reg as one LOP3: bits 4, 5 of both halves of x
// over the bf16 magic.
__device__ __forceinline__ uint32_t lop_bits45(uint32_t x, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00300030, %2, 0xEA;\n" : "=r"(d) : "r"(x), "r"(magic_reg));
  return d;
}
// (x & 0x00100010) | magic_reg as one LOP3: bit 4 of both halves of x over the
// bf16 magic.
__device__ __forceinline__ uint32_t lop_bit4(uint32_t x, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00100010, %2, 0xEA;\n" : "=r"(d) : "r"(x), "r"(magic_reg));
  return d;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// w >> n, as a shift (ALU pipe) or as the high half of w * 2^(32-n) (FMA pipe).
template <int N>
__device__ __forceinline__ uint32_t shr(uint32_t w) {
#if Q4K_STREAM_SHIFT_MUL == 1
  return __umulhi(w, 1u << (32 - N));
#elif Q4K_STREAM_SHIFT_MUL == 2
  return N == 8 ? __umulhi(w, 1u << 24) : w >> N;
#else
  return w >> N;
#endif
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

template <int MT, int NOPS, int NB, int FMT>
__global__ void __launch_bounds__(kWarps * 32, StreamCfg<MT, NB, FMT>::kMinBlocks)
    gemv_stream_kernel(const __grid_constant__ StreamParams<NOPS> p) {
  using C = StreamCfg<MT, NB, FMT>;
  constexpr int TR = C::kRows, ST = C::kStages, NP = C::kPairs;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int KP = p.kp;
  const int kp = warp % KP;                        // this warp's share of each tile
  const int sic = warp / KP;                       // stream within the CTA
  const int sid = blockIdx.x * (kWarps / KP) + sic;  // stream id
  const long long lo = p.total * sid / p.nstreams, hi = p.total * (sid + 1) / p.nstreams;
  const int batch = NB == 1 ? 1 : p.batch;

  uint8_t *wreg = smem + (size_t)warp * C::kWarpBytes;
  uint8_t *ringw = wreg;
  uint8_t *ringx = wreg + C::kOffX;
  uint32_t *perm = reinterpret_cast<uint32_t *>(wreg + C::kOffPerm);
  const uint32_t *zeros = reinterpret_cast<const uint32_t *>(wreg + C::kOffZero);
  float *red = reinterpret_cast<float *>(smem + (size_t)kWarps * C::kWarpBytes);

  if (lane < 16) reinterpret_cast<uint32_t *>(wreg + C::kOffZero)[lane] = 0u;
  uint64_t *full = reinterpret_cast<uint64_t *>(wreg + C::kOffBar);  // TMA ring mbarriers
  if (C::kTma && lane == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // ---- producer: the stream's stages in order, STAGES ahead of the consumer
  Pos pp;
  first_tile(p, TR, lo, hi, pp.op, pp.tile, pp.valid);
  pp.part = 0;
  if (pp.valid) krange(p.op[pp.op].nsb, kp, KP, pp.kb0, pp.kb1);
  else pp.kb0 = pp.kb1 = 0;
  pp.sb = pp.kb0;
  pos_settle<C::kBlock>(p, TR, hi, kp, pp);  // the first stage (when there is one)

  constexpr int SB = C::kSB;
  // Q4_K, Q5_K: lane 0 arms the slot's mbarrier with the stage's bytes (the whole
  // weight tile, out-of-range parts included, and x) and requests the weight
  // tile; lanes b < batch each request x of batch row b.
  // The other formats: a stage's copies are 16-byte cp.async chunks.  Weights: the LPR lanes
  // LPR r .. LPR r + LPR - 1 take row r of the tile, lane LPR r + i its chunks
  // i, i + LPR, ... of the SB super-blocks (with 16-row tiles a lane pair
  // moves 32 contiguous bytes per instruction); x: lane l takes chunk l of
  // each (batch row, super-block).  Each lane closes a stage's copies into one
  // cp.async group, and every ring slot the consumer releases gets one group
  // (empty when the stream has no further stage), so the oldest stage in
  // flight is always the group ST - 1 places back.
  constexpr int LPR = 32 / TR;
  const int crow = lane / LPR, csub = lane % LPR;
  const uint64_t pol = C::kTma ? l2_evict_first_policy() : 0ull;
  auto issue_w = [&](int slot, const Pos &s) {
    const int cnt = min(SB, s.kb1 - s.sb);
    if constexpr (C::kTma) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[slot], (uint32_t)(C::kWBytes + batch * cnt * kXBytes));
        tma_load_2d_hint(ringw + slot * C::kWBytes, &p.map[s.map], &full[slot],
                         s.sb * (C::kBlock / 8), s.tile * TR, pol);
      }
      return;
    }
    if (crow >= s.nrows) return;
    uint8_t *dst = ringw + slot * C::kWBytes + crow * C::kRowBytes + csub * 16;
    const uint8_t *src = s.src + (size_t)crow * s.rstride + (size_t)s.sb * C::kBlock;
    if constexpr (FMT == 2 || FMT == 3 || FMT == 6) {
      // from the row's stage start rounded down to 16 bytes; a chunk that
      // reaches past the matrix takes only the bytes inside it (the rest of
      // the 16 are zero-filled and never read)
      const int lead = (int)(reinterpret_cast<uintptr_t>(src) & 15u);
      const uint8_t *src0 = src - lead + csub * 16;
      const int nch = (lead + cnt * C::kBlock + 15) >> 4;
#pragma unroll
      for (int j = 0; j < (C::kChunks + LPR - 1) / LPR; ++j) {
        if (LPR * j + csub >= nch) break;
        const uint8_t *cs = src0 + 16 * LPR * j;
        const long long left = s.wend - cs;
        cp_async16(dst + 16 * LPR * j, left > 0 ? cs : src0, left >= 16 ? 16 : left > 0 ? (int)left : 0);
      }
    } else {
      constexpr int kFull = (C::kBlock / 16) * SB;  // chunks of a row in a full stage
      if (cnt == SB) {  // (every stage but the last of a warp's share of a tile)
#pragma unroll
        for (int j = 0; j < kFull / LPR; ++j) cp_async16(dst + 16 * LPR * j, src + csub * 16 + 16 * LPR * j);
        constexpr int jt = kFull / LPR;
        if (kFull % LPR != 0 && LPR * jt + csub < kFull)
          cp_async16(dst + 16 * LPR * jt, src + csub * 16 + 16 * LPR * jt);
      } else {
        const int nch = (C::kBlock / 16) * cnt;  // chunks of a row in this stage
#pragma unroll
        for (int j = 0; j < (kFull + LPR - 1) / LPR; ++j)
          if (LPR * j + csub < nch) cp_async16(dst + 16 * LPR * j, src + csub * 16 + 16 * LPR * j);
      }
    }
  };
  // x of batch row b goes to [b][0 .. SB) of the stage's x area.
  auto issue_x = [&](int slot, const Pos &s) {
    const int cnt = min(SB, s.kb1 - s.sb);
    if constexpr (C::kTma) {
      if (lane < batch)
        bulk_load(ringx + slot * C::kXStage + lane * (SB * kXBytes),
                  s.xsrc + (size_t)lane * s.ldx + (size_t)s.sb * kQK, (uint32_t)(cnt * kXBytes),
                  &full[slot]);
      return;
    }
    uint8_t *dst = ringx + slot * C::kXStage + lane * 16;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int u = 0; u < SB; ++u)
        if (b < batch && u < cnt)
          cp_async16(dst + (b * SB + u) * kXBytes,
                     s.xsrc + (size_t)b * s.ldx + (size_t)(s.sb + u) * kQK + lane * 8);
  };

  // With programmatic dependent launch the first p.pre stages' weights go out
  // before the wait (weights are never written by earlier kernels), their x
  // after it.
  int npre = 0;
  {
    Pos q = pp;
    for (; npre < p.pre && npre < ST && q.valid; ++npre) {
      issue_w(npre, q);
      pos_next<SB, C::kBlock>(p, TR, hi, kp, q);
    }
  }
  grid_dependency_wait();
  int inflight = 0;  // TMA stages requested and not yet consumed
  for (int s = 0; s < ST; ++s) {
    if (pp.valid) {
      if (s >= npre) issue_w(s, pp);
      issue_x(s, pp);
      pos_next<SB, C::kBlock>(p, TR, hi, kp, pp);
      ++inflight;
    }
    if constexpr (!C::kTma) cp_async_commit();  // stage s (an empty group past the stream's end)
  }
  grid_launch_dependents();

  // ---- lane constants
  // Scale/min decode of sub-blocks 2t, 2t+1 (branch-free): lanes t < 2 read
  // the low six bits of s[j], s[j+4]; lanes t >= 2 combine a nibble of s[j+4]
  // with the top two bits of s[j-4] (scales) or s[j] (mins).  psel gathers
  // bytes k0, k0+1 of rows g (bytes 0, 1) and g+8 (bytes 2, 3).
  const bool upper = t >= 2;
  const uint32_t k0 = 2 * (t & 1);
  const uint32_t psel = k0 | ((k0 + 1) << 4) | ((k0 + 4) << 8) | ((k0 + 5) << 12);
  const uint32_t mlo4 = upper ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
  const uint32_t mhi4 = upper ? 0x30303030u : 0u;
  // B fragments: lane (g, t) is column g of every MMA; when t == g / 2 its
  // k-slots carry x of batch row 2P + (g & 1) of pair P (sub-block 2t in the E
  // MMAs, 2t+1 in the O MMAs); every other lane, and a row past the batch,
  // reads zeros.  bofs[P]: word offset of that row's sub-block 2t in a
  // permuted-x buffer, or -1.
  const bool own = t == (g >> 1);
  int bofs[NP];
#pragma unroll
  for (int P = 0; P < NP; ++P) {
    const int b = 2 * P + (g & 1);
    bofs[P] = (own && b < batch) ? b * kPermWords + 2 * t * kPermStride : -1;
  }
  uint32_t magic;
  asm volatile("mov.b32 %0, %1;\n" : "=r"(magic) : "n"(kBf16Magic));
  // q2_K, q3_K, Q6_K: x of super-block u of every batch row in B-fragment
  // order (word 2G of a 16-value half holds (x[4G], x[4G+2]), word 2G+1
  // (x[4G+1], x[4G+3])); rows past the batch read as zeros
  auto perm_x_rows = [&](uint32_t *pwb, const uint8_t *xst, int u) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (b < batch) raw = reinterpret_cast<const uint4 *>(xst + (b * C::kSB + u) * kXBytes)[lane];
      uint4 pm;
      pm.x = __byte_perm(raw.x, raw.y, 0x5410u);
      pm.y = __byte_perm(raw.x, raw.y, 0x7632u);
      pm.z = __byte_perm(raw.z, raw.w, 0x5410u);
      pm.w = __byte_perm(raw.z, raw.w, 0x7632u);
      reinterpret_cast<uint4 *>(pwb + b * kPermWords + g * kPermStride)[t] = pm;
    }
  };
  // Q5_K: rotations that bring bit 2t (2t+1) of each qh byte to bit 4.
  const uint32_t rot_e = (uint32_t)(2 * t - 4) & 31u, rot_o = (uint32_t)(2 * t - 3) & 31u;

  // ---- consumer
  int cslot = 0;
  uint32_t phase = 0;  // TMA: parity of the slot's next phase (flips when cslot wraps)
  bool ok = true;      // TMA: false once a wait on a stage has timed out
  int pbuf = 0;
  int op, tile;
  bool tvalid;
  first_tile(p, TR, lo, hi, op, tile, tvalid);
  int par = 0;  // split-K partials buffer parity
  for (; tvalid; next_tile(p, TR, hi, op, tile, tvalid), par ^= 1) {
    const StreamOp &o = p.op[op];
    int kb0, kb1;
    krange(o.nsb, kp, KP, kb0, kb1);
    // per part: rows (g, g+8) of each m-tile and each batch row, partial over
    // sub-blocks 2t, 2t+1
    float yv[2][MT][2][NB];
#pragma unroll
    for (int pt = 0; pt < 2; ++pt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int b = 0; b < NB; ++b) yv[pt][mt][0][b] = yv[pt][mt][1][b] = 0.f;
    for (int part = 0; part < o.parts; ++part) {
      float yacc[MT][2][NB];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int b = 0; b < NB; ++b) yacc[mt][0][b] = yacc[mt][1][b] = 0.f;
      for (int sb = kb0; sb < kb1; sb += SB) {
        if constexpr (C::kTma) {
          // After a timed-out wait the warp walks on without waiting or
          // computing (so that split-K partners meet it at their barriers).
          if (!ok) continue;
          if (!__all_sync(0xffffffffu, mbar_wait(&full[cslot], phase, p.err))) {
            ok = false;
            if (lane == 0) drain_ring(full, ST, cslot, phase, inflight);
            __syncwarp();
            continue;
          }
          --inflight;
        } else {
          cp_async_wait<ST - 1>();  // this lane's copies of the stage have landed
          __syncwarp();             // ... and every lane's are visible
        }
        const int cnt = min(SB, kb1 - sb);
        const uint8_t *wstage = ringw + cslot * C::kWBytes;
        const uint8_t *xstage = ringx + cslot * C::kXStage;
        // Q4_K, Q5_K: the offset forms of this thread's (row, sub-block)
        // pairs for every super-block of the stage first, so that their
        // dependency chains (header loads, reciprocals) run side by side and
        // under the unpack of the first super-block.
        float dsS[SB][MT][2][2], eeS[SB][MT][2][2];
        uint32_t subS[SB][MT][2][2];
        if constexpr (FMT == 4 || FMT == 5) {
#pragma unroll
          for (int u = 0; u < SB; ++u) {
            if (u >= cnt) break;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint8_t *rp = wstage + u * C::kBlock + (mt * 16 + g) * C::kRowBytes;
              const uint4 h0 = *reinterpret_cast<const uint4 *>(rp);
              const uint4 h1 = *reinterpret_cast<const uint4 *>(rp + 8 * C::kRowBytes);
              const uint32_t py = __byte_perm(h0.y, h1.y, psel);
              const uint32_t pz = __byte_perm(h0.z, h1.z, psel);
              const uint32_t pw4 = __byte_perm(h0.w, h1.w, psel);
              const uint32_t sc4 = ((upper ? pw4 : py) & mlo4) | ((py >> 2) & mhi4);
              const uint32_t m4 = ((upper ? (pw4 >> 4) : pz) & mlo4) | ((pz >> 2) & mhi4);
              // rows g, g+8 as the two lanes of the packed fp32 operations
              float2 d2, nd23, dmin2, pdm23;
              scale_pairs(h0.x, h1.x, d2, nd23, dmin2, pdm23);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float2 ds2, ee2;
                offset_form_rows2<FMT == 5 ? 32 : 16>(d2, nd23, dmin2, pdm23, byte_magic(sc4, e),
                                                      byte_magic(sc4, 2 + e), byte_magic_neg(m4, e),
                                                      byte_magic_neg(m4, 2 + e), ds2, ee2,
                                                      subS[u][mt][0][e], subS[u][mt][1][e]);
                dsS[u][mt][0][e] = ds2.x;
                dsS[u][mt][1][e] = ds2.y;
                eeS[u][mt][0][e] = ee2.x;
                eeS[u][mt][1][e] = ee2.y;
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < SB; ++u) {
          if (u >= cnt) break;
          const uint8_t *ws = wstage + u * C::kBlock;
          uint32_t *pw = perm + pbuf * C::kPermBuf;
          if (C::kPermBufs == 1) __syncwarp();  // the previous super-block's reads are done
          if constexpr (FMT == 2) {
            // q2_K: 16 sub-blocks of 16 weights; thread t owns sub-blocks
            // 4t .. 4t+3 (a = 0..3) of rows g, g+8.  Column sums of x per
            // 16 values: the first half of each 32-value block is held by
            // lanes t < 2, the second by t >= 2, so two half-masked pairs of
            // MMAs with A = 1 give thread t the sums X_{4t+a} of each batch
            // row.  The MMA columns of the contraction are (slot, batch row)
            // as for Q4_K.
            float xl[NB][4], xh[NB][4];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              uint4 raw = make_uint4(0u, 0u, 0u, 0u);
              if (b < batch) raw = reinterpret_cast<const uint4 *>(xstage + (b * SB + u) * kXBytes)[lane];
              const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
              const uint4 rl = t < 2 ? raw : z4, rh = t < 2 ? z4 : raw;
              mma_bf16_zc(xl[b], kBf16One, kBf16One, kBf16One, kBf16One, rl.x, rl.y);
              mma_bf16(xl[b], kBf16One, kBf16One, kBf16One, kBf16One, rl.z, rl.w);
              mma_bf16_zc(xh[b], kBf16One, kBf16One, kBf16One, kBf16One, rh.x, rh.y);
              mma_bf16(xh[b], kBf16One, kBf16One, kBf16One, kBf16One, rh.z, rh.w);
              uint4 pm;
              pm.x = __byte_perm(raw.x, raw.y, 0x5410u);
              pm.y = __byte_perm(raw.x, raw.y, 0x7632u);
              pm.z = __byte_perm(raw.z, raw.w, 0x5410u);
              pm.w = __byte_perm(raw.z, raw.w, 0x7632u);
              reinterpret_cast<uint4 *>(pw + b * kPermWords + g * kPermStride)[t] = pm;
            }
            // Rows g, g+8: the stage copy of row r began (row's stage start) &
            // 15 bytes early; with the matrix 16-byte aligned that lead is
            // 4 ((row * nsb + sb) mod 4) (84 = 4 * 21).  Words: d | dmin << 16
            // at 80, the scale | min << 4 bytes of sub-blocks 4t .. 4t+3 at
            // 4t, and quant bytes 16 + 32h .. +31 (h = t / 2).
            uint32_t dw[2], scw[2], qw[2][8];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int row = g + 8 * r;
              const int lead = 4 * (((tile * TR + row) * o.nsb + sb) & 3);
              const uint8_t *bp = wstage + row * C::kRowBytes + lead + u * C::kBlock;
              dw[r] = *reinterpret_cast<const uint32_t *>(bp + 80);
              scw[r] = *reinterpret_cast<const uint32_t *>(bp + 4 * t);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                qw[r][k] = *reinterpret_cast<const uint32_t *>(bp + 16 + 32 * (t >> 1) + 4 * k);
            }
            __syncwarp();  // permuted x visible to every lane; the stage's last reads done
            if (u == cnt - 1) {
              if (pp.valid) {  // refill this slot with the stream's next stage
                issue_w(cslot, pp);
                issue_x(cslot, pp);
                pos_next<SB, C::kBlock>(p, TR, hi, kp, pp);
                ++inflight;
              }
              if constexpr (!C::kTma) cp_async_commit();
            }
            // Offset forms (c in [0, 4]) of the thread's (row, sub-block) pairs.
            float ds2[2][4], ee2[2][4];
            uint32_t sub2[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const float d = half_lo_to_float(dw[r]), dmin = half_hi_to_float(dw[r]);
              const float nd23 = d * -8388608.f, ndm23 = dmin * -8388608.f;
              const uint32_t scl = scw[r] & 0x0F0F0F0Fu, mhi = (scw[r] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
              for (int a = 0; a < 4; ++a)
                offset_form_c<4>(d, nd23, dmin, ndm23, byte_magic(scl, a), byte_magic(mhi, a),
                                 ds2[r][a], ee2[r][a], sub2[r][a]);
            }
            // B fragments: lane (g, t) with t = g / 2 carries sub-block
            // 4t + a (32-value block 2t + a/2, its half a & 1) of batch row
            // 2P + (g & 1) in column g of pair P; every other lane reads
            // zeros.  MMA (a, b): positions 4b .. 4b+3 of the sub-block;
            // acc[P][a] column 2t + i sums (q - c) x over it for batch row
            // 2P + i.
            float acc[NP][4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const uint32_t sh = 2u * (uint32_t)((2 * t + (a >> 1)) & 3);  // quant bits in a byte
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2) {
                uint4 bv[NP];
#pragma unroll
                for (int P = 0; P < NP; ++P) {
                  const bool own = t == (g >> 1) && 2 * P + (g & 1) < batch;
                  const uint32_t *pb = own ? pw + (2 * P + (g & 1)) * kPermWords +
                                                 (2 * t + (a >> 1)) * kPermStride + 8 * (a & 1)
                                           : zeros;
                  bv[P] = reinterpret_cast<const uint4 *>(pb)[own ? c2 : 0];
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int b = 2 * c2 + h, k = 4 * (a & 1) + b;
                  const uint32_t w0 = qw[0][k] >> sh, w1 = qw[1][k] >> sh;
                  const uint32_t a0 = sub_bf16x2(lop_q2(w0, magic), sub2[0][a]);
                  const uint32_t a1 = sub_bf16x2(lop_q2(w1, magic), sub2[1][a]);
                  const uint32_t a2 = sub_bf16x2(lop_q2(w0 >> 8, magic), sub2[0][a]);
                  const uint32_t a3 = sub_bf16x2(lop_q2(w1 >> 8, magic), sub2[1][a]);
#pragma unroll
                  for (int P = 0; P < NP; ++P) {
                    const uint32_t b0 = h ? bv[P].z : bv[P].x, b1 = h ? bv[P].w : bv[P].y;
                    if (b == 0)
                      mma_bf16_zc(acc[P][a], a0, a1, a2, a3, b0, b1);
                    else
                      mma_bf16(acc[P][a], a0, a1, a2, a3, b0, b1);
                  }
                }
              }
            }
            // X_{4t + a} of batch row b: halves lo / hi of 32-value blocks 2t
            // (column 2t) and 2t+1 (column 2t+1) of its column-sum MMAs.
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const float xsa[4] = {xl[b][0], xh[b][0], xl[b][1], xh[b][1]};
                float v = yacc[0][r][b];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                  v = fmaf(ds2[r][a], acc[b >> 1][a][2 * r + (b & 1)], v);
                  v = fmaf(ee2[r][a], xsa[a], v);
                }
                yacc[0][r][b] = v;
              }
            if (C::kPermBufs == 2) pbuf ^= 1;
            continue;
          }
          if constexpr (FMT == 3) {
            // q3_K: 16 sub-blocks of 16 weights, w = d (sc - 32) (u - 4) with u
            // the 3-bit value (two bits in qs, the top bit in the mask bytes)
            // and sc 6 bits: no min term, so the A operand is the exact u - 4
            // and no column sums are needed.  Thread t owns sub-blocks 4t ..
            // 4t+3 (a = 0..3) of rows g, g+8: half h = t / 2, bit pair
            // g2 = (2t + a/2) mod 4 of the qs bytes, mask bit 4h + g2.  The
            // MMA columns are (slot, batch row) as for Q6_K.
            perm_x_rows(pw, xstage, u);
            __syncwarp();  // permuted x visible to every lane
            // Rows g, g+8: the stage copy of row r began (row's stage start) &
            // 15 bytes early; with the matrix 16-byte aligned that lead is
            // 14 ((row * nsb + sb) mod 8) mod 16 (110 = 2 * 55), so the block is
            // only 2-byte aligned: words are read as funnel-shifted aligned pairs.
            auto word_at = [](const uint8_t *q) -> uint32_t {
              const uint32_t *al =
                  reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(q) & ~uintptr_t(3));
              return __funnelshift_r(al[0], al[1], 8u * (uint32_t)(reinterpret_cast<uintptr_t>(q) & 3u));
            };
            const uint8_t *bp[2];
            float ds3[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int row = g + 8 * r;
              const int lead = (14 * (((tile * TR + row) * o.nsb + sb) & 7)) & 15;
              bp[r] = wstage + row * C::kRowBytes + lead + u * C::kBlock;
              // scales of sub-blocks j = 4t .. 4t+3: low nibbles of bytes
              // 4t .. 4t+3 (t < 2) or high nibbles of bytes 4t-8 .. 4t-5
              // (t >= 2) at 96, top two bits in bits 2t of bytes 8 .. 11
              const uint32_t lo4 = (word_at(bp[r] + 96 + 4 * (t & 1)) >> (4 * (t >> 1))) & 0x0F0F0F0Fu;
              const uint32_t hi2 = (word_at(bp[r] + 104) >> (2 * t)) & 0x03030303u;
              const uint32_t sc6 = lo4 | (hi2 << 4);
              const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short *>(bp[r] + 108)));
#pragma unroll
              for (int a = 0; a < 4; ++a)
                ds3[r][a] = d * (float)((int)((sc6 >> (8 * a)) & 0xFFu) - 32);  // exact
            }
            uint32_t sub4;
            asm volatile("mov.b32 %0, %1;\n" : "=r"(sub4) : "n"(0x43044304u));  // bf16 (132, 132)
            float acc[NP][4][4];
#pragma unroll
            for (int ah = 0; ah < 2; ++ah) {  // a & 1: bytes 16 (a & 1) .. +15 of the quant / mask runs
              uint32_t qs[2][4], hm[2][4];
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                  qs[r][b] = word_at(bp[r] + 32 + 32 * (t >> 1) + 16 * ah + 4 * b);
                  hm[r][b] = word_at(bp[r] + 16 * ah + 4 * b);
                }
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2) {
                const int a = 2 * a2 + ah;
                const uint32_t g2 = (uint32_t)((2 * t + a2) & 3);
                const uint32_t qsh = 2u * g2;                                   // quant bits in a byte
                const uint32_t mrot = (4u * (uint32_t)(t >> 1) + g2 - 2u) & 31u;  // mask bit -> bit 2
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                  uint4 bv[NP];
#pragma unroll
                  for (int P = 0; P < NP; ++P) {
                    const bool own = t == (g >> 1) && 2 * P + (g & 1) < batch;
                    const uint32_t *pb = own ? pw + (2 * P + (g & 1)) * kPermWords +
                                                   (2 * t + a2) * kPermStride + 8 * ah
                                             : zeros;
                    bv[P] = reinterpret_cast<const uint4 *>(pb)[own ? c2 : 0];
                  }
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const int b = 2 * c2 + h;
                    uint32_t av[4];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                      const uint32_t lw = qs[r][b] >> qsh;
                      const uint32_t hw = __funnelshift_r(hm[r][b], hm[r][b], mrot);
                      // (128 + u) for bytes 0, 2 and 1, 3: the two low bits over
                      // the top bit at bit 2 and the bf16 magic
                      const uint32_t m02 = lop_bit2(hw, magic), m13 = lop_bit2(hw >> 8, magic);
                      av[r] = sub_bf16x2(lop_q2(lw, m02), sub4);
                      av[2 + r] = sub_bf16x2(lop_q2(lw >> 8, m13), sub4);
                    }
#pragma unroll
                    for (int P = 0; P < NP; ++P) {
                      const uint32_t b0 = h ? bv[P].z : bv[P].x, b1 = h ? bv[P].w : bv[P].y;
                      if (b == 0)
                        mma_bf16_zc(acc[P][a], av[0], av[1], av[2], av[3], b0, b1);
                      else
                        mma_bf16(acc[P][a], av[0], av[1], av[2], av[3], b0, b1);
                    }
                  }
                }
              }
            }
            // column 2t + (b & 1) of pair b / 2 holds batch row b
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                float yv = yacc[0][r][b];
#pragma unroll
                for (int a = 0; a < 4; ++a) yv = fmaf(ds3[r][a], acc[b >> 1][a][2 * r + (b & 1)], yv);
                yacc[0][r][b] = yv;
              }
            __syncwarp();  // every lane's reads of the stage are done
            if (u == cnt - 1) {
              if (pp.valid) {  // refill this slot with the stream's next stage
                issue_w(cslot, pp);
                issue_x(cslot, pp);
                pos_next<SB, C::kBlock>(p, TR, hi, kp, pp);
                ++inflight;
              }
              if constexpr (!C::kTma) cp_async_commit();
            }
            if (C::kPermBufs == 2) pbuf ^= 1;
            continue;
          }
          if constexpr (FMT == 6) {
            // Q6_K: 16 sub-blocks of 16 weights, w = d sc (q - 32) with q the
            // 6-bit value (low nibble in ql, two high bits in qh) and sc an
            // int8: no min term, so the A operand is the exact q - 32 and no
            // column sums are needed.  Thread t owns sub-blocks 4t .. 4t+3
            // (a = 0..3) of rows g, g+8: half h = t / 2 of the block, 32-value
            // group v = (2t + a/2) mod 4 (low nibbles for v < 2, high ones
            // for v >= 2; high bits 2v, 2v+1 of the qh bytes).  The MMA
            // columns are (slot, batch row) as for Q4_K: lane (g, t) with
            // t = g / 2 carries batch row 2P + (g & 1) of pair P.
            perm_x_rows(pw, xstage, u);
            __syncwarp();  // permuted x visible to every lane
            // Rows g, g+8: the stage copy of row r began (row's stage start) &
            // 15 bytes early; with the matrix 16-byte aligned that lead is
            // 2 ((row * nsb + sb) mod 8) (210 = 2 * 105), so the block is only
            // 2-byte aligned: a word at byte offset o is read as the two
            // aligned words around it, funnel-shifted by 8 (o & 3) bits.
            const uint8_t *bp[2];
            uint32_t qh[2][8];
            float ds6[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int row = g + 8 * r;
              const int lead = 2 * (((tile * TR + row) * o.nsb + sb) & 7);
              bp[r] = wstage + row * C::kRowBytes + lead + u * C::kBlock;
              // qh bytes 128 + 32h .. +31
              const uint8_t *qa = bp[r] + 128 + 32 * (t >> 1);
              const uint32_t *al = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(qa) & ~uintptr_t(3));
              const uint32_t fs = 8u * (uint32_t)(reinterpret_cast<uintptr_t>(qa) & 3u);
              uint32_t prev = al[0];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t next = al[k + 1];
                qh[r][k] = __funnelshift_r(prev, next, fs);
                prev = next;
              }
              // scales of sub-blocks 4t .. 4t+3 (int8) at 192 + 4t, d at 208
              const uint8_t *sa = bp[r] + 192 + 4 * t;
              const uint32_t *sl = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(sa) & ~uintptr_t(3));
              const uint32_t scw = __funnelshift_r(sl[0], sl[1], 8u * (uint32_t)(reinterpret_cast<uintptr_t>(sa) & 3u));
              const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short *>(bp[r] + 208)));
#pragma unroll
              for (int a = 0; a < 4; ++a)
                ds6[r][a] = d * (float)(int)(int8_t)(scw >> (8 * a));  // exact
            }
            const uint32_t nsh = (t & 1) ? 4u : 0u;  // high nibbles for v >= 2
            uint32_t sub32;
            asm volatile("mov.b32 %0, %1;\n" : "=r"(sub32) : "n"(0x43204320u));  // bf16 (160, 160)
            float acc[NP][4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const uint32_t v = (uint32_t)((2 * t + (a >> 1)) & 3);
              const uint32_t rot = (2u * v - 4u) & 31u;  // high bits 2v, 2v+1 -> bits 4, 5
              // ql bytes 64h + 16a .. +15 of each row, as four words
              uint32_t ql[2][4];
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const uint8_t *qa = bp[r] + 64 * (t >> 1) + 16 * a;
                const uint32_t *al = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(qa) & ~uintptr_t(3));
                const uint32_t fs = 8u * (uint32_t)(reinterpret_cast<uintptr_t>(qa) & 3u);
                uint32_t prev = al[0];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                  const uint32_t next = al[b + 1];
                  ql[r][b] = __funnelshift_r(prev, next, fs);
                  prev = next;
                }
              }
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2) {
                uint4 bv[NP];
#pragma unroll
                for (int P = 0; P < NP; ++P) {
                  const bool own = t == (g >> 1) && 2 * P + (g & 1) < batch;
                  const uint32_t *pb = own ? pw + (2 * P + (g & 1)) * kPermWords +
                                                 (2 * t + (a >> 1)) * kPermStride + 8 * (a & 1)
                                           : zeros;
                  bv[P] = reinterpret_cast<const uint4 *>(pb)[own ? c2 : 0];
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int b = 2 * c2 + h, kq = 4 * (a & 1) + b;
                  uint32_t av[4];
#pragma unroll
                  for (int r = 0; r < 2; ++r) {
                    const uint32_t lw = ql[r][b] >> nsh;
                    const uint32_t hw = __funnelshift_r(qh[r][kq], qh[r][kq], rot);
                    // (128 + q) for bytes 0, 2 and 1, 3: the nibble over the
                    // two high bits at bits 4, 5 and the bf16 magic
                    const uint32_t m02 = lop_bits45(hw, magic), m13 = lop_bits45(hw >> 8, magic);
                    av[r] = sub_bf16x2(lop_nib(lw, m02), sub32);
                    av[2 + r] = sub_bf16x2(lop_nib(lw >> 8, m13), sub32);
                  }
#pragma unroll
                  for (int P = 0; P < NP; ++P) {
                    const uint32_t b0 = h ? bv[P].z : bv[P].x, b1 = h ? bv[P].w : bv[P].y;
                    if (b == 0)
                      mma_bf16_zc(acc[P][a], av[0], av[1], av[2], av[3], b0, b1);
                    else
                      mma_bf16(acc[P][a], av[0], av[1], av[2], av[3], b0, b1);
                  }
                }
              }
            }
            // column 2t + (b & 1) of pair b / 2 holds batch row b
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                float yv = yacc[0][r][b];
#pragma unroll
                for (int a = 0; a < 4; ++a) yv = fmaf(ds6[r][a], acc[b >> 1][a][2 * r + (b & 1)], yv);
                yacc[0][r][b] = yv;
              }
            __syncwarp();  // every lane's reads of the stage are done
            if (u == cnt - 1) {
              if (pp.valid) {  // refill this slot with the stream's next stage
                issue_w(cslot, pp);
                issue_x(cslot, pp);
                pos_next<SB, C::kBlock>(p, TR, hi, kp, pp);
                ++inflight;
              }
              if constexpr (!C::kTma) cp_async_commit();
            }
            if (C::kPermBufs == 2) pbuf ^= 1;
            continue;
          }
          // X_j of the eight sub-blocks of each batch row: lane (g, t) holds
          // values 8t .. 8t+7 of sub-block g, exactly the B fragment of column
          // g of two MMAs.  Permuted copy: word 2G of a sub-block holds
          // (x[4G], x[4G+2]), word 2G+1 (x[4G+1], x[4G+3]) -- the pairs the
          // nibble operands meet.
          float xs[NB][4];
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (b < batch) raw = reinterpret_cast<const uint4 *>(xstage + (b * SB + u) * kXBytes)[lane];
            mma_bf16_zc(xs[b], kBf16One, kBf16One, kBf16One, kBf16One, raw.x, raw.y);
            mma_bf16(xs[b], kBf16One, kBf16One, kBf16One, kBf16One, raw.z, raw.w);
            uint4 pm;
            pm.x = __byte_perm(raw.x, raw.y, 0x5410u);
            pm.y = __byte_perm(raw.x, raw.y, 0x7632u);
            pm.z = __byte_perm(raw.z, raw.w, 0x5410u);
            pm.w = __byte_perm(raw.z, raw.w, 0x7632u);
            reinterpret_cast<uint4 *>(pw + b * kPermWords + g * kPermStride)[t] = pm;
          }
          uint4 qa[MT][2][2];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const uint8_t *rp = ws + (mt * 16 + g + 8 * r) * C::kRowBytes;
              qa[mt][r][0] = *reinterpret_cast<const uint4 *>(rp + C::kQs + 32 * t);
              qa[mt][r][1] = *reinterpret_cast<const uint4 *>(rp + C::kQs + 32 * t + 16);
            }
          uint8_t *qhb = wreg + C::kOffQh + pbuf * C::kQhBuf;
          if constexpr (FMT == 5) {
            // lanes 2r, 2r+1 copy the 32 fifth-bit bytes of row r (16 each)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const int row = mt * 16 + (lane >> 1);
              *reinterpret_cast<uint4 *>(qhb + row * C::kQhRow + 16 * (lane & 1)) =
                  *reinterpret_cast<const uint4 *>(ws + row * C::kRowBytes + 16 + 16 * (lane & 1));
            }
          }
          __syncwarp();  // permuted x visible to every lane; the stage's last reads done
          if (u == cnt - 1) {
            if (pp.valid) {  // refill this slot with the stream's next stage
              issue_w(cslot, pp);
              issue_x(cslot, pp);
              pos_next<SB, C::kBlock>(p, TR, hi, kp, pp);
              ++inflight;
            }
            if constexpr (!C::kTma) cp_async_commit();
          }

          // this super-block's offset forms (computed above)
          const float(&ds)[MT][2][2] = dsS[u];
          const float(&ee)[MT][2][2] = eeS[u];
          const uint32_t(&sub)[MT][2][2] = subS[u];

          const uint32_t *pe[NP], *po[NP];
#pragma unroll
          for (int P = 0; P < NP; ++P) {
            pe[P] = bofs[P] >= 0 ? pw + bofs[P] : zeros;
            po[P] = bofs[P] >= 0 ? pw + bofs[P] + kPermStride : zeros;
          }
          // accE[mt][P] column 2t + i = sum (q - c) x over sub-block 2t of batch
          // row 2P + i (rows g: [i], g+8: [2 + i]); accO likewise for 2t+1.
          float accE[MT][NP][4], accO[MT][NP][4];
#pragma unroll
          for (int G2 = 0; G2 < 4; ++G2) {
            uint4 be[NP], bo[NP];
#pragma unroll
            for (int P = 0; P < NP; ++P) {
              be[P] = reinterpret_cast<const uint4 *>(pe[P])[G2];  // the zero block is 4 uint4
              bo[P] = reinterpret_cast<const uint4 *>(po[P])[G2];
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int G = 2 * G2 + h;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const uint32_t w0 = word_of(qa[mt][0][G >> 2], G & 3);
                const uint32_t w1 = word_of(qa[mt][1][G >> 2], G & 3);
                // The OR operands of the nibble LOP3s: the bf16 magic, and for
                // Q5_K the fifth bit of each quant at bit 4 of its half.
                uint32_t me0 = magic, me1 = magic, me2 = magic, me3 = magic;
                uint32_t mo0 = magic, mo1 = magic, mo2 = magic, mo3 = magic;
                if constexpr (FMT == 5) {
                  // fifth bits of positions 4G .. 4G+3: bit 2t (sub-block 2t)
                  // and 2t+1 (sub-block 2t+1) of qh bytes 4G .. 4G+3,
                  // rotated to bit 4 of each byte
                  const uint8_t *rq = qhb + (mt * 16 + g) * C::kQhRow + 4 * G;
                  const uint32_t h0 = *reinterpret_cast<const uint32_t *>(rq);
                  const uint32_t h1 = *reinterpret_cast<const uint32_t *>(rq + 8 * C::kQhRow);
                  const uint32_t e0 = __funnelshift_r(h0, h0, rot_e), e1 = __funnelshift_r(h1, h1, rot_e);
                  const uint32_t o0 = __funnelshift_r(h0, h0, rot_o), o1 = __funnelshift_r(h1, h1, rot_o);
                  me0 = lop_bit4(e0, magic);
                  me1 = lop_bit4(e1, magic);
                  me2 = lop_bit4(e0 >> 8, magic);
                  me3 = lop_bit4(e1 >> 8, magic);
                  mo0 = lop_bit4(o0, magic);
                  mo1 = lop_bit4(o1, magic);
                  mo2 = lop_bit4(o0 >> 8, magic);
                  mo3 = lop_bit4(o1 >> 8, magic);
                }
                // low nibbles: sub-block 2t, positions (4G, 4G+2) and (4G+1, 4G+3)
                const uint32_t a0 = sub_bf16x2(lop_nib(w0, me0), sub[mt][0][0]);
                const uint32_t a1 = sub_bf16x2(lop_nib(w1, me1), sub[mt][1][0]);
                const uint32_t a2 = sub_bf16x2(lop_nib(shr<8>(w0), me2), sub[mt][0][0]);
                const uint32_t a3 = sub_bf16x2(lop_nib(shr<8>(w1), me3), sub[mt][1][0]);
                // high nibbles: sub-block 2t+1
                const uint32_t c0 = sub_bf16x2(lop_nib(shr<4>(w0), mo0), sub[mt][0][1]);
                const uint32_t c1 = sub_bf16x2(lop_nib(shr<4>(w1), mo1), sub[mt][1][1]);
                const uint32_t c2 = sub_bf16x2(lop_nib(shr<12>(w0), mo2), sub[mt][0][1]);
                const uint32_t c3 = sub_bf16x2(lop_nib(shr<12>(w1), mo3), sub[mt][1][1]);
#pragma unroll
                for (int P = 0; P < NP; ++P) {
                  const uint32_t be0 = h ? be[P].z : be[P].x, be1 = h ? be[P].w : be[P].y;
                  const uint32_t bo0 = h ? bo[P].z : bo[P].x, bo1 = h ? bo[P].w : bo[P].y;
                  if (G == 0) {
                    mma_bf16_zc(accE[mt][P], a0, a1, a2, a3, be0, be1);
                    mma_bf16_zc(accO[mt][P], c0, c1, c2, c3, bo0, bo1);
                  } else {
                    mma_bf16(accE[mt][P], a0, a1, a2, a3, be0, be1);
                    mma_bf16(accO[mt][P], c0, c1, c2, c3, bo0, bo1);
                  }
                }
              }
            }
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const int P = b >> 1, i = 2 * r + (b & 1);
                float v = yacc[mt][r][b];
                v = fmaf(ds[mt][r][0], accE[mt][P][i], v);
                v = fmaf(ee[mt][r][0], xs[b][0], v);
                v = fmaf(ds[mt][r][1], accO[mt][P][i], v);
                v = fmaf(ee[mt][r][1], xs[b][1], v);
                yacc[mt][r][b] = v;
              }
          if (C::kPermBufs == 2) pbuf ^= 1;
        }
        if (++cslot == ST) {
          cslot = 0;
          phase ^= 1u;
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          yv[part & 1][mt][0][b] = yacc[mt][0][b];
          yv[part & 1][mt][1][b] = yacc[mt][1][b];
        }
    }
    // Rows: add the quad's sub-block pairs (t = 0..3).
#pragma unroll
    for (int pt = 0; pt < 2; ++pt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            float v = yv[pt][mt][r][b];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            yv[pt][mt][r][b] = v;
          }
    const int row0 = tile * TR;
    if (KP == 1) {
      if (t == 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = row0 + mt * 16 + g + 8 * r;
            if (row < o.n) {
#pragma unroll
              for (int b = 0; b < NB; ++b)
                if (b < batch)
                  o.y[(size_t)b * o.ldy + row] =
                      o.parts == 2 ? silu_mul(yv[0][mt][r][b], yv[1][mt][r][b]) : yv[0][mt][r][b];
            }
          }
      }
    } else {
      // Split K: the KP warps of the stream add their partials in warp order.
      // A warp's partials: [part][batch row][row of the tile].
      float *rb = red + ((size_t)(par * kWarps + warp) * 2 * NB) * TR;
      if (t == 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const int rr = mt * 16 + g + 8 * r;
              rb[b * TR + rr] = yv[0][mt][r][b];
              rb[(NB + b) * TR + rr] = yv[1][mt][r][b];
            }
      }
      asm volatile("bar.sync %0, %1;\n" ::"r"(1 + sic), "r"(32 * KP) : "memory");
      if (kp == 0) {
        const float *base = red + ((size_t)(par * kWarps + sic * KP) * 2 * NB) * TR;
        for (int idx = lane; idx < NB * TR; idx += 32) {
          const int b = idx / TR, rr = idx % TR;
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < KP; ++w) {
            gs += base[(w * 2 * NB + b) * TR + rr];
            us += base[(w * 2 * NB + NB + b) * TR + rr];
          }
          const int row = row0 + rr;
          if (row < o.n && b < batch)
            o.y[(size_t)b * o.ldy + row] = o.parts == 2 ? silu_mul(gs, us) : gs;
        }
      }
    }
  }
  // Every stage the warp issued was consumed (or, after a timed-out wait,
  // given the bounded time to land); nothing is left in flight.
  if constexpr (!C::kTma) cp_async_wait<0>();
}

// ---------------------------------------------------------------- host side

std::once_flag g_stream_attr[kMaxDevices];
// Resident CTAs per SM of the kernels ([variant][op table small/large]; the
// variants are NB = 1, 2, 4 for Q4_K (0, 2, 3), NB = 1 for Q5_K, q2_K, Q6_K
// and q3_K (4 .. 7) and NB = 2, 4 for Q5_K (8, 9), q2_K (10, 11), q3_K (12,
// 13) and Q6_K (14, 15); 1 is unused), queried once per device after the
// attributes are set.
int g_occ[kMaxDevices][16][2];

template <int MT, int NOPS, int NB, int FMT = 4>
constexpr auto stream_kernel() {
  return gemv_stream_kernel<MT, NOPS, NB, FMT>;
}

template <int MT, int NOPS, int NB, int FMT = 4>
int stream_setup() {
  cudaFuncSetAttribute(stream_kernel<MT, NOPS, NB, FMT>(),
                       cudaFuncAttributeMaxDynamicSharedMemorySize, StreamCfg<MT, NB, FMT>::kSmem);
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, stream_kernel<MT, NOPS, NB, FMT>(),
                                                    kWarps * 32, StreamCfg<MT, NB, FMT>::kSmem) !=
      cudaSuccess)
    return 0;
  return blocks;
}

void stream_attributes(int dev) {
  g_occ[dev][0][0] = stream_setup<1, 1, 1>();
  g_occ[dev][0][1] = stream_setup<1, kMaxOps, 1>();
  g_occ[dev][2][0] = stream_setup<1, 1, 2>();
  g_occ[dev][2][1] = stream_setup<1, kMaxOps, 2>();
  g_occ[dev][3][0] = stream_setup<1, 1, 4>();
  g_occ[dev][3][1] = stream_setup<1, kMaxOps, 4>();
  g_occ[dev][4][0] = stream_setup<1, 1, 1, 5>();
  g_occ[dev][4][1] = stream_setup<1, kMaxOps, 1, 5>();
  g_occ[dev][5][0] = stream_setup<1, 1, 1, 2>();
  g_occ[dev][5][1] = stream_setup<1, kMaxOps, 1, 2>();
  g_occ[dev][6][0] = stream_setup<1, 1, 1, 6>();
  g_occ[dev][6][1] = stream_setup<1, kMaxOps, 1, 6>();
  g_occ[dev][7][0] = stream_setup<1, 1, 1, 3>();
  g_occ[dev][7][1] = stream_setup<1, kMaxOps, 1, 3>();
  g_occ[dev][8][0] = stream_setup<1, 1, 2, 5>();
  g_occ[dev][8][1] = stream_setup<1, kMaxOps, 2, 5>();
  g_occ[dev][9][0] = stream_setup<1, 1, 4, 5>();
  g_occ[dev][9][1] = stream_setup<1, kMaxOps, 4, 5>();
  g_occ[dev][10][0] = stream_setup<1, 1, 2, 2>();
  g_occ[dev][10][1] = stream_setup<1, kMaxOps, 2, 2>();
  g_occ[dev][11][0] = stream_setup<1, 1, 4, 2>();
  g_occ[dev][11][1] = stream_setup<1, kMaxOps, 4, 2>();
  g_occ[dev][12][0] = stream_setup<1, 1, 2, 3>();
  g_occ[dev][12][1] = stream_setup<1, kMaxOps, 2, 3>();
  g_occ[dev][13][0] = stream_setup<1, 1, 4, 3>();
  g_occ[dev][13][1] = stream_setup<1, kMaxOps, 4, 3>();
  g_occ[dev][14][0] = stream_setup<1, 1, 2, 6>();
  g_occ[dev][14][1] = stream_setup<1, kMaxOps, 2, 6>();
  g_occ[dev][15][0] = stream_setup<1, 1, 4, 6>();
  g_occ[dev][15][1] = stream_setup<1, kMaxOps, 4, 6>();
}

struct StreamPlan {
  int kp = 1, grid = 0;
};

// Split: the least splitting that still gives every resident warp a tile
// (1, 2, else 4 warps per tile).  Tiles are 16 rows (the kernels are written
// for 16*MT; 32-row tiles, with fewer resident warps and twice the registers,
// measured slower on the 27B-class pass and are not instantiated).
StreamPlan plan_stream(long long tiles, int occ, const DeviceFacts *f) {
  StreamPlan best;
  for (const int kp : {1, 2, 4}) {
    if (Q4K_STREAM_FORCE_KP && kp != Q4K_STREAM_FORCE_KP) continue;
    if (occ <= 0) continue;
    const long long warps = (long long)occ * f->sm_count * kWarps;
    best.kp = kp;
    const long long ctas_needed = (tiles * kp + kWarps - 1) / kWarps;
    best.grid = (int)std::min<long long>((long long)occ * f->sm_count, ctas_needed);
    if (tiles * kp >= warps) break;
  }
  return best;
}

template <int MT, int NOPS, int NB, int FMT = 4>
cudaError_t launch_stream_chunk(const StreamOpDesc *ops, int count, int batch, int kp, int grid,
                                bool overlap, cudaStream_t stream) {
  StreamParams<NOPS> prm;
  memset(&prm, 0, sizeof prm);
  const int TR = 16 * MT;
  long long total = 0;
  int nops = 0, nmaps = 0;
  constexpr int kMapCap = (int)(sizeof prm.map / sizeof prm.map[0]);
  // Q4_K, Q5_K: the matrix as a 2-D array of 8-byte words, one row per weight row;
  // a tile is the row slot's words of TR rows
  auto weight_map = [&](const uint8_t *w, int n, int nsb) -> cudaError_t {
    if (nmaps >= kMapCap) return cudaErrorInvalidValue;
    constexpr int kBlk = StreamCfg<MT, NB, FMT>::kBlock;
    const uint64_t dims[2] = {(uint64_t)nsb * (kBlk / 8), (uint64_t)n};
    const uint64_t strides[1] = {(uint64_t)nsb * kBlk};
    const uint32_t box[2] = {(uint32_t)(StreamCfg<MT, NB, FMT>::kRowBytes / 8), (uint32_t)TR};
    const CUresult r = encode_tiled(&prm.map[nmaps++], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2,
                                    const_cast<uint8_t *>(w), dims, strides, box,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
  };
  for (int i = 0; i < count; ++i) {
    const StreamOpDesc &d = ops[i];
    if (d.n <= 0) continue;
    StreamOp &o = prm.op[nops++];
    o.w = static_cast<const uint8_t *>(d.w);
    o.w2 = static_cast<const uint8_t *>(d.w_up);
    o.x = static_cast<const __nv_bfloat16 *>(d.x);
    o.y = d.y;
    o.n = (int)d.n;
    o.nsb = (int)(d.k / kQK);
    o.ntiles = (int)((d.n + TR - 1) / TR);
    o.parts = d.w_up ? 2 : 1;
    o.ldx = (int)d.ldx;
    o.ldy = (int)d.ldy;
    o.byte0 = total;
    o.map = nmaps;
    if (StreamCfg<MT, NB, FMT>::kTma) {
      cudaError_t e = weight_map(o.w, o.n, o.nsb);
      if (e == cudaSuccess && o.w2) e = weight_map(o.w2, o.n, o.nsb);
      if (e != cudaSuccess) return e;
    }
    total += (long long)d.n * o.nsb * kBlockBytes * o.parts;
  }
  if (nops == 0) return cudaSuccess;
  prm.err = device_error_word();
  prm.nops = nops;
  prm.batch = batch;
  prm.kp = kp;
  prm.pre = overlap ? Q4K_STREAM_PRE : 0;
  prm.nstreams = grid * (kWarps / kp);
  prm.total = total;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = (size_t)StreamCfg<MT, NB, FMT>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, stream_kernel<MT, NOPS, NB, FMT>(), prm);
}

template <int NOPS>
cudaError_t launch_stream_nb(const StreamOpDesc *ops, int count, int batch, const StreamPlan &pl,
                             bool overlap, cudaStream_t stream) {
  if (batch == 1) return launch_stream_chunk<1, NOPS, 1>(ops, count, 1, pl.kp, pl.grid, overlap, stream);
  if (batch == 2)
    return launch_stream_chunk<1, NOPS, 2>(ops, count, 2, pl.kp, pl.grid, overlap, stream);
  return launch_stream_chunk<1, NOPS, 4>(ops, count, batch, pl.kp, pl.grid, overlap, stream);
}

// The other k-quant formats (16-row tiles, batch 1..4).
template <int NOPS, int FMT>
cudaError_t launch_stream_kq_nb(const StreamOpDesc *ops, int count, int batch, const StreamPlan &pl,
                                bool overlap, cudaStream_t stream) {
  return batch == 1   ? launch_stream_chunk<1, NOPS, 1, FMT>(ops, count, 1, pl.kp, pl.grid, overlap, stream)
         : batch == 2 ? launch_stream_chunk<1, NOPS, 2, FMT>(ops, count, 2, pl.kp, pl.grid, overlap, stream)
                      : launch_stream_chunk<1, NOPS, 4, FMT>(ops, count, batch, pl.kp, pl.grid, overlap, stream);
}
template <int NOPS>
cudaError_t launch_stream_kq(int fmt, const StreamOpDesc *ops, int count, int batch,
                             const StreamPlan &pl, bool overlap, cudaStream_t stream) {
  switch (fmt) {
    case 2: return launch_stream_kq_nb<NOPS, 2>(ops, count, batch, pl, overlap, stream);
    case 3: return launch_stream_kq_nb<NOPS, 3>(ops, count, batch, pl, overlap, stream);
    case 5: return launch_stream_kq_nb<NOPS, 5>(ops, count, batch, pl, overlap, stream);
    case 6: return launch_stream_kq_nb<NOPS, 6>(ops, count, batch, pl, overlap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int stream_max_batch() { return 4; }

cudaError_t launch_stream(const StreamOpDesc *ops, int64_t count, int batch, bool overlap,
                          cudaStream_t stream, int fmt) {
  if (batch < 1 || batch > stream_max_batch()) return cudaErrorInvalidValue;
  if (fmt < 2 || fmt > 6) return cudaErrorInvalidValue;
  const DeviceFacts *f = device_facts();
  std::call_once(g_stream_attr[f->device], stream_attributes, f->device);
  if (fmt != 4)
    for (int64_t i = 0; i < count; ++i)
      if (ops[i].n > 0 && ops[i].w_up) return cudaErrorInvalidValue;  // no fused gate/up
  // 16-row kernel of this format and batch
  const int nbi = batch == 1 ? 0 : batch == 2 ? 1 : 2;  // NB = 1, 2, 4
  static const int kVar[7][3] = {{0}, {0}, {5, 10, 11}, {7, 12, 13}, {0}, {4, 8, 9}, {6, 14, 15}};
  const int var1 = fmt != 4   ? kVar[fmt][nbi]
                   : batch == 1 ? 0
                   : batch == 2 ? 2
                                : 3;
  // Launches: as few as the kMaxOps weight matrices per launch allow, each
  // taking about the same number of matrices.
  long long mats = 0;
  for (int64_t i = 0; i < count; ++i)
    if (ops[i].n > 0) mats += ops[i].w_up ? 2 : 1;
  const long long nlaunch = (mats + kMaxOps - 1) / kMaxOps;
  const long long per = nlaunch > 0 ? (mats + nlaunch - 1) / nlaunch : kMaxOps;
  int64_t i = 0;
  while (i < count) {
    // a chunk: ops with rows holding at most `per` weight matrices
    int64_t j = i, used = 0, maps = 0;
    long long tiles = 0;
    while (j < count) {
      if (ops[j].n > 0) {
        const int need = ops[j].w_up ? 2 : 1;  // tensor maps of the op's matrices
        if (used > 0 && maps + need > per) break;
        maps += need;
        ++used;
        tiles += (ops[j].n + 15) / 16;
      }
      ++j;
    }
    if (used > 0) {
      const bool single = used == 1;
      const StreamPlan pl = plan_stream(tiles, g_occ[f->device][var1][single ? 0 : 1], f);
      if (pl.grid <= 0) return cudaErrorInvalidConfiguration;
      const StreamOpDesc *chunk = ops + i;
      const int n = (int)(j - i);
      const cudaError_t e =
          fmt != 4 ? (single ? launch_stream_kq<1>(fmt, chunk, n, batch, pl, overlap, stream)
                             : launch_stream_kq<kMaxOps>(fmt, chunk, n, batch, pl, overlap, stream))
          : single ? launch_stream_nb<1>(chunk, n, batch, pl, overlap, stream)
                   : launch_stream_nb<kMaxOps>(chunk, n, batch, pl, overlap, stream);
      if (e != cudaSuccess) return e;
    }
    i = j;
  }
  return cudaGetLastError();
}

}  // namespace q4k
