// q4k_device.cuh -- device-side building blocks shared by the sm_103a kernels:
// the Q4_K block geometry, inline-PTX wrappers (mma.sync, mbarrier, TMA), the
// bounded waits and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

constexpr int kQK = 256;          // weights per super-block
constexpr int kBlockBytes = 144;  // bytes per super-block
constexpr int kQsOffset = 16;     // first quant byte within a super-block

// Device error word (bits Q4K_DEVERR_*): one per device, defined in q4k_api.cu;
// kernels receive its address as an argument.
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrBadExpert = 2u;

__device__ __forceinline__ void set_device_error(unsigned *err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// Wall-clock bound of every wait on an asynchronous copy or MMA (2 s).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mma.sync
// D = A * B + C, m16n8k16, bf16 operands, fp32 accumulate.
// A fragment: a[0] (row g, k 2t..2t+1), a[1] (row g+8, k 2t..), a[2] (row g,
// k 2t+8..), a[3] (row g+8, k 2t+8..); B: b0 (k 2t.., col g), b1 (k 2t+8.., col
// g); C/D: c[0..1] (row g, cols 2t..2t+1), c[2..3] (row g+8); g = lane/4,
// t = lane%4, the lower k / column index in the low half of each register.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with C given separately (starts an accumulation at C).
__device__ __forceinline__ void mma_bf16_c(float (&d)[4], const float (&c)[4], uint32_t a0,
                                           uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                           uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// D = A * B + C, m16n8k16, fp16 operands, fp32 accumulate (same fragments).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A * B + C with C given separately (starts an accumulation at C).
__device__ __forceinline__ void mma_f16_c(float (&d)[4], const float4 &c, uint32_t a0, uint32_t a1,
                                          uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z),
        "f"(c.w));
}
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Same with C = 0 (starts a fresh accumulation).
__device__ __forceinline__ void mma_bf16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// ----------------------------------------------------------------- nibbles
// bf16 0x4300 is 128.0 with a unit last place, so (0x4300 | q) is exactly
// 128 + q for q < 16.  These turn the low nibbles of bytes 0 and 2 of a word
// (or the nibbles selected by a prior shift) into a bf16 pair (128+q0, 128+q2).
constexpr uint32_t kBf16Magic = 0x43004300u;
constexpr uint32_t kBf16Neg128 = 0xC300C300u;  // bf16 -128 in both halves
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return (w & 0x000F000Fu) | kBf16Magic; }
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) {
  return ((w >> 4) & 0x000F000Fu) | kBf16Magic;
}
// (w & 0x000F000F) | magic as one LOP3 (lookup 0xEA = (a & b) | c), with the
// magic held in a register so that the mask can be the immediate operand.
__device__ __forceinline__ uint32_t lop_nib(uint32_t w, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;\n" : "=r"(d) : "r"(w), "r"(magic_reg));
  return d;
}
// fp16 0x6400 is 1024.0 with a unit last place and ten mantissa bits, so
// (w & 0x000F000F) | 0x64006400 is the pair (1024+q0, 1024+q2) of the low
// nibbles of bytes 0 and 2, and (w & 0x00F000F0) | 0x64006400 the pair
// (1024+16 q0', 1024+16 q2') of their high nibbles -- no shift needed.
constexpr uint32_t kF16Magic = 0x64006400u;
__device__ __forceinline__ uint32_t lop_nib_hi16(uint32_t w, uint32_t magic_reg) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;\n" : "=r"(d) : "r"(w), "r"(magic_reg));
  return d;
}

// (128 + q) - (128 + c) for both bf16 halves: with q in [0, 15] and c in
// [0, 16] every input and the result are exact in bf16, so this is the exact
// small integer q - c.
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Reciprocal, hardware approximation (about 1 ulp; +inf for +0).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}
constexpr uint32_t kBf16One = 0x3F803F80u;  // bf16 1.0 in both halves

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// One poll of phase `parity`; the thread may sleep in the hardware until the
// phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity,
                                              uint32_t hint_ns = 1000000u) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar`.  Gives up once kWaitLimitNs of wall time
// have passed (checked every 32 polls), sets the timeout bit of the device
// error word and returns false.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, unsigned *err) {
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) break;
  }
  set_device_error(err, kDevErrTimeout);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, err);
}
// After a timed-out wait on a ring of TMA stages: give the copies still in
// flight (the `inflight` stages from slot `slot` on, whose next phase has
// parity `phase`) the same bounded time to land before the caller moves on
// and its CTA exits.
__device__ __noinline__ inline void drain_ring(uint64_t *bars, int stages, int slot,
                                               uint32_t phase, int inflight) {
  const uint64_t t0 = global_ns();
  for (int j = 0; j < inflight; ++j) {
    while (!mbar_try_wait(&bars[slot], phase, 1000u))
      if (global_ns() - t0 > kWaitLimitNs) return;
    if (++slot == stages) {
      slot = 0;
      phase ^= 1u;
    }
  }
}
// ----------------------------------------------------------------- cp.async
// 16-byte copy global -> shared by this thread (both addresses 16-byte
// aligned), L1 bypassed; the first src_bytes (0..16) bytes come from src, the
// rest of the 16 are zero-filled.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Close this thread's cp.async copies issued so far into a group; wait until
// at most N of its groups are still in flight (their data is then visible to
// the thread; other threads see it after a barrier).
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------- TMA
// Untiled bulk copy global -> shared of `bytes` bytes (both addresses 16-byte
// aligned, bytes a multiple of 16), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// The same with an L2 cache policy (createpolicy) for the source bytes.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Tiled tensor copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// L2 policy for data read exactly once (weights streamed from HBM).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}

// Prefetch a tensor map descriptor into the constant cache.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}


// ----------------------------------------------------------------- PDL
// Programmatic dependent launch: wait until the grids this one depends on have
// completed and flushed memory (a no-op when launched without the attribute),
// and let dependent grids start their own prologue early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ----------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}
// Address of the same shared-memory byte in CTA `rank` of the cluster, and
// loads from there (distributed shared memory).
__device__ __forceinline__ uint32_t peer_smem(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 16-byte store into the shared memory of a peer CTA (`addr` and `bar` mapped
// with peer_smem); its bytes complete a transaction on the peer's mbarrier
// `bar`, which is how the peer learns that they have landed.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(
          addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
      "r"(__float_as_uint(v.w)), "r"(bar)
      : "memory");
}
// Tiled 2-D copy global -> shared of every CTA in `mask` (same smem offset, same
// mbarrier offset in each destination CTA).
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *map, uint64_t *bar,
                                               int c0, int c1, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(mask)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05
// Tensor memory allocation (one warp, .sync.aligned); the base address is
// written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 out).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Same, arriving on the barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_mc(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05, K-major operand stored in the
// 128-byte swizzle layout (8 rows x 128 bytes per 1024-byte atom, atoms
// stacked along M/N).  Start address and strides in 16-byte units; bits 46-47
// hold the descriptor version (1), bits 61-63 the layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                                  // leading byte offset (unused)
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;        // stride byte offset
  d |= (uint64_t)1u << 46;                                  // version
  d |= (uint64_t)2u << 61;                                  // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// ----------------------------------------------------------------- scales
// Scales and mins of sub-blocks 2t and 2t+1 (t = 0..3) of one super-block,
// from its header words h1 = s[0..3], h2 = s[4..7], h3 = s[8..11].
// Returns sc_{2t} | sc_{2t+1} << 8 in *sc2 and the mins likewise in *m2.
__device__ __forceinline__ void scales_pair(uint32_t h1, uint32_t h2, uint32_t h3, int t,
                                            uint32_t *sc2, uint32_t *m2) {
  const uint32_t sh = (t & 1) * 16;  // byte 2(t&1) of the word
  const uint32_t p1 = h1 >> sh, p2 = h2 >> sh, p3 = h3 >> sh;
  if (t < 2) {  // sub-blocks 0..3: low six bits of s[j], s[j+4]
    *sc2 = p1 & 0x3F3Fu;
    *m2 = p2 & 0x3F3Fu;
  } else {  // sub-blocks 4..7: low/high nibble of s[j+4], top two bits of s[j-4], s[j]
    *sc2 = (p3 & 0x0F0Fu) | ((p1 >> 2) & 0x3030u);
    *m2 = ((p3 >> 4) & 0x0F0Fu) | ((p2 >> 2) & 0x3030u);
  }
}

// All eight scales/mins of a super-block: sc_j = byte j of (*sc_lo, *sc_hi)
// (bytes 0..3 in lo, 4..7 in hi), mins likewise.
__device__ __forceinline__ void scales_all(uint32_t h1, uint32_t h2, uint32_t h3, uint32_t *sc_lo,
                                           uint32_t *sc_hi, uint32_t *m_lo, uint32_t *m_hi) {
  *sc_lo = h1 & 0x3F3F3F3Fu;
  *m_lo = h2 & 0x3F3F3F3Fu;
  *sc_hi = (h3 & 0x0F0F0F0Fu) | ((h1 >> 2) & 0x30303030u);
  *m_hi = ((h3 >> 4) & 0x0F0F0F0Fu) | ((h2 >> 2) & 0x30303030u);
}

// ----------------------------------------------------------------- offset form
// Every weight of sub-block j of a super-block is w = ds (q - c) + e with
//   ds = d sc_j,  dm = dmin m_j,  c = an integer in [0, CMAX] nearest to dm / ds
//   (clamped; CMAX = 16 for 4-bit quants, 32 for Q5_K's 5-bit ones, 4 for
//   q2_K's 2-bit ones),
//   e = ds c - dm rounded once,
// so  sum_i w_i x_i = ds sum_i (q_i - c) x_i + e sum_i x_i.  The tensor cores
// take the small integers q - c (exact in bf16) against x, so a weight that is
// exactly zero (ds q = dm) contributes an exact zero product, and the rounding
// error of the whole sum stays proportional to sum |w| |x|: |ds (q - c)| <=
// 2 |w| and |e| <= |w| for every weight of the sub-block.
//
// sc_magic / m_magic hold 0x4B000000 | byte (the float 2^23 + byte), nd23 /
// ndm23 = -d 2^23 / -dmin 2^23: fma(d, 2^23 + sc, -d 2^23) is d sc exactly.
// Outputs: ds, e, and sub = (128 + c) as bf16 in both halves (the value to
// subtract from the 128 + q nibble operands).
template <int CMAX>
__device__ __forceinline__ void offset_form_c(float d, float nd23, float dmin, float ndm23,
                                              uint32_t sc_magic, uint32_t m_magic, float &ds,
                                              float &e, uint32_t &sub) {
  static_assert(CMAX == 4 || CMAX == 16 || CMAX == 32, "128 + c must stay in bf16's unit-step range");
  ds = fmaf(d, __uint_as_float(sc_magic), nd23);
  const float dm = fmaf(dmin, __uint_as_float(m_magic), ndm23);
  // u = (dm/ds + 0.5) / CMAX saturated to [0, 1] (NaN -> 0), v = 128 + CMAX u
  // in [128, 128 + CMAX]: the bf16 truncation of v is 128 + c with
  // c = floor(dm/ds + 0.5) clamped to [0, CMAX] (exact for an integer ratio:
  // the approximate reciprocal moves 128.5 + c by less than half an fp32
  // ulp).  ds = 0 makes the ratio NaN or +-inf, which the saturation maps to
  // c = 0 or CMAX.
  const float u = __saturatef(fmaf(dm, rcp_approx((float)CMAX * ds), 0.5f / (float)CMAX));
  const uint32_t vb = __float_as_uint(fmaf(u, (float)CMAX, 128.f));
  sub = __byte_perm(vb, 0u, 0x3232u);
  e = fmaf(ds, __uint_as_float(vb & 0xFFFF0000u) - 128.f, -dm);
}
// The offset forms of one sub-block in each of two rows (x: the first row,
// y: the second) with the paired operations on the packed fp32 pipe; the same
// c as offset_form_c (v_*: the fp32 128 + CMAX u, whose bf16 truncation is
// 128 + c), and ds, e as exact or as singly rounded.  d and
// dmin are the two rows' scales, nd23 = -2^23 d and pdm23 = 2^23 dmin; sc_*
// are the scale bytes as the float 2^23 + sc (byte_magic) and nm_* the min
// bytes as -(2^23 + m) (byte_magic_neg), so that the fmas below give d sc and
// -dmin m exactly.  (-dm) * rcp(-CMAX ds) is the ratio of offset_form_c with
// both signs flipped; ds = +-0 and dm = 0 map to c = 0 or CMAX as there.
template <int CMAX>
__device__ __forceinline__ void offset_form_rows2_v(float2 d, float2 nd23, float2 dmin, float2 pdm23,
                                                    uint32_t sc_x, uint32_t sc_y, uint32_t nm_x,
                                                    uint32_t nm_y, float2 &ds, float2 &e,
                                                    uint32_t &v_x, uint32_t &v_y) {
  static_assert(CMAX == 4 || CMAX == 16 || CMAX == 32, "128 + c must stay in bf16's unit-step range");
  ds = __ffma2_rn(d, make_float2(__uint_as_float(sc_x), __uint_as_float(sc_y)), nd23);
  const float2 ndm = __ffma2_rn(dmin, make_float2(__uint_as_float(nm_x), __uint_as_float(nm_y)), pdm23);
  const float2 t = __fmul2_rn(make_float2(-(float)CMAX, -(float)CMAX), ds);
  const float ux = __saturatef(fmaf(ndm.x, rcp_approx(t.x), 0.5f / (float)CMAX));
  const float uy = __saturatef(fmaf(ndm.y, rcp_approx(t.y), 0.5f / (float)CMAX));
  const float2 v = __ffma2_rn(make_float2(ux, uy), make_float2((float)CMAX, (float)CMAX),
                              make_float2(128.f, 128.f));
  v_x = __float_as_uint(v.x);
  v_y = __float_as_uint(v.y);
  const float2 c = __fadd2_rn(make_float2(__uint_as_float(v_x & 0xFFFF0000u), __uint_as_float(v_y & 0xFFFF0000u)),
                              make_float2(-128.f, -128.f));
  e = __ffma2_rn(ds, c, ndm);
}
// ... with the subtrahends as bf16 pairs (128 + c, 128 + c) of each row.
template <int CMAX>
__device__ __forceinline__ void offset_form_rows2(float2 d, float2 nd23, float2 dmin, float2 pdm23,
                                                  uint32_t sc_x, uint32_t sc_y, uint32_t nm_x,
                                                  uint32_t nm_y, float2 &ds, float2 &e,
                                                  uint32_t &sub_x, uint32_t &sub_y) {
  uint32_t v_x, v_y;
  offset_form_rows2_v<CMAX>(d, nd23, dmin, pdm23, sc_x, sc_y, nm_x, nm_y, ds, e, v_x, v_y);
  sub_x = __byte_perm(v_x, 0u, 0x3232u);
  sub_y = __byte_perm(v_y, 0u, 0x3232u);
}
// ... with the subtrahends of both rows packed in one word: (128 + c_x, 128 + c_y).
template <int CMAX>
__device__ __forceinline__ void offset_form_rows2_packed(float2 d, float2 nd23, float2 dmin,
                                                         float2 pdm23, uint32_t sc_x, uint32_t sc_y,
                                                         uint32_t nm_x, uint32_t nm_y, float2 &ds,
                                                         float2 &e, uint32_t &sub_xy) {
  uint32_t v_x, v_y;
  offset_form_rows2_v<CMAX>(d, nd23, dmin, pdm23, sc_x, sc_y, nm_x, nm_y, ds, e, v_x, v_y);
  sub_xy = __byte_perm(v_x, v_y, 0x7632u);
}
// d, dmin of two rows' super-blocks (the first words of their headers) as the
// pairs offset_form_rows2 takes, with nd23 = -2^23 d and pdm23 = 2^23 dmin.
__device__ __forceinline__ void scale_pairs(uint32_t h_x, uint32_t h_y, float2 &d, float2 &nd23,
                                            float2 &dmin, float2 &pdm23) {
  d = make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h_x & 0xFFFFu))),
                  __half2float(__ushort_as_half(static_cast<unsigned short>(h_y & 0xFFFFu))));
  dmin = make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h_x >> 16))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h_y >> 16))));
  nd23 = __fmul2_rn(d, make_float2(-8388608.f, -8388608.f));
  pdm23 = __fmul2_rn(dmin, make_float2(8388608.f, 8388608.f));
}
// Q4_K: q in [0, 15], c in [0, 16].
__device__ __forceinline__ void offset_form(float d, float nd23, float dmin, float ndm23,
                                            uint32_t sc_magic, uint32_t m_magic, float &ds,
                                            float &e, uint32_t &sub) {
  offset_form_c<16>(d, nd23, dmin, ndm23, sc_magic, m_magic, ds, e, sub);
}
// Byte i of w as the float 2^23 + byte (bit pattern 0x4B0000bb).
__device__ __forceinline__ uint32_t byte_magic(uint32_t w, int i) {
  return __byte_perm(w, 0x4B000000u, 0x7540u + (uint32_t)i);
}
// Byte i of w as the float -(2^23 + byte) (bit pattern 0xCB0000bb).
__device__ __forceinline__ uint32_t byte_magic_neg(uint32_t w, int i) {
  return __byte_perm(w, 0xCB000000u, 0x7540u + (uint32_t)i);
}

__device__ __forceinline__ float half_lo_to_float(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi_to_float(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
}

}  // namespace q4k
