// q4k_api.cu -- the extern "C" boundary of libq4k.so (declared in
// include/q4k.h): argument checks, device checks, launch, error mapping.
//
// "spec: specialized model runtimes", section "Architecture": the runtime is
// loaded in-process behind a C ABI; section "Prototype ABI scope": every
// failure returns a clean value its caller already handles (no exceptions, no
// aborts cross this boundary); section "Correctness and control": FFI pointer,
// length and error-path behaviour is tested.
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <mutex>
#include <vector>

#include "../../include/q4k.h"
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {

__device__ unsigned int g_device_error = 0u;

namespace {

DeviceFacts g_facts[kMaxDevices];
std::once_flag g_facts_once[kMaxDevices];
unsigned *g_err_ptr[kMaxDevices];
std::once_flag g_err_once[kMaxDevices];

void resolve_error_word(int dev) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) g_err_ptr[dev] = static_cast<unsigned *>(p);
}

void query_facts(int dev) {
  DeviceFacts &f = g_facts[dev];
  f.device = dev;
  cudaDeviceGetAttribute(&f.major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&f.minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&f.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&f.max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&f.l2_bytes, cudaDevAttrL2CacheSize, dev);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encode() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device check shared by every compute entry point.
int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4K_ERR_CUDA;
  const DeviceFacts *f = device_facts();
  if (f->major != 10 || f->minor != 3) return Q4K_ERR_DEVICE;
  return Q4K_OK;
}

int map_launch(cudaError_t e) { return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA; }

// Q4K_OK when every non-null pointer is memory of the current device
// (cudaMalloc'd, not host, pinned, managed or another GPU's memory).  The
// kernels' TMA copies, and the prefill GEMM's cluster-multicast copy of X, are
// built over these addresses; they must read this GPU's own memory only.
int check_device_memory(std::initializer_list<const void *> ptrs) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
  for (const void *p : ptrs) {
    if (!p) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      (void)cudaGetLastError();  // the failed query leaves no error behind
      return Q4K_ERR_MEMORY;
    }
    if (at.type != cudaMemoryTypeDevice || at.device != dev) return Q4K_ERR_MEMORY;
  }
  return Q4K_OK;
}

static_assert(kMoeScratchBytes == Q4K_MOE_NOALLOC_SCRATCH_BYTES,
              "the allocation-free MoE array and its documented size must agree");

}  // namespace

const DeviceFacts *device_facts() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(g_facts_once[dev], query_facts, dev);
  return &g_facts[dev];
}

unsigned *device_error_word() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_err_once[dev], resolve_error_word, dev);
  return g_err_ptr[dev];
}

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, void *addr,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  std::call_once(g_encode_once, resolve_encode);
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  return g_encode(map, type, rank, addr, reinterpret_cast<const cuuint64_t *>(dims),
                  reinterpret_cast<const cuuint64_t *>(strides_bytes),
                  reinterpret_cast<const cuuint32_t *>(box), elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {
// One warp waits, through the same bounded wait every kernel uses, on an
// mbarrier that no thread ever arrives at.  After the wall-clock limit the wait
// gives up, sets the timeout bit of the device error word and the kernel ends.
__global__ void selftest_wait_timeout_kernel(unsigned *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  (void)mbar_wait(&bar, 0, err);
}
}  // namespace

}  // namespace q4k

using namespace q4k;

extern "C" {

int q4k_abi_version(void) { return Q4K_ABI_VERSION; }

const char *q4k_status_str(int status) {
  switch (status) {
    case Q4K_OK: return "ok";
    case Q4K_ERR_NULL: return "null pointer";
    case Q4K_ERR_SHAPE: return "bad shape";
    case Q4K_ERR_ALIGN: return "misaligned pointer or stride";
    case Q4K_ERR_WORKSPACE: return "workspace missing or too small";
    case Q4K_ERR_DEVICE: return "device is not sm_103";
    case Q4K_ERR_CUDA: return "CUDA error";
    case Q4K_ERR_DATA: return "a kernel reported bad data";
    case Q4K_ERR_MEMORY: return "a pointer is not device memory of the current device";
    default: return "unknown status";
  }
}

int q4k_dequant(const void *w, int64_t n, int64_t k, void *out, int out_dtype, void *stream) {
  if (n < 0 || k <= 0 || (k % kQK) != 0 || (out_dtype != 0 && out_dtype != 1)) return Q4K_ERR_SHAPE;
  if (n == 0) return Q4K_OK;
  if (!w || !out) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(out, 16)) return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, out});
  if (st != Q4K_OK) return st;
  return map_launch(launch_dequant(w, n, k, out, out_dtype, static_cast<cudaStream_t>(stream)));
}

namespace {
// Argument checks of one projection; Q4K_OK with *empty set when there is
// nothing to compute.
int check_gemv(const void *w, int64_t n, int64_t k, const void *x, int64_t batch, int64_t ldx,
               const float *y, int64_t ldy, uint32_t flags, bool *empty) {
  *empty = false;
  if (n < 0 || k <= 0 || (k % kQK) != 0 || batch < 0 || batch > 16) return Q4K_ERR_SHAPE;
  if (n > INT32_MAX / 2 || k / kQK > INT32_MAX / kBlockBytes) return Q4K_ERR_SHAPE;
  if (flags & ~(uint32_t)Q4K_FLAG_OVERLAP_WEIGHTS) return Q4K_ERR_SHAPE;
  if (n == 0 || batch == 0) {
    *empty = true;
    return Q4K_OK;
  }
  if (ldx < k || ldy < n) return Q4K_ERR_SHAPE;
  if (!w || !x || !y) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4) || (ldx % 8) != 0) return Q4K_ERR_ALIGN;
  return Q4K_OK;
}
}  // namespace

namespace {
// Batch sizes the stream kernel takes (its batch-row strides are 32-bit; at
// batch 1 they are not used).
bool stream_batch(int64_t batch, int64_t ldx, int64_t ldy) {
  return batch == 1 || (batch <= stream_max_batch() && ldx <= INT32_MAX && ldy <= INT32_MAX);
}
int64_t stream_stride(int64_t batch, int64_t ld) { return batch == 1 ? 0 : ld; }

// One projection (plain, or fused gate/up when w_up is set) after its
// arguments were checked: batch 1..4 runs in the stream kernel; 5..16 in the
// 64-row tile kernel when the op has enough tiles to occupy the GPU, else in
// the per-op batched kernel.
int run_gemv(const void *w, const void *w_up, int64_t n, int64_t k, const void *x, int64_t batch,
             int64_t ldx, float *y, int64_t ldy, uint32_t flags, void *stream) {
  const bool overlap = (flags & Q4K_FLAG_OVERLAP_WEIGHTS) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const StreamOpDesc d = {w, w_up, x, y, n, k, stream_stride(batch, ldx), stream_stride(batch, ldy)};
  if (stream_batch(batch, ldx, ldy)) return map_launch(launch_stream(&d, 1, (int)batch, overlap, s));
  if (ldx <= INT32_MAX && ldy <= INT32_MAX && wide_worth_it(&d, 1, (int)batch))
    return map_launch(launch_wide(&d, 1, (int)batch, overlap, s));
  return map_launch(launch_gemv(w, w_up, n, k, x, batch, ldx, y, ldy, overlap, s));
}
}  // namespace

int q4k_gemv_ex(const void *w, int64_t n, int64_t k, const void *x, int64_t batch, int64_t ldx,
                float *y, int64_t ldy, uint32_t flags, void *stream) {
  bool empty = false;
  int st = check_gemv(w, n, k, x, batch, ldx, y, ldy, flags, &empty);
  if (st != Q4K_OK || empty) return st;
  st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, x, y});
  if (st != Q4K_OK) return st;
  return run_gemv(w, nullptr, n, k, x, batch, ldx, y, ldy, flags, stream);
}

int q4k_gemv(const void *w, int64_t n, int64_t k, const void *x, int64_t batch, int64_t ldx,
             float *y, int64_t ldy, void *stream) {
  return q4k_gemv_ex(w, n, k, x, batch, ldx, y, ldy, 0u, stream);
}

int q4k_gemv_glu(const void *w_gate, const void *w_up, int64_t n, int64_t k, const void *x,
                 int64_t batch, int64_t ldx, float *h, int64_t ldh, uint32_t flags, void *stream) {
  bool empty = false;
  int st = check_gemv(w_gate, n, k, x, batch, ldx, h, ldh, flags, &empty);
  if (st != Q4K_OK || empty) return st;
  if (!w_up) return Q4K_ERR_NULL;
  if (!aligned(w_up, 16)) return Q4K_ERR_ALIGN;
  st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w_gate, w_up, x, h});
  if (st != Q4K_OK) return st;
  return run_gemv(w_gate, w_up, n, k, x, batch, ldx, h, ldh, flags, stream);
}

int q4k_gemv_seq(const q4k_gemv_op *ops, int64_t count, int64_t batch, uint32_t flags,
                 void *stream) {
  if (count < 0) return Q4K_ERR_SHAPE;
  if (count == 0) return Q4K_OK;
  if (!ops) return Q4K_ERR_NULL;
  bool any = false;
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    bool empty = false;
    const int st = check_gemv(o.w, o.n, o.k, o.x, batch, o.ldx, o.y, o.ldy, flags, &empty);
    if (st != Q4K_OK) return st;
    if (!empty && o.w_up && !aligned(o.w_up, 16)) return Q4K_ERR_ALIGN;
    any = any || !empty;
  }
  if (!any) return Q4K_OK;
  int st = check_device();
  if (st != Q4K_OK) return st;
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    if (o.n == 0) continue;
    st = check_device_memory({o.w, o.w_up, o.x, o.y});
    if (st != Q4K_OK) return st;
  }
  const bool overlap = (flags & Q4K_FLAG_OVERLAP_WEIGHTS) != 0;
  bool strides32 = true;
  for (int64_t i = 0; i < count; ++i)
    strides32 = strides32 && (ops[i].n == 0 || (ops[i].ldx <= INT32_MAX && ops[i].ldy <= INT32_MAX));
  if (strides32 || batch == 1) {
    std::vector<StreamOpDesc> d;
    d.reserve((size_t)count);
    for (int64_t i = 0; i < count; ++i) {
      const q4k_gemv_op &o = ops[i];
      d.push_back(StreamOpDesc{o.w, o.w_up, o.x, o.y, o.n, o.k, stream_stride(batch, o.ldx),
                               stream_stride(batch, o.ldy)});
    }
    // one persistent launch streams every op's weights back to back
    if (batch <= stream_max_batch())
      return map_launch(
          launch_stream(d.data(), count, (int)batch, overlap, static_cast<cudaStream_t>(stream)));
    if (wide_worth_it(d.data(), count, (int)batch))
      return map_launch(
          launch_wide(d.data(), count, (int)batch, overlap, static_cast<cudaStream_t>(stream)));
  }
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    if (o.n == 0) continue;
    st = map_launch(launch_gemv(o.w, o.w_up, o.n, o.k, o.x, batch, o.ldx, o.y, o.ldy, overlap,
                                static_cast<cudaStream_t>(stream)));
    if (st != Q4K_OK) return st;
  }
  return Q4K_OK;
}

int q4k_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx, void *y,
             int64_t ldy, void *stream) {
  if (n < 0 || k <= 0 || (k % kQK) != 0 || m < 0) return Q4K_ERR_SHAPE;
  if (n > INT32_MAX / 2 || m > INT32_MAX / 2 || k > INT32_MAX / 2) return Q4K_ERR_SHAPE;
  if (n == 0 || m == 0) return Q4K_OK;
  if (ldx < k || ldy < n) return Q4K_ERR_SHAPE;
  if (!w || !x || !y) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 16) || (ldx % 8) != 0 || (ldy % 8) != 0)
    return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, x, y});
  if (st != Q4K_OK) return st;
  return map_launch(launch_gemm(w, n, k, x, m, ldx, y, ldy, static_cast<cudaStream_t>(stream)));
}

int q4k_gemm_rmsnorm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                     const float *gamma, float eps, float *rinv, void *y, int64_t ldy,
                     void *stream) {
  if (n < 0 || k <= 0 || (k % kQK) != 0 || m < 0) return Q4K_ERR_SHAPE;
  if (n > INT32_MAX / 2 || m > INT32_MAX / 2 || k > INT32_MAX / 2) return Q4K_ERR_SHAPE;
  if (!(eps >= 0.f) || eps > 3.0e38f) return Q4K_ERR_SHAPE;  // negative, NaN or infinite
  if (n == 0 || m == 0) return Q4K_OK;
  if (ldx < k || ldy < n) return Q4K_ERR_SHAPE;
  if (!w || !x || !y || !gamma || !rinv) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 16) || (ldx % 8) != 0 || (ldy % 8) != 0 ||
      !aligned(gamma, 16) || !aligned(rinv, 4))
    return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, x, y, gamma, rinv});
  if (st != Q4K_OK) return st;
  return map_launch(launch_gemm_rmsnorm(w, n, k, x, m, ldx, gamma, eps, rinv, y, ldy,
                                        static_cast<cudaStream_t>(stream)));
}

int q4k_kq_block_bytes(int32_t format) {
  return format == 4 ? kBlockBytes : kq_block_bytes(format);
}

int q4k_kq_dequant(int32_t format, const void *w, int64_t n, int64_t k, void *out, int out_dtype,
                   void *stream) {
  if (format == 4) return q4k_dequant(w, n, k, out, out_dtype, stream);
  if (kq_block_bytes(format) == 0) return Q4K_ERR_SHAPE;
  if (n < 0 || k <= 0 || (k % kQK) != 0 || (out_dtype != 0 && out_dtype != 1)) return Q4K_ERR_SHAPE;
  if (n == 0) return Q4K_OK;
  if (!w || !out) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(out, 16)) return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, out});
  if (st != Q4K_OK) return st;
  return map_launch(
      launch_kq_dequant(format, w, n, k, out, out_dtype, static_cast<cudaStream_t>(stream)));
}

namespace {
// The k-quant projections the tensor-core stream kernel takes: batch 1..4
// (with 32-bit batch-row strides beyond batch 1), as for Q4_K.
bool kq_stream(int32_t format, int64_t batch, int64_t ldx, int64_t ldy) {
  (void)format;
  return stream_batch(batch, ldx, ldy);
}
// Argument checks of one k-quant projection (format != 4), before any launch.
int check_kq(int32_t format, const void *w, int64_t n, int64_t k, const void *x, int64_t batch,
             int64_t ldx, const float *y, int64_t ldy, bool *empty) {
  *empty = false;
  if (kq_block_bytes(format) == 0) return Q4K_ERR_SHAPE;
  if (n < 0 || k <= 0 || (k % kQK) != 0 || batch < 0 || batch > 16) return Q4K_ERR_SHAPE;
  if (n > INT32_MAX / 2 || kq_gemv_smem(format, k) > 227 * 1024) return Q4K_ERR_SHAPE;
  if (n == 0 || batch == 0) {
    *empty = true;
    return Q4K_OK;
  }
  if (ldx < k || ldy < n) return Q4K_ERR_SHAPE;
  if (!w || !x || !y) return Q4K_ERR_NULL;
  if (!aligned(w, 16) || !aligned(x, 16) || (ldx % 8) != 0 || !aligned(y, 4)) return Q4K_ERR_ALIGN;
  return Q4K_OK;
}
}  // namespace

int q4k_kq_gemv(int32_t format, const void *w, int64_t n, int64_t k, const void *x, int64_t batch,
                int64_t ldx, float *y, int64_t ldy, void *stream) {
  if (format == 4) return q4k_gemv(w, n, k, x, batch, ldx, y, ldy, stream);
  bool empty = false;
  int st = check_kq(format, w, n, k, x, batch, ldx, y, ldy, &empty);
  if (st != Q4K_OK || empty) return st;
  st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w, x, y});
  if (st != Q4K_OK) return st;
  if (kq_stream(format, batch, ldx, ldy)) {  // tensor cores, as Q4_K
    const StreamOpDesc d = {w, nullptr, x, y, n, k, stream_stride(batch, ldx), stream_stride(batch, ldy)};
    return map_launch(
        launch_stream(&d, 1, (int)batch, false, static_cast<cudaStream_t>(stream), format));
  }
  return map_launch(launch_kq_gemv(format, w, n, k, x, batch, ldx, y, ldy,
                                   static_cast<cudaStream_t>(stream)));
}

int q4k_kq_gemv_seq(int32_t format, const q4k_gemv_op *ops, int64_t count, int64_t batch,
                    uint32_t flags, void *stream) {
  if (format == 4) return q4k_gemv_seq(ops, count, batch, flags, stream);
  if (kq_block_bytes(format) == 0 || count < 0) return Q4K_ERR_SHAPE;
  if (flags & ~(uint32_t)Q4K_FLAG_OVERLAP_WEIGHTS) return Q4K_ERR_SHAPE;
  if (count == 0) return Q4K_OK;
  if (!ops) return Q4K_ERR_NULL;
  bool any = false;
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    bool empty = false;
    const int st = check_kq(format, o.w, o.n, o.k, o.x, batch, o.ldx, o.y, o.ldy, &empty);
    if (st != Q4K_OK) return st;
    if (o.w_up) return Q4K_ERR_SHAPE;  // no fused gate/up for these formats
    any = any || !empty;
  }
  if (!any) return Q4K_OK;
  int st = check_device();
  if (st != Q4K_OK) return st;
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    if (o.n == 0) continue;
    st = check_device_memory({o.w, o.x, o.y});
    if (st != Q4K_OK) return st;
  }
  const bool overlap = (flags & Q4K_FLAG_OVERLAP_WEIGHTS) != 0;
  bool on_stream = true;
  for (int64_t i = 0; i < count; ++i)
    on_stream = on_stream && (ops[i].n == 0 || kq_stream(format, batch, ops[i].ldx, ops[i].ldy));
  if (on_stream) {  // persistent launches of the tensor-core stream kernel
    std::vector<StreamOpDesc> d;
    d.reserve((size_t)count);
    for (int64_t i = 0; i < count; ++i) {
      const q4k_gemv_op &o = ops[i];
      d.push_back(StreamOpDesc{o.w, nullptr, o.x, o.y, o.n, o.k, stream_stride(batch, o.ldx),
                               stream_stride(batch, o.ldy)});
    }
    return map_launch(launch_stream(d.data(), count, (int)batch, overlap,
                                    static_cast<cudaStream_t>(stream), format));
  }
  for (int64_t i = 0; i < count; ++i) {
    const q4k_gemv_op &o = ops[i];
    if (o.n == 0) continue;
    st = map_launch(launch_kq_gemv(format, o.w, o.n, o.k, o.x, batch, o.ldx, o.y, o.ldy,
                                   static_cast<cudaStream_t>(stream)));
    if (st != Q4K_OK) return st;
  }
  return Q4K_OK;
}

size_t q4k_moe_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                              int64_t ffn) {
  if (n_experts <= 0 || n_tokens < 0 || top_k <= 0 || hidden <= 0 || ffn <= 0) return 0;
  return moe_workspace_size(n_experts, n_tokens, top_k, hidden, ffn);
}

int q4k_moe_workspace_views(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                            int64_t ffn, uint64_t offsets[5]) {
  if (!offsets) return Q4K_ERR_NULL;
  if (n_experts <= 0 || n_tokens <= 0 || top_k <= 0 || hidden <= 0 || ffn <= 0) return Q4K_ERR_SHAPE;
  moe_workspace_views(n_experts, n_tokens, top_k, hidden, ffn, offsets);
  return Q4K_OK;
}

int q4k_moe_gemv(const void *w_gate, const void *w_up, const void *w_down, int64_t expert_stride,
                 int32_t n_experts, int64_t hidden, int64_t ffn, const void *x, int32_t n_tokens,
                 int64_t ldx, const int32_t *ids, const float *wts, int32_t top_k, float *y,
                 int64_t ldy, void *workspace, size_t workspace_bytes, void *stream) {
  return q4k_moe_gemv_ex(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn, x, n_tokens,
                         ldx, ids, wts, top_k, y, ldy, 0u, workspace, workspace_bytes, stream);
}

int q4k_moe_gemv_ex(const void *w_gate, const void *w_up, const void *w_down,
                    int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                    const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                    const float *wts, int32_t top_k, float *y, int64_t ldy, uint32_t flags,
                    void *workspace, size_t workspace_bytes, void *stream) {
  if (flags & ~(uint32_t)Q4K_MOE_WEIGHTED_DOWN) return Q4K_ERR_SHAPE;
  if (n_experts <= 0 || n_experts > 2048 || hidden <= 0 || ffn <= 0 || (hidden % kQK) ||
      (ffn % kQK) || n_tokens < 0 || n_tokens > 64 || top_k < 1 || top_k > 16)
    return Q4K_ERR_SHAPE;
  if (hidden > (1 << 20) || ffn > (1 << 20)) return Q4K_ERR_SHAPE;
  if (expert_stride < (ffn * hidden / kQK) * kBlockBytes) return Q4K_ERR_SHAPE;
  if (n_tokens == 0) return Q4K_OK;
  if (ldx < hidden || ldy < hidden) return Q4K_ERR_SHAPE;
  if (!w_gate || !w_up || !w_down || !x || !ids || !wts || !y) return Q4K_ERR_NULL;
  if (!workspace ||
      workspace_bytes < moe_workspace_size(n_experts, n_tokens, top_k, hidden, ffn))
    return Q4K_ERR_WORKSPACE;
  if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || (expert_stride % 16) ||
      !aligned(x, 16) || (ldx % 8) || !aligned(y, 4) || !aligned(ids, 4) || !aligned(wts, 4) ||
      !aligned(workspace, 16))
    return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w_gate, w_up, w_down, x, ids, wts, y, workspace});
  if (st != Q4K_OK) return st;
  return map_launch(launch_moe(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn, x,
                               n_tokens, ldx, ids, wts, top_k, y, ldy, workspace,
                               (flags & Q4K_MOE_WEIGHTED_DOWN) != 0,
                               static_cast<cudaStream_t>(stream)));
}

size_t q4k_moe_prefill_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k,
                                      int64_t hidden, int64_t ffn) {
  if (n_experts <= 0 || n_tokens < 0 || top_k <= 0 || hidden <= 0 || ffn <= 0) return 0;
  return moe_prefill_workspace_size(n_experts, n_tokens, top_k, hidden, ffn);
}

int q4k_moe_prefill(const void *w_gate, const void *w_up, const void *w_down,
                    int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                    const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                    const float *wts, int32_t top_k, float *y, int64_t ldy, void *workspace,
                    size_t workspace_bytes, void *stream) {
  if (n_experts <= 0 || n_experts > 2048 || hidden <= 0 || ffn <= 0 || (hidden % kQK) ||
      (ffn % kQK) || n_tokens < 0 || n_tokens > 65535 || top_k < 1 || top_k > 16)
    return Q4K_ERR_SHAPE;
  if (hidden > (1 << 20) || ffn > (1 << 20)) return Q4K_ERR_SHAPE;
  if ((int64_t)n_tokens * top_k * (hidden > ffn ? hidden : ffn) > ((int64_t)1 << 31))
    return Q4K_ERR_SHAPE;
  if (expert_stride < (ffn * hidden / kQK) * kBlockBytes) return Q4K_ERR_SHAPE;
  if (n_tokens == 0) return Q4K_OK;
  if (ldx < hidden || ldy < hidden) return Q4K_ERR_SHAPE;
  if (!w_gate || !w_up || !w_down || !x || !ids || !wts || !y) return Q4K_ERR_NULL;
  if (!workspace ||
      workspace_bytes < moe_prefill_workspace_size(n_experts, n_tokens, top_k, hidden, ffn))
    return Q4K_ERR_WORKSPACE;
  if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || (expert_stride % 16) ||
      !aligned(x, 16) || (ldx % 8) || !aligned(y, 4) || !aligned(ids, 4) || !aligned(wts, 4) ||
      !aligned(workspace, 16))
    return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w_gate, w_up, w_down, x, ids, wts, y, workspace});
  if (st != Q4K_OK) return st;
  return map_launch(launch_moe_prefill(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn,
                                       x, n_tokens, ldx, ids, wts, top_k, y, ldy, workspace,
                                       static_cast<cudaStream_t>(stream)));
}

int q4k_moe_gemv_noalloc(const void *w_gate, const void *w_up, const void *w_down,
                         int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                         const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                         const float *wts, int32_t top_k, float *y, int64_t ldy, void *stream) {
  if (n_experts <= 0 || n_experts > 2048 || hidden <= 0 || ffn <= 0 || (hidden % kQK) ||
      (ffn % kQK) || n_tokens < 0 || n_tokens > 64 || top_k < 1 || top_k > 16)
    return Q4K_ERR_SHAPE;
  if (hidden > (1 << 20) || ffn > (1 << 20)) return Q4K_ERR_SHAPE;
  if (expert_stride < (ffn * hidden / kQK) * kBlockBytes) return Q4K_ERR_SHAPE;
  if (n_tokens == 0) return Q4K_OK;
  if (ldx < hidden || ldy < hidden) return Q4K_ERR_SHAPE;
  if (!w_gate || !w_up || !w_down || !x || !ids || !wts || !y) return Q4K_ERR_NULL;
  if (moe_workspace_size(n_experts, n_tokens, top_k, hidden, ffn) > kMoeScratchBytes)
    return Q4K_ERR_WORKSPACE;
  if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || (expert_stride % 16) ||
      !aligned(x, 16) || (ldx % 8) || !aligned(y, 4) || !aligned(ids, 4) || !aligned(wts, 4))
    return Q4K_ERR_ALIGN;
  int st = check_device();
  if (st != Q4K_OK) return st;
  st = check_device_memory({w_gate, w_up, w_down, x, ids, wts, y});
  if (st != Q4K_OK) return st;
  return map_launch(launch_moe_scratch(w_gate, w_up, w_down, expert_stride, n_experts, hidden, ffn,
                                       x, n_tokens, ldx, ids, wts, top_k, y, ldy,
                                       static_cast<cudaStream_t>(stream)));
}

int q4k_selftest_wait_timeout(void *stream) {
  int st = check_device();
  if (st != Q4K_OK) return st;
  selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_error_word());
  return map_launch(cudaGetLastError());
}

int q4k_get_device_error(void *stream, uint32_t *bits) {
  if (!bits) return Q4K_ERR_NULL;
  *bits = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return Q4K_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return Q4K_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return Q4K_ERR_CUDA;
  *bits = v;
  return v ? Q4K_ERR_DATA : Q4K_OK;
}

}  // extern "C"
