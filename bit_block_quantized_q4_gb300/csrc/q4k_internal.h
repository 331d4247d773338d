// q4k_internal.h -- host-side declarations shared by the library's translation
// units (launchers and the per-device facts they size their grids with).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace q4k {

// Devices the per-device tables below cover (device ordinals 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

struct DeviceFacts {
  int device = -1;
  int major = 0, minor = 0;
  int sm_count = 0;
  int max_smem_optin = 0;     // bytes of dynamic shared memory a block may opt into
  int max_smem_per_sm = 0;
  int l2_bytes = 0;
};

// Facts of the current device (queried once per device).  Kernel attributes
// (shared-memory opt-in) are per device as well: each launcher sets them once
// per device ordinal, device_facts()->device.
const DeviceFacts *device_facts();

// Device address of the current device's error word (Q4K_DEVERR_* bits).
unsigned *device_error_word();

// cuTensorMapEncodeTiled, resolved from the driver once.
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, void *addr,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swizzle,
                      CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

cudaError_t launch_dequant(const void *w, int64_t n, int64_t k, void *out, int out_dtype,
                           cudaStream_t stream);
// Batch 2..16: Y = W X, or with w_up != nullptr Y = silu(W X) * (W_up X).
cudaError_t launch_gemv(const void *w, const void *w_up, int64_t n, int64_t k, const void *x,
                        int64_t batch, int64_t ldx, float *y, int64_t ldy, bool overlap,
                        cudaStream_t stream);
// One projection of a stream launch (batch 1..4): Y[b] = W X[b], or for a
// fused gate/up op (w_up != nullptr) Y[b] = silu(W X[b]) * (W_up X[b]).
struct StreamOpDesc {
  const void *w;     // weights; the gate matrix of a fused gate/up op
  const void *w_up;  // up matrix of a fused gate/up op, nullptr otherwise
  const void *x;     // bf16 [batch][ldx]
  float *y;          // fp32 [batch][ldy]
  int64_t n, k;
  int64_t ldx, ldy;  // batch-row strides (elements, < 2^31)
};
// The ops, in order, as one persistent launch (several when count exceeds the
// kernel's op table); ops with n == 0 are skipped.  batch 1..stream_max_batch().
// fmt 4 (Q4_K, batch 1..4), or 2, 3, 5, 6 (q2_K, q3_K, Q5_K, Q6_K; batch 1:
// a decode projection of the k-quant entry points).
cudaError_t launch_stream(const StreamOpDesc *ops, int64_t count, int batch, bool overlap,
                          cudaStream_t stream, int fmt = 4);
int stream_max_batch();
// Batch 5..16 as one persistent launch of 64-row tiles (q4k_wide.cu), for
// lists of ops with enough tiles to occupy the GPU (wide_worth_it).
bool wide_worth_it(const StreamOpDesc *ops, int64_t count, int batch);
cudaError_t launch_wide(const StreamOpDesc *ops, int64_t count, int batch, bool overlap,
                        cudaStream_t stream);
cudaError_t launch_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                        void *y, int64_t ldy, cudaStream_t stream);
// Grouped expert GEMM (routed-MoE prefill): for each work slot s < meta[0],
// rows [slot_start[s], slot_start[s+1]) (at most 256) of the expert-sorted X
// (rows x k bf16, row stride ldx) times the n x k Q4_K matrix of expert
// slot_expert[s] (at byte slot_expert[s] * expert_stride of w) into the same
// rows of Y (bf16, row stride ldy).  Grid: n-tiles x max_slots.
cudaError_t launch_gemm_grouped(const void *w, int64_t expert_stride, int n_experts, int64_t n,
                                int64_t k, const void *x, int64_t rows, int64_t ldx, void *y,
                                int64_t ldy, const int *slot_expert, const int *slot_start,
                                const int *meta, int max_slots, cudaStream_t stream);

// The same with an RMSNorm prologue (gamma non-null): rinv (m floats) is
// written first, then Y = rinv (X (W diag(gamma))^T).
cudaError_t launch_gemm_rmsnorm(const void *w, int64_t n, int64_t k, const void *x, int64_t m,
                                int64_t ldx, const float *gamma, float eps, float *rinv, void *y,
                                int64_t ldy, cudaStream_t stream);
size_t moe_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                          int64_t ffn);
// Byte offsets in the MoE workspace of: the pair index of every (token, slot)
// (int32), g, u, h (fp32 [pair][ffn]) and the down outputs (fp32 [pair][hidden]).
void moe_workspace_views(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                         int64_t ffn, uint64_t out[5]);
cudaError_t launch_moe(const void *w_gate, const void *w_up, const void *w_down,
                       int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                       const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                       const float *wts, int32_t top_k, float *y, int64_t ldy, void *workspace,
                       bool weighted_down, cudaStream_t stream);

// Routed-MoE prefill: route, gather, grouped gate/up GEMMs, SiLU, grouped
// down GEMM, weighted sum (see q4k_moe.cu).
size_t moe_prefill_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k,
                                  int64_t hidden, int64_t ffn);
cudaError_t launch_moe_prefill(const void *w_gate, const void *w_up, const void *w_down,
                               int64_t expert_stride, int32_t n_experts, int64_t hidden,
                               int64_t ffn, const void *x, int32_t n_tokens, int64_t ldx,
                               const int32_t *ids, const float *wts, int32_t top_k, float *y,
                               int64_t ldy, void *workspace, cudaStream_t stream);

// Other k-quant formats (2 q2_K, 3 q3_K, 5 Q5_K, 6 Q6_K; q4k_kquant.cu).
int kq_block_bytes(int format);  // 0 for an unknown format
size_t kq_gemv_smem(int format, int64_t k);
cudaError_t launch_kq_dequant(int format, const void *w, int64_t n, int64_t k, void *out,
                              int out_dtype, cudaStream_t stream);
cudaError_t launch_kq_gemv(int format, const void *w, int64_t n, int64_t k, const void *x,
                           int64_t batch, int64_t ldx, float *y, int64_t ldy, cudaStream_t stream);

// Workspace of the allocation-free MoE call (bytes of its device array).
constexpr size_t kMoeScratchBytes = 8u << 20;

cudaError_t launch_moe_scratch(const void *w_gate, const void *w_up, const void *w_down,
                               int64_t expert_stride, int32_t n_experts, int64_t hidden,
                               int64_t ffn, const void *x, int32_t n_tokens, int64_t ldx,
                               const int32_t *ids, const float *wts, int32_t top_k, float *y,
                               int64_t ldy, cudaStream_t stream);

}  // namespace q4k
