/*
 * q4k.h -- C ABI of the GB300 (sm_103a) Q4_K quantized-weight projection
 * library (libq4k.so).
 *
 * What the library computes
 *   The projection step of LLM serving with block-quantized weights: a weight
 *   matrix stored as GGUF Q4_K super-blocks is dequantized and contracted with
 *   bf16 activations.
 *   - "spec: specialized model runtimes", section "Architecture": the kernel
 *     tier T0 ("GEMM, attention/GDN, quant/dequant, norms, RoPE") is the source
 *     of the expected speedup; the runtime is loaded in-process behind a C ABI;
 *     section "Non-goals": no CPU offload and no multi-GPU inside one
 *     specialization.
 *   - "spec: specialized model runtimes", section "Prototype ABI scope": a
 *     failing call returns a clean failure value that its caller handles.
 *   - "Layer Package Repository Spec", sections "Repository Identity" and
 *     "Repository Layout": the weight artifact is a Q4_K ("UD-Q4_K_XL") GGUF
 *     model split into per-layer tensors, loaded directly.
 *   - "Layer Package Repository Spec", section "Policy Resolution" (GLM MoE
 *     fixture): a routed-FFN decode layer is dominated (96%) by the routed
 *     gate/up/down expert matmuls, followed by a fused SwiGLU and the
 *     route-weighted sum.
 *
 * Q4_K super-block (256 weights in 144 bytes, little-endian; the GGUF layout)
 *    bytes   0..1   d     binary16      bytes 2..3  dmin  binary16
 *    bytes   4..15  12 bytes holding eight 6-bit scales sc_j and mins m_j:
 *                   j < 4:  sc_j = s[j] & 63,  m_j = s[j+4] & 63
 *                   j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4)
 *                           m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 *    bytes  16..143 128 bytes of 4-bit quants: byte 32c+l holds weight 64c+l
 *                   (low nibble) and weight 64c+32+l (high nibble)
 *    weight i (sub-block j = i/32):  w = d * sc_j * q - dmin * m_j
 *
 * Matrix layout: an N x K weight matrix (N outputs, K inputs, K a multiple of
 * 256) is N rows of K/256 consecutive super-blocks, rows contiguous, so row r
 * starts at byte r * (K/256) * 144.  y = W x.
 *
 * Conventions for every call
 *   - All pointers are DEVICE pointers unless stated otherwise: memory of the
 *     CURRENT device (cudaMalloc or a pool on it).  Host, pinned, managed or
 *     another GPU's memory is rejected with Q4K_ERR_MEMORY before anything is
 *     launched.  The caller owns every buffer.  Outputs must not alias inputs.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on that stream and never synchronize, except
 *     q4k_get_device_error.  They keep no per-call state and are thread-safe.
 *   - Strides (ldx, ldy) are in elements.
 *   - Argument errors are reported before anything is launched (nothing runs).
 *     An empty problem (n == 0, batch/m/tokens == 0) returns Q4K_OK and
 *     launches nothing.
 *   - Kernels never trap.  Bad data found on the device (an expert id out of
 *     range, a wait that gave up) sets a device-side error word, read and
 *     cleared with q4k_get_device_error.
 *   - Numerics: dequantized weights are the exact value rounded once to fp32
 *     (q4k_dequant is bit-exact).  Contractions accumulate in fp32; GEMV and
 *     MoE results satisfy |y - y_ref| <= 2e-3 * sum_k |w_k| |x_k| per element,
 *     the prefill GEMM (bf16 tensor-core operands) 1e-2 * sum_k |w_k||x_k|,
 *     for every finite input whose products and sums stay in fp32 range.  The
 *     decode kernels take sub-block j of a row as w = ds (q - c) + e (ds =
 *     d sc_j, c the integer in [0, 16] nearest to dmin m_j / ds, e = ds c -
 *     dmin m_j), so exactly-zero weights give exactly-zero products and a row
 *     whose weights all cancel gives exactly 0; x enters the tensor cores as
 *     bf16, unscaled.
 */
#ifndef Q4K_H
#define Q4K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4K_ABI_VERSION 2

/* Return codes of every entry point. */
enum q4k_status {
    Q4K_OK = 0,
    Q4K_ERR_NULL = 1,      /* a required pointer is NULL                              */
    Q4K_ERR_SHAPE = 2,     /* K not a positive multiple of 256, negative size, batch
                              out of range, stride smaller than the row              */
    Q4K_ERR_ALIGN = 3,     /* a pointer or stride breaks the alignment stated below   */
    Q4K_ERR_WORKSPACE = 4, /* workspace NULL or smaller than the size query says      */
    Q4K_ERR_DEVICE = 5,    /* current device is not sm_103 (GB300)                    */
    Q4K_ERR_CUDA = 6,      /* a CUDA call or kernel launch failed                      */
    Q4K_ERR_DATA = 7,      /* q4k_get_device_error: a kernel reported bad data         */
    Q4K_ERR_MEMORY = 8     /* a pointer is not device memory of the current device     */
};

/* Bits of the device error word (q4k_get_device_error). */
#define Q4K_DEVERR_TIMEOUT 1u    /* a bounded wait on an asynchronous copy gave up */
#define Q4K_DEVERR_BAD_EXPERT 2u /* an expert id outside [0, n_experts) was skipped */

int q4k_abi_version(void);
const char *q4k_status_str(int status);

/*
 * q4k_dequant -- expand an N x K Q4_K matrix to dense weights.
 * ("spec: specialized model runtimes", section "Architecture": the
 *  quant/dequant op of kernel tier T0.)
 *   w       device, N x K Q4_K (16-byte aligned)
 *   out     device, N x K row-major; out_dtype 0 = fp32 (bit-exact: the exact
 *           weight rounded once to nearest even), 1 = bf16 (that fp32 value
 *           rounded to nearest even bf16).  16-byte aligned.
 * Errors: NULL, SHAPE (k % 256, n < 0, out_dtype not 0/1), ALIGN, DEVICE, MEMORY,
 * CUDA.
 */
int q4k_dequant(const void *w, int64_t n, int64_t k, void *out, int out_dtype, void *stream);

/*
 * q4k_gemv -- decode projection, Y[b, :] = W X[b, :] for b < batch, batch 1..16.
 * ("spec: specialized model runtimes", sections "Architecture" (T0 GEMM) and
 *  "Development sequence" (decode throughput is the metric); batching of decode
 *  steps: "PRD: Performant Concurrent Distributed GGUF Runtime", DGR-012.)
 * Each super-block is read from memory once and contracted with every batch row.
 *   w       device, N x K Q4_K, 16-byte aligned
 *   x       device, batch x K bf16, row stride ldx >= K; x 16-byte aligned and
 *           ldx a multiple of 8
 *   y       device, batch x N fp32, row stride ldy >= N; 4-byte aligned
 * Errors: NULL, SHAPE, ALIGN, DEVICE, MEMORY, CUDA.
 */
int q4k_gemv(const void *w, int64_t n, int64_t k, const void *x, int64_t batch, int64_t ldx,
             float *y, int64_t ldy, void *stream);

/*
 * q4k_gemv_ex -- q4k_gemv with flags.
 *   Q4K_FLAG_OVERLAP_WEIGHTS: the kernel is launched as a programmatic
 *     dependent of the kernel launched before it on `stream` and starts
 *     streaming W while that kernel is still finishing.  X is read and Y
 *     written only after the earlier kernel has completed, so stream order
 *     holds for them; the caller guarantees that no kernel still running ahead
 *     of this call on the stream writes W (true for model weights, which are
 *     loaded once).  Consecutive decode projections overlap their start-up
 *     latency this way ("spec: specialized model runtimes", section
 *     "Development sequence": graph-captured decode).
 * Other flag bits -> Q4K_ERR_SHAPE.  Everything else as q4k_gemv.
 */
#define Q4K_FLAG_OVERLAP_WEIGHTS 1u
int q4k_gemv_ex(const void *w, int64_t n, int64_t k, const void *x, int64_t batch, int64_t ldx,
                float *y, int64_t ldy, uint32_t flags, void *stream);

/*
 * q4k_gemv_glu -- fused gate/up decode projection of a dense (or shared-expert)
 * FFN: H[b, i] = silu((Wg X[b])_i) * (Wu X[b])_i, silu(g) = g / (1 + exp(-g)),
 * for b < batch (1..16), computed in fp32 from the two fp32 projections.
 * ("Layer Package Repository Spec", sections "Policy Resolution" and
 *  "Execution Policy": merged shared gate/up.)  Both matrices are streamed in
 * one pass and only H is written.
 *   w_gate, w_up  device, each N x K Q4_K, 16-byte aligned
 *   x             as q4k_gemv
 *   h             device, batch x N fp32, row stride ldh >= N
 *   flags         as q4k_gemv_ex
 * Each of g = Wg x and u = Wu x is accurate to the GEMV bound; H is silu(g) u
 * of those values.  Errors: as q4k_gemv_ex (NULL also for w_up == NULL).
 */
int q4k_gemv_glu(const void *w_gate, const void *w_up, int64_t n, int64_t k, const void *x,
                 int64_t batch, int64_t ldx, float *h, int64_t ldh, uint32_t flags, void *stream);

/*
 * q4k_gemv_seq -- a sequence of decode projections run in order on one stream
 * by one call: the same results as calling q4k_gemv_ex (or q4k_gemv_glu for an
 * op whose w_up is set) for ops[0], ops[1], .. with the same batch, flags and
 * stream.  A decode step runs every projection of every layer ("spec:
 * specialized model runtimes", section "Development sequence": decode
 * throughput is the metric).
 *   ops     host array of `count` q4k_gemv_op, read during the call only; each
 *           op's w, n, k, x, ldx, y, ldy mean what they mean for q4k_gemv; w_up
 *           NULL for a plain projection, the up matrix of a fused gate/up op
 *           (w is then the gate matrix and y receives silu(W x) * (W_up x))
 *   count   >= 0 (0: nothing to do)
 *   batch   1..16, shared by all ops
 *   flags   as q4k_gemv_ex
 * At batch 1..4, and at 5..16 when the ops hold at least two 64-row tiles per
 * resident CTA of the GPU, the ops run as persistent launches that stream
 * their weights back to back, one launch per Q4K_SEQ_MATRICES_PER_LAUNCH
 * weight matrices (a fused gate/up op counts two; the ops are split evenly
 * over the launches), and ops may run concurrently; otherwise each op is its
 * own launch.  At every batch: no op of
 * a sequence may read what another op of the same sequence writes (split
 * dependent projections into separate calls; stream order holds between
 * calls).
 * Every op is checked before the first launch: on a NULL, SHAPE, ALIGN or
 * MEMORY error nothing is launched.  A launch failure (CUDA) stops the
 * sequence; the launches before it stay enqueued.
 * Errors: NULL (also ops == NULL with count > 0), SHAPE, ALIGN, DEVICE, MEMORY,
 * CUDA.
 */
#define Q4K_SEQ_MATRICES_PER_LAUNCH 160
typedef struct q4k_gemv_op {
  const void *w;
  int64_t n, k;
  const void *x;
  int64_t ldx;
  float *y;
  int64_t ldy;
  const void *w_up; /* NULL, or the up matrix of a fused gate/up op (ABI 2) */
} q4k_gemv_op;
int q4k_gemv_seq(const q4k_gemv_op *ops, int64_t count, int64_t batch, uint32_t flags,
                 void *stream);

/*
 * q4k_gemm -- prefill projection, Y = X W^T for m tokens (any m >= 1).
 * ("spec: specialized model runtimes", section "Feasibility gate": one
 *  quantized GEMM; prefill throughput and TTFT are reported metrics in "PRD:
 *  Performant Concurrent Distributed GGUF Runtime", DGR-001.)
 * Weight tiles are dequantized to bf16 in shared memory and multiplied on the
 * tensor cores (tcgen05) with fp32 accumulation; the output is rounded to bf16.
 *   w       device, N x K Q4_K, 16-byte aligned
 *   x       device, m x K bf16, row stride ldx >= K (ldx multiple of 8, x 16-byte
 *           aligned)
 *   y       device, m x N bf16, row stride ldy >= N (ldy multiple of 8, y 16-byte
 *           aligned)
 * Stream order holds: the kernel is launched as a programmatic dependent of the
 * kernel before it on `stream` (its set-up overlaps that kernel's tail) but
 * reads X and W and writes Y only after that kernel has completed.  Should a
 * bounded wait inside the kernel time out, the affected output tiles are left
 * unwritten and q4k_get_device_error reports it.
 * The CTAs of a cluster that share X receive it by one TMA multicast copy; the
 * tensor map of that copy covers only x, which must be memory of the current
 * device (checked: Q4K_ERR_MEMORY otherwise).  A call involves one GPU only.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, MEMORY, CUDA.
 */
int q4k_gemm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
             void *y, int64_t ldy, void *stream);

/*
 * q4k_gemm_rmsnorm -- prefill projection of RMS-normalised activations
 * ("spec: specialized model runtimes", section "Feasibility gate": one
 *  quantized GEMM plus fused RMSNorm, the norm as the GEMM's prologue):
 *     rinv[t] = 1 / sqrt( (1/K) sum_i X[t,i]^2 + eps )          (fp32, written)
 *     Y[t, j] = bf16( rinv[t] * sum_i W[j,i] gamma[i] X[t,i] )
 * The normalised activations are never formed: gamma scales each weight as it
 * is dequantized (bf16(w * gamma[i])), and rinv scales the accumulators of
 * token t.  A first kernel (one warp per token, programmatic dependent of the
 * kernel before it) writes rinv; the GEMM follows as its programmatic
 * dependent.  Accuracy: |Y - Y_ref| <= 1e-2 * sum_i |W[j,i]| |xh[t,i]| per
 * element, xh = X rinv gamma (the q4k_gemm bound on the normalised input).
 *   gamma   device, K fp32, 16-byte aligned
 *   eps     finite, >= 0
 *   rinv    device, m fp32, 4-byte aligned (written; also an output)
 *   other arguments as q4k_gemm
 * Errors: NULL, SHAPE (also a negative, NaN or infinite eps), ALIGN, DEVICE,
 *         MEMORY, CUDA.
 */
int q4k_gemm_rmsnorm(const void *w, int64_t n, int64_t k, const void *x, int64_t m, int64_t ldx,
                     const float *gamma, float eps, float *rinv, void *y, int64_t ldy,
                     void *stream);

/*
 * Other k-quant formats ("Layer Package Repository Spec", section "Policy
 * Resolution": q2_K / q3_K routed-down recipes; Q5_K / Q6_K tensors of "_XL"
 * mixes).  The pages name the formats; the layouts are the GGUF k-quant
 * super-blocks of 256 weights (all little-endian, binary16 scales):
 *   Q4K_FMT_Q2_K  84 bytes: 16 scale bytes (scale | min << 4) of 16-weight
 *                 sub-blocks, 64 bytes of 2-bit quants, d, dmin;
 *                 w = d * scale * q - dmin * min.
 *   Q4K_FMT_Q3_K 110 bytes: 32 high-bit mask bytes, 64 bytes of 2-bit quants,
 *                 12 bytes of sixteen 6-bit scales, d;
 *                 w = d * (scale - 32) * (2 bits - (mask bit ? 0 : 4)).
 *   Q4K_FMT_Q4_K 144 bytes: the Q4_K of every other call in this header.
 *   Q4K_FMT_Q5_K 176 bytes: d, dmin, the Q4_K scale bytes, 32 fifth-bit bytes,
 *                 128 nibble bytes; w = d * sc * (nibble + 16 bit) - dmin * m.
 *   Q4K_FMT_Q6_K 210 bytes: 128 low-nibble bytes, 64 bytes of 2-bit high
 *                 parts, 16 int8 scales of 16-weight sub-blocks, d;
 *                 w = d * scale * (6-bit value - 32).
 * Dequantized weights are the exact value rounded once to fp32 (bit-exact);
 * GEMV results satisfy |y - y_ref| <= 2e-3 * sum_k |w_k||x_k| (fp32 products
 * of the rounded weights with x, fp32 accumulation; q2_K, Q5_K and Q6_K at
 * batch 1: the Q4_K kernels' exact small-integer operands on the tensor
 * cores, so a row whose weights are all zero gives exactly 0).
 */
#define Q4K_FMT_Q2_K 2
#define Q4K_FMT_Q3_K 3
#define Q4K_FMT_Q4_K 4
#define Q4K_FMT_Q5_K 5
#define Q4K_FMT_Q6_K 6
/* Bytes per 256-weight super-block of a format (0: not a format). */
int q4k_kq_block_bytes(int32_t format);
/*
 * q4k_kq_dequant -- q4k_dequant for any of the formats (rows of K/256
 * super-blocks of the format; format 4 is q4k_dequant itself).
 * Errors: as q4k_dequant, and SHAPE for an unknown format.
 */
int q4k_kq_dequant(int32_t format, const void *w, int64_t n, int64_t k, void *out, int out_dtype,
                   void *stream);
/*
 * q4k_kq_gemv -- q4k_gemv for any of the formats: Y[b, :] = W X[b, :],
 * batch 1..16, arguments and layouts as q4k_gemv (format 4 is q4k_gemv
 * itself).  Each weight row is read once for all batch rows.  Batch 1..4 runs
 * on the tensor cores (exact small-integer operands, as Q4_K), batch 5..16
 * forms each weight in fp32 and contracts in fp32.  K is limited so
 * that 8 rows fit in shared memory: K/256 * block bytes <= 29040 (e.g.
 * K <= 35328 for Q6_K, 88320 for q2_K).
 * Errors: as q4k_gemv, and SHAPE for an unknown format or too long a row.
 */
int q4k_kq_gemv(int32_t format, const void *w, int64_t n, int64_t k, const void *x, int64_t batch,
                int64_t ldx, float *y, int64_t ldy, void *stream);

/*
 * q4k_kq_gemv_seq -- a sequence of q4k_kq_gemv projections of one format,
 * run in order on one stream by one call: the same results as calling
 * q4k_kq_gemv(format, ...) for ops[0], ops[1], .. with the same batch (a
 * decode step of a model whose layers are stored in that format: "Layer
 * Package Repository Spec", section "Repository Identity").
 *   format  Q4K_FMT_* (Q4K_FMT_Q4_K is q4k_gemv_seq itself)
 *   ops     host array of `count` q4k_gemv_op as for q4k_gemv_seq, each w
 *           in `format`; w_up must be NULL (no fused gate/up here)
 *   batch   1..16, shared by all ops
 *   flags   as q4k_gemv_ex
 * At batch 1..4 the ops run as persistent launches of the tensor-core kernel
 * (one per Q4K_SEQ_MATRICES_PER_LAUNCH ops, split evenly)
 * that stream their weights back to back, and ops may run concurrently: no op
 * may read what another op of the same sequence writes.  At larger batches
 * each op is its own
 * launch.  Every op is checked before the first launch.
 * Errors: as q4k_kq_gemv; SHAPE also for w_up != NULL or unknown flags; NULL
 * for ops == NULL with count > 0.
 */
int q4k_kq_gemv_seq(int32_t format, const q4k_gemv_op *ops, int64_t count, int64_t batch,
                    uint32_t flags, void *stream);

/*
 * q4k_moe_workspace_size -- bytes of device workspace q4k_moe_gemv needs.
 */
size_t q4k_moe_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                              int64_t ffn);

/*
 * q4k_moe_workspace_views -- where q4k_moe_gemv leaves its intermediate
 * results in the workspace (no counterpart on the pages; for inspection and
 * stage-by-stage checks).  After a call has completed, the workspace holds at
 * these byte offsets:
 *   offsets[0]  int32 [n_tokens * top_k]: the pair index of (token t, slot j)
 *               at t * top_k + j, or -1 for a skipped (bad) expert id
 *   offsets[1]  fp32 [pairs][ffn]: g = Wg_e x_t of each pair
 *   offsets[2]  fp32 [pairs][ffn]: u = Wu_e x_t
 *   offsets[3]  fp32 [pairs][ffn]: h = silu(g) * u
 *   offsets[4]  fp32 [pairs][hidden]: Wd_e h (before the route weight;
 *               Wd_e (wts * h) in the weighted-down order)
 * Errors: NULL, SHAPE.
 */
int q4k_moe_workspace_views(int32_t n_experts, int32_t n_tokens, int32_t top_k, int64_t hidden,
                            int64_t ffn, uint64_t offsets[5]);

/*
 * q4k_moe_gemv -- routed mixture-of-experts FFN for decode tokens.
 * ("Layer Package Repository Spec", section "Policy Resolution": routed
 *  gate/up/down expert matmuls, fused SwiGLU, route-weighted sum.)
 * For token t and slot j with expert e = ids[t*top_k + j]:
 *     h = silu(Wg_e x_t) * (Wu_e x_t)           (ffn values, fp32)
 *     Y[t, :] = sum_j wts[t*top_k + j] * (Wd_e h)   (slots summed in order j)
 * Tokens are grouped per expert so each active expert's weights are read once
 * for all of its tokens.
 *   w_gate, w_up   device; expert e's ffn x hidden Q4_K matrix starts at byte
 *                  e * expert_stride
 *   w_down         device; expert e's hidden x ffn Q4_K matrix starts at byte
 *                  e * expert_stride
 *   n_experts      1..2048
 *   expert_stride  bytes, >= (ffn * hidden / 256) * 144, multiple of 16
 *   hidden, ffn    multiples of 256
 *   x              device, n_tokens x hidden bf16, row stride ldx (mult. of 8)
 *   ids, wts       device, n_tokens x top_k int32 / fp32 (top_k 1..16, n_tokens
 *                  1..64).  An id outside [0, n_experts) contributes nothing and
 *                  sets Q4K_DEVERR_BAD_EXPERT.
 *   y              device, n_tokens x hidden fp32, row stride ldy
 *   workspace      device, >= q4k_moe_workspace_size(...) bytes, 16-byte aligned;
 *                  no initial contents needed; calls sharing one workspace
 *                  must not overlap on the GPU.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, DEVICE, MEMORY, CUDA.
 */
int q4k_moe_gemv(const void *w_gate, const void *w_up, const void *w_down, int64_t expert_stride,
                 int32_t n_experts, int64_t hidden, int64_t ffn, const void *x, int32_t n_tokens,
                 int64_t ldx, const int32_t *ids, const float *wts, int32_t top_k, float *y,
                 int64_t ldy, void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4k_moe_gemv_ex -- q4k_moe_gemv with flags (flags 0: q4k_moe_gemv).
 *   Q4K_MOE_WEIGHTED_DOWN: the weighted-down order ("Layer Package Repository
 *     Spec", section "Execution Policy", experimental.moe_weighted_down): the
 *     route weight scales h before the routed down projection and the slots'
 *     down outputs are summed unweighted,
 *         Y[t, :] = sum_j Wd_e (wts[t*top_k + j] * h)     (slots in order j).
 *     Equal to q4k_moe_gemv's result in exact arithmetic; within the same
 *     bound.  The workspace's h view keeps silu(g) * u; its down-output view
 *     holds Wd_e (wts * h).
 * Other flag bits: Q4K_ERR_SHAPE.  Everything else as q4k_moe_gemv.
 */
#define Q4K_MOE_WEIGHTED_DOWN 1u
int q4k_moe_gemv_ex(const void *w_gate, const void *w_up, const void *w_down,
                    int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                    const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                    const float *wts, int32_t top_k, float *y, int64_t ldy, uint32_t flags,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4k_moe_prefill -- routed mixture-of-experts FFN for a block of tokens
 * (prefill), the expert matmuls as grouped tensor-core GEMMs.
 * ("Layer Package Repository Spec", section "Policy Resolution": routed
 *  gate/up/down expert matmuls (the MUL_MAT_ID path), fused SwiGLU,
 *  route-weighted sum.)
 * The same result as q4k_moe_gemv for any number of tokens: the (token, slot)
 * pairs are sorted by expert into work slots of at most 256 pairs, and each
 * active expert's weights are dequantized to bf16 once per slot and multiplied
 * on the tensor cores (tcgen05, fp32 accumulation) with all of the slot's
 * token rows.  Intermediates in bf16: g = Wg_e x and u = Wu_e x (rounded once
 * from fp32), h = silu(g) * u (computed in fp32), p = Wd_e h; Y in fp32.
 * Accuracy: each GEMM stage within 1e-2 * sum |w||x| of its exact result on
 * its own inputs, propagated through SiLU and the weighted sum.
 *   arguments as q4k_moe_gemv, except n_tokens 1..65535 (with
 *   n_tokens * top_k * max(hidden, ffn) <= 2^31) and the workspace:
 *   workspace   device, >= q4k_moe_prefill_workspace_size(...) bytes, 16-byte
 *               aligned (it holds the sorted token rows and the intermediates)
 * Seven launches on `stream`, each a programmatic dependent of the one before.
 * Errors: NULL, SHAPE, ALIGN, WORKSPACE, DEVICE, MEMORY, CUDA.
 */
size_t q4k_moe_prefill_workspace_size(int32_t n_experts, int32_t n_tokens, int32_t top_k,
                                      int64_t hidden, int64_t ffn);
int q4k_moe_prefill(const void *w_gate, const void *w_up, const void *w_down,
                    int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                    const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                    const float *wts, int32_t top_k, float *y, int64_t ldy, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * q4k_moe_gemv_noalloc -- q4k_moe_gemv without a caller-provided workspace.
 * (The pages have no counterpart of this call; it is a convenience of this
 *  library.)  For callers that cannot allocate device memory per call: engines
 * that carve all device memory into their own arena at start-up, or plugin and
 * host code that does not own the allocator.  The workspace is instead a
 * device array inside the library of Q4K_MOE_NOALLOC_SCRATCH_BYTES bytes,
 * held on every GPU that loads the library until the process exits.
 *   - Arguments, results and errors as q4k_moe_gemv; a problem whose
 *     q4k_moe_workspace_size(...) exceeds the array returns Q4K_ERR_WORKSPACE
 *     before anything runs.  It allocates nothing (no cudaMalloc, no cudaFree,
 *     no allocating library routine).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     Should that look-up fail, the call returns Q4K_ERR_CUDA and the next
 *     call on the device tries again.
 *   - All calls on a device share the one array: calls that overlap on the
 *     GPU (different streams, or concurrent host threads) race on it.  Each
 *     call writes every workspace byte it reads, so no clearing is needed.
 */
#define Q4K_MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int q4k_moe_gemv_noalloc(const void *w_gate, const void *w_up, const void *w_down,
                         int64_t expert_stride, int32_t n_experts, int64_t hidden, int64_t ffn,
                         const void *x, int32_t n_tokens, int64_t ldx, const int32_t *ids,
                         const float *wts, int32_t top_k, float *y, int64_t ldy, void *stream);

/*
 * q4k_get_device_error -- synchronize `stream`, return the device error word
 * (Q4K_DEVERR_* bits) in *bits and clear it.  Returns Q4K_ERR_DATA when any bit
 * was set, Q4K_OK otherwise, Q4K_ERR_NULL if bits is NULL, Q4K_ERR_CUDA on a
 * CUDA failure.  The word is per device and shared by all calls on it.
 */
int q4k_get_device_error(void *stream, uint32_t *bits);

/* Failure-path self test (no counterpart on the pages).  Launches one warp that
 * waits, through the same bounded wait every kernel uses, on an mbarrier that
 * nothing ever arrives at.  After the wait's wall-clock limit (about 2 s) it
 * gives up, sets Q4K_DEVERR_TIMEOUT in the device error word and the kernel
 * ends normally: the GPU context stays usable.  Asynchronous on `stream`; read
 * the result with q4k_get_device_error.  Returns Q4K_ERR_DEVICE off sm_103 and
 * Q4K_ERR_CUDA if the launch fails. */
int q4k_selftest_wait_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4K_H */
