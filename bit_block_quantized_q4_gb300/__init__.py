"""Python binding of libq4k.so, the GB300 (sm_103a) Q4_K projection library.

The functions here carry the C entry points' names and only marshal
arguments: torch tensors in, raw device pointers, sizes and the current CUDA
stream out.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback.  If libq4k.so is missing, importing works but every call
raises.  Build it with ``python -m bit_block_quantized_q4_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libq4k.so")
Q4K_VALUES = 256
Q4K_BYTES = 144

STATUS = {0: "Q4K_OK", 1: "Q4K_ERR_NULL", 2: "Q4K_ERR_SHAPE", 3: "Q4K_ERR_ALIGN",
          4: "Q4K_ERR_WORKSPACE", 5: "Q4K_ERR_DEVICE", 6: "Q4K_ERR_CUDA", 7: "Q4K_ERR_DATA",
          8: "Q4K_ERR_MEMORY"}
Q4K_FLAG_OVERLAP_WEIGHTS = 1
Q4K_SEQ_MATRICES_PER_LAUNCH = 160
Q4K_MOE_WEIGHTED_DOWN = 1
EXPORTS = ("q4k_abi_version", "q4k_status_str", "q4k_dequant", "q4k_gemv", "q4k_gemv_ex",
           "q4k_gemv_glu", "q4k_gemv_seq", "q4k_gemm", "q4k_gemm_rmsnorm",
           "q4k_kq_block_bytes", "q4k_kq_dequant", "q4k_kq_gemv", "q4k_kq_gemv_seq",
           "q4k_moe_workspace_size", "q4k_moe_workspace_views", "q4k_moe_gemv",
           "q4k_moe_gemv_ex", "q4k_moe_gemv_noalloc", "q4k_moe_prefill",
           "q4k_moe_prefill_workspace_size",
           "q4k_get_device_error", "q4k_selftest_wait_timeout")

_lock = threading.Lock()
_lib = None


class GemvOp(ctypes.Structure):
    """One entry of q4k_gemv_seq's op array (struct q4k_gemv_op); w_up is NULL
    for a plain projection, the up matrix of a fused gate/up op otherwise."""
    _fields_ = [("w", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("y", ctypes.c_void_p),
                ("ldy", ctypes.c_int64), ("w_up", ctypes.c_void_p)]


class Q4KError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_str(status)})")


def lib() -> ctypes.CDLL:
    """The loaded libq4k.so with argument types declared (raises if not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run python -m bit_block_quantized_q4_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        L.q4k_abi_version.restype = ctypes.c_int
        L.q4k_abi_version.argtypes = []
        L.q4k_status_str.restype = ctypes.c_char_p
        L.q4k_status_str.argtypes = [ctypes.c_int]
        L.q4k_dequant.restype = ctypes.c_int
        L.q4k_dequant.argtypes = [P, I64, I64, P, ctypes.c_int, P]
        L.q4k_gemv.restype = ctypes.c_int
        L.q4k_gemv.argtypes = [P, I64, I64, P, I64, I64, P, I64, P]
        L.q4k_gemv_ex.restype = ctypes.c_int
        L.q4k_gemv_ex.argtypes = [P, I64, I64, P, I64, I64, P, I64, ctypes.c_uint32, P]
        L.q4k_gemv_glu.restype = ctypes.c_int
        L.q4k_gemv_glu.argtypes = [P, P, I64, I64, P, I64, I64, P, I64, ctypes.c_uint32, P]
        L.q4k_gemv_seq.restype = ctypes.c_int
        L.q4k_gemv_seq.argtypes = [ctypes.POINTER(GemvOp), I64, I64, ctypes.c_uint32, P]
        L.q4k_gemm.restype = ctypes.c_int
        L.q4k_gemm.argtypes = [P, I64, I64, P, I64, I64, P, I64, P]
        L.q4k_kq_block_bytes.restype = ctypes.c_int
        L.q4k_kq_block_bytes.argtypes = [I32]
        L.q4k_kq_dequant.restype = ctypes.c_int
        L.q4k_kq_dequant.argtypes = [I32, P, I64, I64, P, ctypes.c_int, P]
        L.q4k_kq_gemv.restype = ctypes.c_int
        L.q4k_kq_gemv.argtypes = [I32, P, I64, I64, P, I64, I64, P, I64, P]
        L.q4k_kq_gemv_seq.restype = ctypes.c_int
        L.q4k_kq_gemv_seq.argtypes = [I32, ctypes.POINTER(GemvOp), I64, I64, ctypes.c_uint32, P]
        L.q4k_gemm_rmsnorm.restype = ctypes.c_int
        L.q4k_gemm_rmsnorm.argtypes = [P, I64, I64, P, I64, I64, P, ctypes.c_float, P, P, I64, P]
        L.q4k_moe_workspace_size.restype = SZ
        L.q4k_moe_workspace_size.argtypes = [I32, I32, I32, I64, I64]
        L.q4k_moe_workspace_views.restype = ctypes.c_int
        L.q4k_moe_workspace_views.argtypes = [I32, I32, I32, I64, I64, ctypes.POINTER(ctypes.c_uint64)]
        L.q4k_moe_gemv.restype = ctypes.c_int
        L.q4k_moe_gemv.argtypes = [P, P, P, I64, I32, I64, I64, P, I32, I64, P, P, I32, P, I64,
                                   P, SZ, P]
        L.q4k_moe_gemv_ex.restype = ctypes.c_int
        L.q4k_moe_gemv_ex.argtypes = [P, P, P, I64, I32, I64, I64, P, I32, I64, P, P, I32, P, I64,
                                      ctypes.c_uint32, P, SZ, P]
        L.q4k_moe_prefill_workspace_size.restype = SZ
        L.q4k_moe_prefill_workspace_size.argtypes = [I32, I32, I32, I64, I64]
        L.q4k_moe_prefill.restype = ctypes.c_int
        L.q4k_moe_prefill.argtypes = [P, P, P, I64, I32, I64, I64, P, I32, I64, P, P, I32, P, I64,
                                      P, SZ, P]
        L.q4k_moe_gemv_noalloc.restype = ctypes.c_int
        L.q4k_moe_gemv_noalloc.argtypes = [P, P, P, I64, I32, I64, I64, P, I32, I64, P, P, I32, P,
                                           I64, P]
        L.q4k_get_device_error.restype = ctypes.c_int
        L.q4k_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        L.q4k_selftest_wait_timeout.restype = ctypes.c_int
        L.q4k_selftest_wait_timeout.argtypes = [P]
        _lib = L
        return L


def status_str(status: int) -> str:
    try:
        return lib().q4k_status_str(int(status)).decode()
    except RuntimeError:
        return "library not built"


def _check(status: int, what: str) -> None:
    if status != 0:
        raise Q4KError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def q4k_abi_version() -> int:
    return int(lib().q4k_abi_version())


def q4k_dequant(w: torch.Tensor, n: int, k: int, out_dtype=torch.float32, out=None, stream=None):
    """Dense N x K weights (fp32 or bf16) from an N x K Q4_K matrix on the GPU."""
    if out is None:
        out = torch.empty((n, k), dtype=out_dtype, device=w.device)
    code = {torch.float32: 0, torch.bfloat16: 1}[out.dtype]
    _check(lib().q4k_dequant(_ptr(w), n, k, _ptr(out), code, _stream(stream)), "q4k_dequant")
    return out


def q4k_gemv(w: torch.Tensor, n: int, k: int, x: torch.Tensor, out=None, stream=None):
    """Y[b] = W X[b] for X of shape [batch, K] (or [K]) bf16; returns fp32 [batch, N]."""
    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    _check(lib().q4k_gemv(_ptr(w), n, k, _ptr(x2), batch, x2.stride(0), _ptr(out), out.stride(0),
                          _stream(stream)), "q4k_gemv")
    return out[0] if x.dim() == 1 else out


def q4k_gemv_ex(w: torch.Tensor, n: int, k: int, x: torch.Tensor, flags: int, out=None,
                stream=None):
    """q4k_gemv with flags (Q4K_FLAG_OVERLAP_WEIGHTS)."""
    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    _check(lib().q4k_gemv_ex(_ptr(w), n, k, _ptr(x2), batch, x2.stride(0), _ptr(out),
                             out.stride(0), flags, _stream(stream)), "q4k_gemv_ex")
    return out[0] if x.dim() == 1 else out


def q4k_gemv_glu(w_gate: torch.Tensor, w_up: torch.Tensor, n: int, k: int, x: torch.Tensor,
                 flags: int = 0, out=None, stream=None):
    """H[b] = silu(Wg X[b]) * (Wu X[b]) for X [batch, K] (or [K]) bf16; fp32 [batch, N]."""
    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    _check(lib().q4k_gemv_glu(_ptr(w_gate), _ptr(w_up), n, k, _ptr(x2), batch, x2.stride(0),
                              _ptr(out), out.stride(0), flags, _stream(stream)), "q4k_gemv_glu")
    return out[0] if x.dim() == 1 else out


def gemv_ops(ops) -> ctypes.Array:
    """The op array of q4k_gemv_seq from (w, n, k, x, y) tuples, or
    (w_gate, n, k, x, y, w_up) for a fused gate/up op: x [batch, K] bf16 and
    y [batch, N] fp32 on the device.  The array holds raw pointers; keep the
    tensors alive while it is used.  Build it once and reuse it."""
    arr = (GemvOp * len(ops))()
    for i, op in enumerate(ops):
        w, n, k, x, y = op[:5]
        w_up = op[5] if len(op) > 5 else None
        x2 = x.unsqueeze(0) if x.dim() == 1 else x
        y2 = y.unsqueeze(0) if y.dim() == 1 else y
        arr[i] = GemvOp(_ptr(w), n, k, _ptr(x2), x2.stride(0), _ptr(y2), y2.stride(0), _ptr(w_up))
    return arr


def q4k_gemv_seq(ops, batch: int, flags: int = 0, stream=None) -> None:
    """Launch a sequence of projections in order (ops: gemv_ops(...) or a
    list of (w, n, k, x, y) tuples), as q4k_gemv_ex for each in turn."""
    arr = ops if isinstance(ops, ctypes.Array) else gemv_ops(ops)
    _check(lib().q4k_gemv_seq(arr, len(arr), batch, flags, _stream(stream)), "q4k_gemv_seq")


def q4k_gemm(w: torch.Tensor, n: int, k: int, x: torch.Tensor, out=None, stream=None):
    """Y = X W^T for X [M, K] bf16; returns bf16 [M, N]."""
    m = x.shape[0]
    if out is None:  # the C ABI wants a row stride that is a multiple of 8
        ld = (n + 7) // 8 * 8
        out = torch.empty((m, ld), dtype=torch.bfloat16, device=x.device)[:, :n]
    _check(lib().q4k_gemm(_ptr(w), n, k, _ptr(x), m, x.stride(0), _ptr(out), out.stride(0),
                          _stream(stream)), "q4k_gemm")
    return out


Q4K_FMT_Q2_K, Q4K_FMT_Q3_K, Q4K_FMT_Q4_K, Q4K_FMT_Q5_K, Q4K_FMT_Q6_K = 2, 3, 4, 5, 6


def q4k_kq_block_bytes(fmt: int) -> int:
    return int(lib().q4k_kq_block_bytes(fmt))


def q4k_kq_dequant(fmt: int, w: torch.Tensor, n: int, k: int, dtype=torch.float32, stream=None):
    """Dense weights of an n x k matrix of k-quant format fmt (fp32 or bf16)."""
    out = torch.empty((n, k), dtype=dtype, device=w.device)
    _check(lib().q4k_kq_dequant(fmt, _ptr(w), n, k, _ptr(out), 1 if dtype == torch.bfloat16 else 0,
                                _stream(stream)), "q4k_kq_dequant")
    return out


def q4k_kq_gemv(fmt: int, w: torch.Tensor, n: int, k: int, x: torch.Tensor, out=None, stream=None):
    """Y = X W^T for x [batch, k] bf16 and a k-quant matrix of format fmt; fp32 [batch, n]."""
    x2 = x if x.dim() == 2 else x.view(1, -1)
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    _check(lib().q4k_kq_gemv(fmt, _ptr(w), n, k, _ptr(x2), batch, x2.stride(0), _ptr(out),
                             out.stride(0), _stream(stream)), "q4k_kq_gemv")
    return out


def q4k_kq_gemv_seq(fmt: int, ops, batch: int, flags: int = 0, stream=None) -> None:
    """q4k_gemv_seq for k-quant matrices of format fmt (ops: gemv_ops(...) of
    (w, n, k, x, y) tuples, or such a list), as q4k_kq_gemv for each in turn."""
    arr = ops if isinstance(ops, ctypes.Array) else gemv_ops(ops)
    _check(lib().q4k_kq_gemv_seq(fmt, arr, len(arr), batch, flags, _stream(stream)),
           "q4k_kq_gemv_seq")


def q4k_gemm_rmsnorm(w: torch.Tensor, n: int, k: int, x: torch.Tensor, gamma: torch.Tensor,
                     eps: float, out=None, rinv=None, stream=None):
    """Y = rinv * (X (W diag(gamma))^T), rinv = 1/sqrt(mean(X^2) + eps) per token;
    returns (Y bf16 [M, N], rinv fp32 [M])."""
    m = x.shape[0]
    if out is None:
        ld = (n + 7) // 8 * 8
        out = torch.empty((m, ld), dtype=torch.bfloat16, device=x.device)[:, :n]
    if rinv is None:
        rinv = torch.empty(m, dtype=torch.float32, device=x.device)
    _check(lib().q4k_gemm_rmsnorm(_ptr(w), n, k, _ptr(x), m, x.stride(0), _ptr(gamma), float(eps),
                                  _ptr(rinv), _ptr(out), out.stride(0), _stream(stream)),
           "q4k_gemm_rmsnorm")
    return out, rinv


def q4k_moe_workspace_size(n_experts: int, n_tokens: int, top_k: int, hidden: int, ffn: int) -> int:
    return int(lib().q4k_moe_workspace_size(n_experts, n_tokens, top_k, hidden, ffn))


def q4k_moe_workspace_views(n_experts: int, n_tokens: int, top_k: int, hidden: int,
                            ffn: int) -> dict:
    """Byte offsets of the intermediate results q4k_moe_gemv leaves in its
    workspace: pair index per (token, slot), g, u, h and the down outputs."""
    arr = (ctypes.c_uint64 * 5)()
    _check(lib().q4k_moe_workspace_views(n_experts, n_tokens, top_k, hidden, ffn, arr),
           "q4k_moe_workspace_views")
    return dict(zip(("tj_pair", "g", "u", "h", "p"), (int(v) for v in arr)))


def q4k_moe_gemv(w_gate, w_up, w_down, expert_stride: int, n_experts: int, hidden: int, ffn: int,
                 x: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor, out=None, workspace=None,
                 stream=None):
    """Routed-expert FFN for decode tokens; returns fp32 [T, hidden]."""
    T, top_k = ids.shape
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    ws_bytes = q4k_moe_workspace_size(n_experts, T, top_k, hidden, ffn)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    _check(lib().q4k_moe_gemv(_ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride, n_experts,
                              hidden, ffn, _ptr(x), T, x.stride(0), _ptr(ids), _ptr(wts), top_k,
                              _ptr(out), out.stride(0), _ptr(workspace), workspace.numel(),
                              _stream(stream)), "q4k_moe_gemv")
    return out


def q4k_moe_gemv_ex(w_gate, w_up, w_down, expert_stride: int, n_experts: int, hidden: int,
                    ffn: int, x: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor, flags: int = 0,
                    out=None, workspace=None, stream=None):
    """q4k_moe_gemv with flags (Q4K_MOE_WEIGHTED_DOWN); returns fp32 [T, hidden]."""
    T, top_k = ids.shape
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    ws_bytes = q4k_moe_workspace_size(n_experts, T, top_k, hidden, ffn)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    _check(lib().q4k_moe_gemv_ex(_ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride, n_experts,
                                 hidden, ffn, _ptr(x), T, x.stride(0), _ptr(ids), _ptr(wts), top_k,
                                 _ptr(out), out.stride(0), flags, _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "q4k_moe_gemv_ex")
    return out


def q4k_moe_prefill_workspace_size(n_experts: int, n_tokens: int, top_k: int, hidden: int,
                                   ffn: int) -> int:
    return int(lib().q4k_moe_prefill_workspace_size(n_experts, n_tokens, top_k, hidden, ffn))


def q4k_moe_prefill(w_gate, w_up, w_down, expert_stride: int, n_experts: int, hidden: int,
                    ffn: int, x: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor, out=None,
                    workspace=None, stream=None):
    """Routed-expert FFN for a block of tokens (grouped tensor-core GEMMs);
    returns fp32 [T, hidden]."""
    T, top_k = ids.shape
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    ws_bytes = q4k_moe_prefill_workspace_size(n_experts, T, top_k, hidden, ffn)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    _check(lib().q4k_moe_prefill(_ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride, n_experts,
                                 hidden, ffn, _ptr(x), T, x.stride(0), _ptr(ids), _ptr(wts), top_k,
                                 _ptr(out), out.stride(0), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "q4k_moe_prefill")
    return out


def q4k_moe_gemv_noalloc(w_gate, w_up, w_down, expert_stride: int, n_experts: int, hidden: int,
                         ffn: int, x: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor, out=None,
                         stream=None):
    """q4k_moe_gemv with the library's own fixed device workspace (no allocation)."""
    T, top_k = ids.shape
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    _check(lib().q4k_moe_gemv_noalloc(_ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride,
                                      n_experts, hidden, ffn, _ptr(x), T, x.stride(0), _ptr(ids),
                                      _ptr(wts), top_k, _ptr(out), out.stride(0), _stream(stream)),
           "q4k_moe_gemv_noalloc")
    return out


def q4k_get_device_error(stream=None) -> int:
    """Synchronizes the stream, returns and clears the device error word."""
    bits = ctypes.c_uint32(0)
    st = lib().q4k_get_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (0, 7):
        raise Q4KError(st, "q4k_get_device_error")
    return int(bits.value)


def q4k_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self test (a wait nothing completes; ~2 s)."""
    _check(lib().q4k_selftest_wait_timeout(_stream(stream)), "q4k_selftest_wait_timeout")
