"""CPU oracle for the Q4_K quantized-weight projection path.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``bit_block_quantized_q4_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``q4k_oracle.c`` (plain C, fp64); this module only
builds it with gcc and marshals numpy arrays through ctypes.  Every function
cites the passage it follows in ``q4k_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q4K_VALUES = 256
Q4K_BYTES = 144


def build(force: bool = False) -> str:
    """Compile q4k_oracle.c into liboracle.so (gcc, -O2, OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_fp16_to_f64.restype = ctypes.c_double
        lib.oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_unpack_scales.argtypes = [P, P, P]
        lib.oracle_quant.restype = ctypes.c_int
        lib.oracle_quant.argtypes = [P, ctypes.c_int]
        lib.oracle_dequant_block_f64.argtypes = [P, P]
        lib.oracle_dequant_f64.argtypes = [P, I64, I64, P]
        lib.oracle_dequant_f32.argtypes = [P, I64, I64, P]
        lib.oracle_dequant_bf16.argtypes = [P, I64, I64, P]
        lib.oracle_gemv_bf16.argtypes = [P, I64, I64, P, I64, I64, P, I64, P, P]
        lib.oracle_gemv_f64.argtypes = [P, I64, I64, P, I64, I64, ctypes.c_int, P]
        lib.oracle_gemv_glu.argtypes = [P, P, I64, I64, P, I64, I64, P, P, P, P, P]
        lib.oracle_moe.argtypes = [P, P, P, I64, I32, I64, I64, P, I32, I64, P, P, I32,
                                   P, P, P, P, ctypes.c_int]
        lib.oracle_rmsnorm_gemv.argtypes = [P, I64, I64, P, I64, I64, P, ctypes.c_float, P, P, P]
        lib.oracle_kq_block_bytes.restype = ctypes.c_int
        lib.oracle_kq_block_bytes.argtypes = [ctypes.c_int]
        for fn in ("oracle_kq_dequant_f64", "oracle_kq_dequant_f32", "oracle_kq_dequant_bf16"):
            getattr(lib, fn).argtypes = [ctypes.c_int, P, I64, I64, P]
        lib.oracle_kq_gemv_bf16.argtypes = [ctypes.c_int, P, I64, I64, P, I64, I64, P, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(w) -> np.ndarray:
    if isinstance(w, (bytes, bytearray, memoryview)):
        w = np.frombuffer(bytes(w), dtype=np.uint8)
    a = np.ascontiguousarray(np.asarray(w), dtype=np.uint8)
    return a.reshape(-1)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# --- scalar decoders (q4k_oracle.c: oracle_fp16_to_f64 / oracle_bf16_to_f64) ---

def fp16_to_f64(bits: int) -> float:
    return float(_load().oracle_fp16_to_f64(int(bits) & 0xFFFF))


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def f32_to_bf16(value: float) -> int:
    """fp32 -> bf16 bits, round to nearest even (oracle_f32_to_bf16_rne)."""
    return int(_load().oracle_f32_to_bf16_rne(float(np.float32(value))))


def unpack_scales(s12) -> tuple[list[int], list[int]]:
    """12 packed scale bytes -> ([sc_0..sc_7], [m_0..m_7]) (oracle_unpack_scales)."""
    s = _u8(s12)
    assert s.size == 12
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    _load().oracle_unpack_scales(_ptr(s), _ptr(sc), _ptr(m))
    return sc.tolist(), m.tolist()


def quant(qs128, i: int) -> int:
    qs = _u8(qs128)
    assert qs.size == 128
    return int(_load().oracle_quant(_ptr(qs), int(i)))


# --- matrix level ---

def _check_w(w, n: int, k: int) -> np.ndarray:
    if k % Q4K_VALUES:
        raise ValueError("k must be a multiple of 256")
    a = _u8(w)
    if a.size != n * (k // Q4K_VALUES) * Q4K_BYTES:
        raise ValueError("weight byte count does not match n x k")
    return a


def dequant_f64(w, n: int, k: int) -> np.ndarray:
    """Exact weights (fp64), [n, k] (oracle_dequant_f64)."""
    a = _check_w(w, n, k)
    out = np.empty((n, k), np.float64)
    _load().oracle_dequant_f64(_ptr(a), n, k, _ptr(out))
    return out


def dequant_f32(w, n: int, k: int) -> np.ndarray:
    """Weights rounded once to fp32, [n, k] (oracle_dequant_f32)."""
    a = _check_w(w, n, k)
    out = np.empty((n, k), np.float32)
    _load().oracle_dequant_f32(_ptr(a), n, k, _ptr(out))
    return out


def dequant_bf16(w, n: int, k: int) -> np.ndarray:
    """Weights as bf16 bits (uint16), fp32 then RNE to bf16 (oracle_dequant_bf16)."""
    a = _check_w(w, n, k)
    out = np.empty((n, k), np.uint16)
    _load().oracle_dequant_bf16(_ptr(a), n, k, _ptr(out))
    return out


def gemv(w, n: int, k: int, x_bf16, rows=None) -> tuple[np.ndarray, np.ndarray]:
    """y = W x and s = |W| |x| in fp64 for bf16 activations (oracle_gemv_bf16).

    x_bf16: uint16 array [batch, k] (or [k]).  Returns (y, s) of shape
    [batch, n] (or [batch, len(rows)] when rows is given).
    """
    a = _check_w(w, n, k)
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16)))
    assert x.shape[1] == k
    batch = x.shape[0]
    r = None
    count = n
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert r.size == 0 or (r.min() >= 0 and r.max() < n)
        count = r.size
    y = np.empty((batch, count), np.float64)
    s = np.empty((batch, count), np.float64)
    if count:
        _load().oracle_gemv_bf16(_ptr(a), n, k, _ptr(x), batch, k,
                                 _ptr(r) if r is not None else None, count, _ptr(y), _ptr(s))
    return y, s


def gemv_f64(w, n: int, k: int, x, use_abs: bool = False) -> np.ndarray:
    """y = W x (or |W| x) for fp64 activations [batch, k] (oracle_gemv_f64)."""
    a = _check_w(w, n, k)
    xv = np.ascontiguousarray(np.atleast_2d(np.asarray(x, dtype=np.float64)))
    assert xv.shape[1] == k
    y = np.empty((xv.shape[0], n), np.float64)
    _load().oracle_gemv_f64(_ptr(a), n, k, _ptr(xv), xv.shape[0], k, 1 if use_abs else 0, _ptr(y))
    return y


def gemv_glu(w_gate, w_up, n: int, k: int, x_bf16):
    """Fused gate/up (oracle_gemv_glu): returns (h, g, u, sg, su), each
    [batch, n] fp64: h = silu(g) * u, g = Wg x, u = Wu x, sg = |Wg||x|,
    su = |Wu||x|."""
    a = _check_w(w_gate, n, k)
    b = _check_w(w_up, n, k)
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16)))
    assert x.shape[1] == k
    batch = x.shape[0]
    outs = [np.empty((batch, n), np.float64) for _ in range(5)]
    if n:
        _load().oracle_gemv_glu(_ptr(a), _ptr(b), n, k, _ptr(x), batch, k, *(_ptr(o) for o in outs))
    return tuple(outs)


def rmsnorm_gemv(w, n: int, k: int, x_bf16, gamma, eps: float):
    """Projection of RMS-normalised activations (oracle_rmsnorm_gemv): returns
    (y, s, rinv) with y = W xh, s = |W| |xh| ([batch, n] fp64) and rinv
    ([batch] fp64), xh = x * rinv * gamma, rinv = 1 / sqrt(mean(x^2) + eps)."""
    a = _check_w(w, n, k)
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16)))
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float32))
    assert x.shape[1] == k and g.shape == (k,)
    batch = x.shape[0]
    y = np.empty((batch, n), np.float64)
    s = np.empty((batch, n), np.float64)
    rinv = np.empty(batch, np.float64)
    if batch and n:
        _load().oracle_rmsnorm_gemv(_ptr(a), n, k, _ptr(x), batch, k, _ptr(g), float(eps), _ptr(y),
                                    _ptr(s), _ptr(rinv))
    return y, s, rinv


# ---------------------------------------------------------------- other k-quants
# format ids: 2 q2_K, 3 q3_K, 4 Q4_K, 5 Q5_K, 6 Q6_K (oracle_kq_*)
KQ_FORMATS = {"q2_K": 2, "q3_K": 3, "Q4_K": 4, "Q5_K": 5, "Q6_K": 6}


def kq_block_bytes(fmt: int) -> int:
    return int(_load().oracle_kq_block_bytes(int(fmt)))


def _check_kq(fmt: int, w, n: int, k: int) -> np.ndarray:
    if k % 256:
        raise ValueError("k must be a multiple of 256")
    bb = kq_block_bytes(fmt)
    if bb == 0:
        raise ValueError("unknown format")
    a = _u8(w)
    if a.size != n * (k // 256) * bb:
        raise ValueError("weight byte count does not match n x k")
    return a


def kq_dequant_f64(fmt: int, w, n: int, k: int) -> np.ndarray:
    """Exact weights (fp64) [n, k] of format fmt (oracle_kq_dequant_f64)."""
    a = _check_kq(fmt, w, n, k)
    out = np.empty((n, k), np.float64)
    _load().oracle_kq_dequant_f64(int(fmt), _ptr(a), n, k, _ptr(out))
    return out


def kq_dequant_f32(fmt: int, w, n: int, k: int) -> np.ndarray:
    """Weights rounded once to fp32 (oracle_kq_dequant_f32)."""
    a = _check_kq(fmt, w, n, k)
    out = np.empty((n, k), np.float32)
    _load().oracle_kq_dequant_f32(int(fmt), _ptr(a), n, k, _ptr(out))
    return out


def kq_dequant_bf16(fmt: int, w, n: int, k: int) -> np.ndarray:
    """Weights as bf16 bits: fp32, then RNE to bf16 (oracle_kq_dequant_bf16)."""
    a = _check_kq(fmt, w, n, k)
    out = np.empty((n, k), np.uint16)
    _load().oracle_kq_dequant_bf16(int(fmt), _ptr(a), n, k, _ptr(out))
    return out


def kq_gemv(fmt: int, w, n: int, k: int, x_bf16) -> tuple[np.ndarray, np.ndarray]:
    """(y, s) = (W x, |W| |x|) in fp64 for bf16 activations [batch, k] (oracle_kq_gemv_bf16)."""
    a = _check_kq(fmt, w, n, k)
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16)))
    assert x.shape[1] == k
    batch = x.shape[0]
    y = np.empty((batch, n), np.float64)
    s = np.empty((batch, n), np.float64)
    if n and batch:
        _load().oracle_kq_gemv_bf16(int(fmt), _ptr(a), n, k, _ptr(x), batch, k, _ptr(y), _ptr(s))
    return y, s


def moe(w_gate, w_up, w_down, expert_stride: int, n_experts: int, hidden: int, ffn: int,
        x_bf16, ids, wts, return_stages: bool = False, weighted_down: bool = False):
    """Routed-expert FFN for decode tokens (oracle_moe).

    x_bf16 uint16 [T, hidden]; ids int32 [T, top_k]; wts float32 [T, top_k].
    Returns y [T, hidden] fp64, plus (g, u, h), each [T*top_k, ffn], when
    return_stages is set.  weighted_down: the route weight scales h before the
    down projection and the slots' outputs are summed unweighted.
    """
    g8, u8, d8 = _u8(w_gate), _u8(w_up), _u8(w_down)
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16)))
    ids_a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    wts_a = np.ascontiguousarray(np.asarray(wts, dtype=np.float32))
    T, top_k = ids_a.shape
    assert x.shape == (T, hidden) and wts_a.shape == (T, top_k)
    y = np.empty((T, hidden), np.float64)
    if return_stages:
        g = np.empty((T * top_k, ffn), np.float64)
        u = np.empty_like(g)
        h = np.empty_like(g)
        gp, up, hp = _ptr(g), _ptr(u), _ptr(h)
    else:
        gp = up = hp = None
    _load().oracle_moe(_ptr(g8), _ptr(u8), _ptr(d8), int(expert_stride), int(n_experts),
                       int(hidden), int(ffn), _ptr(x), int(T), int(hidden), _ptr(ids_a),
                       _ptr(wts_a), int(top_k), _ptr(y), gp, up, hp, int(bool(weighted_down)))
    if return_stages:
        return y, (g, u, h)
    return y
