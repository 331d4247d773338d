"""The C-ABI boundary: the library loads, exports what include/q4k.h declares,
and rejects bad arguments before launching anything ("spec: specialized model
runtimes", section "Correctness and control": FFI pointer, length and
error-path tests).  The CPU-only tests never reach a CUDA call: every argument
error is reported before the device is touched.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4k.h")


@pytest.fixture(scope="module")
def L():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as q4k
    return q4k.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4k_\w+)\s*\(", text)))


def test_header_declares_the_four_calls_and_helpers():
    names = _declared()
    for n in ("q4k_dequant", "q4k_gemv", "q4k_gemv_glu", "q4k_gemv_seq", "q4k_gemm",
              "q4k_moe_gemv", "q4k_moe_workspace_size", "q4k_get_device_error", "q4k_abi_version",
              "q4k_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_binding_names_match_the_c_entry_points():
    import bit_block_quantized_q4_gb300 as q4k
    for name in _declared():
        if name in ("q4k_status_str",):
            continue
        assert hasattr(q4k, name), name


def test_abi_version_and_status_strings(L):
    assert L.q4k_abi_version() == 2
    for s in range(9):
        assert L.q4k_status_str(s).decode()
    assert L.q4k_status_str(99).decode() == "unknown status"


P = 0x10000  # a non-null, 64 KiB-aligned pointer value; never dereferenced


def test_dequant_argument_errors(L):
    assert L.q4k_dequant(P, 4, 255, P, 0, None) == 2
    assert L.q4k_dequant(P, -1, 256, P, 0, None) == 2
    assert L.q4k_dequant(P, 4, 256, P, 2, None) == 2
    assert L.q4k_dequant(P, 0, 256, P, 0, None) == 0          # empty: no-op
    assert L.q4k_dequant(None, 4, 256, P, 0, None) == 1
    assert L.q4k_dequant(P, 4, 256, None, 0, None) == 1
    assert L.q4k_dequant(P + 8, 4, 256, P, 0, None) == 3
    assert L.q4k_dequant(P, 4, 256, P + 4, 0, None) == 3


def test_gemv_argument_errors(L):
    assert L.q4k_gemv(P, 4, 0, P, 1, 256, P, 4, None) == 2
    assert L.q4k_gemv(P, 4, 300, P, 1, 304, P, 4, None) == 2
    assert L.q4k_gemv(P, 4, 256, P, 17, 256, P, 4, None) == 2
    assert L.q4k_gemv(P, 4, 256, P, -1, 256, P, 4, None) == 2
    assert L.q4k_gemv(P, 4, 256, P, 1, 128, P, 4, None) == 2    # ldx < k
    assert L.q4k_gemv(P, 4, 256, P, 1, 256, P, 2, None) == 2    # ldy < n
    assert L.q4k_gemv(P, 0, 256, P, 1, 256, P, 4, None) == 0
    assert L.q4k_gemv(P, 4, 256, P, 0, 256, P, 4, None) == 0
    assert L.q4k_gemv(None, 4, 256, P, 1, 256, P, 4, None) == 1
    assert L.q4k_gemv(P, 4, 256, None, 1, 256, P, 4, None) == 1
    assert L.q4k_gemv(P, 4, 256, P, 1, 256, None, 4, None) == 1
    assert L.q4k_gemv(P + 4, 4, 256, P, 1, 256, P, 4, None) == 3
    assert L.q4k_gemv(P, 4, 256, P + 2, 1, 256, P, 4, None) == 3
    assert L.q4k_gemv(P, 4, 256, P, 2, 260, P, 4, None) == 3     # ldx not a multiple of 8
    assert L.q4k_gemv(P, 4, 256, P, 1, 256, P + 2, 4, None) == 3


def test_gemv_glu_argument_errors(L):
    assert L.q4k_gemv_glu(P, P, 4, 300, P, 1, 304, P, 4, 0, None) == 2
    assert L.q4k_gemv_glu(P, P, 4, 256, P, 17, 256, P, 4, 0, None) == 2
    assert L.q4k_gemv_glu(P, P, 4, 256, P, 1, 256, P, 4, 2, None) == 2   # unknown flag bit
    assert L.q4k_gemv_glu(P, P, 0, 256, P, 1, 256, P, 4, 0, None) == 0   # empty: no-op
    assert L.q4k_gemv_glu(None, P, 4, 256, P, 1, 256, P, 4, 0, None) == 1
    assert L.q4k_gemv_glu(P, None, 4, 256, P, 1, 256, P, 4, 0, None) == 1
    assert L.q4k_gemv_glu(P, P + 8, 4, 256, P, 1, 256, P, 4, 0, None) == 3
    assert L.q4k_gemv_glu(P, P, 4, 256, P + 2, 1, 256, P, 4, 0, None) == 3


def test_gemv_op_struct_layout_matches_the_header():
    # q4k_gemv_op: w, n, k, x, ldx, y, ldy, w_up -- eight 8-byte fields
    from bit_block_quantized_q4_gb300 import GemvOp
    assert ctypes.sizeof(GemvOp) == 64
    assert [f[0] for f in GemvOp._fields_] == ["w", "n", "k", "x", "ldx", "y", "ldy", "w_up"]
    assert GemvOp.w_up.offset == 56


def test_binding_constants_match_the_header():
    import bit_block_quantized_q4_gb300 as q4k
    text = open(HEADER).read()
    for name in ("Q4K_ABI_VERSION", "Q4K_FLAG_OVERLAP_WEIGHTS", "Q4K_MOE_WEIGHTED_DOWN",
                 "Q4K_SEQ_MATRICES_PER_LAUNCH"):
        m = re.search(r"#define %s (\d+)u?\b" % name, text)
        assert m, name
        if hasattr(q4k, name):
            assert getattr(q4k, name) == int(m.group(1)), name


def test_gemv_seq_checks_every_op_before_launching(L):
    from bit_block_quantized_q4_gb300 import GemvOp
    good = GemvOp(P, 4, 256, P, 256, P, 4)
    ops = (GemvOp * 3)(good, good, good)
    assert L.q4k_gemv_seq(ops, 0, 1, 0, None) == 0          # nothing to do
    assert L.q4k_gemv_seq(None, 3, 1, 0, None) == 1
    assert L.q4k_gemv_seq(ops, -1, 1, 0, None) == 2
    assert L.q4k_gemv_seq(ops, 3, 17, 0, None) == 2         # batch shared by all ops
    assert L.q4k_gemv_seq(ops, 3, 1, 2, None) == 2          # unknown flag bit
    # an error in the last op is found before anything is launched (a launch
    # on this GPU-less machine would report the device instead)
    for bad, status in ((GemvOp(None, 4, 256, P, 256, P, 4), 1),
                        (GemvOp(P, 4, 300, P, 304, P, 4), 2),
                        (GemvOp(P, 4, 256, P, 128, P, 4), 2),
                        (GemvOp(P + 4, 4, 256, P, 256, P, 4), 3),
                        (GemvOp(P, 4, 256, P, 256, P + 2, 4), 3),
                        (GemvOp(P, 4, 256, P, 256, P, 4, P + 8), 3)):   # misaligned w_up
        ops[2] = bad
        assert L.q4k_gemv_seq(ops, 3, 1, 0, None) == status
    # empty ops only: nothing to launch
    ops[0] = ops[1] = ops[2] = GemvOp(P, 0, 256, P, 256, P, 4)
    assert L.q4k_gemv_seq(ops, 3, 1, 0, None) == 0


def test_gemm_argument_errors(L):
    assert L.q4k_gemm(P, 4, 100, P, 8, 104, P, 8, None) == 2
    assert L.q4k_gemm(P, 8, 256, P, -2, 256, P, 8, None) == 2
    assert L.q4k_gemm(P, 8, 256, P, 0, 256, P, 8, None) == 0
    assert L.q4k_gemm(P, 8, 256, P, 4, 256, P, 4, None) == 2     # ldy < n
    assert L.q4k_gemm(None, 8, 256, P, 4, 256, P, 8, None) == 1
    assert L.q4k_gemm(P, 8, 256, P, 4, 256, P + 8, 8, None) == 3
    assert L.q4k_gemm(P, 8, 256, P, 4, 260, P, 8, None) == 3


def test_moe_argument_errors(L):
    E, H, F = 8, 256, 512
    stride = F * H // 256 * 144
    ws = L.q4k_moe_workspace_size(E, 4, 2, H, F)
    assert ws > 0
    args = [P, P, P, stride, E, H, F, P, 4, H, P, P, 2, P, H, P, ws, None]

    def call(**kw):
        a = list(args)
        names = ["wg", "wu", "wd", "stride", "E", "H", "F", "x", "T", "ldx", "ids", "wts", "k",
                 "y", "ldy", "ws", "wsb", "stream"]
        for key, v in kw.items():
            a[names.index(key)] = v
        return L.q4k_moe_gemv(*a)

    assert call(H=300) == 2
    assert call(k=0) == 2
    assert call(k=17) == 2
    assert call(T=65) == 2
    assert call(stride=stride - 16) == 2
    assert call(T=0) == 0
    assert call(ids=None) == 1
    assert call(ws=None) == 4
    assert call(wsb=ws - 1) == 4
    assert call(stride=stride + 8) == 3
    assert call(x=P + 2) == 3


def test_moe_ex_flags(L):
    # flags sit between ldy and the workspace; bits other than
    # Q4K_MOE_WEIGHTED_DOWN are a SHAPE error before anything else is looked at
    E, H, F = 8, 256, 512
    stride = F * H // 256 * 144
    ws = L.q4k_moe_workspace_size(E, 4, 2, H, F)

    def call(flags, **kw):
        a = dict(wg=P, wu=P, wd=P, stride=stride, E=E, H=H, F=F, x=P, T=4, ldx=H, ids=P, wts=P,
                 k=2, y=P, ldy=H, flags=flags, ws=P, wsb=ws, stream=None)
        a.update(kw)
        return L.q4k_moe_gemv_ex(*a.values())

    assert call(2) == 2
    assert call(0x80000000) == 2
    assert call(2, ids=None) == 2
    assert call(1, ids=None) == 1
    assert call(0, ids=None) == 1
    assert call(1, T=0) == 0
    assert call(1, ws=None) == 4
    assert call(1, H=300) == 2


def test_gemm_rmsnorm_argument_errors(L):
    m, n, k = 8, 128, 256

    def call(**kw):
        a = dict(w=P, n=n, k=k, x=P, m=m, ldx=k, gamma=P, eps=1e-6, rinv=P, y=P, ldy=n, stream=None)
        a.update(kw)
        return L.q4k_gemm_rmsnorm(*a.values())

    assert call(eps=-1.0) == 2
    assert call(eps=float("nan")) == 2
    assert call(eps=float("inf")) == 2
    assert call(k=300) == 2
    assert call(m=0) == 0
    assert call(gamma=None) == 1
    assert call(rinv=None) == 1
    assert call(gamma=P + 4) == 3
    assert call(rinv=P + 2) == 3
    assert call(x=P + 8) == 3


def test_moe_prefill_argument_errors(L):
    E, H, F, T, K = 8, 256, 512, 40, 2
    stride = F * H // 256 * 144
    ws = L.q4k_moe_prefill_workspace_size(E, T, K, H, F)
    P_ = T * K   # sorted token rows and down outputs (P x H bf16), g, u, h (P x F bf16)
    assert ws >= 2 * P_ * H * 2 + 3 * P_ * F * 2

    def call(**kw):
        a = dict(wg=P, wu=P, wd=P, stride=stride, E=E, H=H, F=F, x=P, T=T, ldx=H, ids=P, wts=P,
                 k=K, y=P, ldy=H, ws=P, wsb=ws, stream=None)
        a.update(kw)
        return L.q4k_moe_prefill(*a.values())

    assert call(H=300) == 2
    assert call(T=70000) == 2
    assert call(k=17) == 2
    assert call(E=0) == 2
    assert call(T=0) == 0
    assert call(ids=None) == 1
    assert call(ws=None) == 4
    assert call(wsb=ws - 1) == 4
    assert call(stride=stride + 8) == 3
    assert call(x=P + 2) == 3


def test_kq_argument_errors(L):
    assert [L.q4k_kq_block_bytes(f) for f in (2, 3, 4, 5, 6)] == [84, 110, 144, 176, 210]
    assert L.q4k_kq_block_bytes(1) == 0 and L.q4k_kq_block_bytes(7) == 0
    assert L.q4k_kq_dequant(1, P, 4, 256, P, 0, None) == 2
    assert L.q4k_kq_dequant(2, P, 4, 300, P, 0, None) == 2
    assert L.q4k_kq_dequant(2, P, 4, 256, P, 2, None) == 2
    assert L.q4k_kq_dequant(3, None, 4, 256, P, 0, None) == 1
    assert L.q4k_kq_dequant(5, P + 2, 4, 256, P, 0, None) == 3
    assert L.q4k_kq_dequant(6, P, 0, 256, P, 0, None) == 0

    def gemv(fmt=2, n=8, k=512, x=P, batch=1, ldx=512, y=P, ldy=8, w=P):
        return L.q4k_kq_gemv(fmt, w, n, k, x, batch, ldx, y, ldy, None)

    assert gemv(fmt=7) == 2
    assert gemv(batch=17) == 2
    assert gemv(k=300) == 2
    assert gemv(fmt=6, k=35328, ldx=35328, n=0) == 0       # the longest Q6_K row is accepted
    assert gemv(fmt=6, k=35328 + 256, ldx=35584) == 2     # 8 rows no longer fit in shared memory
    assert gemv(batch=0) == 0
    assert gemv(x=None) == 1
    assert gemv(ldx=500) == 2
    assert gemv(x=P + 8) == 3
    assert gemv(ldx=516) == 3


def test_kq_gemv_seq_checks_every_op_before_launching(L):
    from bit_block_quantized_q4_gb300 import GemvOp
    good = GemvOp(P, 4, 512, P, 512, P, 4)
    ops = (GemvOp * 3)(good, good, good)
    assert L.q4k_kq_gemv_seq(2, ops, 0, 1, 0, None) == 0       # nothing to do
    assert L.q4k_kq_gemv_seq(7, ops, 3, 1, 0, None) == 2       # unknown format
    assert L.q4k_kq_gemv_seq(3, None, 3, 1, 0, None) == 1
    assert L.q4k_kq_gemv_seq(5, ops, -1, 1, 0, None) == 2
    assert L.q4k_kq_gemv_seq(6, ops, 3, 17, 0, None) == 2      # batch shared by all ops
    assert L.q4k_kq_gemv_seq(2, ops, 3, 1, 2, None) == 2       # unknown flag bit
    # an error in the last op is found before anything is launched (a launch
    # on this GPU-less machine would report the device instead)
    for bad, status in ((GemvOp(None, 4, 512, P, 512, P, 4), 1),
                        (GemvOp(P, 4, 300, P, 304, P, 4), 2),
                        (GemvOp(P, 4, 512, P, 256, P, 4), 2),
                        (GemvOp(P + 4, 4, 512, P, 512, P, 4), 3),
                        (GemvOp(P, 4, 512, P + 8, 512, P, 4), 3),
                        (GemvOp(P, 4, 512, P, 512, P, 4, P), 2)):   # no fused gate/up
        ops[2] = bad
        for fmt in (2, 3, 5, 6):
            assert L.q4k_kq_gemv_seq(fmt, ops, 3, 1, 0, None) == status, (fmt, status)
    ops[2] = GemvOp(P, 0, 512, None, 512, None, 4)              # an empty op is skipped
    assert L.q4k_kq_gemv_seq(2, ops, 3, 1, 0, None) != 2


def test_get_device_error_rejects_null(L):
    assert L.q4k_get_device_error(None, None) == 1


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import bit_block_quantized_q4_gb300 as q4k
    monkeypatch.setattr(q4k, "_lib", None)
    monkeypatch.setattr(q4k, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        q4k.lib()


def test_header_compiles_as_c99_and_a_c_program_links(L, tmp_path):
    # The boundary is a plain C ABI: a C99 program that calls every entry point
    # compiles warning-free against include/q4k.h and links against libq4k.so
    # (it is only built here, not run: running needs a GPU).
    import shutil
    import subprocess
    import bit_block_quantized_q4_gb300 as q4k
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_q4k.c"
    src.write_text(r'''
#include "q4k.h"
#include <stdio.h>
int main(void) {
  q4k_gemv_op ops[1] = {{0, 4, 256, 0, 256, 0, 4, 0}};
  uint32_t bits = 0;
  int st = q4k_abi_version() == Q4K_ABI_VERSION ? Q4K_OK : -1;
  st |= q4k_dequant(0, 4, 256, 0, 0, 0);
  st |= q4k_gemv(0, 4, 256, 0, 1, 256, 0, 4, 0);
  st |= q4k_gemv_ex(0, 4, 256, 0, 1, 256, 0, 4, Q4K_FLAG_OVERLAP_WEIGHTS, 0);
  st |= q4k_gemv_glu(0, 0, 4, 256, 0, 1, 256, 0, 4, 0u, 0);
  st |= q4k_gemv_seq(ops, 1, 1, 0u, 0);
  st |= q4k_gemm(0, 4, 256, 0, 1, 256, 0, 8, 0);
  st |= q4k_kq_block_bytes(Q4K_FMT_Q2_K) == 84 ? 0 : 1 << 21;
  st |= q4k_kq_dequant(Q4K_FMT_Q3_K, 0, 4, 256, 0, 0, 0);
  st |= q4k_kq_gemv(Q4K_FMT_Q6_K, 0, 4, 256, 0, 1, 256, 0, 4, 0);
  st |= q4k_gemm_rmsnorm(0, 4, 256, 0, 1, 256, 0, 1e-6f, 0, 0, 8, 0);
  st |= (int)q4k_moe_workspace_size(8, 1, 2, 256, 256);
  st |= q4k_moe_gemv(0, 0, 0, 0, 8, 256, 256, 0, 1, 256, 0, 0, 2, 0, 256, 0, 0, 0);
  st |= q4k_moe_gemv_ex(0, 0, 0, 0, 8, 256, 256, 0, 1, 256, 0, 0, 2, 0, 256,
                        Q4K_MOE_WEIGHTED_DOWN, 0, 0, 0);
  st |= q4k_moe_gemv_noalloc(0, 0, 0, 0, 8, 256, 256, 0, 1, 256, 0, 0, 2, 0, 256, 0);
  st |= (int)q4k_moe_prefill_workspace_size(8, 40, 2, 256, 256);
  st |= q4k_moe_prefill(0, 0, 0, 0, 8, 256, 256, 0, 40, 256, 0, 0, 2, 0, 256, 0, 0, 0);
  st |= q4k_get_device_error(0, &bits);
  st |= q4k_selftest_wait_timeout(0);
  st |= (int)sizeof(q4k_gemv_op) == 64 ? 0 : 1 << 20;
  printf("%s %d\n", q4k_status_str(st), st);
  return 0;
}
''')
    exe = tmp_path / "use_q4k"
    lib_dir = os.path.dirname(q4k.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", lib_dir, "-lq4k", "-Wl,-rpath," + lib_dir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
