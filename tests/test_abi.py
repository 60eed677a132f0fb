"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, its struct layout matches the ctypes mirror, and argument
errors come back as the documented status codes before anything launches."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def _build_library():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_attn_build", os.path.join(ROOT, "attn_fwd_03_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="module")
def binding():
    _build_library()
    import attn_fwd_03_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_entry_points(binding):
    assert _declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(binding):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(binding.lib, name)


def test_struct_layout_matches_c(binding):
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "attn.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(attn_fwd_params),
         offsetof(attn_fwd_params, q), offsetof(attn_fwd_params, mask_stride), sizeof(attn_bwd_params),
         offsetof(attn_bwd_params, dout), offsetof(attn_bwd_params, workspace_bytes), sizeof(attn_decode_params),
         offsetof(attn_decode_params, q), offsetof(attn_decode_params, num_splits),
         offsetof(attn_decode_params, workspace_bytes), sizeof(attn_fwd_fp8_params),
         offsetof(attn_fwd_fp8_params, q_descale), offsetof(attn_fwd_fp8_params, reserved1));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "l.c")
        exe = os.path.join(td, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    F, B, Dp, F8 = binding.FwdParams, binding.BwdParams, binding.DecodeParams, binding.Fp8Params
    want = [ctypes.sizeof(F), F.q.offset, F.mask_stride.offset, ctypes.sizeof(B), B.dout.offset,
            B.workspace_bytes.offset, ctypes.sizeof(Dp), Dp.q.offset, Dp.num_splits.offset,
            Dp.workspace_bytes.offset, ctypes.sizeof(F8), F8.q_descale.offset, F8.reserved1.offset]
    assert got == want


def _params(binding, **kw):
    p = binding.FwdParams()
    p.B, p.H, p.N, p.d = kw.get("B", 1), kw.get("H", 1), kw.get("N", 128), kw.get("d", 64)
    p.dtype = kw.get("dtype", binding.ATTN_BF16)
    p.causal = kw.get("causal", 0)
    p.scale = kw.get("scale", 0.125)
    p.reserved0 = kw.get("reserved0", 0)
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    for name in ("q", "k", "v", "o", "lse"):
        setattr(p, name, kw.get(name, fake))
    st = kw.get("stride", (128 * 64, 128 * 64, 64))
    for name in ("q_stride", "k_stride", "v_stride", "o_stride"):
        setattr(p, name, (ctypes.c_int64 * 3)(*st))
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), "ATTN_ERR_UNSUPPORTED"),
    (dict(d=512), "ATTN_ERR_UNSUPPORTED"),
    (dict(d=256, dtype=1), "ATTN_ERR_UNSUPPORTED"),  # head dim 256: 16-bit inputs only
    (dict(B=-1), "ATTN_ERR_INVALID"),
    (dict(N=-5), "ATTN_ERR_INVALID"),
    (dict(dtype=7), "ATTN_ERR_INVALID"),
    (dict(causal=2), "ATTN_ERR_INVALID"),
    (dict(reserved0=1), "ATTN_ERR_INVALID"),
    (dict(scale=float("nan")), "ATTN_ERR_INVALID"),
    (dict(scale=0.0), "ATTN_ERR_INVALID"),
    (dict(scale=-0.5), "ATTN_ERR_INVALID"),
    (dict(q=0), "ATTN_ERR_INVALID"),
    (dict(lse=0), "ATTN_ERR_INVALID"),
    (dict(q=(1 << 20) + 8), "ATTN_ERR_ALIGN"),
    (dict(stride=(128 * 64, 128 * 64, 60)), "ATTN_ERR_ALIGN"),
    (dict(stride=(128 * 64, 0, 64)), "ATTN_ERR_INVALID"),
    (dict(B=70000), "ATTN_ERR_UNSUPPORTED"),
])
def test_fwd_argument_errors(binding, kw, status):
    p = _params(binding, **kw)
    rc = binding.lib.attn_fwd(ctypes.byref(p), None)
    assert rc == getattr(binding, status)
    assert binding.last_error() != ""


def test_null_params(binding):
    assert binding.lib.attn_fwd(None, None) == binding.ATTN_ERR_INVALID
    assert binding.lib.attn_bwd(None, None) == binding.ATTN_ERR_INVALID
    assert binding.lib.attn_bwd_deterministic(None, None) == binding.ATTN_ERR_INVALID
    assert binding.lib.attn_bwd_workspace_size(None) == 0


@pytest.mark.parametrize("shape", [(0, 2, 128), (2, 0, 128), (1, 1, 0)])
def test_empty_problem_is_a_no_op(binding, shape):
    B, H, N = shape
    p = _params(binding, B=B, H=H, N=N, q=0, k=0, v=0, o=0, lse=0)
    assert binding.lib.attn_fwd(ctypes.byref(p), None) == binding.ATTN_OK
    bp = binding.BwdParams()
    bp.fwd = p
    assert binding.lib.attn_bwd(ctypes.byref(bp), None) == binding.ATTN_OK
    assert binding.lib.attn_bwd_deterministic(ctypes.byref(bp), None) == binding.ATTN_OK
    assert binding.lib.attn_bwd_workspace_size(ctypes.byref(p)) == 0


@pytest.mark.parametrize("entry", ["attn_bwd", "attn_bwd_deterministic"])
def test_bwd_argument_errors(binding, entry):
    call = getattr(binding.lib, entry)
    bp = binding.BwdParams()
    bp.fwd = _params(binding, dtype=binding.ATTN_F32)
    assert call(ctypes.byref(bp), None) == binding.ATTN_ERR_UNSUPPORTED
    bp.fwd = _params(binding, d=256)  # built for attn_bwd; the deterministic backward stops at 128
    want = binding.ATTN_ERR_UNSUPPORTED if entry == "attn_bwd_deterministic" else binding.ATTN_ERR_INVALID
    assert call(ctypes.byref(bp), None) == want
    bp.fwd = _params(binding)
    assert call(ctypes.byref(bp), None) == binding.ATTN_ERR_INVALID  # dout NULL
    fake = 1 << 20
    st = (ctypes.c_int64 * 3)(128 * 64, 128 * 64, 64)
    bp.dout, bp.dq, bp.dk, bp.dv = fake, fake, fake, fake
    bp.do_stride, bp.dq_stride, bp.dk_stride, bp.dv_stride = st, st, st, st
    bp.workspace, bp.workspace_bytes = fake, 16
    assert call(ctypes.byref(bp), None) == binding.ATTN_ERR_WORKSPACE
    assert "needed" in binding.last_error()


def test_workspace_size(binding):
    # per (b, h) and 128-row tile: 2 x 128 fp32 statistics; then the fp32 dQ accumulator
    for N in (100, 128, 300):
        for d in (64, 128, 256):
            p = _params(binding, B=2, H=3, N=N, d=d)
            tiles = 2 * 3 * ((N + 127) // 128)
            assert binding.lib.attn_bwd_workspace_size(ctypes.byref(p)) == tiles * 1024 + 2 * 3 * N * d * 4


def test_version_and_timeout_knobs(binding):
    assert binding.version() >= 100
    binding.set_wait_timeout_ns(5)  # clamped, must not crash
    binding.set_wait_timeout_ns(2_000_000_000)
    binding.debug_set_producer_stall(0)


def _decode_params(binding, **kw):
    p = binding.DecodeParams()
    p.B, p.H, p.nq, p.nk, p.d = kw.get("B", 1), kw.get("H", 2), kw.get("nq", 1), kw.get("nk", 4096), kw.get("d", 128)
    p.dtype = kw.get("dtype", binding.ATTN_BF16)
    p.causal = kw.get("causal", 0)
    p.scale = kw.get("scale", 0.088)
    p.reserved0 = kw.get("reserved0", 0)
    p.num_splits = kw.get("num_splits", 0)
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    for name in ("q", "k", "v", "o", "lse"):
        setattr(p, name, kw.get(name, fake))
    st = kw.get("stride", (4096 * 128, 4096 * 128, 128))
    for name in ("q_stride", "k_stride", "v_stride", "o_stride"):
        setattr(p, name, (ctypes.c_int64 * 3)(*st))
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(nq=129), "ATTN_ERR_UNSUPPORTED"),
    (dict(nq=-1), "ATTN_ERR_INVALID"),
    (dict(nk=0), "ATTN_ERR_INVALID"),
    (dict(d=96), "ATTN_ERR_UNSUPPORTED"),
    (dict(dtype=1), "ATTN_ERR_UNSUPPORTED"),  # fp32
    (dict(dtype=7), "ATTN_ERR_INVALID"),
    (dict(causal=2), "ATTN_ERR_INVALID"),
    (dict(reserved0=1), "ATTN_ERR_INVALID"),
    (dict(num_splits=-1), "ATTN_ERR_INVALID"),
    (dict(scale=0.0), "ATTN_ERR_INVALID"),
    (dict(B=300, H=300), "ATTN_ERR_UNSUPPORTED"),
    (dict(k=0), "ATTN_ERR_INVALID"),
    (dict(lse=0), "ATTN_ERR_INVALID"),
    (dict(v=(1 << 20) + 8), "ATTN_ERR_ALIGN"),
    (dict(stride=(4096 * 128, 4096 * 128, 100)), "ATTN_ERR_ALIGN"),
])
def test_decode_argument_errors(binding, kw, status):
    p = _decode_params(binding, **kw)
    assert binding.lib.attn_decode(ctypes.byref(p), None) == getattr(binding, status)
    assert binding.last_error() != ""
    assert binding.lib.attn_decode_workspace_size(ctypes.byref(p)) == 0


@pytest.mark.parametrize("shape", [(0, 2, 1), (2, 0, 1), (1, 1, 0)])
def test_decode_empty_problem_is_a_no_op(binding, shape):
    B, H, nq = shape
    p = _decode_params(binding, B=B, H=H, nq=nq, q=0, k=0, v=0, o=0, lse=0)
    assert binding.lib.attn_decode(ctypes.byref(p), None) == binding.ATTN_OK


def _fp8_params(binding, **kw):
    p = binding.Fp8Params()
    p.f = _params(binding, **{"d": 128, "dtype": binding.ATTN_E4M3, "stride": (128 * 128, 128 * 128, 128), **kw})
    p.q_descale, p.k_descale, p.v_descale = kw.get("descale", (0.5, 0.5, 0.5))
    p.reserved1 = kw.get("reserved1", 0)
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(d=64), "ATTN_ERR_UNSUPPORTED"),
    (dict(d=192), "ATTN_ERR_UNSUPPORTED"),
    (dict(dtype=0), "ATTN_ERR_UNSUPPORTED"),  # a 16-bit dtype goes through attn_fwd
    (dict(descale=(0.5, 0.0, 0.5)), "ATTN_ERR_INVALID"),
    (dict(descale=(0.5, 0.5, float("inf"))), "ATTN_ERR_INVALID"),
    (dict(reserved1=3), "ATTN_ERR_INVALID"),
    (dict(causal=2), "ATTN_ERR_INVALID"),
    (dict(N=-1), "ATTN_ERR_INVALID"),
    (dict(stride=(128 * 128, 128 * 128, 120)), "ATTN_ERR_ALIGN"),  # rows of 120 bytes
])
def test_fp8_argument_errors(binding, kw, status):
    p = _fp8_params(binding, **kw)
    assert binding.lib.attn_fwd_fp8(ctypes.byref(p), None) == getattr(binding, status)
    assert binding.last_error()


def test_fp8_null_and_empty(binding):
    assert binding.lib.attn_fwd_fp8(None, None) == binding.ATTN_ERR_INVALID
    p = _fp8_params(binding, B=0)
    assert binding.lib.attn_fwd_fp8(ctypes.byref(p), None) == binding.ATTN_OK
    # E4M3 given to the 16-bit entry point is refused
    f = _params(binding, d=128, dtype=binding.ATTN_E4M3)
    assert binding.lib.attn_fwd(ctypes.byref(f), None) == binding.ATTN_ERR_UNSUPPORTED
