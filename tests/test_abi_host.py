"""Host-side tests of the C ABI: the library loads, exports every entry point
include/gbfuse.h declares, and rejects bad arguments with the documented status
before touching a device.  No test here launches a kernel (the pointers are
fake addresses that the validation must never dereference)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gbfuse.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GBF_API\s+[\w\s\*]+?\b(gbf_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def test_header_declares_the_entry_points():
    assert declared_symbols() == sorted(["gbf_add_rmsnorm_fp8", "gbf_qkv_split_norm_rope",
                                         "gbf_qkv_split_layernorm_rope", "gbf_linear_bias_gelu", "gbf_gated_act",
                                         "gbf_linear_fp8_act", "gbf_fold_norm_weight",
                                         "gbf_bn_fold", "gbf_copy", "gbf_device_status", "gbf_last_error",
                                         "gbf_version", "gbf_selftest_bounded_wait"])


def test_library_exports_every_declared_symbol(gbf):
    out = subprocess.run(["nm", "-D", "--defined-only", gbf.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gbf_\w+)", out))
    assert set(declared_symbols()) <= exported
    # nothing but the documented C entry points leaks out of the library
    assert {s for s in exported if s.startswith("gbf")} == set(declared_symbols())
    for s in declared_symbols():
        assert hasattr(gbf.raw(), s)
    assert set(gbf.EXPORTED) == set(declared_symbols())


def test_version(gbf):
    assert gbf.version() == 10000


F = 0x10000          # fake, 16-byte aligned "device" addresses; never dereferenced


def A(i):
    return ctypes.c_void_p(F * (i + 1))


def last(gbf):
    return gbf.raw().gbf_last_error().decode()


def test_add_rmsnorm_validation(gbf):
    L = gbf.raw()
    call = lambda **k: L.gbf_add_rmsnorm_fp8(*[k.get(n, d) for n, d in [           # noqa: E731
        ("x", A(0)), ("res_in", A(1)), ("res_out", A(2)), ("gate", None), ("mode", 0), ("weight", A(3)),
        ("scale", None), ("shift", None), ("q", A(4)), ("rows", 4), ("hidden", 64), ("eps", 1e-6),
        ("s", 0.05), ("stream", None)]])
    assert call(rows=0) == gbf.OK                         # empty: nothing enqueued
    assert call(hidden=60) == gbf.EALIGN and "multiple of 8" in last(gbf)
    assert call(hidden=65536) == gbf.EUNSUPPORTED
    assert call(hidden=0) == gbf.EINVAL
    assert call(rows=-1) == gbf.EINVAL
    assert call(mode=7) == gbf.EINVAL
    assert call(x=None) == gbf.EINVAL
    assert call(weight=None) == gbf.EINVAL                # WEIGHT mode needs a weight
    assert call(mode=2) == gbf.EINVAL                     # ADA needs scale and shift
    assert call(eps=-1.0) == gbf.EINVAL
    assert call(s=0.0) == gbf.EINVAL
    assert call(s=float("inf")) == gbf.EINVAL
    assert call(eps=float("nan")) == gbf.EINVAL
    assert call(x=ctypes.c_void_p(F + 8)) == gbf.EALIGN
    # res_out may alias res_in exactly, but not overlap x or partially overlap res_in
    assert call(res_out=A(0)) == gbf.EINVAL
    assert call(res_out=ctypes.c_void_p(2 * F + 16)) == gbf.EINVAL
    assert call(q=A(1)) == gbf.EINVAL


def test_qkv_validation(gbf):
    L = gbf.raw()
    sec_ok = (ctypes.c_int32 * 3)(44, 42, 42)
    sec_bad = (ctypes.c_int32 * 3)(44, 42, 41)
    call = lambda **k: L.gbf_qkv_split_norm_rope(*[k.get(n, d) for n, d in [       # noqa: E731
        ("qkv", A(0)), ("tokens", 4), ("hq", 2), ("hkv", 1), ("d", 128), ("norm", 0), ("qw", A(1)),
        ("kw", A(2)), ("eps", 1e-6), ("rope", 0), ("pos", A(3)), ("sec", None), ("theta", 1e4),
        ("q", A(4)), ("k", A(5)), ("v", A(6)), ("slots", None), ("rows", 4), ("stream", None)]])
    assert call(tokens=0) == gbf.OK
    assert call(d=100) == gbf.EUNSUPPORTED
    assert call(d=512) == gbf.EUNSUPPORTED
    assert call(d=96, norm=0) == gbf.EUNSUPPORTED          # per-head needs a power of two
    assert call(norm=5) == gbf.EINVAL
    assert call(rope=1) == gbf.EINVAL                       # 3D without sections
    assert call(rope=1, sec=ctypes.cast(sec_bad, ctypes.c_void_p)) == gbf.EINVAL
    assert call(rope=1, sec=ctypes.cast(sec_ok, ctypes.c_void_p), d=64) == gbf.EINVAL   # sum != head_dim
    assert call(rows=3) == gbf.EINVAL                       # cache too small without slots
    assert call(theta=0.0) == gbf.EINVAL
    assert call(pos=None) == gbf.EINVAL
    assert call(q=ctypes.c_void_p(5 * F + 4)) == gbf.EALIGN
    assert call(q=A(0)) == gbf.EINVAL                       # Q overlaps the packed input
    assert call(k=A(6)) == gbf.EINVAL                       # K and V caches overlap
    # the staged (shared-memory) path bounds the row width; the per-head 1D kernel does not
    assert call(norm=1, hq=220, hkv=40) == gbf.EUNSUPPORTED  # (6*220 + 8*40) * 128 > 196608
    assert call(norm=0, hq=220, hkv=40, tokens=0) == gbf.OK
    assert call(norm=1, hq=220, hkv=40, tokens=0) == gbf.EUNSUPPORTED


def test_qkv_layernorm_validation(gbf):
    L = gbf.raw()
    call = lambda **k: L.gbf_qkv_split_layernorm_rope(*[k.get(n, d) for n, d in [       # noqa: E731
        ("qkv", A(0)), ("tokens", 4), ("hq", 2), ("hkv", 1), ("d", 128), ("qw", A(1)), ("qb", A(7)),
        ("kw", A(2)), ("kb", A(8)), ("eps", 1e-5), ("pos", A(3)), ("theta", 1e4),
        ("q", A(4)), ("k", A(5)), ("v", A(6)), ("slots", None), ("rows", 4), ("stream", None)]])
    assert call(tokens=0) == gbf.OK
    assert call(tokens=0, qb=None, kb=None) == gbf.OK
    assert call(d=96) == gbf.EUNSUPPORTED                    # only 64, 128, 256
    assert call(d=512) == gbf.EUNSUPPORTED
    assert call(eps=-1.0) == gbf.EINVAL
    assert call(qw=None) == gbf.EINVAL
    assert call(qb=ctypes.c_void_p(7 * F + 2)) == gbf.EALIGN
    assert call(q=A(7)) == gbf.EINVAL                       # Q overlaps the Q bias
    # the RMSNorm entry point does not take the LayerNorm mode
    assert L.gbf_qkv_split_norm_rope(A(0), 4, 2, 1, 128, 2, A(1), A(2), ctypes.c_float(1e-6), 0, A(3), None,
                                     ctypes.c_float(1e4), A(4), A(5), A(6), None, 4, None) == gbf.EINVAL


def test_gated_act_validation(gbf):
    L = gbf.raw()
    call = lambda x=A(0), y=A(1), rows=4, d=64, act=gbf.ACT_SILU: L.gbf_gated_act(x, y, rows, d, act, None)  # noqa
    assert call(rows=0) == gbf.OK
    for act in (gbf.ACT_SILU, gbf.ACT_GELU_TANH, gbf.ACT_GELU_ERF):
        assert call(rows=0, act=act) == gbf.OK
    assert call(act=gbf.ACT_NONE) == gbf.EINVAL
    assert call(act=9) == gbf.EINVAL
    assert call(d=60) == gbf.EALIGN
    assert call(d=0) == gbf.EINVAL
    assert call(rows=-1) == gbf.EINVAL
    assert call(x=None) == gbf.EINVAL
    assert call(y=ctypes.c_void_p(F + 8)) == gbf.EALIGN
    assert call(y=ctypes.c_void_p(F + 256)) == gbf.EINVAL     # y overlaps x


def test_linear_fp8_and_norm_fold_validation(gbf):
    L = gbf.raw()
    lin = lambda **k: L.gbf_linear_fp8_act(*[k.get(n, d) for n, d in [              # noqa: E731
        ("x", A(0)), ("xs", 0.05), ("w", A(1)), ("ws", A(2)), ("b", A(3)), ("y", A(4)), ("m", 128), ("n", 256),
        ("k", 256), ("act", 1), ("s", None)]])
    assert lin(m=0) == gbf.OK
    assert lin(k=192) == gbf.EUNSUPPORTED                    # K % 128
    assert lin(n=8) == gbf.EUNSUPPORTED
    assert lin(xs=0.0) == gbf.EINVAL
    assert lin(xs=float("nan")) == gbf.EINVAL
    assert lin(ws=None) == gbf.EINVAL
    assert lin(act=6) == gbf.EINVAL
    assert lin(ws=ctypes.c_void_p(2 * F + 4)) == gbf.EALIGN
    assert lin(y=A(2)) == gbf.EINVAL                         # Y overlaps w_scale
    fold = lambda **k: L.gbf_fold_norm_weight(*[k.get(n, d) for n, d in [          # noqa: E731
        ("w", A(0)), ("g", A(1)), ("gemma", 1), ("oc", 8), ("inner", 64), ("wo", A(2)), ("s", None)]])
    assert fold(oc=0) == gbf.OK
    assert fold(inner=0) == gbf.EINVAL
    assert fold(gemma=2) == gbf.EINVAL
    assert fold(g=None) == gbf.EINVAL
    assert fold(wo=ctypes.c_void_p(F + 16)) == gbf.EINVAL    # partial overlap with W
    assert fold(wo=A(1)) == gbf.EINVAL                       # overlaps gamma


def test_linear_and_fold_and_copy_validation(gbf):
    L = gbf.raw()
    lin = lambda **k: L.gbf_linear_bias_gelu(*[k.get(n, d) for n, d in [          # noqa: E731
        ("x", A(0)), ("w", A(1)), ("b", A(2)), ("y", A(3)), ("m", 128), ("n", 256), ("k", 128), ("act", 1),
        ("s", None)]])
    assert lin(m=0) == gbf.OK
    for act in (gbf.ACT_NONE, gbf.ACT_GELU_TANH, gbf.ACT_GELU_ERF, gbf.ACT_SILU):
        assert lin(m=0, act=act) == gbf.OK
    assert lin(m=0, act=7) == gbf.EINVAL
    assert lin(k=100) == gbf.EUNSUPPORTED
    assert lin(n=8) == gbf.EUNSUPPORTED
    assert lin(act=5) == gbf.EINVAL
    assert lin(x=None) == gbf.EINVAL
    assert lin(y=ctypes.c_void_p(4 * F + 2)) == gbf.EALIGN
    assert lin(y=A(0)) == gbf.EINVAL
    # int32 extents inside the kernel: 2^31 itself is refused, as is a tile count past 2^31 - 1
    assert lin(m=1 << 31) == gbf.EUNSUPPORTED
    assert lin(n=1 << 31) == gbf.EUNSUPPORTED
    assert lin(k=1 << 31) == gbf.EUNSUPPORTED
    assert lin(m=(1 << 31) - 1, n=(1 << 31) - 16) == gbf.EUNSUPPORTED
    fold = lambda **k: L.gbf_bn_fold(*[k.get(n, d) for n, d in [                   # noqa: E731
        ("w", A(0)), ("b", None), ("g", A(1)), ("be", A(2)), ("mu", A(3)), ("var", A(4)), ("eps", 1e-2),
        ("oc", 8), ("inner", 27), ("wo", A(5)), ("bo", A(6)), ("s", None)]])
    assert fold(oc=0) == gbf.OK
    assert fold(eps=-1.0) == gbf.EINVAL
    assert fold(inner=0) == gbf.EINVAL
    assert fold(g=None) == gbf.EINVAL
    assert fold(bo=A(1)) == gbf.EINVAL                      # b_out overlaps gamma
    assert fold(wo=ctypes.c_void_p(F + 2)) == gbf.EINVAL    # partial overlap with W
    assert L.gbf_copy(A(0), A(1), -1, None) == gbf.EINVAL
    assert L.gbf_copy(A(0), A(1), 0, None) == gbf.OK
    assert L.gbf_copy(A(0), ctypes.c_void_p(2 * F + 8), 64, None) == gbf.EALIGN
    assert L.gbf_copy(A(0), ctypes.c_void_p(F + 16), 64, None) == gbf.EINVAL


def test_python_binding_raises_with_message(gbf):
    """A non-OK status from the library becomes GbfError with the status and the
    library's message: hidden = 60 is not a multiple of 8 (GBF_EALIGN), found on
    the host before any launch (the pointers are distinct, aligned, never read)."""
    import ctypes
    p = [ctypes.c_void_p(a) for a in (1 << 20, 2 << 20, 3 << 20, 4 << 20)]
    with pytest.raises(gbf.GbfError) as e:
        gbf._check(gbf.raw().gbf_add_rmsnorm_fp8(p[0], p[1], p[2], None, gbf.NORM_NOWEIGHT, None, None, None, p[3],
                                                 4, 60, 1e-6, 0.05, None))
    assert e.value.status == gbf.EALIGN and len(str(e.value)) > len("status -2: ")
