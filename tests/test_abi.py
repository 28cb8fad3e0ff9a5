"""CPU-only checks of the C ABI: the library loads, exports every declared symbol, and rejects bad
arguments on the host before touching any pointer or the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")
LIB = os.path.join(ROOT, "block_scaled_fp8_moe_gb300", "libmoe.so")


def declared():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def B():
    if not os.path.exists(LIB):
        from block_scaled_fp8_moe_gb300 import build
        build.build()
    from block_scaled_fp8_moe_gb300 import binding
    return binding


def test_header_declares_the_five_layer_entry_points():
    names = set(declared())
    for n in ("moe_route_topk", "moe_quant_mxfp8", "moe_w13_swiglu_grouped", "moe_w2_combine_grouped",
              "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(LIB)
    for n in declared():
        assert hasattr(lib, n), n
    assert sorted(declared()) == sorted(B.EXPORTED)


def test_status_strings(B):
    for c in range(7):
        assert B.lib.moe_status_string(c) != b"unknown status"
    assert B.lib.moe_status_string(99) == b"unknown status"


@pytest.mark.parametrize("bad", [
    dict(H=100), dict(I=96), dict(k=0), dict(k=33), dict(E=2000), dict(k=9, E=8), dict(T=-1), dict(H=32768),
])
def test_unsupported_shapes_rejected_on_host(B, bad):
    args = dict(T=4, H=256, E=8, k=2, I=128)
    args.update(bad)
    shp = B.shape(**args)
    assert B.moe_workspace_bytes(shp) == 0
    n = ctypes.c_void_p(0)
    rc = B.lib.moe_route_topk(ctypes.byref(shp), *([n] * 10), n, 0, n)
    assert rc in (B.MOE_ERR_UNSUPPORTED_SHAPE, B.MOE_ERR_INVALID_ARG)
    rc = B.lib.moe_forward(ctypes.byref(shp), *([n] * 9), None, n, 0, n)
    assert rc in (B.MOE_ERR_UNSUPPORTED_SHAPE, B.MOE_ERR_INVALID_ARG)


def test_workspace_checks_on_host(B):
    shp = B.shape(6, 4096, 256, 8, 2048)
    need = B.moe_workspace_bytes(shp)
    assert need > 0 and need % 256 == 0
    n = ctypes.c_void_p(0)
    # null workspace
    assert B.lib.moe_w13_swiglu_grouped(ctypes.byref(shp), *([n] * 9), n, need, n) == B.MOE_ERR_WORKSPACE
    # misaligned / too small workspace (never dereferenced: checks precede any launch)
    fake = ctypes.c_void_p(0x1000 + 8)
    assert B.lib.moe_w2_combine_grouped(ctypes.byref(shp), *([n] * 10), fake, need, n) == B.MOE_ERR_WORKSPACE
    # the split down projection / combine only need the status word, but it must be there
    assert B.lib.moe_w2_grouped(ctypes.byref(shp), *([n] * 7), n, 256, n) == B.MOE_ERR_WORKSPACE
    assert B.lib.moe_combine(ctypes.byref(shp), *([n] * 5), ctypes.c_void_p(0x1000), 128, n) == B.MOE_ERR_WORKSPACE
    assert B.lib.moe_combine(ctypes.byref(shp), *([n] * 5), ctypes.c_void_p(0x1000), 256, n) == B.MOE_ERR_INVALID_ARG
    fake = ctypes.c_void_p(0x1000)
    assert B.lib.moe_forward(ctypes.byref(shp), *([n] * 9), None, fake, need - 256, n) == B.MOE_ERR_WORKSPACE


def test_null_pointers_rejected(B):
    shp = B.shape(6, 4096, 256, 8, 2048)
    need = B.moe_workspace_bytes(shp)
    n = ctypes.c_void_p(0)
    fake_ws = ctypes.c_void_p(0x10000)
    assert B.lib.moe_forward(ctypes.byref(shp), *([n] * 9), None, fake_ws, need, n) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_quant_mxfp8(4, 64, n, n, n, n) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_quant_mxfp8(4, 48, n, n, n, n) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert B.lib.moe_quant_mxfp8(0, 64, n, n, n, n) == B.MOE_OK          # empty is a no-op


def test_packed_sizes(B):
    shp = B.shape(1, 4096, 256, 8, 576)
    q13, s13 = B.moe_packed_w13_bytes(shp)
    q2, s2 = B.moe_packed_w2_bytes(shp)
    assert q13 == 256 * (576 // 64) * (4096 // 128) * 8192 and s13 == q13 // 16
    assert q2 == 256 * (4096 // 128) * 5 * 8192 and s2 == q2 // 16     # K = 576 -> 5 chunks of 128


def test_dead_from_survival_host_checks(B):
    n = ctypes.c_void_p(0)
    assert B.lib.moe_dead_from_survival(0, n, 0.2, n, n) == B.MOE_OK           # empty is a no-op
    assert B.lib.moe_dead_from_survival(-1, n, 0.2, n, n) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_dead_from_survival(4, n, 0.2, n, n) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_dead_from_survival(4, n, float("nan"), n, n) == B.MOE_ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x1002)                                               # not 4-byte aligned
    assert B.lib.moe_dead_from_survival(4, odd, 0.2, ctypes.c_void_p(0x2000), n) == B.MOE_ERR_INVALID_ARG


def _prototypes():
    """name -> number of parameters, from the declarations in include/moe.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_the_header(B):
    protos = _prototypes()
    assert set(protos) == set(B.EXPORTED)
    for name, n in protos.items():
        fn = getattr(B.lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == n, (name, n, fn.argtypes)
