"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function declared in include/moe.h, and rejects bad arguments on the
host before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from int4_grouped_gemm_gb300 import _lib, build
    build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("moe_prefill", "moe_decode", "pack_int4", "moe_workspace_bytes",
                     "moe_route_logits", "moe_read_device_status", "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from int4_grouped_gemm_gb300 import _lib
    names = header_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"
    # the binding marshals every declared call, under the same name
    assert sorted(_lib.SIGNATURES) == names


def test_status_strings(lib):
    from int4_grouped_gemm_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "NULL" in _lib.status_string(_lib.MOE_ERR_NULL)
    assert "bounded wait" in _lib.status_string(_lib.MOE_ERR_TIMEOUT - 3)


def _desc(E=256, k=8, H=2048, I=512, G=64, shared=1):
    from int4_grouped_gemm_gb300._lib import moe_layer_desc
    return moe_layer_desc(E, k, H, I, G, shared, None, None)


def test_workspace_sizes_and_shape_checks(lib):
    from int4_grouped_gemm_gb300 import _lib
    d = _desc()
    n512 = _lib.moe_workspace_bytes(d, 512)
    n4096 = _lib.moe_workspace_bytes(d, 4096)
    assert 0 < n512 < n4096
    # h [T*(k+1)][I] bf16 and the fp32 combine accumulator dominate
    assert n4096 >= 4096 * 9 * 512 * 2 + 4096 * 2048 * 4
    for bad in (_desc(E=0), _desc(E=257), _desc(k=9), _desc(k=0), _desc(E=4, k=5), _desc(H=200),
                _desc(I=100), _desc(I=192), _desc(G=16), _desc(H=32768), _desc(shared=2)):
        assert _lib.moe_workspace_bytes(bad, 16) == 0
    assert _lib.moe_workspace_bytes(d, 0) == 0
    # x[T][H] must hold at most 2^32 elements (32-bit offsets in the token copier)
    wide = _desc(H=16384)
    assert _lib.moe_workspace_bytes(wide, (1 << 32) // 16384) > 0
    assert _lib.moe_workspace_bytes(wide, (1 << 32) // 16384 + 1) == 0


def test_argument_errors_are_caught_on_the_host(lib):
    from int4_grouped_gemm_gb300 import _lib
    d = _desc()
    rc = lib.moe_prefill(None, None, 16, None, None, 0, None)
    assert rc == _lib.MOE_ERR_NULL
    rc = lib.moe_prefill(ctypes.byref(d), None, 16, None, None, 0, None)   # weights NULL
    assert rc == _lib.MOE_ERR_NULL
    bad = _desc(k=9)
    assert lib.moe_decode(ctypes.byref(bad), None, None, None, 0, None) == _lib.MOE_ERR_SHAPE
    # misaligned pointer
    assert lib.pack_int4(ctypes.c_void_p(8), 4, 64, 32, ctypes.c_void_p(16), ctypes.c_void_p(32),
                         ctypes.c_void_p(48), None) == _lib.MOE_ERR_ALIGN
    # group must divide K and be a multiple of 8
    assert lib.pack_int4(ctypes.c_void_p(16), 4, 64, 24, ctypes.c_void_p(16), ctypes.c_void_p(32),
                         ctypes.c_void_p(48), None) == _lib.MOE_ERR_SHAPE
    assert lib.moe_read_device_status(None, None) == _lib.MOE_ERR_NULL


def test_router_split_sizes_and_host_checks(lib):
    from int4_grouped_gemm_gb300 import _lib
    assert _lib.moe_router_split_bytes(256, 2048) == 2 * 256 * 2048 * 2
    assert _lib.moe_router_split_bytes(40, 256) == 2 * 48 * 256 * 2      # rows padded to 16
    for E, H in ((0, 2048), (257, 2048), (16, 200), (16, 32768)):
        assert _lib.moe_router_split_bytes(E, H) == 0
        assert lib.moe_split_router(ctypes.c_void_p(16), E, H, ctypes.c_void_p(32), None) == _lib.MOE_ERR_SHAPE
    assert lib.moe_split_router(None, 16, 256, ctypes.c_void_p(32), None) == _lib.MOE_ERR_NULL
    assert lib.moe_split_router(ctypes.c_void_p(16), 16, 256, ctypes.c_void_p(40), None) == _lib.MOE_ERR_ALIGN
    # a misaligned split in the layer is refused before anything runs
    q = _lib.moe_qweight(1024, 1024, 1024)
    d = _lib.moe_layer_desc(256, 8, 2048, 512, 64, 1, 1024, None, q, q, q)
    d.router_split = 8
    assert lib.moe_prefill(ctypes.byref(d), ctypes.c_void_p(1024), 16, ctypes.c_void_p(2048),
                           ctypes.c_void_p(4096), 1 << 40, None) == _lib.MOE_ERR_ALIGN


def test_pipelined_host_call_rejects_bad_arguments_on_the_host(lib):
    from int4_grouped_gemm_gb300 import _lib
    d = _desc()
    two = (ctypes.c_void_p * 2)(16, 32)
    one = (ctypes.c_void_p * 1)(64)
    none = (ctypes.c_void_p * 1)(None)
    f = lib.moe_forward_host_stream
    # no calls, no arrays, a NULL host buffer, a misaligned staging buffer
    assert f(ctypes.byref(d), one, one, 0, 16, two, two, None, 0, None) == _lib.MOE_ERR_TOKENS
    assert f(ctypes.byref(d), None, one, 1, 16, two, two, None, 0, None) == _lib.MOE_ERR_NULL
    assert f(ctypes.byref(d), none, one, 1, 16, two, two, None, 0, None) == _lib.MOE_ERR_NULL
    assert f(ctypes.byref(d), one, one, 1, 16, (ctypes.c_void_p * 2)(16, 40), two, None, 0, None) == \
        _lib.MOE_ERR_ALIGN
    assert f(ctypes.byref(d), one, one, 1, 0, two, two, None, 0, None) == _lib.MOE_ERR_TOKENS
    bad = _desc(k=9)
    assert f(ctypes.byref(bad), one, one, 1, 16, two, two, None, 0, None) == _lib.MOE_ERR_SHAPE


def test_routing_views_layout(lib):
    from int4_grouped_gemm_gb300 import _lib
    d = _desc()
    v = _lib.moe_routing_views_for(d, 4096)
    offs = [v.logits, v.topk_idx, v.topk_w, v.counts, v.offsets, v.perm, v.inv_perm, v.tile_group,
            v.tile_row, v.tile_rows, v.tile_sched, v.num_tiles]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert v.tile_size == 128
    assert v.max_tiles >= (4096 * 9) // 128 + 257


def test_small_batch_decode_checks_on_the_host(lib):
    from int4_grouped_gemm_gb300 import _lib
    # 16-byte aligned stand-in pointers: every case below must be rejected on
    # the host, before a device or any of the pointers is touched
    q = _lib.moe_qweight(256, 512, 768)
    d = _lib.moe_layer_desc(256, 8, 2048, 512, 64, 1, 1024, None, q, q, q)
    f = lib.moe_decode_batch
    x, y, ws = ctypes.c_void_p(2048), ctypes.c_void_p(4096), ctypes.c_void_p(8192)
    n = _lib.moe_workspace_bytes(d, 1)
    # the union of 8 tokens' picks (at most 64 experts) + the shared expert:
    # per-slot SwiGLU rows [8][I] bf16, and per group of slots (one slot per
    # group at most) the weighted outputs [8][H] fp32
    assert n >= 65 * 8 * (512 * 2 + 2048 * 4)
    assert f(ctypes.byref(d), x, 0, y, ws, n, None) == _lib.MOE_ERR_TOKENS
    assert f(ctypes.byref(d), x, 9, y, ws, n, None) == _lib.MOE_ERR_TOKENS
    assert f(ctypes.byref(d), x, 4, y, ws, 4096, None) == _lib.MOE_ERR_WORKSPACE
    assert f(ctypes.byref(d), ctypes.c_void_p(2056), 4, y, ws, n, None) == _lib.MOE_ERR_ALIGN
    assert f(ctypes.byref(d), None, 4, y, ws, n, None) == _lib.MOE_ERR_NULL
    wide = _lib.moe_layer_desc(256, 8, 8192, 512, 64, 1, 1024, None, q, q, q)   # above the decode limit
    assert f(ctypes.byref(wide), x, 4, y, ws, 1 << 30, None) == _lib.MOE_ERR_SHAPE
    bad = _lib.moe_layer_desc(256, 9, 2048, 512, 64, 1, 1024, None, q, q, q)
    assert f(ctypes.byref(bad), x, 4, y, ws, n, None) == _lib.MOE_ERR_SHAPE


def test_decoder_block_checks_on_the_host(lib):
    from int4_grouped_gemm_gb300 import _lib
    q = _lib.moe_qweight(256, 512, 768)
    d = _lib.moe_layer_desc(256, 8, 2048, 512, 64, 1, 1024, None, q, q, q)
    a, r, w, out, ws = (ctypes.c_void_p(v) for v in (2048, 4096, 8192, 16384, 32768))
    n = _lib.moe_workspace_bytes(d, 16)
    # the residual stream and the normalised input ([T][H] bf16 each) come
    # after the layer's own tables, the last of which follow y_acc
    v = _lib.moe_routing_views_for(d, 16)
    assert n >= v.y_acc + 16 * 2048 * 4 + 2 * 16 * 2048 * 2
    for f, T in ((lib.moe_prefill_block, 16), (lib.moe_decode_batch_block, 4)):
        assert f(ctypes.byref(d), a, r, w, ctypes.c_float(-1.0), T, out, ws, n, None) == _lib.MOE_ERR_SHAPE
        assert f(ctypes.byref(d), a, r, w, ctypes.c_float(float("nan")), T, out, ws, n, None) == _lib.MOE_ERR_SHAPE
        assert f(ctypes.byref(d), a, r, ctypes.c_void_p(8196), ctypes.c_float(1e-6), T, out, ws, n, None) == \
            _lib.MOE_ERR_ALIGN
        assert f(ctypes.byref(d), a, None, w, ctypes.c_float(1e-6), T, out, ws, n, None) == _lib.MOE_ERR_NULL
        assert f(ctypes.byref(d), a, r, w, ctypes.c_float(1e-6), T, out, ws, 4096, None) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_decode_batch_block(ctypes.byref(d), a, r, w, ctypes.c_float(1e-6), 9, out, ws, n, None) == \
        _lib.MOE_ERR_TOKENS
    assert lib.moe_prefill_block(ctypes.byref(d), a, r, w, ctypes.c_float(1e-6), 0, out, ws, n, None) == \
        _lib.MOE_ERR_TOKENS
