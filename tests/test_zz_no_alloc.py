"""moe_decode_static_scratch: batch-1 decode on the library's fixed scratch
array, with no caller workspace.  Compared with moe_decode (caller workspace)
on the same layer and tokens, over consecutive calls, so that whatever one
call leaves in the shared array cannot leak into the next; compared with the
CPU oracle; and its failure path: a device-side timeout stays readable
through moe_read_static_scratch_status until it is read.  The file name
keeps it last in collection order, after every other test has used the
library; it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import PackedLayer

from moe_helpers import assert_close


def _fake_desc(E, k, H, I, G):
    # 16-byte aligned stand-in pointers: the call must reject the shape on
    # the host, before it reads any of them or touches a device.
    q = _lib.moe_qweight(256, 512, 768)
    return _lib.moe_layer_desc(E, k, H, I, G, 1, 1024, None, q, q, q)


def test_oversized_layer_rejected_on_host():
    from int4_grouped_gemm_gb300 import build
    build.build()
    lib = _lib.load()
    # at E=256, k=8 the 64 KiB array holds I <= 3328; each of these needs more
    for E, k, H, I, G in [(256, 8, 2048, 3456, 64), (256, 8, 4096, 4096, 32), (128, 8, 2048, 4096, 64)]:
        d = _fake_desc(E, k, H, I, G)
        rc = lib.moe_decode_static_scratch(ctypes.byref(d), ctypes.c_void_p(2048), ctypes.c_void_p(4096), None)
        assert rc == _lib.MOE_ERR_WORKSPACE, (E, k, H, I, G, rc)
    assert "workspace" in _lib.status_string(_lib.MOE_ERR_WORKSPACE)
    # shape errors are still shape errors
    d = _fake_desc(256, 9, 2048, 512, 64)
    assert lib.moe_decode_static_scratch(ctypes.byref(d), ctypes.c_void_p(2048), ctypes.c_void_p(4096),
                                         None) == _lib.MOE_ERR_SHAPE
    assert lib.moe_decode_static_scratch(None, None, None, None) == _lib.MOE_ERR_NULL


def _layer(name, layer=0):
    cfg = synthetic.CONFIGS[name]
    L = synthetic.make_layer(cfg, layer=layer, device="cuda", with_x=False)
    packed = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    del L
    return cfg, packed


def _static(layer: PackedLayer, x: torch.Tensor) -> torch.Tensor:
    y = torch.empty_like(x)
    rc = _lib.load().moe_decode_static_scratch(ctypes.byref(layer.desc), ctypes.c_void_p(x.data_ptr()),
                                               ctypes.c_void_p(y.data_ptr()),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.MOE_OK, _lib.status_string(rc)
    return y


@pytest.mark.gpu
def test_static_scratch_matches_workspace_decode():
    cfg, big = _layer("decode40", layer=5)
    tcfg, tiny = _layer("tiny")
    ws_big = big.workspace(1)
    ws_tiny = tiny.workspace(1)
    xs = synthetic.make_tokens(cfg.H, 3, seed=71).cuda()
    xt = synthetic.make_tokens(tcfg.H, 2, seed=72).cuda()
    # consecutive calls: two tokens of the large layer, then the small layer
    # (a different scratch layout), then the large layer again
    calls = [(big, ws_big, xs[0:1]), (big, ws_big, xs[1:2]), (tiny, ws_tiny, xt[0:1]),
             (tiny, ws_tiny, xt[1:2]), (big, ws_big, xs[2:3])]
    for i, (layer, ws, x) in enumerate(calls):
        x = x.contiguous()
        got = _static(layer, x)
        want = layer.decode(x, ws)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert_close(got.float().cpu().numpy(), want.float().cpu().numpy(), f"call {i}")
    # the same token twice in a row gives the same output
    a = _static(big, xs[0:1].contiguous())
    b = _static(big, xs[0:1].contiguous())
    torch.cuda.synchronize()
    assert_close(b.float().cpu().numpy(), a.float().cpu().numpy(), "repeat")
    assert _lib.moe_read_device_status(ws_big.buf) == 0


@pytest.mark.gpu
def test_static_scratch_matches_the_oracle():
    """The static-scratch decode against the CPU oracle itself (not only
    against moe_decode), token by token on the small layer."""
    from moe_helpers import oracle_layer
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ref = oracle_layer(L, L.x)
    for t in range(cfg.T):
        y = _static(layer, L.x[t:t + 1].cuda().contiguous())
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy(), ref["y"][t:t + 1], f"token {t}")
    assert _lib.moe_read_static_scratch_status() == 0


@pytest.mark.gpu
def test_static_scratch_timeout_is_reported_then_cleared():
    """With a one-cycle wait limit the decode kernel's grid-barrier waits run
    out (no block waits for the others): the call still returns MOE_OK (the
    failure happens on the device), the status stays in the array through a
    second failing call, moe_read_static_scratch_status reports it and
    clears it, and the next normal call matches the oracle."""
    from moe_helpers import oracle_layer
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    x = L.x[0:1].cuda().contiguous()
    _lib.moe_read_static_scratch_status()  # start from a cleared status
    old = _lib.moe_set_wait_limit(1)
    try:
        _static(layer, x)
        _static(layer, x)
        torch.cuda.synchronize()
    finally:
        _lib.moe_set_wait_limit(old)
    st = _lib.moe_read_static_scratch_status()
    assert _lib.MOE_ERR_TIMEOUT - 100 < st <= _lib.MOE_ERR_TIMEOUT, st
    assert _lib.moe_read_static_scratch_status() == 0   # the read cleared it
    y = _static(layer, x)
    torch.cuda.synchronize()
    assert _lib.moe_read_static_scratch_status() == 0
    assert_close(y.float().cpu().numpy(), oracle_layer(L, L.x)["y"][0:1], "after the timeout")
