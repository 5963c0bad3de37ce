"""Failure paths without a GPU fault: a bounded device wait that runs out
reports a status instead of hanging, and bad arguments are rejected on the
host before any launch."""
import pytest
import torch

from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import PackedLayer

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    _lib.moe_workspace_init(ws)
    _lib.moe_selftest_wait_timeout(ws, 20000)
    st = _lib.moe_read_device_status(ws)
    assert st == _lib.MOE_ERR_TIMEOUT
    assert _lib.moe_read_device_status(ws) == 0       # read clears it
    # the context is still usable
    assert float(torch.ones(4, device="cuda").sum()) == 4.0


def test_workspace_too_small_and_bad_tokens():
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    x = L.x.cuda()
    y = torch.empty_like(x)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MoEError) as e:
        _lib.moe_prefill(layer.desc, x, cfg.T, y, small)
    assert e.value.code == _lib.MOE_ERR_WORKSPACE
    ws = layer.workspace(cfg.T)
    with pytest.raises(_lib.MoEError) as e:
        _lib.moe_prefill(layer.desc, x, 0, y, ws.buf)
    assert e.value.code == _lib.MOE_ERR_TOKENS
    with pytest.raises(_lib.MoEError) as e:
        _lib.moe_prefill(layer.desc, x[:, 1:], cfg.T, y, ws.buf)   # misaligned by 2 bytes
    assert e.value.code == _lib.MOE_ERR_ALIGN


def test_decode_grid_barrier_timeout_is_reported_and_the_context_survives():
    """With a wait limit of one clock cycle the decode kernel's grid-barrier
    waits run out (no block waits for the others): the first block to give
    up records the status and raises the abort flag, every block drains its
    own staging copies and returns.  Then a normal call still matches the
    oracle."""
    from int4_grouped_gemm_gb300.moe import DecodeChain
    from moe_helpers import assert_close, oracle_layer
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(1)
    x = L.x[0:1].cuda().contiguous()
    layers = []
    for l in range(3):
        Ll = synthetic.make_layer(cfg, layer=l, with_x=False)
        layers.append(PackedLayer.from_fp32(cfg, Ll.router_w, Ll.router_bias, Ll.w_gate, Ll.w_up, Ll.w_down))
    chain = DecodeChain(layers)
    old = _lib.moe_set_wait_limit(1)
    try:
        layer.decode(x, ws)
        chain.set_input(x)
        chain.step_eager()
        torch.cuda.synchronize()
    finally:
        _lib.moe_set_wait_limit(old)
    for buf in (ws.buf, chain.ws.buf):
        st = _lib.moe_read_device_status(buf)
        assert _lib.MOE_ERR_TIMEOUT - 100 < st <= _lib.MOE_ERR_TIMEOUT, st
    # the context is usable and the kernel is correct again with the normal limit
    y = layer.decode(x, ws)
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), oracle_layer(L, L.x)["y"][0:1], "after the timeout")
    assert _lib.moe_read_device_status(ws.buf) == 0
