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
