"""Parity at shapes the benchmark does not exercise: the widest hidden size
the decode kernel serves (4096, its second register-tile instance), a wide
expert (I = 1024: longer down rows), both at once with k = 8 (the decode
kernel's register fallback for the gate/up rows), group 32 along a long K,
and decode stacks longer than one kernel launch (more than 64 layers)."""
import pytest
import torch

from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import DecodeChain, PackedLayer

from moe_helpers import assert_close, oracle_layer
from test_gpu_prefill import check_layer

pytestmark = pytest.mark.gpu

WIDE_H = synthetic.MoEConfig("wideH", T=300, H=4096, E=8, k=2, I=256, group=32, seed=21)
WIDE_I = synthetic.MoEConfig("wideI", T=200, H=512, E=8, k=2, I=1024, group=64, seed=22)
# widest hidden and expert sizes with k = 8: the decode kernel's gate/up rows
# no longer fit in shared memory (they go through registers) and its down rows
# are wider than one 16-element span per lane
WIDE_HI = synthetic.MoEConfig("wideHI", T=6, H=4096, E=8, k=8, I=1024, group=64, seed=23)


@pytest.mark.parametrize("cfg", [WIDE_H, WIDE_I], ids=lambda c: c.name)
def test_prefill_wide_shapes(cfg):
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


@pytest.mark.parametrize("cfg", [WIDE_H, WIDE_I, WIDE_HI], ids=lambda c: c.name)
def test_decode_wide_shapes(cfg):
    L = synthetic.make_layer(cfg, T=6)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(1)
    ref = oracle_layer(L, L.x)
    for t in range(L.x.shape[0]):
        y = layer.decode(L.x[t:t + 1].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy(), ref["y"][t:t + 1], f"{cfg.name} token {t}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_decode_stack_longer_than_one_launch():
    """70 layers: the stack runs as two kernel launches (64 + 6 layers); its
    output equals running the layers one moe_decode call at a time."""
    cfg = synthetic.CONFIGS["tiny"]
    layers = []
    for l in range(70):
        L = synthetic.make_layer(cfg, layer=l, with_x=False)
        layers.append(PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down))
    chain = DecodeChain(layers)
    x0 = synthetic.make_tokens(cfg.H, 1, seed=77).cuda() * 4  # keeps the chain away from 0 for longer
    eager = chain.layer_outputs_eager(x0)
    chain.set_input(x0)
    chain.step_eager()
    torch.cuda.synchronize()
    assert torch.equal(chain.output(), eager[-1])
    assert _lib.moe_read_device_status(chain.ws.buf) == 0
