"""Batch-1 decode parity: dequant-GEMV path against the CPU oracle, per layer
and through the 40-layer CUDA-graph chain that the benchmark replays."""
import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import DecodeChain, PackedLayer

from moe_helpers import assert_close, oracle_layer, x_bits

pytestmark = pytest.mark.gpu


def _packed(cfg, l, device="cuda"):
    L = synthetic.make_layer(cfg, layer=l, device=device, with_x=False)
    return L, PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)


def _oracle_touched(L, xb: np.ndarray, cfg):
    """Oracle for one token: route with the oracle's own logits, then quantise
    only the touched experts (oracle quantiser) and evaluate them."""
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    logits = oracle.router_logits(xb, L.router_w.cpu().numpy(), bias)
    idx, w = oracle.topk(logits, cfg.k)
    sel = torch.tensor([int(e) for e in idx[0]] + [cfg.E], device=L.w_gate.device)
    gate = oracle.quantize_stack(L.w_gate[sel].cpu().numpy(), cfg.group)
    up = oracle.quantize_stack(L.w_up[sel].cpu().numpy(), cfg.group)
    down = oracle.quantize_stack(L.w_down[sel].cpu().numpy(), cfg.group)
    local = np.arange(cfg.k, dtype=np.int32)[None, :]
    return oracle.experts_given_routing(xb, gate, up, down, cfg.k, True, local, w)


def test_tiny_decode_tokens():
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(1)
    ref = oracle_layer(L, L.x)
    for t in range(cfg.T):
        y = layer.decode(L.x[t:t + 1].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy(), ref["y"][t:t + 1], f"token {t}")
    assert _lib.moe_read_device_status(ws.buf) == 0


@pytest.fixture(scope="module")
def chain40():
    cfg = synthetic.CONFIGS["decode40"]
    layers = [_packed(cfg, l)[1] for l in range(cfg.layers)]
    torch.cuda.empty_cache()
    return cfg, DecodeChain(layers)


def test_every_layer_fresh_token(chain40):
    """All 40 layers of the decode stack, each on its own fresh token."""
    cfg, chain = chain40
    x = synthetic.make_tokens(cfg.H, cfg.layers, seed=33)
    for l in range(cfg.layers):
        L = synthetic.make_layer(cfg, layer=l, device="cuda", with_x=False)
        y = chain.layers[l].decode(x[l:l + 1].cuda().contiguous(), chain.ws)
        torch.cuda.synchronize()
        ref = _oracle_touched(L, x_bits(x[l:l + 1]), cfg)
        assert_close(y.float().cpu().numpy(), ref, f"layer {l}")
        del L
    assert _lib.moe_read_device_status(chain.ws.buf) == 0


def test_graph_step_equals_eager_and_first_layers_match_oracle(chain40):
    """The bench's decode step (40 layers through moe_decode_layers, captured
    in a CUDA graph) equals the layers run one call at a time, and the first
    two layers match the oracle chain."""
    cfg, chain = chain40
    x0 = synthetic.make_tokens(cfg.H, 1, seed=cfg.seed).cuda()
    eager = chain.layer_outputs_eager(x0)
    chain.set_input(x0)
    chain.step()                      # captures on first use, then replays
    torch.cuda.synchronize()
    assert torch.equal(chain.output(), eager[-1])
    chain.set_input(x0)
    chain.step()
    torch.cuda.synchronize()
    assert torch.equal(chain.output(), eager[-1]), "graph replay != eager"
    assert _lib.moe_read_device_status(chain.ws.buf) == 0
    # layers 0 and 1 against the oracle chain (relative errors roughly double
    # per layer through the quadratic SwiGLU, so deeper layers are checked on
    # fresh tokens instead)
    xb = x_bits(x0.cpu())
    for l in range(2):
        L = synthetic.make_layer(cfg, layer=l, device="cuda", with_x=False)
        ref = _oracle_touched(L, xb, cfg)
        assert_close(eager[l].float().cpu().numpy(), ref, f"chain layer {l}")
        xb = oracle.bf16_round(ref.astype(np.float32))


# Routing shapes of the decode kernel beyond the benchmark's: no shared expert
# (8 slots, not 9), a single pick, and expert counts that fill the top-k
# kernel's 32-key warps only partly (padding keys must never be picked).
DECODE_SHAPES = [
    synthetic.MoEConfig("dec_noshared", T=5, H=256, E=16, k=2, I=128, group=32, seed=31, has_shared=False),
    synthetic.MoEConfig("dec_k1", T=5, H=512, E=8, k=1, I=256, group=64, seed=32),
    synthetic.MoEConfig("dec_e40_k3", T=5, H=256, E=40, k=3, I=128, group=32, seed=33),
    synthetic.MoEConfig("dec_e200_k8_noshared", T=4, H=512, E=200, k=8, I=128, group=64, seed=34,
                        has_shared=False),
]


@pytest.mark.parametrize("cfg", DECODE_SHAPES, ids=lambda c: c.name)
def test_decode_routing_shapes(cfg):
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(1)
    ref = oracle_layer(L, L.x)
    for t in range(cfg.T):
        y = layer.decode(L.x[t:t + 1].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy(), ref["y"][t:t + 1], f"{cfg.name} token {t}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_decode_stack_without_shared_expert():
    """A 3-layer stack of the no-shared shape: one launch runs all three and
    equals three single-layer calls."""
    cfg = DECODE_SHAPES[0]
    layers = []
    for l in range(3):
        L = synthetic.make_layer(cfg, layer=l, with_x=False)
        layers.append(PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down))
    chain = DecodeChain(layers)
    x0 = synthetic.make_tokens(cfg.H, 1, seed=35).cuda() * 4
    eager = chain.layer_outputs_eager(x0)
    chain.set_input(x0)
    chain.step_eager()
    torch.cuda.synchronize()
    assert torch.equal(chain.output(), eager[-1])
    assert _lib.moe_read_device_status(chain.ws.buf) == 0
