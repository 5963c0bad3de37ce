"""Routing variants of the layer on the GPU against the oracle: picked
weights without renormalisation, and a shared expert gated per token by
sigmoid(x . g), in prefill (routing kernel + combine) and in decode (the
persistent kernel's top-k, its first-layer router phase and the next-layer
score sums of a stack)."""
import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import DecodeChain, PackedLayer

from moe_helpers import assert_close, check_topk_exact, oracle_stacks, reference_under_gpu_routing, x_bits

pytestmark = pytest.mark.gpu

VARIANTS = [(True, False), (False, True), (True, True)]  # (no_renorm, gated)


def _gate_vec(H, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(H, generator=g) * 0.05


def _oracle(L, x, stacks, no_renorm, sg):
    cfg = L.cfg
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    return oracle.moe_layer(x_bits(x), L.router_w.cpu().numpy(), bias, *stacks, cfg.E, cfg.k, cfg.has_shared,
                            renorm=not no_renorm, shared_gate_w=None if sg is None else sg.numpy())


def _layer(L, no_renorm, sg):
    cfg = L.cfg
    return PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down, no_renorm=no_renorm,
                                 shared_gate=sg)


@pytest.mark.parametrize("no_renorm,gated", VARIANTS, ids=["no_renorm", "gated", "both"])
def test_prefill_variants(no_renorm, gated):
    cfg = synthetic.MoEConfig("variants", T=200, H=512, E=24, k=4, I=128, group=64, seed=51)
    L = synthetic.make_layer(cfg)
    sg = _gate_vec(cfg.H, 52) if gated else None
    layer = _layer(L, no_renorm, sg)
    ws = layer.workspace(cfg.T)
    y = layer.prefill(L.x.cuda(), ws)
    torch.cuda.synchronize()
    assert _lib.moe_read_device_status(ws.buf) == 0
    stacks = oracle_stacks(L, cfg.group)
    ref = _oracle(L, L.x, stacks, no_renorm, sg)
    rt = ws.routing(layer.desc, cfg.T)
    g_logits = rt["logits"].cpu().numpy()
    g_idx = rt["topk_idx"].cpu().numpy()
    g_w = rt["topk_w"].cpu().numpy()
    assert np.abs(g_logits - ref["logits"]).max() <= 1e-5 * np.abs(ref["logits"]).max()
    # picks bit-exact and weights (renormalised or not) of the GPU's own logits
    idx, w = check_topk_exact(g_logits, g_idx, g_w, cfg.k, renorm=not no_renorm, what="prefill variant")
    if no_renorm:
        assert np.all(g_w.sum(axis=1) < 1.0)
    want = reference_under_gpu_routing(ref["y"], ref["idx"], x_bits(L.x), stacks, cfg.E, cfg.has_shared, idx, w,
                                       shared_w=ref["shared_w"])
    assert_close(y.float().cpu().numpy(), want, f"prefill no_renorm={no_renorm} gated={gated}")


@pytest.mark.parametrize("no_renorm,gated", VARIANTS, ids=["no_renorm", "gated", "both"])
def test_decode_variants(no_renorm, gated):
    cfg = synthetic.MoEConfig("variants_dec", T=5, H=512, E=24, k=4, I=128, group=64, seed=53)
    L = synthetic.make_layer(cfg)
    sg = _gate_vec(cfg.H, 54) if gated else None
    layer = _layer(L, no_renorm, sg)
    ws = layer.workspace(1)
    ref = _oracle(L, L.x, oracle_stacks(L, cfg.group), no_renorm, sg)
    for t in range(cfg.T):
        y = layer.decode(L.x[t:t + 1].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy(), ref["y"][t:t + 1], f"decode token {t}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_decode_stack_of_gated_layers():
    """A 4-layer stack in one launch, gated layers with no renormalisation:
    the gate scores of layers 2-4 come from the previous layer's blocks
    (fp64 sums of partials), which must equal layer-by-layer calls, whose
    gate score comes from the first-layer router phase; layer 3 is ungated."""
    cfg = synthetic.MoEConfig("variants_stack", T=1, H=512, E=24, k=4, I=128, group=64, seed=55)
    layers = []
    for l in range(4):
        Ll = synthetic.make_layer(cfg, layer=l, with_x=False)
        sg = None if l == 2 else _gate_vec(cfg.H, 60 + l)
        layers.append(_layer(Ll, True, sg))
    chain = DecodeChain(layers)
    x0 = synthetic.make_tokens(cfg.H, 1, seed=56).cuda() * 4
    eager = chain.layer_outputs_eager(x0)
    chain.set_input(x0)
    chain.step_eager()
    torch.cuda.synchronize()
    # the stack sums the next layer's scores in another order than one layer's
    # router phase: compare within the output tolerance, not bit for bit
    assert_close(chain.output().float().cpu().numpy(), eager[-1].float().cpu().numpy(), "gated stack")
    assert _lib.moe_read_device_status(chain.ws.buf) == 0


def test_variant_arguments_rejected_on_the_host():
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = _layer(L, False, None)
    ws = layer.workspace(cfg.T)
    d = layer.desc
    d.no_renorm = 2
    x = L.x.cuda()
    assert _lib.moe_workspace_bytes(d, cfg.T) == 0
    with pytest.raises(_lib.MoEError) as e:
        _lib.moe_prefill(d, x, cfg.T, torch.empty_like(x), ws.buf)
    assert e.value.code == _lib.MOE_ERR_SHAPE
    d.no_renorm = 0
    g = torch.zeros(cfg.H + 4, device="cuda")
    d.shared_gate = g.data_ptr() + 4  # misaligned
    with pytest.raises(_lib.MoEError) as e:
        _lib.moe_prefill(d, x, cfg.T, torch.empty_like(x), ws.buf)
    assert e.value.code == _lib.MOE_ERR_ALIGN
