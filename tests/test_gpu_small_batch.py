"""Small-batch decode (moe_decode_batch, 1 to 8 tokens) against the CPU
oracle: every batch size on small layers, the full-size layer with the
oracle on the union of the touched experts, the routing variants, layers
without a shared expert, the widest hidden size, group 32, and agreement
with moe_decode (B = 1) and moe_prefill on the same tokens."""
import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import PackedLayer

from moe_helpers import assert_close, batch_routing, oracle_layer, oracle_stacks, reference_under_gpu_routing, x_bits

pytestmark = pytest.mark.gpu

MID = synthetic.MoEConfig("sbmid", T=8, H=512, E=24, k=4, I=128, group=64, seed=61)
NOSHARED = synthetic.MoEConfig("sbnoshared", T=8, H=512, E=40, k=6, I=256, group=32, seed=62, has_shared=False)
ODD = synthetic.MoEConfig("sbodd", T=8, H=256, E=33, k=3, I=128, group=64, seed=63, bias="normal")
WIDE = synthetic.MoEConfig("sbwide", T=8, H=4096, E=8, k=8, I=1024, group=32, seed=64)


def _packed(L, **kw):
    cfg = L.cfg
    return PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down, **kw)


def _check_rows(y, ref, what, layer, ws, renorm=True, gated=False):
    """Routing checked exactly against the GPU's logits, then every token's
    output against the oracle under that routing."""
    B = y.shape[0]
    idx, w = batch_routing(layer, ws, B, renorm, gated)
    want = reference_under_gpu_routing(ref["y"], ref["idx"], ref["xb"], ref["stacks"], ref["E"], ref["has_shared"],
                                       idx, w, shared_w=ref.get("shared_w"))
    assert_close(y.float().cpu().numpy(), want, what)


def _oracle_full(L, x, stacks=None):
    stacks = stacks if stacks is not None else oracle_stacks(L, L.cfg.group)
    r = oracle_layer(L, x, stacks=stacks)
    r.update(k=L.cfg.k, E=L.cfg.E, has_shared=L.cfg.has_shared, stacks=stacks, xb=x_bits(x))
    return r


@pytest.mark.parametrize("cfg", [synthetic.CONFIGS["tiny"], MID, NOSHARED, ODD], ids=lambda c: c.name)
def test_every_batch_size(cfg):
    L = synthetic.make_layer(cfg, T=8)
    layer = _packed(L)
    ws = layer.workspace(1)
    x = L.x.cuda()
    stacks = oracle_stacks(L, cfg.group)
    for B in range(1, 9):
        xb = x[:B].contiguous()
        y = layer.decode_batch(xb, ws)
        torch.cuda.synchronize()
        _check_rows(y, _oracle_full(L, L.x[:B], stacks), f"{cfg.name} B={B}", layer, ws)
    assert _lib.moe_read_device_status(ws.buf) == 0


def _oracle_union(L, x, gpu_idx=None):
    """Oracle for a few tokens of a full-size layer: the oracle's own logits
    and top-k, then only the experts in the union of the picks (and of the
    GPU's picks, when given; plus the shared expert) quantised and
    evaluated.  Expert indices in the result are local to that union."""
    cfg = L.cfg
    xb = x_bits(x)
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    logits = oracle.router_logits(xb, L.router_w.cpu().numpy(), bias)
    idx, w = oracle.topk(logits, cfg.k)
    picked = set(int(e) for e in idx.ravel())
    union = sorted(picked | (set(int(e) for e in gpu_idx.ravel()) if gpu_idx is not None else set()))
    pos = {e: i for i, e in enumerate(union)}
    sel = torch.tensor(union + [cfg.E], device=L.w_gate.device)
    gate = oracle.quantize_stack(L.w_gate[sel].cpu().numpy(), cfg.group)
    up = oracle.quantize_stack(L.w_up[sel].cpu().numpy(), cfg.group)
    down = oracle.quantize_stack(L.w_down[sel].cpu().numpy(), cfg.group)
    local = np.vectorize(pos.get)(idx).astype(np.int32)
    y = oracle.experts_given_routing(xb, gate, up, down, len(union), True, local, w)
    return {"y": y, "logits": logits, "idx": local, "k": cfg.k, "E": len(union), "has_shared": True,
            "stacks": (gate, up, down), "xb": xb, "union": len(picked), "local": pos}


def _check_union(y, L, x, layer, ws, what):
    """_check_rows for a full-size layer with the oracle on the union of the
    oracle's and the GPU's picks (GPU routing mapped into that union)."""
    B = y.shape[0]
    idx, w = batch_routing(layer, ws, B)
    ref = _oracle_union(L, x, gpu_idx=idx)
    local = np.vectorize(ref["local"].get)(idx).astype(np.int32)
    want = reference_under_gpu_routing(ref["y"], ref["idx"], ref["xb"], ref["stacks"], ref["E"], True, local, w)
    assert_close(y.float().cpu().numpy(), want, what)
    return ref


@pytest.fixture(scope="module")
def full_layer():
    cfg = synthetic.CONFIGS["decode40"]
    L = synthetic.make_layer(cfg, layer=7, device="cuda", with_x=False)
    return L, _packed(L)


@pytest.mark.parametrize("B", [2, 5, 8])
def test_full_size_layer(full_layer, B):
    L, layer = full_layer
    ws = layer.workspace(1)
    x = synthetic.make_tokens(L.cfg.H, B, seed=90 + B)
    y = layer.decode_batch(x.cuda().contiguous(), ws)
    torch.cuda.synchronize()
    ref = _check_union(y, L, x, layer, ws, f"decode40 layer B={B}")
    assert ref["union"] > L.cfg.k  # the tokens pick different experts
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_one_token_agrees_with_decode_and_batch_with_prefill(full_layer):
    L, layer = full_layer
    ws = layer.workspace(8)
    x = synthetic.make_tokens(L.cfg.H, 8, seed=97).cuda()
    y1 = layer.decode_batch(x[:1].contiguous(), ws)
    g1 = batch_routing(layer, ws, 1)[0]
    yd = layer.decode(x[:1].contiguous(), ws)
    yb = layer.decode_batch(x, ws)
    gb = batch_routing(layer, ws, 8)[0]
    yp = layer.prefill(x, ws)
    torch.cuda.synchronize()
    gp = ws.routing(layer.desc, 8)["topk_idx"].cpu().numpy()
    # where both paths' routings agree (no near tie decided differently by
    # their fp32 summation orders) the outputs agree within the tolerance
    if np.array_equal(g1[0], gb[0]):
        assert_close(y1.float().cpu().numpy(), yd.float().cpu().numpy(), "B=1 vs moe_decode")
    same = np.all(np.sort(gb, axis=1) == np.sort(gp, axis=1), axis=1)
    assert same.mean() >= 0.75
    assert_close(yb.float().cpu().numpy()[same], yp.float().cpu().numpy()[same], "batch vs prefill")
    # a token's row does not depend on the other tokens of the batch beyond
    # the fp32 order of the slot sums (slots are grouped by the batch's union)
    np.testing.assert_allclose(yb[:1].float().cpu().numpy(), y1.float().cpu().numpy(), rtol=1e-2, atol=1e-4)


def test_same_token_repeated_and_repeat_calls_are_identical():
    cfg = MID
    L = synthetic.make_layer(cfg, T=1)
    layer = _packed(L)
    ws = layer.workspace(1)
    x = L.x.cuda().repeat(8, 1).contiguous()
    a = layer.decode_batch(x, ws)
    b = layer.decode_batch(x, ws)
    torch.cuda.synchronize()
    for t in range(8):
        assert torch.equal(a[t], a[0])
    assert torch.equal(a, b)
    _check_rows(b, _oracle_full(L, L.x.repeat(8, 1)), "repeated token", layer, ws)


def test_wide_hidden_and_expert_group32():
    L = synthetic.make_layer(WIDE, T=8)
    layer = _packed(L)
    ws = layer.workspace(1)
    stacks = oracle_stacks(L, WIDE.group)
    for B in (3, 8):
        y = layer.decode_batch(L.x[:B].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        _check_rows(y, _oracle_full(L, L.x[:B], stacks), f"wide B={B}", layer, ws)


@pytest.mark.parametrize("no_renorm,gated", [(True, False), (False, True), (True, True)],
                         ids=["no_renorm", "gated", "both"])
def test_routing_variants(no_renorm, gated):
    cfg = MID
    L = synthetic.make_layer(cfg, T=8)
    sg = torch.randn(cfg.H, generator=torch.Generator().manual_seed(65)) * 0.05 if gated else None
    layer = _packed(L, no_renorm=no_renorm, shared_gate=sg)
    ws = layer.workspace(1)
    y = layer.decode_batch(L.x.cuda(), ws)
    torch.cuda.synchronize()
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    stacks = oracle_stacks(L, cfg.group)
    ref = oracle.moe_layer(x_bits(L.x), L.router_w.cpu().numpy(), bias, *stacks, cfg.E, cfg.k,
                           cfg.has_shared, renorm=not no_renorm,
                           shared_gate_w=None if sg is None else sg.numpy())
    ref.update(k=cfg.k, E=cfg.E, has_shared=cfg.has_shared, stacks=stacks, xb=x_bits(L.x))
    _check_rows(y, ref, f"variant no_renorm={no_renorm} gated={gated}", layer, ws, renorm=not no_renorm,
                gated=gated)
