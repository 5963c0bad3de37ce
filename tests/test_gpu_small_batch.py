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

from moe_helpers import ambiguous, assert_close, oracle_layer, oracle_stacks, x_bits

pytestmark = pytest.mark.gpu

MID = synthetic.MoEConfig("sbmid", T=8, H=512, E=24, k=4, I=128, group=64, seed=61)
NOSHARED = synthetic.MoEConfig("sbnoshared", T=8, H=512, E=40, k=6, I=256, group=32, seed=62, has_shared=False)
ODD = synthetic.MoEConfig("sbodd", T=8, H=256, E=33, k=3, I=128, group=64, seed=63, bias="normal")
WIDE = synthetic.MoEConfig("sbwide", T=8, H=4096, E=8, k=8, I=1024, group=32, seed=64)


def _packed(L, **kw):
    cfg = L.cfg
    return PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down, **kw)


def _check_rows(y, ref, what):
    """Compare the tokens whose top-k set is not ambiguous (nearly tied k-th
    and (k+1)-th oracle logits may route the other way in fp32)."""
    cfg_k, E = ref["k"], ref["E"]
    ok = ~ambiguous(ref["logits"], cfg_k, E)
    assert ok.any()
    assert_close(y.float().cpu().numpy()[ok], ref["y"][ok], what)


def _oracle_full(L, x):
    r = oracle_layer(L, x)
    r["k"], r["E"] = L.cfg.k, L.cfg.E
    return r


@pytest.mark.parametrize("cfg", [synthetic.CONFIGS["tiny"], MID, NOSHARED, ODD], ids=lambda c: c.name)
def test_every_batch_size(cfg):
    L = synthetic.make_layer(cfg, T=8)
    layer = _packed(L)
    ws = layer.workspace(1)
    x = L.x.cuda()
    for B in range(1, 9):
        xb = x[:B].contiguous()
        y = layer.decode_batch(xb, ws)
        torch.cuda.synchronize()
        _check_rows(y, _oracle_full(L, L.x[:B]), f"{cfg.name} B={B}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def _oracle_union(L, x):
    """Oracle for a few tokens of a full-size layer: the oracle's own logits
    and top-k, then only the experts in the union of the picks (and the
    shared expert) quantised and evaluated."""
    cfg = L.cfg
    xb = x_bits(x)
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    logits = oracle.router_logits(xb, L.router_w.cpu().numpy(), bias)
    idx, w = oracle.topk(logits, cfg.k)
    union = sorted(set(int(e) for e in idx.ravel()))
    pos = {e: i for i, e in enumerate(union)}
    sel = torch.tensor(union + [cfg.E], device=L.w_gate.device)
    gate = oracle.quantize_stack(L.w_gate[sel].cpu().numpy(), cfg.group)
    up = oracle.quantize_stack(L.w_up[sel].cpu().numpy(), cfg.group)
    down = oracle.quantize_stack(L.w_down[sel].cpu().numpy(), cfg.group)
    local = np.vectorize(pos.get)(idx).astype(np.int32)
    y = oracle.experts_given_routing(xb, gate, up, down, len(union), True, local, w)
    return {"y": y, "logits": logits, "k": cfg.k, "E": cfg.E, "union": len(union)}


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
    ref = _oracle_union(L, x)
    assert ref["union"] > L.cfg.k  # the tokens pick different experts
    _check_rows(y, ref, f"decode40 layer B={B}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_one_token_agrees_with_decode_and_batch_with_prefill(full_layer):
    L, layer = full_layer
    ws = layer.workspace(8)
    x = synthetic.make_tokens(L.cfg.H, 8, seed=97).cuda()
    ref = _oracle_union(L, x.cpu())
    ok = ~ambiguous(ref["logits"], L.cfg.k, L.cfg.E)
    y1 = layer.decode_batch(x[:1].contiguous(), ws)
    yd = layer.decode(x[:1].contiguous(), ws)
    yb = layer.decode_batch(x, ws)
    yp = layer.prefill(x, ws)
    torch.cuda.synchronize()
    if ok[0]:
        assert_close(y1.float().cpu().numpy(), yd.float().cpu().numpy(), "B=1 vs moe_decode")
    assert_close(yb.float().cpu().numpy()[ok], yp.float().cpu().numpy()[ok], "batch vs prefill")
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
    _check_rows(a[:1], _oracle_full(L, L.x), "repeated token")


def test_wide_hidden_and_expert_group32():
    L = synthetic.make_layer(WIDE, T=8)
    layer = _packed(L)
    ws = layer.workspace(1)
    for B in (3, 8):
        y = layer.decode_batch(L.x[:B].cuda().contiguous(), ws)
        torch.cuda.synchronize()
        _check_rows(y, _oracle_full(L, L.x[:B]), f"wide B={B}")


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
    ref = oracle.moe_layer(x_bits(L.x), L.router_w.cpu().numpy(), bias, *oracle_stacks(L, cfg.group), cfg.E, cfg.k,
                           cfg.has_shared, renorm=not no_renorm,
                           shared_gate_w=None if sg is None else sg.numpy())
    ref["k"], ref["E"] = cfg.k, cfg.E
    _check_rows(y, ref, f"variant no_renorm={no_renorm} gated={gated}")
