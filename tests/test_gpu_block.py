"""The layer inside a pre-norm decoder block (moe_prefill_block,
moe_decode_batch_block) against the oracle's moe_block: h = attn + residual,
x = RMSNorm(h) * w as the layer's input, out = bf16(MoE(x) + h).  With a
small residual stream the layer dominates the output and the usual
tolerance checks the whole chain; at full scale the output is compared
within bf16 rounding of h plus the layer's tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import PackedLayer

from moe_helpers import (assert_close, batch_routing, check_topk_exact, oracle_stacks, reference_under_gpu_routing,
                         x_bits)

pytestmark = pytest.mark.gpu

MID = synthetic.MoEConfig("blkmid", T=200, H=512, E=24, k=4, I=128, group=64, seed=71)


def _inputs(cfg, T, scale, seed):
    g = torch.Generator().manual_seed(seed)
    attn = (torch.randn(T, cfg.H, generator=g) * scale).to(torch.bfloat16)
    resid = (torch.randn(T, cfg.H, generator=g) * scale).to(torch.bfloat16)
    w = (torch.rand(cfg.H, generator=g) + 0.5).float()
    return attn, resid, w


def _oracle(L, attn, resid, w, eps, stacks=None):
    cfg = L.cfg
    gate, up, down = stacks if stacks is not None else oracle_stacks(L, cfg.group)
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    return oracle.moe_block(x_bits(attn), x_bits(resid), w.numpy(), eps, L.router_w.cpu().numpy(), bias, gate, up,
                            down, cfg.E, cfg.k, cfg.has_shared)


def _floats(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _check_intermediates(layer, ws, T, small_batch, ref, what):
    """The residual stream h in the workspace equals the oracle's bit for bit
    (one fp32 add, one rounding), and the normalised input x is within one
    bf16 ulp of it (fp32 against fp64 statistics)."""
    hoff, xoff = _lib.moe_block_views_for(layer.desc, T, small_batch)
    H = layer.desc.H
    gh = ws.view(hoff, torch.int16, T * H).view(T, H).cpu().numpy().view(np.uint16)
    gx = ws.view(xoff, torch.int16, T * H).view(T, H).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(gh, ref["h"], err_msg=f"{what}: residual stream h")
    a, b = _floats(gx), _floats(ref["x"])
    mag = np.maximum(np.abs(a), np.abs(b))
    ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7), 0.0)
    assert np.all(np.abs(a - b) <= ulp), f"{what}: normalised input x beyond one bf16 ulp"


def _check(out, ref, cfg, what, small, idx, w, stacks):
    """Output against the oracle's block under the GPU's routing (the
    oracle's own layer where the picks agree)."""
    got = out.float().cpu().numpy()
    y = reference_under_gpu_routing(ref["y"], ref["idx"], ref["x"], stacks, cfg.E, cfg.has_shared, idx, w)
    want = _floats(oracle.residual_out(ref["h"], y))
    if small:
        assert_close(got, want, what)
    else:
        # both sides round h + y once to bf16: allow two ulps of the result
        # (2^-6 of its magnitude at most) on top of the layer's own tolerance
        h = _floats(ref["h"])
        bound = 2.0 ** -6 * np.abs(want) + 2e-2 * np.abs(want - h).max()
        err = np.abs(got - want)
        assert (err <= bound).all(), f"{what}: max excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("cfg", [synthetic.CONFIGS["tiny"], MID], ids=lambda c: c.name)
@pytest.mark.parametrize("scale", [0.01, 1.0], ids=["small_stream", "unit_stream"])
def test_prefill_block(cfg, scale):
    L = synthetic.make_layer(cfg, with_x=False)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    attn, resid, w = _inputs(cfg, cfg.T, scale, seed=cfg.seed + 5)
    ws = layer.workspace(cfg.T)
    out = layer.prefill_block(attn.cuda(), resid.cuda(), w.cuda(), ws, eps=1e-6)
    torch.cuda.synchronize()
    assert _lib.moe_read_device_status(ws.buf) == 0
    stacks = oracle_stacks(L, cfg.group)
    ref = _oracle(L, attn, resid, w, 1e-6, stacks)
    what = f"prefill block {cfg.name}"
    _check_intermediates(layer, ws, cfg.T, False, ref, what)
    rt = ws.routing(layer.desc, cfg.T)
    idx, wt = check_topk_exact(rt["logits"].cpu().numpy(), rt["topk_idx"].cpu().numpy(),
                               rt["topk_w"].cpu().numpy(), cfg.k, what=what)
    _check(out, ref, cfg, what, scale < 0.1, idx, wt, stacks)


@pytest.mark.parametrize("scale", [0.01, 1.0], ids=["small_stream", "unit_stream"])
def test_decode_batch_block_every_size(scale):
    cfg = MID
    L = synthetic.make_layer(cfg, with_x=False)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    attn, resid, w = _inputs(cfg, 8, scale, seed=81)
    ws = layer.workspace(1)
    stacks = oracle_stacks(L, cfg.group)
    for B in range(1, 9):
        out = layer.decode_batch_block(attn[:B].cuda(), resid[:B].cuda(), w.cuda(), ws, eps=1e-5)
        torch.cuda.synchronize()
        ref = _oracle(L, attn[:B], resid[:B], w, 1e-5, stacks)
        what = f"batch block B={B}"
        _check_intermediates(layer, ws, B, True, ref, what)
        idx, wt = batch_routing(layer, ws, B)
        _check(out, ref, cfg, what, scale < 0.1, idx, wt, stacks)


def test_block_in_place_and_full_size_small_batch():
    """Full-size layer, 8 tokens through the small-batch block form, output
    written over attn; the oracle evaluates only the experts the tokens pick."""
    cfg = synthetic.CONFIGS["decode40"]
    L = synthetic.make_layer(cfg, layer=11, device="cuda", with_x=False)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    attn, resid, w = _inputs(cfg, 8, 0.01, seed=83)
    ws = layer.workspace(1)
    buf = attn.cuda().contiguous()
    want_gpu = layer.decode_batch_block(buf, resid.cuda(), w.cuda(), ws)
    layer.decode_batch_block(buf, resid.cuda(), w.cuda(), ws, out=buf)
    torch.cuda.synchronize()
    assert torch.equal(buf, want_gpu)  # deterministic, and in place reads attn before writing
    g_idx, g_w = batch_routing(layer, ws, 8)
    # oracle on the union of the oracle's and the GPU's picks
    h, x = oracle.residual_rmsnorm(x_bits(attn), x_bits(resid), w.numpy(), 1e-6)
    _check_intermediates(layer, ws, 8, True, {"h": h, "x": x}, "full-size batch block")
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    logits = oracle.router_logits(x, L.router_w.cpu().numpy(), bias)
    idx, wt = oracle.topk(logits, cfg.k)
    union = sorted(set(int(e) for e in idx.ravel()) | set(int(e) for e in g_idx.ravel()))
    pos = {e: i for i, e in enumerate(union)}
    sel = torch.tensor(union + [cfg.E], device=L.w_gate.device)
    stacks = [oracle.quantize_stack(m[sel].cpu().numpy(), cfg.group) for m in (L.w_gate, L.w_up, L.w_down)]
    local = np.vectorize(pos.get)(idx).astype(np.int32)
    y = oracle.experts_given_routing(x, *stacks, len(union), True, local, wt)
    sub = dataclasses.replace(cfg, E=len(union))
    ref = {"y": y, "idx": local, "h": h, "x": x}
    _check(buf, ref, sub, "full-size batch block", True, np.vectorize(pos.get)(g_idx).astype(np.int32), g_w, stacks)
