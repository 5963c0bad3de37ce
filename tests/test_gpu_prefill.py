"""Prefill parity: the whole MoE layer on the GPU (router, routing tables,
grouped int4 GEMMs with SwiGLU, weighted combine) against the CPU oracle."""
import dataclasses

import numpy as np
import pytest
import torch

from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.moe import PackedLayer

from moe_helpers import (assert_close, check_topk_exact, oracle_layer, oracle_stacks, reference_under_gpu_routing,
                         sample_tokens, x_bits)

pytestmark = pytest.mark.gpu


def run_gpu(L, x):
    cfg = L.cfg
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(x.shape[0])
    y = layer.prefill(x.cuda(), ws)
    torch.cuda.synchronize()
    assert _lib.moe_read_device_status(ws.buf) == 0
    return layer, ws, y.float().cpu().numpy()


def check_layer(L, x, tokens=None):
    """Every listed token: GPU logits within fp32 summation error of the
    oracle's, GPU picks bit-exact (weights within fp32 rounding) of the
    oracle's top-k of those GPU logits, and the output against the oracle
    under that routing (the oracle's own layer wherever its picks agree)."""
    cfg = L.cfg
    T = x.shape[0]
    layer, ws, y = run_gpu(L, x)
    stacks = oracle_stacks(L, cfg.group)
    ref = oracle_layer(L, x, tokens=tokens, stacks=stacks)
    toks = ref["tokens"]
    rt = ws.routing(layer.desc, T)
    g_logits = rt["logits"].cpu().numpy()[toks]
    # logits agree with the oracle's fp32 router up to summation order
    assert np.abs(g_logits - ref["logits"]).max() <= 1e-5 * np.abs(ref["logits"]).max()
    g_idx = rt["topk_idx"].cpu().numpy()[toks]
    g_w = rt["topk_w"].cpu().numpy()[toks]
    idx, w = check_topk_exact(g_logits, g_idx, g_w, cfg.k, what=cfg.name)
    want = reference_under_gpu_routing(ref["y"], ref["idx"], x_bits(x)[toks], stacks, cfg.E, cfg.has_shared, idx, w)
    return assert_close(y[toks], want, cfg.name)


def test_tiny_all_tokens():
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


@pytest.mark.parametrize("T", [1, 3, 17, 100, 300])
def test_tiny_shapes_ragged_T(T):
    cfg = dataclasses.replace(synthetic.CONFIGS["tiny"], T=T, seed=100 + T)
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


def test_mid_shapes_multi_tile_groups():
    """E=8 experts with ~300 rows each and a 600-row shared group: several
    token tiles per group with ragged tails."""
    cfg = synthetic.MoEConfig("mid", T=600, H=512, E=8, k=4, I=128, group=64, seed=7)
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


def test_no_shared_expert():
    cfg = synthetic.MoEConfig("noshared", T=70, H=256, E=16, k=2, I=128, group=32, seed=8, has_shared=False)
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


@pytest.mark.parametrize("cfg", [
    synthetic.MoEConfig("e40_k3", T=150, H=256, E=40, k=3, I=128, group=32, seed=36),
    synthetic.MoEConfig("e200_k8", T=90, H=512, E=200, k=8, I=128, group=64, seed=37),
], ids=lambda c: c.name)
def test_expert_counts_not_a_multiple_of_16(cfg):
    """The router GEMM pads the expert rows to 16 (zero rows) and the top-k
    must never pick a padding column."""
    L = synthetic.make_layer(cfg)
    check_layer(L, L.x)


def test_one_expert_takes_all_tokens_and_empty_experts():
    cfg = synthetic.MoEConfig("skewtiny", T=300, H=256, E=16, k=2, I=128, group=32, seed=9)
    L = synthetic.make_layer(cfg)
    bias = torch.full((cfg.E,), -30.0)
    bias[3] = 30.0          # every token picks expert 3
    bias[5] = 0.0
    bias[11] = 0.0          # the second slot goes to 5 or 11; the rest stay empty
    L.router_bias = bias
    check_layer(L, L.x)


@pytest.mark.parametrize("E,H", [(16, 256), (40, 256), (256, 2048)])
def test_router_split_is_its_definition_and_both_router_paths_agree(E, H):
    """moe_split_router writes hi = bf16(w) and lo = bf16(w - hi) with zero
    padding rows; a layer that carries the split and one that leaves it to
    each call (router_split NULL) give the same logits, picks and weights bit
    for bit, and outputs within one bf16 ulp (the combine's fp32 additions
    land in no fixed order)."""
    cfg = synthetic.MoEConfig(f"split{E}", T=130, H=H, E=E, k=2, I=128, group=64, seed=300 + E)
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    E16 = (E + 15) // 16 * 16
    assert layer.router_split.numel() == _lib.moe_router_split_bytes(E, H) == 2 * E16 * H * 2
    parts = layer.router_split.view(torch.bfloat16).view(2, E16, H).cpu()
    w = L.router_w.float()
    hi = w.to(torch.bfloat16)
    lo = (w - hi.float()).to(torch.bfloat16)
    assert torch.equal(parts[0, :E].view(torch.int16), hi.view(torch.int16))
    assert torch.equal(parts[1, :E].view(torch.int16), lo.view(torch.int16))
    assert not parts[:, E:].view(torch.int16).any()
    x = L.x.cuda()
    ws = layer.workspace(cfg.T)
    y_split = layer.prefill(x, ws).clone()
    rt = {n: v.clone() for n, v in ws.routing(layer.desc, cfg.T).items() if n in ("logits", "topk_idx", "topk_w")}
    d = _lib.moe_layer_desc.from_buffer_copy(layer.desc)
    d.router_split = None
    y_call = torch.empty_like(x)
    _lib.moe_prefill(d, x, cfg.T, y_call, ws.buf)
    torch.cuda.synchronize()
    assert _lib.moe_read_device_status(ws.buf) == 0
    rt2 = ws.routing(layer.desc, cfg.T)
    for n, v in rt.items():
        assert torch.equal(v, rt2[n]), n
    # one bf16 rounding step, plus the fp32 reassociation error of the k + 1
    # terms where they cancel
    a, b = y_split.float(), y_call.float()
    bound = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7 + 1e-5 * b.abs().max()
    assert ((a - b).abs() <= bound).all()


def test_graph_replay_matches_eager():
    """The layer captured in a CUDA graph (its kernels launched as
    programmatic dependents) and replayed twice gives the eager call's
    routing tables bit for bit and its output within one bf16 step (the
    combine's fp32 additions land in no fixed order)."""
    cfg = dataclasses.replace(synthetic.CONFIGS["prefill512"], T=700, seed=91)
    L = synthetic.make_layer(cfg, device="cuda")
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(cfg.T)
    x = L.x.cuda()
    y_eager = layer.prefill(x, ws).clone()
    names = ("logits", "topk_idx", "topk_w", "counts", "offsets", "perm", "tile_sched")
    rt = {n: ws.routing(layer.desc, cfg.T)[n].clone() for n in names}
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _lib.moe_prefill(layer.desc, x, cfg.T, y, ws.buf)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _lib.moe_prefill(layer.desc, x, cfg.T, y, ws.buf)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert _lib.moe_read_device_status(ws.buf) == 0
        rt2 = ws.routing(layer.desc, cfg.T)
        for n in names:
            assert torch.equal(rt[n], rt2[n]), n
        a, b = y.float(), y_eager.float()
        bound = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7 + 1e-5 * b.abs().max()
        assert ((a - b).abs() <= bound).all()


@pytest.mark.parametrize("T", [1, 2, 8])
def test_full_shapes_small_batches(T):
    """The speculative-verify shape: a few tokens through the full-size
    layer (most experts empty, one short tile per touched expert)."""
    cfg = dataclasses.replace(synthetic.CONFIGS["prefill512"], T=T, seed=70 + T)
    L = synthetic.make_layer(cfg, device="cuda")
    check_layer(L, L.x)


@pytest.mark.parametrize("name,n", [("prefill512", 40), ("prefill4096", 40)])
def test_full_size_sampled(name, n):
    cfg = synthetic.CONFIGS[name]
    L = synthetic.make_layer(cfg, device="cuda")
    toks = sample_tokens(cfg.T, n, seed=cfg.seed)
    check_layer(L, L.x, tokens=toks)


@pytest.mark.slow
def test_full_size_skew16384_sampled():
    cfg = synthetic.CONFIGS["skew16384"]
    L = synthetic.make_layer(cfg, device="cuda")
    toks = sample_tokens(cfg.T, 32, seed=cfg.seed)
    check_layer(L, L.x, tokens=toks)


def test_pipelined_host_calls_match_the_oracle():
    """moe_forward_host_stream: five calls on three different inputs (one host
    buffer given twice, as a serving loop may), two device staging sets
    alternating; every output against the oracle, with a decode-sized call
    (T = 1) through the same entry point."""
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer = PackedLayer.from_fp32(cfg, L.router_w, L.router_bias, L.w_gate, L.w_up, L.w_down)
    ws = layer.workspace(cfg.T)
    xs = [synthetic.make_tokens(cfg.H, cfg.T, seed=40 + i) for i in range(3)]
    order = [0, 1, 2, 1, 0]
    x_hosts = [xs[i].clone().pin_memory() for i in order]
    x_hosts[3] = x_hosts[1]  # the same host buffer for two calls
    y_hosts = [torch.empty_like(x).pin_memory() for x in x_hosts]
    x_devs = [torch.empty_like(xs[0], device="cuda") for _ in range(2)]
    y_devs = [torch.empty_like(xs[0], device="cuda") for _ in range(2)]
    _lib.moe_forward_host_stream(layer.desc, x_hosts, cfg.T, y_hosts, x_devs, y_devs, ws.buf)
    refs = [oracle_layer(L, x)["y"] for x in xs]
    for c, i in enumerate(order):
        assert_close(y_hosts[c].float().numpy(), refs[i], f"call {c}")
    # T = 1 goes to the decode kernel
    one = [x[0:1].clone().pin_memory() for x in xs]
    outs = [torch.empty_like(o).pin_memory() for o in one]
    x1 = [torch.empty_like(xs[0][0:1], device="cuda") for _ in range(2)]
    y1 = [torch.empty_like(xs[0][0:1], device="cuda") for _ in range(2)]
    _lib.moe_forward_host_stream(layer.desc, one, 1, outs, x1, y1, ws.buf)
    for i in range(3):
        assert_close(outs[i].float().numpy(), refs[i][0:1], f"decode call {i}")
    assert _lib.moe_read_device_status(ws.buf) == 0


def test_host_buffers_end_to_end_equals_device_path():
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    layer, ws, y_dev = run_gpu(L, L.x)
    x_host = L.x.clone().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    xd = torch.empty_like(L.x, device="cuda")
    yd = torch.empty_like(xd)
    _lib.moe_forward_host(layer.desc, x_host, cfg.T, y_host, xd, yd, ws.buf)
    got = y_host.float().numpy()
    # the weighted combine adds fp32 partial sums with reductions whose order
    # is not fixed: two runs may differ by one bf16 rounding step (at most
    # 2^-7 of the value) plus the fp32 reassociation error of a sum of k+1
    # terms, which matters only where the terms cancel (1e-5 of the scale)
    bound = 2.0 ** -7 * np.maximum(np.abs(got), np.abs(y_dev)) + 1e-5 * np.abs(y_dev).max()
    assert np.all(np.abs(got - y_dev) <= bound)
    ref = oracle_layer(L, L.x)
    assert_close(got, ref["y"], "host buffers")
