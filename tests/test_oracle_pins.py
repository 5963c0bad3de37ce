"""Pins for the CPU oracle: each check compares it with something other than
itself (hand-worked examples, library routines, brute force, closed forms and
invariants), so that a dropped term, a wrong index, sign or tie-break, or a
transposed operand in the oracle fails at least one of them."""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from int4_grouped_gemm_gb300 import synthetic


def _fx(fixture_loader, name):
    return fixture_loader(name)


# ------------------------------------------------------------------ bf16


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(11)
    vals = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 10)
    edge = torch.tensor([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40, 1e-45],
                        dtype=torch.float32)
    ties = torch.tensor([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF, 0x00008000],
                        dtype=torch.int64).to(torch.int32).view(torch.float32)
    x = torch.cat([vals.float(), edge, ties])
    ours = oracle.bf16_round(x.numpy())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------- quantiser


def test_quantize_hand_packed(fixture_loader):
    fx = fixture_loader("quant_hand_packed.txt")
    G = int(fx["G"][0])
    w = np.array([fx["w_row0"], fx["w_row1"]], np.float32)
    q, s, b = oracle.quantize(w, G)
    np.testing.assert_array_equal(q, np.array([fx["q_row0"], fx["q_row1"]], np.uint32))
    np.testing.assert_array_equal(s, np.array([fx["scale_row0"], fx["scale_row1"]], np.uint16))
    np.testing.assert_array_equal(b, np.array([fx["bias_row0"], fx["bias_row1"]], np.uint16))
    deq = oracle.dequant(q, s, b, 16, G)
    np.testing.assert_array_equal(deq, np.array([fx["deq_row0"], fx["deq_row1"]], np.float64))


def test_nibble_order_even_elements_low():
    # word k/8 holds element 2j of the word in nibble j and 2j+1 in nibble j+4
    s_bits = 0x3F80  # scale 1, bias 0 -> w == code
    w = np.array([[0, 15, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14]], np.float32)
    q, s, b = oracle.quantize(w, 16)
    assert s[0, 0] == s_bits and b[0, 0] == 0
    # word 0: elements 0 15 1 2 3 4 5 6 -> nibbles (low to high) 0 1 3 5 | 15 2 4 6
    # word 1: elements 7 .. 14            -> nibbles 7 9 11 13 | 8 10 12 14
    assert q[0, 0] == 0x642F_5310 and q[0, 1] == 0xECA8_DB97


def _bf16_of(x):
    return torch.tensor(np.float32(x)).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF


@pytest.mark.parametrize("G", [32, 64])
def test_quantize_scale_bias_and_nearest_code(G):
    rng = np.random.default_rng(5)
    rows, K = 24, 256
    w = (rng.standard_normal((rows, K)) * 0.02).astype(np.float32)
    w[3, :G] = 0.125                       # constant group -> s = 0, codes 0
    q, s, b = oracle.quantize(w, G)
    deq = oracle.dequant(q, s, b, K, G)
    for r in range(rows):
        for g in range(K // G):
            v = w[r, g * G:(g + 1) * G]
            mn, mx = np.float32(v.min()), np.float32(v.max())
            assert s[r, g] == _bf16_of(np.float32(mx - mn) / np.float32(15.0))
            assert b[r, g] == _bf16_of(mn)
            sv = float(torch.tensor(int(s[r, g]), dtype=torch.int32).to(torch.int16)
                       .view(torch.bfloat16).float())
            bv = float(torch.tensor(int(b[r, g]), dtype=torch.int32).to(torch.int16)
                       .view(torch.bfloat16).float())
            grid = bv + sv * np.arange(16, dtype=np.float64)
            d = deq[r, g * G:(g + 1) * G]
            # each dequantised value is one of the 16 grid points and (brute
            # force over all codes) a nearest one to the input
            for vi, di in zip(v.astype(np.float64), d):
                assert np.any(grid == di)
                assert abs(vi - di) <= np.min(np.abs(grid - vi)) + 1e-7 * abs(vi) + 1e-12
            # closed-form bound on the round-trip error
            bound = sv / 2 + 2.0 ** -8 * (float(mx - mn) + abs(float(mn))) + 1e-7
            assert np.max(np.abs(d - v)) <= bound


def test_quantize_constant_group_is_code_zero():
    w = np.full((1, 64), -0.7, np.float32)
    q, s, b = oracle.quantize(w, 64)
    assert s[0, 0] == 0 and b[0, 0] == _bf16_of(-0.7)
    assert np.all(q == 0)


# ---------------------------------------------------------------- router


def test_router_logits_within_fp32_bound():
    rng = np.random.default_rng(7)
    T, H, E = 32, 512, 24
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    xb = synthetic.bf16_bits(x).numpy().view(np.uint16)
    Wr = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    l = oracle.router_logits(xb, Wr, bias)
    xf = x.float().numpy().astype(np.float64)
    exact = xf @ Wr.astype(np.float64).T + bias.astype(np.float64)
    gamma = (H + 1) * 2.0 ** -24 / (1 - (H + 1) * 2.0 ** -24)
    bound = gamma * (np.abs(xf) @ np.abs(Wr.astype(np.float64)).T + np.abs(bias))
    assert np.all(np.abs(l - exact) <= bound)
    # an operand mix-up (Wr read transposed, bias dropped) is far outside the bound
    assert np.max(np.abs(l - exact)) < 1e-4


# ----------------------------------------------------------------- top-k


def test_topk_hand_ties(fixture_loader):
    fx = fixture_loader("topk_ties.txt")
    l = np.array([fx["logits"]], np.float32)
    for k in (3, 4):
        idx, w = oracle.topk(l, k)
        np.testing.assert_array_equal(idx[0], np.array(fx[f"k{k}_idx"], np.int32))
        np.testing.assert_allclose(w[0], np.array(fx[f"k{k}_w"]), rtol=1e-15, atol=1e-16)


@pytest.mark.parametrize("kind", ["normal", "ties"])
@pytest.mark.parametrize("E,k", [(16, 2), (16, 4), (8, 8), (256, 8)])
def test_topk_brute_force(kind, E, k):
    l = synthetic.make_logits(64, E, seed=E * 10 + k, kind=kind).numpy()
    idx, w = oracle.topk(l, k)
    for t in range(l.shape[0]):
        row = l[t]
        # rank = competitors strictly greater, plus equal ones with a lower index
        rank = np.array([np.sum(row > row[e]) + np.sum((row == row[e]) & (np.arange(E) < e))
                         for e in range(E)])
        expect = np.argsort(rank, kind="stable")[:k]
        np.testing.assert_array_equal(idx[t], expect)
        assert set(idx[t]) == set(np.nonzero(rank < k)[0])
        # library cross-check: lexsort by (-logit, index)
        np.testing.assert_array_equal(idx[t], np.lexsort((np.arange(E), -row.astype(np.float64)))[:k])
        # weights: softmax over the picked logits (library), summing to one
        ref = scipy.special.softmax(row[idx[t]].astype(np.float64))
        np.testing.assert_allclose(w[t], ref, rtol=1e-12, atol=1e-15)
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_topk_all_equal_picks_lowest_indices():
    l = np.zeros((5, 256), np.float32)
    idx, w = oracle.topk(l, 8)
    assert np.all(idx == np.arange(8, dtype=np.int32))
    np.testing.assert_allclose(w, 1.0 / 8, rtol=1e-15)


def test_topk_weights_equal_full_softmax_renormalised():
    l = synthetic.make_logits(16, 32, seed=3).numpy()
    idx, w = oracle.topk(l, 4)
    p = scipy.special.softmax(l.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


# ----------------------------------------------------- routing tables


def _random_idx(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,BN,shared", [(37, 16, 2, 8, True), (64, 256, 8, 16, True),
                                              (5, 8, 8, 4, False), (1, 256, 8, 256, True)])
def test_route_invariants_and_brute_force(T, E, k, BN, shared):
    idx = _random_idx(T, E, k, seed=T + E)
    R = oracle.route(idx, E, shared, BN)
    counts, offsets, perm, inv = R["counts"], R["offsets"], R["perm"], R["inv_perm"]
    G = E + (1 if shared else 0)
    assert counts[:E].sum() == T * k
    assert offsets[E] == T * k and offsets[G] == T * k + (T if shared else 0)
    if shared:
        assert counts[E] == T
    np.testing.assert_array_equal(np.bincount(idx.ravel(), minlength=E), counts[:E])
    assert sorted(perm.tolist()) == list(range(T * k))           # bijection
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))   # inverse
    # brute force: sort every (expert, token, slot) triple
    triples = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
    np.testing.assert_array_equal(perm, np.array([t * k + j for _, t, j in triples]))
    # tiles cover every group's rows exactly once, in blocks of at most BN
    covered = np.zeros(offsets[G], np.int32)
    for g_, r0, n in zip(R["tile_group"], R["tile_row"], R["tile_rows"]):
        assert 1 <= n <= BN and offsets[g_] <= r0 and r0 + n <= offsets[g_ + 1]
        covered[r0:r0 + n] += 1
    assert np.all(covered == 1)
    assert len(R["tile_group"]) == sum(-(-int(c) // BN) for c in counts)


# ------------------------------------------------------------- experts


def _dense_swiglu(xf, Wg, Wu, Wd):
    g = xf @ Wg.T
    u = xf @ Wu.T
    return (g / (1.0 + np.exp(-g)) * u) @ Wd.T


@pytest.mark.parametrize("shared", [False, True])
def test_single_expert_reduces_to_dense_swiglu(shared):
    """E = 1, k = 1: the layer is a dense SwiGLU MLP (plus the shared one)."""
    cfg = synthetic.MoEConfig("dense", T=6, H=128, E=1, k=1, I=64, group=32, seed=21,
                              has_shared=shared)
    L = synthetic.make_layer(cfg)
    gate = oracle.quantize_stack(L.w_gate.numpy(), 32)
    up = oracle.quantize_stack(L.w_up.numpy(), 32)
    down = oracle.quantize_stack(L.w_down.numpy(), 32)
    xb = synthetic.bf16_bits(L.x).numpy().view(np.uint16)
    out = oracle.moe_layer(xb, L.router_w.numpy(), None, gate, up, down, E=1, k=1,
                           has_shared=shared)
    assert np.all(out["idx"] == 0) and np.allclose(out["w"], 1.0)
    xf = L.x.float().numpy().astype(np.float64)
    nexp = 2 if shared else 1
    ref = np.zeros((cfg.T, cfg.H))
    for e in range(nexp):
        Wg = oracle.dequant(gate.q[e], gate.s[e], gate.b[e], cfg.H, 32)
        Wu = oracle.dequant(up.q[e], up.s[e], up.b[e], cfg.H, 32)
        Wd = oracle.dequant(down.q[e], down.s[e], down.b[e], cfg.I, 32)
        ref += _dense_swiglu(xf, Wg, Wu, Wd)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-12)


def test_identity_experts_pass_input_through():
    T, E, k, H = 40, 16, 4, 64
    l = synthetic.make_logits(T, E, seed=9).numpy()
    idx, w = oracle.topk(l, k)
    x = synthetic.make_tokens(H, T, seed=4)
    xb = synthetic.bf16_bits(x).numpy().view(np.uint16)
    y = oracle.dispatch_combine_identity(xb, E, True, idx, w)
    np.testing.assert_allclose(y, x.float().numpy().astype(np.float64), rtol=1e-14, atol=0)


def test_tiny_layer_against_numpy_evaluation():
    """Whole tiny layer vs an independent numpy evaluation (library sort and
    matmul) of the same definition, on the oracle's own quantised weights."""
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    G = cfg.group
    gate = oracle.quantize_stack(L.w_gate.numpy(), G)
    up = oracle.quantize_stack(L.w_up.numpy(), G)
    down = oracle.quantize_stack(L.w_down.numpy(), G)
    xb = synthetic.bf16_bits(L.x).numpy().view(np.uint16)
    out = oracle.moe_layer(xb, L.router_w.numpy(), None, gate, up, down, cfg.E, cfg.k, True)
    xf = L.x.float().numpy().astype(np.float64)
    logits = xf @ L.router_w.numpy().astype(np.float64).T
    y = np.zeros((cfg.T, cfg.H))
    deq = {}
    for e in range(cfg.E + 1):
        deq[e] = (oracle.dequant(gate.q[e], gate.s[e], gate.b[e], cfg.H, G),
                  oracle.dequant(up.q[e], up.s[e], up.b[e], cfg.H, G),
                  oracle.dequant(down.q[e], down.s[e], down.b[e], cfg.I, G))
    for t in range(cfg.T):
        order = np.lexsort((np.arange(cfg.E), -logits[t]))[:cfg.k]
        np.testing.assert_array_equal(out["idx"][t], order)
        p = scipy.special.softmax(logits[t][order])
        for j, e in enumerate(order):
            y[t] += p[j] * _dense_swiglu(xf[t:t + 1], *deq[e])[0]
        y[t] += _dense_swiglu(xf[t:t + 1], *deq[cfg.E])[0]
    # the oracle's router is fp32 (weights move by ~1e-7 relative), the numpy
    # evaluation's is fp64
    np.testing.assert_allclose(out["y"], y, rtol=1e-5, atol=1e-6 * np.abs(y).max())


# ------------------------------------------------------- routing variants


def test_topk_without_renormalisation_keeps_full_softmax_probabilities():
    """renorm=False: the picked weights are the softmax over all E as they
    are (scipy), so they sum below 1; the picks themselves do not change."""
    rng = np.random.default_rng(41)
    logits = rng.normal(size=(40, 24)).astype(np.float32)
    idx_r, _ = oracle.topk(logits, 5)
    idx, w = oracle.topk(logits, 5, renorm=False)
    np.testing.assert_array_equal(idx, idx_r)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), axis=1), rtol=1e-12)
    assert np.all(w.sum(axis=1) < 1.0)


def _gated_inputs(seed=43):
    cfg = synthetic.MoEConfig("gated", T=7, H=128, E=6, k=2, I=64, group=32, seed=seed)
    L = synthetic.make_layer(cfg)
    stacks = [oracle.quantize_stack(w.numpy(), 32) for w in (L.w_gate, L.w_up, L.w_down)]
    xb = synthetic.bf16_bits(L.x).numpy().view(np.uint16)
    g = torch.Generator().manual_seed(seed)
    sg = (torch.randn(cfg.H, generator=g) * 0.05).numpy().astype(np.float32)
    return cfg, L, stacks, xb, sg


def test_shared_gate_weight_is_the_sigmoid_of_the_gate_score():
    """sigmoid(x . g) with the dot in float64 (numpy): the oracle's fp32 sum
    differs by at most a few fp32 roundings of the terms."""
    cfg, L, stacks, xb, sg = _gated_inputs()
    out = oracle.moe_layer(xb, L.router_w.numpy(), None, *stacks, cfg.E, cfg.k, True, shared_gate_w=sg)
    xf = L.x.float().numpy().astype(np.float64)
    s = xf @ sg.astype(np.float64)
    bound = cfg.H * 2.0 ** -23 * (np.abs(xf) @ np.abs(sg.astype(np.float64)))
    ref_lo, ref_hi = 1.0 / (1.0 + np.exp(-(s - bound))), 1.0 / (1.0 + np.exp(-(s + bound)))
    assert np.all((out["shared_w"] >= ref_lo - 1e-15) & (out["shared_w"] <= ref_hi + 1e-15))
    np.testing.assert_array_equal(oracle.shared_gate(xb, sg), out["shared_w"])
    ungated = oracle.moe_layer(xb, L.router_w.numpy(), None, *stacks, cfg.E, cfg.k, True)
    assert np.all(ungated["shared_w"] == 1.0)


def test_gated_shared_expert_scales_only_the_shared_part():
    """y(gated) = y(no shared) + c * (y(shared, weight 1) - y(no shared)) per
    token: the gate multiplies the shared expert's output and nothing else.
    A zero gate vector gives c = 1/2 exactly."""
    cfg, L, stacks, xb, sg = _gated_inputs(44)
    Wr = L.router_w.numpy()
    none = oracle.moe_layer(xb, Wr, None, *stacks, cfg.E, cfg.k, False)["y"]
    one = oracle.moe_layer(xb, Wr, None, *stacks, cfg.E, cfg.k, True)["y"]
    for vec in (sg, np.zeros_like(sg)):
        out = oracle.moe_layer(xb, Wr, None, *stacks, cfg.E, cfg.k, True, shared_gate_w=vec)
        c = out["shared_w"][:, None]
        np.testing.assert_allclose(out["y"], none + c * (one - none), rtol=1e-9, atol=1e-12)
    assert np.all(out["shared_w"] == 0.5)


def test_experts_given_routing_equals_the_layer_under_its_own_routing():
    """The experts-only evaluation under a given routing reproduces the whole
    layer when handed the layer's own picks and weights (also with the gated
    shared expert's per-token weights), and with no shared expert it drops
    exactly the shared part: the path the GPU tests use for rows whose
    near-tied picks the GPU decided the other way."""
    cfg, L, stacks, xb, sg = _gated_inputs(45)
    Wr = L.router_w.numpy()
    for vec in (None, sg):
        out = oracle.moe_layer(xb, Wr, None, *stacks, cfg.E, cfg.k, True, shared_gate_w=vec)
        sw = None if vec is None else out["shared_w"]
        y = oracle.experts_given_routing(xb, *stacks, cfg.E, True, out["idx"], out["w"], shared_w=sw)
        np.testing.assert_array_equal(y, out["y"])
    none = oracle.moe_layer(xb, Wr, None, *stacks, cfg.E, cfg.k, False)
    y = oracle.experts_given_routing(xb, *stacks, cfg.E, False, none["idx"], none["w"])
    np.testing.assert_array_equal(y, none["y"])


# ------------------------------------------- steps either side of the layer

def _bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _floats(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def test_residual_add_rounds_to_nearest_even():
    # 1 + 2^-9 (a quarter ulp) and 1 + 2^-8 (a tie, even neighbour below) stay
    # 1; (1 + 2^-7) + 2^-8 is a tie whose even neighbour is 1 + 2^-6
    a = np.array([[0x3F80, 0x3F80, 0x3F81]], np.uint16)
    r = np.array([[0x3B00, 0x3B80, 0x3B80]], np.uint16)
    h, _ = oracle.residual_rmsnorm(a, r, np.ones(3, np.float32), 0.0)
    assert h.tolist() == [[0x3F80, 0x3F80, 0x3F82]]


def test_rmsnorm_worked_example():
    # h = (3, 4): mean square 12.5, x = (3, 4) / sqrt(12.5) = (0.84853, 1.13137),
    # to bf16: 0.84765625 (0x3F59) and 1.1328125 (0x3F91)
    h, x = oracle.residual_rmsnorm(_bits([[3.0, 4.0]]), _bits([[0.0, 0.0]]), np.ones(2, np.float32), 0.0)
    assert h.tolist() == [[0x4040, 0x4080]]
    assert x.tolist() == [[0x3F59, 0x3F91]]
    # alternating signs of one magnitude: the RMS is that magnitude, x = w
    w = np.array([0.5, -2.0, 3.0, 0.25], np.float32)
    _, x = oracle.residual_rmsnorm(_bits([[6.0, -6.0, 6.0, -6.0]]), _bits([[0.0] * 4]), w, 0.0)
    assert np.array_equal(_floats(x)[0], w * np.array([1, -1, 1, -1], np.float32))


def test_rmsnorm_against_torch_and_invariants():
    g = torch.Generator().manual_seed(41)
    T, H = 6, 512
    a = _bits(torch.randn(T, H, generator=g).numpy())
    r = _bits((torch.randn(T, H, generator=g) * 0.5).numpy())
    w = (torch.rand(H, generator=g) + 0.5).numpy().astype(np.float32)
    eps = 1e-6
    h, x = oracle.residual_rmsnorm(a, r, w, eps)
    # residual: the fp32 sum of the two bf16 values, rounded by torch
    hv = torch.from_numpy(_floats(a)) + torch.from_numpy(_floats(r))
    assert np.array_equal(h, hv.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    # norm: float64 torch reference (its bf16 cast goes through fp32, so a rare
    # element may differ by one ulp from the oracle's single rounding)
    hd = torch.from_numpy(_floats(h)).double()
    ref = hd / torch.sqrt((hd * hd).mean(dim=1, keepdim=True) + eps) * torch.from_numpy(w).double()
    ref_bits = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    diff = np.abs(x.astype(np.int32) - ref_bits.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
    # doubling h changes nothing (eps = 0); doubling w doubles x exactly
    _, x1 = oracle.residual_rmsnorm(h, np.zeros_like(h), w, 0.0)
    _, x2 = oracle.residual_rmsnorm(_bits(2 * _floats(h)), np.zeros_like(h), w, 0.0)
    assert np.array_equal(x1, x2)
    _, x3 = oracle.residual_rmsnorm(h, np.zeros_like(h), 2 * w, 0.0)
    assert np.array_equal(_floats(x3), 2 * _floats(x1))


def test_rmsnorm_eps_dominates_a_tiny_row():
    # h = 2^-10 everywhere, eps = 1: x = 2^-10 / sqrt(1 + 2^-20), which rounds to 2^-10
    c = np.float32(2.0 ** -10)
    _, x = oracle.residual_rmsnorm(_bits([[c] * 8]), _bits([[0.0] * 8]), np.ones(8, np.float32), 1.0)
    assert np.array_equal(_floats(x)[0], np.full(8, c, np.float32))
    # without eps the same row normalises to 1
    _, x = oracle.residual_rmsnorm(_bits([[c] * 8]), _bits([[0.0] * 8]), np.ones(8, np.float32), 0.0)
    assert np.array_equal(_floats(x)[0], np.ones(8, np.float32))


def test_residual_out_adds_h_and_rounds_once():
    h = _bits([[1.0, 1.0, 1.0, -2.0]])
    y = np.array([[2.0 ** -9, 3 * 2.0 ** -9, -1.0, 0.5]])
    out = oracle.residual_out(h, y)
    # 1 + 2^-9 -> 1; 1 + 3 * 2^-9 -> 1 + 2^-7; 1 - 1 -> 0; -2 + 0.5 -> -1.5
    assert out.tolist() == [[0x3F80, 0x3F81, 0x0000, 0xBFC0]]
    # just above a tie: 1 + 2^-8 + 2^-30 rounds up to 1 + 2^-7 when rounded
    # once (through fp32 it would become the tie 1 + 2^-8 and then 1)
    assert oracle.residual_out(_bits([[1.0]]), np.array([[2.0 ** -8 + 2.0 ** -30]])).tolist() == [[0x3F81]]


def test_block_with_zero_experts_is_the_residual_stream():
    # all expert weights zero: the layer adds nothing, out is h bit for bit
    cfg = synthetic.CONFIGS["tiny"]
    L = synthetic.make_layer(cfg)
    zero = oracle.quantize_stack(np.zeros_like(L.w_gate.numpy()), cfg.group)
    zdown = oracle.quantize_stack(np.zeros_like(L.w_down.numpy()), cfg.group)
    g = torch.Generator().manual_seed(5)
    a = _bits(torch.randn(cfg.T, cfg.H, generator=g).numpy())
    r = _bits(torch.randn(cfg.T, cfg.H, generator=g).numpy())
    w = np.ones(cfg.H, np.float32)
    blk = oracle.moe_block(a, r, w, 1e-6, L.router_w.numpy(), None, zero, zero, zdown, cfg.E, cfg.k, True)
    assert np.array_equal(blk["out"], blk["h"])
    # and with the real experts, out - h is the layer on the normalised input
    gate, up, down = (oracle.quantize_stack(m.numpy(), cfg.group) for m in (L.w_gate, L.w_up, L.w_down))
    blk = oracle.moe_block(a, r, w, 1e-6, L.router_w.numpy(), None, gate, up, down, cfg.E, cfg.k, True)
    plain = oracle.moe_layer(blk["x"], L.router_w.numpy(), None, gate, up, down, cfg.E, cfg.k, True)
    assert np.array_equal(blk["out"], oracle.residual_out(blk["h"], plain["y"]))


# ------------------------------------------------ GQA decode attention (second workload)

def _attn_inputs(Hq, Hkv, D, L_cap, seed, scale_kv=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Hq, D, generator=g).to(torch.bfloat16)
    k = (torch.randn(Hkv, L_cap, D, generator=g) * scale_kv).to(torch.bfloat16)
    v = torch.randn(Hkv, L_cap, D, generator=g).to(torch.bfloat16)
    bits = lambda t: synthetic.bf16_bits(t).numpy().view(np.uint16)  # noqa: E731
    return q, k, v, bits(q), bits(k), bits(v)


def test_attention_single_position_returns_its_value():
    """L = 1: the only position gets probability 1, so every query head of a
    group returns that position's value row exactly."""
    q, k, v, qb, kb, vb = _attn_inputs(16, 2, 64, 3, seed=101)
    o = oracle.gqa_attention(qb, kb, vb, 1, 0.125)
    for h in range(16):
        np.testing.assert_array_equal(o[h], v[h // 8, 0].float().numpy().astype(np.float64))


def test_attention_equal_keys_average_the_values():
    """Identical keys (or scale 0) give every position the same probability:
    the output is the plain mean of the value rows."""
    q, k, v, qb, kb, vb = _attn_inputs(8, 2, 32, 20, seed=102)
    kb_same = np.broadcast_to(kb[:, :1, :], kb.shape).copy()
    mean = v[:, :13].float().numpy().astype(np.float64).mean(axis=1)
    for o in (oracle.gqa_attention(qb, kb_same, vb, 13, 0.177), oracle.gqa_attention(qb, kb, vb, 13, 0.0)):
        for h in range(8):
            np.testing.assert_allclose(o[h], mean[h // 4], rtol=1e-12, atol=1e-14)


def test_attention_against_scipy_softmax():
    """Random heads against an independent float64 evaluation with the
    library softmax: scores K q * scale, probabilities softmax, output p V."""
    from scipy.special import softmax
    Hq, Hkv, D, L = 16, 2, 128, 37
    q, k, v, qb, kb, vb = _attn_inputs(Hq, Hkv, D, 50, seed=103)
    scale = 1.0 / np.sqrt(D)
    o = oracle.gqa_attention(qb, kb, vb, L, scale)
    qf, kf, vf = (t.float().numpy().astype(np.float64) for t in (q, k, v))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        p = softmax(kf[g, :L] @ qf[h] * scale)
        np.testing.assert_allclose(o[h], p @ vf[g, :L], rtol=1e-11, atol=1e-13)


def test_attention_query_heads_share_consecutive_groups():
    """Query heads 0-7 read key-value head 0 and heads 8-15 head 1: zeroing
    head 1's values zeroes exactly heads 8-15, and swapping the two key-value
    heads swaps the two halves of the output."""
    q, k, v, qb, kb, vb = _attn_inputs(16, 2, 64, 9, seed=104)
    vz = vb.copy()
    vz[1] = 0
    o = oracle.gqa_attention(qb, kb, vz, 9, 0.125)
    assert np.all(o[8:] == 0.0) and np.all(np.abs(o[:8]).sum(axis=1) > 0)
    q_sw = np.concatenate([qb[8:], qb[:8]])
    o_sw = oracle.gqa_attention(q_sw, kb[::-1].copy(), vb[::-1].copy(), 9, 0.125)
    base = oracle.gqa_attention(qb, kb, vb, 9, 0.125)
    np.testing.assert_array_equal(o_sw, np.concatenate([base[8:], base[:8]]))


def test_attention_ignores_positions_past_L_and_their_order():
    """Only the first L cached positions count (huge values past them change
    nothing), and permuting those positions (keys and values together)
    leaves the output unchanged up to summation order."""
    q, k, v, qb, kb, vb = _attn_inputs(8, 1, 32, 40, seed=105)
    o = oracle.gqa_attention(qb, kb, vb, 29, 0.2)
    big = synthetic.bf16_bits(torch.full((1, 11, 32), 1e4).to(torch.bfloat16)).numpy().view(np.uint16)
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[:, 29:], vb2[:, 29:] = big, big
    np.testing.assert_array_equal(oracle.gqa_attention(qb, kb2, vb2, 29, 0.2), o)
    perm = np.random.default_rng(7).permutation(29)
    kp, vp = kb.copy(), vb.copy()
    kp[:, :29], vp[:, :29] = kb[:, perm], vb[:, perm]
    np.testing.assert_allclose(oracle.gqa_attention(qb, kp, vp, 29, 0.2), o, rtol=1e-12, atol=1e-14)
