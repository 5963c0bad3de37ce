"""GPU routing (top-k, weights, histogram, scan, permutation, tile map) is
bit-exact against the oracle given the same fp32 router logits."""
import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300._lib import moe_layer_desc
from int4_grouped_gemm_gb300.moe import Workspace

pytestmark = pytest.mark.gpu


def expected_schedule(tg, tr, tn, BN):
    """Grouped-GEMM work units: each group's tiles in pairs (the last alone
    if odd), given by their first tile; units of two full tiles first in
    canonical order, then the rest by rows descending (ties: lower group)."""
    units = []
    first = {}
    for i, g in enumerate(tg):
        first.setdefault(g, i)
    for i, g in enumerate(tg):
        if (i - first[g]) % 2 == 0:
            rows = tn[i] + (tn[i + 1] if i + 1 < len(tg) and tg[i + 1] == g else 0)
            units.append((i, g, rows))
    full = [u for u in units if u[2] == 2 * BN]
    part = sorted([u for u in units if u[2] < 2 * BN], key=lambda u: (-u[2], u[1]))
    return np.array([u[0] for u in full + part], np.int32)


def run_case(T, E, k, shared, kind, seed):
    desc = moe_layer_desc(E, k, 256, 128, 32, int(shared), None, None)
    ws = Workspace(desc, T)
    logits = synthetic.make_logits(T, E, seed, kind)
    _lib.moe_route_logits(desc, logits.cuda(), T, ws.buf)
    torch.cuda.synchronize()
    assert _lib.moe_read_device_status(ws.buf) == 0
    keys = ("topk_idx", "topk_w", "counts", "offsets", "perm", "inv_perm", "tile_group", "tile_row", "tile_rows",
            "tile_sched")
    views = ws.routing(desc, T)
    g = {key: views[key].cpu().numpy() for key in keys}
    g["tile_size"] = views["tile_size"]
    idx, w = oracle.topk(logits.numpy(), k)
    R = oracle.route(idx, E, shared, g["tile_size"])
    np.testing.assert_array_equal(g["topk_idx"], idx)
    np.testing.assert_allclose(g["topk_w"], w, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(g["counts"], R["counts"])
    np.testing.assert_array_equal(g["offsets"], R["offsets"])
    np.testing.assert_array_equal(g["perm"], R["perm"])
    np.testing.assert_array_equal(g["inv_perm"], R["inv_perm"])
    np.testing.assert_array_equal(g["tile_group"], R["tile_group"])
    np.testing.assert_array_equal(g["tile_row"], R["tile_row"])
    np.testing.assert_array_equal(g["tile_rows"], R["tile_rows"])
    np.testing.assert_array_equal(g["tile_sched"], expected_schedule(R["tile_group"], R["tile_row"],
                                                                     R["tile_rows"], g["tile_size"]))


@pytest.mark.parametrize("kind", ["normal", "ties", "equal"])
@pytest.mark.parametrize("T,E,k,shared", [(1, 256, 8, True), (16, 16, 2, True), (37, 16, 2, False),
                                          (64, 8, 8, True), (65, 256, 8, True), (1000, 33, 3, True)])
def test_route_small(T, E, k, shared, kind):
    run_case(T, E, k, shared, kind, seed=T * 7 + E)


@pytest.mark.parametrize("T,kind", [(512, "normal"), (4096, "normal"), (4096, "ties"), (16384, "normal"),
                                    (16384, "equal")])
def test_route_full_sizes(T, kind):
    run_case(T, 256, 8, True, kind, seed=T)


def _decode_logits(T, E, k, kind, seed):
    """Logit rows for the decode top-k: the shared kinds, plus 'signed_zero'
    (values from {-0, +0, 0.5, -0.5}: many ties between the two zeros) and
    'kth_tie' (normal rows in which the (k+1)-th largest value is set equal
    to the k-th, on an expert index below or above it)."""
    if kind in ("normal", "ties", "equal"):
        return synthetic.make_logits(T, E, seed, kind)
    g = torch.Generator().manual_seed(seed)
    if kind == "signed_zero":
        grid = torch.tensor([-0.0, 0.0, 0.5, -0.5])
        return grid[torch.randint(0, 4, (T, E), generator=g)]
    if kind == "kth_tie":
        x = torch.randn(T, E, generator=g)
        if k < E:
            order = torch.argsort(-x, dim=1)
            for t in range(T):
                x[t, order[t, k]] = x[t, order[t, k - 1]]
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("renorm", [True, False], ids=["renorm", "no_renorm"])
@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "signed_zero", "kth_tie"])
@pytest.mark.parametrize("E,k", [(16, 1), (16, 8), (40, 3), (200, 8), (256, 8), (256, 1), (9, 8)])
def test_decode_topk_given_logits(E, k, kind, renorm):
    """The batch-1 decode kernel's own top-k (bitonic sort, rank, softmax)
    on given logits: picks bit-exact with oracle.topk, weights within fp32
    rounding, the logits echoed bit for bit."""
    T = 64
    logits = _decode_logits(T, E, k, kind, seed=E * 31 + k)
    desc = moe_layer_desc(E, k, 256, 128, 32, 1, None, None)
    desc.no_renorm = 0 if renorm else 1
    ld = E + 2 * k + 1
    out = torch.zeros(T, ld, dtype=torch.float32, device="cuda")
    _lib.moe_decode_topk_logits(desc, logits.cuda().contiguous(), out)
    rec = out.cpu().numpy()
    assert np.array_equal(rec[:, :E].view(np.uint32), logits.numpy().view(np.uint32))
    idx = rec[:, E:E + k].copy().view(np.int32)
    w = rec[:, E + k:E + 2 * k]
    oi, ow = oracle.topk(logits.numpy(), k, renorm)
    np.testing.assert_array_equal(idx, oi)
    np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)
    assert np.all(rec[:, E + 2 * k] == 1.0)
