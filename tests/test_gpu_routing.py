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
