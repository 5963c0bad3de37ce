"""Shared helpers of the parity tests: build one layer for both sides from the
same seeded fp32 inputs (the GPU packs them with pack_int4, the oracle with
its own quantiser) and compare outputs under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic

# Output tolerance: max|gpu - oracle| <= 2e-2 * max|oracle| and
# sum|gpu - oracle| / sum|oracle| <= 5e-3 (gpu output bf16, oracle fp64).
MAX_REL = 2e-2
L1_REL = 5e-3
# A token whose oracle logits put the k-th and (k+1)-th largest closer than
# this (relative to max |logit|) has an ambiguous top-k set: the GPU's fp32
# router sums in another order and may pick the other expert.
AMBIGUOUS_REL = 1e-4


def x_bits(x: torch.Tensor) -> np.ndarray:
    return synthetic.bf16_bits(x.cpu()).numpy().view(np.uint16)


def oracle_stacks(L: synthetic.LayerInputs, group: int):
    gate = oracle.quantize_stack(L.w_gate.cpu().numpy(), group)
    up = oracle.quantize_stack(L.w_up.cpu().numpy(), group)
    down = oracle.quantize_stack(L.w_down.cpu().numpy(), group)
    return gate, up, down


def oracle_layer(L: synthetic.LayerInputs, x: torch.Tensor, tokens=None, stacks=None) -> dict:
    cfg = L.cfg
    gate, up, down = stacks if stacks is not None else oracle_stacks(L, cfg.group)
    bias = None if L.router_bias is None else L.router_bias.cpu().numpy()
    return oracle.moe_layer(x_bits(x), L.router_w.cpu().numpy(), bias, gate, up, down, cfg.E, cfg.k,
                            cfg.has_shared, tokens=tokens)


def ambiguous(logits: np.ndarray, k: int, E: int) -> np.ndarray:
    """Tokens whose k-th / (k+1)-th largest oracle logits nearly tie."""
    if k >= E:
        return np.zeros(logits.shape[0], bool)
    srt = -np.sort(-logits.astype(np.float64), axis=1)
    gap = srt[:, k - 1] - srt[:, k]
    scale = np.abs(logits).max(axis=1) + 1e-30
    return gap < AMBIGUOUS_REL * scale


def compare(got: np.ndarray, want: np.ndarray):
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    scale = np.abs(want).max()
    err = np.abs(got - want)
    max_rel = err.max() / scale if scale > 0 else err.max()
    l1 = err.sum() / max(np.abs(want).sum(), 1e-300)
    return max_rel, l1


def assert_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    max_rel, l1 = compare(got, want)
    assert max_rel <= MAX_REL, f"{what}: max error {max_rel:.3e} of max|oracle| (bound {MAX_REL})"
    assert l1 <= L1_REL, f"{what}: L1 ratio {l1:.3e} (bound {L1_REL})"
    return max_rel, l1


def sample_tokens(T: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pick.update({0, T - 1})
    return np.array(sorted(pick), np.int32)


def check_topk_exact(gpu_logits: np.ndarray, gpu_idx: np.ndarray, gpu_w: np.ndarray, k: int, renorm: bool = True,
                     what: str = ""):
    """The GPU's picks are bit-exact, and its weights within fp32 rounding, of
    the oracle's top-k of the GPU's own fp32 logits; returns the oracle's
    (idx, w) for those logits."""
    idx, w = oracle.topk(gpu_logits, k, renorm)
    np.testing.assert_array_equal(gpu_idx, idx, err_msg=f"{what}: picks differ from oracle.topk of the GPU logits")
    np.testing.assert_allclose(gpu_w, w, rtol=2e-6, atol=1e-7, err_msg=f"{what}: weights")
    return idx, w


def flipped(ref_idx: np.ndarray, gpu_idx: np.ndarray) -> np.ndarray:
    """Rows whose set of picked experts differs between the oracle's own
    logits and the GPU's (a near tie at the k-th place decided the other way
    by the fp32 summation order)."""
    return ~np.all(np.sort(ref_idx, axis=1) == np.sort(gpu_idx, axis=1), axis=1)


def reference_under_gpu_routing(ref_y: np.ndarray, ref_idx: np.ndarray, xb_rows: np.ndarray, stacks, E: int,
                                has_shared: bool, idx: np.ndarray, w: np.ndarray, shared_w=None,
                                max_flipped: float = 0.05) -> np.ndarray:
    """Oracle outputs to compare the GPU's against: the oracle's own layer
    where its picks agree with the GPU's, and, for the rows whose near-tied
    picks went the other way, the oracle's experts and combine evaluated
    under the routing that the GPU's logits give (idx, w from oracle.topk of
    the GPU logits, already checked bit-exact against the GPU's picks)."""
    flip = flipped(ref_idx, idx)
    assert flip.mean() <= max_flipped, f"{flip.sum()} of {len(flip)} rows picked other experts"
    want = np.array(ref_y, dtype=np.float64, copy=True)
    if flip.any():
        sw = None if shared_w is None else np.asarray(shared_w, np.float64)[flip]
        want[flip] = oracle.experts_given_routing(xb_rows[flip], *stacks, E, has_shared, idx[flip], w[flip],
                                                  shared_w=sw)
    return want


def batch_routing(layer, ws, B, renorm=True, gated=False):
    """What the small-batch kernels decided, read from the workspace views, and
    checked against the oracle given the GPU's own fp32 logits: the slots are
    bit-exactly the union of oracle.topk's picks in ascending expert order
    (then the shared expert), and each slot's per-token weight is the oracle
    weight of that pick (0 where the token did not pick it; the shared
    slot's 1, or the sigmoid of the gate score).  Returns the oracle's
    (idx, w) for the GPU logits."""
    d = layer.desc
    E, k = d.E, d.k
    v = _lib.moe_batch_views_for(d)
    logits = ws.view(v.logits, torch.float32, v.max_tokens * v.logit_ld).view(v.max_tokens, v.logit_ld)
    logits = logits[:B].cpu().numpy()
    slots = ws.view(v.slots, torch.int32, 1 + v.S_max).cpu().numpy()
    slot_w = ws.view(v.slot_w, torch.float32, v.S_max * v.max_tokens).view(v.S_max, v.max_tokens)
    slot_w = slot_w[:, :B].cpu().numpy()
    idx, w = oracle.topk(logits[:, :E], k, renorm)
    union = sorted(set(int(e) for e in idx.ravel()))
    expect = union + ([E] if d.has_shared else [])
    n = int(slots[0])
    assert n == len(expect) and slots[1:1 + n].tolist() == expect, "slot list != union of oracle.topk picks"
    want = np.zeros((n, B))
    pos = {e: i for i, e in enumerate(union)}
    for t in range(B):
        for j in range(k):
            want[pos[int(idx[t, j])], t] = w[t, j]
    if d.has_shared:
        want[n - 1] = 1.0 / (1.0 + np.exp(-logits[:, E].astype(np.float64))) if gated else 1.0
    np.testing.assert_allclose(slot_w[:n], want, rtol=2e-6, atol=1e-7, err_msg="per-slot token weights")
    return idx, w
