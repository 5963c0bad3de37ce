"""Shared helpers of the parity tests: build one layer for both sides from the
same seeded fp32 inputs (the GPU packs them with pack_int4, the oracle with
its own quantiser) and compare outputs under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from int4_grouped_gemm_gb300 import synthetic

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
