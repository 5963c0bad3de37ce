"""GQA decode attention (the second workload) against the CPU oracle: one
token's attention over a key-value cache, query heads sharing key-value
heads, packed (each key-value row read once for its query heads) and per
head; ragged cache lengths around the kernel's 16-position tiles, partly
filled caches, group sizes 1-8, head dimensions 64 and 128, a peaked softmax,
the uniform case, and the full 32K-position cache of the benchmark."""
import math

import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import _lib, synthetic
from int4_grouped_gemm_gb300.synthetic import AttnConfig

from moe_helpers import assert_close

pytestmark = pytest.mark.gpu


def _bits(t):
    return synthetic.bf16_bits(t.cpu()).numpy().view(np.uint16)


def _run(cfg, per_head=False, scale=None):
    q, k, v = synthetic.make_attention(cfg)
    scale = 1.0 / math.sqrt(cfg.D) if scale is None else scale
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    ws = torch.empty(_lib.gqa_attention_workspace_bytes(cfg.Hq, cfg.Hkv, cfg.D, cfg.L), dtype=torch.uint8,
                     device="cuda")
    _lib.gqa_decode_attention(qd, kd, vd, cfg.L, scale, out, ws, per_head=per_head)
    torch.cuda.synchronize()
    ref = oracle.gqa_attention(_bits(q), _bits(k), _bits(v), cfg.L, scale)
    return out.float().cpu().numpy(), ref, (qd, kd, vd, ws)


SHAPES = [
    AttnConfig("one", Hq=16, Hkv=2, D=128, L=1, seed=201),
    AttnConfig("seven_of_twelve", Hq=16, Hkv=2, D=128, L=7, L_cap=12, seed=202),
    AttnConfig("one_subchunk", Hq=16, Hkv=2, D=128, L=64, seed=203),
    AttnConfig("sixty_five", Hq=16, Hkv=2, D=128, L=65, seed=204),
    AttnConfig("ragged_1000", Hq=16, Hkv=2, D=128, L=1000, L_cap=1100, seed=205),
    AttnConfig("ragged_4097", Hq=16, Hkv=2, D=128, L=4097, seed=206),
    AttnConfig("d64_group8", Hq=8, Hkv=1, D=64, L=333, seed=207),
    AttnConfig("group3", Hq=12, Hkv=4, D=128, L=300, seed=208),
    AttnConfig("mha_group1", Hq=16, Hkv=16, D=64, L=150, seed=209),
    AttnConfig("peaked", Hq=16, Hkv=2, D=128, L=2000, seed=210, k_scale=6.0),
    # one position past a 16-position tile; 256 query heads, whose per-head
    # blocks each take all 257 positions (17 tiles: two or three rounds of
    # the eight warps, the last tile one position long)
    AttnConfig("tile_plus_one", Hq=16, Hkv=2, D=128, L=17, seed=211),
    AttnConfig("heads256_range257", Hq=256, Hkv=32, D=64, L=257, L_cap=300, seed=212),
]


@pytest.mark.parametrize("per_head", [False, True], ids=["packed", "per_head"])
@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
def test_attention_against_the_oracle(cfg, per_head):
    got, ref, _ = _run(cfg, per_head)
    assert_close(got, ref, f"{cfg.name} {'per head' if per_head else 'packed'}")


def test_full_32k_cache_and_repeat_calls_are_identical():
    cfg = synthetic.ATTN_CONFIGS["gqa32k"]
    got, ref, (qd, kd, vd, ws) = _run(cfg)
    max_rel, l1 = assert_close(got, ref, "32K cache")
    assert l1 < 2e-3
    again = torch.empty_like(qd)
    _lib.gqa_decode_attention(qd, kd, vd, cfg.L, 1.0 / math.sqrt(cfg.D), again, ws)
    torch.cuda.synchronize()
    assert np.array_equal(again.float().cpu().numpy(), got)
    per_head, _, _ = _run(cfg, per_head=True)
    assert_close(per_head, ref, "32K cache per head")


def test_scale_zero_averages_the_values():
    """scale 0: every position weighs 1/L, the output is the mean of the
    value rows (the oracle's closed form, checked by the pins)."""
    cfg = AttnConfig("uniform", Hq=16, Hkv=2, D=128, L=777, seed=211)
    got, ref, _ = _run(cfg, scale=0.0)
    _, _, v = synthetic.make_attention(cfg)
    mean = v.float().numpy().astype(np.float64).mean(axis=1)
    np.testing.assert_allclose(ref, np.repeat(mean, 8, axis=0), rtol=1e-10, atol=1e-12)
    assert_close(got, ref, "uniform")


def test_attention_arguments_rejected_on_the_host():
    q = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MoEError) as e:
        _lib.gqa_decode_attention(q, kv, kv, 65, 0.1, out, ws)           # L > L_cap
    assert e.value.code == _lib.MOE_ERR_TOKENS
    with pytest.raises(_lib.MoEError) as e:
        _lib.gqa_decode_attention(q[:, :96].contiguous(), kv[:, :, :96].contiguous(), kv[:, :, :96].contiguous(),
                                  10, 0.1, out, ws)                      # D = 96
    assert e.value.code == _lib.MOE_ERR_SHAPE
    with pytest.raises(_lib.MoEError) as e:
        _lib.gqa_decode_attention(q, kv, kv, 10, 0.1, out, ws[:16])      # workspace too small
    assert e.value.code == _lib.MOE_ERR_WORKSPACE
