"""pack_int4 on the GPU is bit-exact against the oracle quantiser."""
import numpy as np
import pytest
import torch

import oracle
from int4_grouped_gemm_gb300 import synthetic
from int4_grouped_gemm_gb300.moe import pack_matrix

pytestmark = pytest.mark.gpu


def _gpu_pack(w: torch.Tensor, group: int):
    """GPU pack; returns words and the scale/bias without the row-pitch padding
    (after checking that the padding is zero)."""
    qm = pack_matrix(w.cuda(), group)
    torch.cuda.synchronize()
    ng = w.shape[-1] // group
    s = qm.scale.cpu().numpy().view(np.uint16)
    b = qm.bias.cpu().numpy().view(np.uint16)
    assert s.shape[-1] % 8 == 0 and s.shape[-1] >= ng
    assert np.all(s[..., ng:] == 0) and np.all(b[..., ng:] == 0)
    return qm.q.cpu().numpy().view(np.uint32), s[..., :ng], b[..., :ng]


def test_hand_packed_fixture(fixture_loader):
    fx = fixture_loader("quant_hand_packed.txt")
    w = torch.tensor([fx["w_row0"], fx["w_row1"]], dtype=torch.float32)
    q, s, b = _gpu_pack(w, int(fx["G"][0]))
    np.testing.assert_array_equal(q, np.array([fx["q_row0"], fx["q_row1"]], np.uint32))
    np.testing.assert_array_equal(s, np.array([fx["scale_row0"], fx["scale_row1"]], np.uint16))
    np.testing.assert_array_equal(b, np.array([fx["bias_row0"], fx["bias_row1"]], np.uint16))


@pytest.mark.parametrize("rows,K,G,std", [(7, 64, 32, 0.02), (33, 256, 64, 0.02), (5, 2048, 64, 1.0),
                                          (3, 512, 32, 1e-3)])
def test_random_matrices(rows, K, G, std):
    w = synthetic.make_weight_matrix(rows, K, seed=rows * K + G, std=std)
    w[0, :G] = 0.25  # constant group
    w[1, G:2 * G] = w[1, G:2 * G].round(decimals=1)  # repeated values, exact ties in codes
    q, s, b = _gpu_pack(w, G)
    oq, os_, ob = oracle.quantize(w.numpy(), G)
    np.testing.assert_array_equal(s, os_)
    np.testing.assert_array_equal(b, ob)
    np.testing.assert_array_equal(q, oq)


def test_full_layer_prefill512():
    """Every gate/up/down matrix of the T=512 layer (257 experts), bit for bit."""
    cfg = synthetic.CONFIGS["prefill512"]
    L = synthetic.make_layer(cfg, device="cuda", with_x=False)
    for name in ("w_gate", "w_up", "w_down"):
        w = getattr(L, name)
        q, s, b = _gpu_pack(w, cfg.group)
        n, rows, K = w.shape
        oq, os_, ob = oracle.quantize(w.reshape(n * rows, K).cpu().numpy(), cfg.group)
        np.testing.assert_array_equal(s.reshape(n * rows, -1), os_, err_msg=name)
        np.testing.assert_array_equal(b.reshape(n * rows, -1), ob, err_msg=name)
        np.testing.assert_array_equal(q.reshape(n * rows, -1), oq, err_msg=name)
