"""Device-resident int4 MoE layers on top of the C ABI.

``PackedLayer`` owns one layer's weights in HBM in the library's int4 format
(packed on the GPU by ``pack_int4``) and the ``moe_layer_desc`` that points at
them; ``Workspace`` owns the scratch buffer a layer call needs.  PyTorch only
provides device memory and streams here.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib
from ._lib import moe_layer_desc, moe_qweight


def ld_groups(K: int, group: int) -> int:
    """Row pitch (in groups) of the scale/bias arrays: K/group rounded up to 8."""
    return (K // group + 7) // 8 * 8


@dataclass
class QMatrix:
    """One stacked int4 matrix set [n_exp][rows][K] in the library format."""
    q: torch.Tensor      # int32 view of uint32 words [n_exp, rows, K/8]
    scale: torch.Tensor  # int16 view of bf16 bits [n_exp, rows, ld_groups(K, G)] (zero padded)
    bias: torch.Tensor
    rows: int
    K: int
    group: int

    def as_c(self) -> moe_qweight:
        return moe_qweight(self.q.data_ptr(), self.scale.data_ptr(), self.bias.data_ptr())


def pack_matrix(w: torch.Tensor, group: int, stream=None) -> QMatrix:
    """Quantise fp32 w [..., rows, K] on the GPU (pack_int4)."""
    assert w.is_cuda and w.dtype == torch.float32
    w = w.contiguous()
    *lead, rows, K = w.shape
    total_rows = w.numel() // K
    q = torch.empty(*lead, rows, K // 8, dtype=torch.int32, device=w.device)
    s = torch.empty(*lead, rows, ld_groups(K, group), dtype=torch.int16, device=w.device)
    b = torch.empty_like(s)
    _lib.pack_int4(w, total_rows, K, group, q, s, b, stream)
    return QMatrix(q, s, b, rows, K, group)


class PackedLayer:
    def __init__(self, E: int, k: int, H: int, I: int, group: int, has_shared: bool,
                 router_w: torch.Tensor, router_bias: Optional[torch.Tensor],
                 gate: QMatrix, up: QMatrix, down: QMatrix, no_renorm: bool = False,
                 shared_gate: Optional[torch.Tensor] = None):
        self.E, self.k, self.H, self.I, self.group, self.has_shared = E, k, H, I, group, bool(has_shared)
        self.router_w = router_w.contiguous()
        self.router_bias = None if router_bias is None else router_bias.contiguous()
        self.shared_gate = None if shared_gate is None else shared_gate.contiguous()
        self.gate, self.up, self.down = gate, up, down
        # the router weights' bf16 hi/lo parts for the prefill's tensor-core
        # router, split once here instead of on every call
        self.router_split = torch.empty(_lib.moe_router_split_bytes(E, H), dtype=torch.uint8,
                                        device=self.router_w.device)
        _lib.moe_split_router(self.router_w, E, H, self.router_split)
        self.desc = moe_layer_desc(E, k, H, I, group, int(has_shared), self.router_w.data_ptr(),
                                   None if self.router_bias is None else self.router_bias.data_ptr(),
                                   gate.as_c(), up.as_c(), down.as_c(), int(no_renorm),
                                   None if self.shared_gate is None else self.shared_gate.data_ptr(),
                                   self.router_split.data_ptr())

    @classmethod
    def from_fp32(cls, cfg, router_w, router_bias, w_gate, w_up, w_down, stream=None, no_renorm: bool = False,
                  shared_gate: Optional[torch.Tensor] = None) -> "PackedLayer":
        """Pack fp32 expert weights (on the GPU) into a device-resident layer
        (routing variants: no_renorm, shared_gate [H] fp32)."""
        dev = torch.device("cuda")
        router_w = router_w.to(dev, torch.float32)
        router_bias = None if router_bias is None else router_bias.to(dev, torch.float32)
        shared_gate = None if shared_gate is None else shared_gate.to(dev, torch.float32)
        gate = pack_matrix(w_gate.to(dev), cfg.group, stream)
        up = pack_matrix(w_up.to(dev), cfg.group, stream)
        down = pack_matrix(w_down.to(dev), cfg.group, stream)
        return cls(cfg.E, cfg.k, cfg.H, cfg.I, cfg.group, cfg.has_shared, router_w, router_bias,
                   gate, up, down, no_renorm, shared_gate)

    def workspace(self, T_max: int) -> "Workspace":
        return Workspace(self.desc, T_max)

    def prefill(self, x: torch.Tensor, ws: "Workspace", y: Optional[torch.Tensor] = None, stream=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        _lib.moe_prefill(self.desc, x, T, y, ws.buf, stream)
        return y

    def decode(self, x: torch.Tensor, ws: "Workspace", y: Optional[torch.Tensor] = None, stream=None):
        if y is None:
            y = torch.empty_like(x)
        _lib.moe_decode(self.desc, x, y, ws.buf, stream)
        return y

    def prefill_block(self, attn: torch.Tensor, residual: torch.Tensor, norm_w: torch.Tensor, ws: "Workspace",
                      eps: float = 1e-6, out: Optional[torch.Tensor] = None, stream=None):
        """The layer in a pre-norm decoder block: out = MoE(RMSNorm(h) w) + h, h = attn + residual."""
        if out is None:
            out = torch.empty_like(attn)
        _lib.moe_prefill_block(self.desc, attn, residual, norm_w, eps, out, ws.buf, stream)
        return out

    def decode_batch_block(self, attn: torch.Tensor, residual: torch.Tensor, norm_w: torch.Tensor, ws: "Workspace",
                           eps: float = 1e-6, out: Optional[torch.Tensor] = None, stream=None):
        """prefill_block for 1 to 8 tokens through the small-batch path."""
        if out is None:
            out = torch.empty_like(attn)
        _lib.moe_decode_batch_block(self.desc, attn, residual, norm_w, eps, out, ws.buf, stream)
        return out

    def decode_batch(self, x: torch.Tensor, ws: "Workspace", y: Optional[torch.Tensor] = None, stream=None):
        """1 to 8 tokens: each picked expert is read once for all of them."""
        if y is None:
            y = torch.empty_like(x)
        _lib.moe_decode_batch(self.desc, x, y, ws.buf, stream)
        return y


class Workspace:
    """Scratch memory for one layer call (routing tables, h, fp32 combine)."""

    def __init__(self, desc: moe_layer_desc, T_max: int, device="cuda"):
        nbytes = _lib.moe_workspace_bytes(desc, T_max)
        if nbytes == 0:
            raise _lib.MoEError(_lib.MOE_ERR_SHAPE, "moe_workspace_bytes")
        self.T_max = T_max
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _lib.moe_workspace_init(self.buf)

    def view(self, offset: int, dtype, n: int) -> torch.Tensor:
        item = torch.empty(0, dtype=dtype).element_size()
        return self.buf[offset:offset + n * item].view(dtype)

    def routing(self, desc: moe_layer_desc, T: int) -> dict:
        """The routing tables of the last call with T tokens (device tensors)."""
        v = _lib.moe_routing_views_for(desc, T)
        E, k = desc.E, desc.k
        ng = E + desc.has_shared
        n_tiles, n_units = (int(c) for c in self.view(v.num_tiles, torch.int32, 2).tolist())
        return dict(
            logits=self.view(v.logits, torch.float32, T * E).view(T, E),
            topk_idx=self.view(v.topk_idx, torch.int32, T * k).view(T, k),
            topk_w=self.view(v.topk_w, torch.float32, T * k).view(T, k),
            counts=self.view(v.counts, torch.int32, ng),
            offsets=self.view(v.offsets, torch.int32, ng + 1),
            perm=self.view(v.perm, torch.int32, T * k),
            inv_perm=self.view(v.inv_perm, torch.int32, T * k),
            tile_group=self.view(v.tile_group, torch.int32, n_tiles),
            tile_row=self.view(v.tile_row, torch.int32, n_tiles),
            tile_rows=self.view(v.tile_rows, torch.int32, n_tiles),
            tile_sched=self.view(v.tile_sched, torch.int32, n_units),
            tile_size=v.tile_size,
            h=self.view(v.h, torch.bfloat16, (T * k + T) * desc.I).view(T * k + T, desc.I),
            y_acc=self.view(v.y_acc, torch.float32, T * desc.H).view(T, desc.H),
        )


class DecodeChain:
    """Batch-1 decode through a stack of independent layers.

    One step runs every layer once (``moe_decode_layers``): the token in
    ``tok`` goes through all layers and the last layer's output is written
    back into ``tok``, so the next step's input is already in place on the
    device, with no host round trip between tokens.  ``capture()`` records
    one step as a CUDA graph.
    """

    def __init__(self, layers, device="cuda", norm_w=None, eps: float = 1e-6):
        """norm_w: one [H] fp32 device tensor per layer for the decoder-block
        form (residual stream and RMS norm around every layer), or None."""
        self.layers = list(layers)
        H = self.layers[0].H
        self.descs = (moe_layer_desc * len(self.layers))(*[l.desc for l in self.layers])
        self.ws = Workspace(self.layers[0].desc, 1, device=device)
        self.tok = torch.zeros(1, H, dtype=torch.bfloat16, device=device)
        self.norm_w = None if norm_w is None else [w.contiguous() for w in norm_w]
        self.eps = eps
        self.graph = None

    def set_input(self, x: torch.Tensor):
        self.tok.copy_(x.reshape(self.tok.shape))

    def step_eager(self, stream=None):
        if self.norm_w is None:
            _lib.moe_decode_layers(self.descs, self.tok, self.tok, self.ws.buf, stream)
        else:
            _lib.moe_decode_layers_block(self.descs, self.norm_w, self.eps, self.tok, self.tok, self.ws.buf, stream)

    def layer_outputs_eager(self, x: torch.Tensor):
        """Run the layers one moe_decode call at a time and keep every output."""
        outs = []
        cur = x.reshape(self.tok.shape).contiguous()
        for layer in self.layers:
            nxt = torch.empty_like(cur)
            _lib.moe_decode(layer.desc, cur, nxt, self.ws.buf)
            outs.append(nxt)
            cur = nxt
        return outs

    def capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        saved = self.tok.clone()
        with torch.cuda.stream(s):
            self.step_eager(s)  # warm-up outside the graph (lazy init, module load)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.tok.copy_(saved)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step_eager(torch.cuda.current_stream())
        self.graph = g
        return g

    def step(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def output(self) -> torch.Tensor:
        return self.tok
