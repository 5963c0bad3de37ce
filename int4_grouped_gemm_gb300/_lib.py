"""ctypes binding of libmoe_gb300.so: same names as the C ABI in include/moe.h.

Argument marshalling only: torch tensors are passed as raw device pointers and
every step of the layer runs in the library's CUDA kernels.  There is no CPU
fallback; loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

c_i32, c_i64, c_p, c_sz, c_ll = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_longlong

MOE_OK = 0
MOE_ERR_NULL = -1
MOE_ERR_ALIGN = -2
MOE_ERR_SHAPE = -3
MOE_ERR_TOKENS = -4
MOE_ERR_WORKSPACE = -5
MOE_ERR_CUDA = -6
MOE_ERR_TENSOR_MAP = -7
MOE_ERR_DEVICE = -8
MOE_ERR_TIMEOUT = -100


class moe_qweight(ctypes.Structure):
    _fields_ = [("q", c_p), ("scale", c_p), ("bias", c_p)]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("E", c_i32), ("k", c_i32), ("H", c_i32), ("I", c_i32), ("group", c_i32),
                ("has_shared", c_i32), ("router_w", c_p), ("router_bias", c_p),
                ("gate", moe_qweight), ("up", moe_qweight), ("down", moe_qweight),
                ("no_renorm", c_i32), ("shared_gate", c_p), ("router_split", c_p)]


class moe_routing_views(ctypes.Structure):
    _fields_ = [(n, c_i64) for n in ("logits", "topk_idx", "topk_w", "counts", "offsets", "perm",
                                      "inv_perm", "tile_group", "tile_row", "tile_rows", "tile_sched",
                                      "num_tiles", "h", "y_acc")] + \
        [("max_tiles", c_i32), ("tile_size", c_i32)]


class moe_batch_views(ctypes.Structure):
    _fields_ = [(n, c_i64) for n in ("logits", "slots", "slot_w", "h")] + \
        [("S_max", c_i32), ("logit_ld", c_i32), ("max_tokens", c_i32)]


MOE_DECODE_PHASES = 8
MOE_DECODE_TRACE_BLOCKS = 256


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


_lib = None

# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_workspace_bytes": (c_sz, [c_p, c_i32]),
    "moe_workspace_init": (ctypes.c_int, [c_p, c_sz, c_p]),
    "moe_router_split_bytes": (c_sz, [c_i32, c_i32]),
    "moe_split_router": (ctypes.c_int, [c_p, c_i32, c_i32, c_p, c_p]),
    "moe_routing_views_for": (ctypes.c_int, [c_p, c_i32, c_p]),
    "moe_prefill": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p, c_sz, c_p]),
    "moe_prefill_profiled": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p, c_sz, c_p, c_p]),
    "moe_decode": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_sz, c_p]),
    "moe_decode_layers": (ctypes.c_int, [c_p, c_i32, c_p, c_p, c_p, c_sz, c_p]),
    "moe_decode_batch": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p, c_sz, c_p]),
    "moe_prefill_block": (ctypes.c_int, [c_p, c_p, c_p, c_p, ctypes.c_float, c_i32, c_p, c_p, c_sz, c_p]),
    "moe_decode_batch_block": (ctypes.c_int, [c_p, c_p, c_p, c_p, ctypes.c_float, c_i32, c_p, c_p, c_sz, c_p]),
    "moe_decode_static_scratch": (ctypes.c_int, [c_p, c_p, c_p, c_p]),
    "moe_read_static_scratch_status": (ctypes.c_int, [c_p]),
    "moe_decode_layers_traced": (ctypes.c_int, [c_p, c_p, ctypes.c_float, c_i32, c_p, c_p, c_p, c_sz, c_p, c_p, c_p]),
    "moe_decode_layers_block": (ctypes.c_int, [c_p, c_p, ctypes.c_float, c_i32, c_p, c_p, c_p, c_sz, c_p]),
    "moe_decode_topk_logits": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p]),
    "moe_batch_views_for": (ctypes.c_int, [c_p, c_p]),
    "moe_block_views_for": (ctypes.c_int, [c_p, c_i32, c_i32, c_p, c_p]),
    "moe_route_logits": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_sz, c_p]),
    "pack_int4": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_p, c_p, c_p, c_p]),
    "moe_read_device_status": (ctypes.c_int, [c_p, c_p]),
    "moe_set_wait_limit": (c_ll, [c_ll]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [c_p, c_sz, c_ll, c_p]),
    "moe_forward_host": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "moe_forward_host_stream": (ctypes.c_int, [c_p, c_p, c_p, c_i32, c_i32, c_p, c_p, c_p, c_sz, c_p]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gqa_attention_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32]),
    "gqa_decode_attention": (ctypes.c_int, [c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.c_float, c_p,
                                            c_p, c_sz, c_p]),
    "gqa_decode_attention_per_head": (ctypes.c_int, [c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i32, c_i32,
                                                     ctypes.c_float, c_p, c_p, c_sz, c_p]),
}


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} not found: build it first (python -m int4_grouped_gemm_gb300.build)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoEError(rc, what)


def _ptr(t):
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


# --------------------------------------------------------------- calls


def moe_workspace_bytes(desc: moe_layer_desc, T_max: int) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(desc), T_max))


def moe_workspace_init(ws, stream=None):
    _check(load().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def moe_router_split_bytes(E: int, H: int) -> int:
    return int(load().moe_router_split_bytes(E, H))


def moe_split_router(router_w, E: int, H: int, out, stream=None):
    """out [2][E16][H] bf16 (a uint8 device tensor of moe_router_split_bytes
    bytes) = the hi/lo bf16 parts of router_w [E][H] fp32."""
    if out.numel() * out.element_size() < moe_router_split_bytes(E, H):
        raise MoEError(MOE_ERR_WORKSPACE, "moe_split_router: output too small")
    _check(load().moe_split_router(_ptr(router_w), E, H, _ptr(out), _stream(stream)), "moe_split_router")


def moe_routing_views_for(desc: moe_layer_desc, T: int) -> moe_routing_views:
    v = moe_routing_views()
    _check(load().moe_routing_views_for(ctypes.byref(desc), T, ctypes.byref(v)), "moe_routing_views_for")
    return v


def moe_prefill(desc: moe_layer_desc, x, T: int, y, ws, stream=None):
    _check(load().moe_prefill(ctypes.byref(desc), _ptr(x), T, _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_prefill")


def moe_prefill_profiled(desc: moe_layer_desc, x, T: int, y, ws, events, stream=None):
    """events: 6 torch.cuda.Event(enable_timing=True) recorded at the stage boundaries."""
    arr = (c_p * 6)(*[int(e.cuda_event) if e is not None else None for e in events])
    _check(load().moe_prefill_profiled(ctypes.byref(desc), _ptr(x), T, _ptr(y), _ptr(ws),
                                       ws.numel() * ws.element_size(), arr, _stream(stream)),
           "moe_prefill_profiled")


def moe_decode(desc: moe_layer_desc, x, y, ws, stream=None):
    _check(load().moe_decode(ctypes.byref(desc), _ptr(x), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "moe_decode")


def moe_decode_batch(desc: moe_layer_desc, x, y, ws, stream=None):
    """x, y: [B][H] bf16 with 1 <= B <= 8."""
    _check(load().moe_decode_batch(ctypes.byref(desc), _ptr(x), x.shape[0], _ptr(y), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)), "moe_decode_batch")


def moe_prefill_block(desc: moe_layer_desc, attn, residual, norm_w, eps, out, ws, stream=None):
    """out = bf16(MoE(RMSNorm(attn + residual) * norm_w) + (attn + residual))."""
    _check(load().moe_prefill_block(ctypes.byref(desc), _ptr(attn), _ptr(residual), _ptr(norm_w), float(eps),
                                    attn.shape[0], _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "moe_prefill_block")


def moe_decode_batch_block(desc: moe_layer_desc, attn, residual, norm_w, eps, out, ws, stream=None):
    """The decoder-block form of moe_decode_batch (1 to 8 tokens)."""
    _check(load().moe_decode_batch_block(ctypes.byref(desc), _ptr(attn), _ptr(residual), _ptr(norm_w), float(eps),
                                         attn.shape[0], _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "moe_decode_batch_block")


def moe_decode_layers(descs, x, y, ws, stream=None):
    """descs: a ctypes array of moe_layer_desc (one per layer)."""
    _check(load().moe_decode_layers(ctypes.cast(descs, c_p), len(descs), _ptr(x), _ptr(y), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "moe_decode_layers")


def moe_decode_static_scratch(desc: moe_layer_desc, x, y, stream=None):
    """moe_decode on the library's fixed scratch array (no workspace)."""
    _check(load().moe_decode_static_scratch(ctypes.byref(desc), _ptr(x), _ptr(y), _stream(stream)),
           "moe_decode_static_scratch")


def moe_read_static_scratch_status(stream=None) -> int:
    """Read and clear the status word of the static-scratch decode on the current device."""
    return int(load().moe_read_static_scratch_status(_stream(stream)))


def _norm_ptrs(norm_w):
    """A ctypes array of the layers' norm-weight device pointers (or None)."""
    if norm_w is None:
        return None
    return (c_p * len(norm_w))(*[_ptr(w) for w in norm_w])


def moe_decode_layers_traced(descs, x, y, ws, routing_trace=None, time_trace=None, norm_w=None, eps=1e-6,
                             stream=None):
    """moe_decode_layers (or, with norm_w, moe_decode_layers_block) that also
    records each layer's routing (routing_trace: float32 [n_layers][E + 2k + 1])
    and per-block phase time stamps (time_trace: int64 [n_layers]
    [MOE_DECODE_TRACE_BLOCKS][MOE_DECODE_PHASES])."""
    nw = _norm_ptrs(norm_w)
    _check(load().moe_decode_layers_traced(ctypes.cast(descs, c_p), nw, float(eps), len(descs), _ptr(x), _ptr(y),
                                           _ptr(ws), ws.numel() * ws.element_size(), _ptr(routing_trace),
                                           _ptr(time_trace), _stream(stream)), "moe_decode_layers_traced")


def moe_decode_layers_block(descs, norm_w, eps, x, y, ws, stream=None):
    """The decoder-block form of moe_decode_layers: norm_w holds one [H] fp32
    device tensor per layer; the token is the residual stream."""
    if len(norm_w) != len(descs):
        raise ValueError("moe_decode_layers_block: one norm weight per layer")
    _check(load().moe_decode_layers_block(ctypes.cast(descs, c_p), _norm_ptrs(norm_w), float(eps), len(descs),
                                          _ptr(x), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)), "moe_decode_layers_block")


def moe_decode_topk_logits(desc: moe_layer_desc, logits, out, stream=None):
    """The decode kernel's top-k on given logits [n][E]; out float32 [n][E + 2k + 1]."""
    _check(load().moe_decode_topk_logits(ctypes.byref(desc), _ptr(logits), logits.shape[0], _ptr(out),
                                         _stream(stream)), "moe_decode_topk_logits")


def moe_batch_views_for(desc: moe_layer_desc) -> moe_batch_views:
    v = moe_batch_views()
    _check(load().moe_batch_views_for(ctypes.byref(desc), ctypes.byref(v)), "moe_batch_views_for")
    return v


def moe_block_views_for(desc: moe_layer_desc, T: int, small_batch: bool):
    h, x = c_i64(), c_i64()
    _check(load().moe_block_views_for(ctypes.byref(desc), T, int(small_batch), ctypes.byref(h), ctypes.byref(x)),
           "moe_block_views_for")
    return h.value, x.value


def moe_route_logits(desc: moe_layer_desc, logits, T: int, ws, stream=None):
    _check(load().moe_route_logits(ctypes.byref(desc), _ptr(logits), T, _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)), "moe_route_logits")


def pack_int4(w, rows: int, K: int, group: int, q, scale, bias, stream=None):
    _check(load().pack_int4(_ptr(w), rows, K, group, _ptr(q), _ptr(scale), _ptr(bias), _stream(stream)),
           "pack_int4")


def moe_read_device_status(ws, stream=None) -> int:
    return int(load().moe_read_device_status(_ptr(ws), _stream(stream)))


def moe_set_wait_limit(cycles: int) -> int:
    return int(load().moe_set_wait_limit(int(cycles)))


def moe_selftest_wait_timeout(ws, limit_cycles: int, stream=None):
    _check(load().moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(limit_cycles),
                                            _stream(stream)), "moe_selftest_wait_timeout")


def moe_forward_host(desc: moe_layer_desc, x_host, T: int, y_host, x_dev, y_dev, ws, stream=None):
    _check(load().moe_forward_host(ctypes.byref(desc), _ptr(x_host), T, _ptr(y_host), _ptr(x_dev), _ptr(y_dev),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward_host")


def moe_forward_host_stream(desc: moe_layer_desc, x_hosts, T: int, y_hosts, x_devs, y_devs, ws, stream=None):
    """len(x_hosts) pipelined calls; x_devs / y_devs: two device staging tensors each."""
    n = len(x_hosts)
    if len(y_hosts) != n or len(x_devs) != 2 or len(y_devs) != 2:
        raise ValueError("moe_forward_host_stream: n host inputs and outputs, two device staging buffers each")
    arr = ctypes.c_void_p * n
    pair = ctypes.c_void_p * 2
    xs = arr(*[_ptr(t) for t in x_hosts])
    ys = arr(*[_ptr(t) for t in y_hosts])
    xd = pair(*[_ptr(t) for t in x_devs])
    yd = pair(*[_ptr(t) for t in y_devs])
    _check(load().moe_forward_host_stream(ctypes.byref(desc), xs, ys, n, T, xd, yd, _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward_host_stream")


# ---------------------------------------------------- GQA decode attention


def gqa_attention_workspace_bytes(Hq: int, Hkv: int, D: int, L: int) -> int:
    return int(load().gqa_attention_workspace_bytes(Hq, Hkv, D, L))


def gqa_decode_attention(q, k_cache, v_cache, L: int, scale: float, out, ws, per_head: bool = False, stream=None):
    """q [Hq, D], k_cache / v_cache [Hkv, L_cap, D] bf16 (device); out [Hq, D]."""
    Hq, D = q.shape
    Hkv, L_cap, _ = k_cache.shape
    fn = load().gqa_decode_attention_per_head if per_head else load().gqa_decode_attention
    _check(fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), Hq, Hkv, D, L, L_cap, float(scale), _ptr(out), _ptr(ws),
              ws.numel() * ws.element_size(), _stream(stream)), "gqa_decode_attention")
