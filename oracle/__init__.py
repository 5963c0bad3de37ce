"""CPU oracle for the int4 MoE layer (ctypes wrapper around ``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the CPU-baseline leg of ``bench.py``; never by the library.  It shares no code
with the CUDA path.  Every function here only marshals numpy arrays; the
arithmetic is in ``moe_oracle.c`` (whose header cites the passages it follows).

Parity status: quantiser, dequant, router, top-k, routing tables, the
dense single-expert case, the residual add / RMS norm steps around the
layer and the GQA decode attention of the second workload are pinned by
``tests/test_oracle_pins.py``; the
whole layer beyond those pins is "parity unpinned" (the pages print no worked
example or output value).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP, no contraction)."""
    stamp = _LIB + ".host"
    host = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != host:
        force = True
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
        with open(stamp, "w") as f:
            f.write(host + "\n")
    return _LIB


_lib = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


def lib():
    """The compiled oracle.  MOE_ORACLE_LIB names another build of the same
    source to load instead (the mutation tests load deliberately broken
    copies that way, to show that the pins catch them)."""
    global _lib
    if _lib is None:
        path = os.environ.get("MOE_ORACLE_LIB")
        if not path:
            build()
            path = _LIB
        L = ctypes.CDLL(path)
        L.oracle_bf16_round.argtypes = [_p, _i64, _p]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_quantize.argtypes = [_p, _i64, _i32, _i32, _p, _p, _p]
        L.oracle_dequant.argtypes = [_p, _p, _p, _i64, _i32, _i32, _p]
        L.oracle_router_logits.argtypes = [_p, _i32, _i32, _p, _p, _i32, _p]
        L.oracle_topk.argtypes = [_p, _i32, _i32, _i32, _p, _p]
        L.oracle_topk_opt.argtypes = [_p, _i32, _i32, _i32, _i32, _p, _p]
        L.oracle_shared_gate.argtypes = [_p, _i32, _i32, _p, _p]
        L.oracle_route.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p, _p, _p, _i32]
        L.oracle_route.restype = _i32
        L.oracle_moe_layer.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p] + [_p] * 9 + \
            [_p, _i32, _p, _p, _p, _p]
        L.oracle_moe_layer_opt.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p] + \
            [_p] * 9 + [_p, _i32, _p, _p, _p, _p, _p]
        L.oracle_experts_given_routing.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, _i32, _i32] + [_p] * 9 + \
            [_p, _p, _p, _p]
        L.oracle_dispatch_combine_identity.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, _p, _p, _p]
        L.oracle_residual_rmsnorm.argtypes = [_p, _p, _i32, _i32, _p, ctypes.c_double, _p, _p]
        L.oracle_residual_out.argtypes = [_p, _p, _i64, _p]
        L.oracle_gqa_attention.argtypes = [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, ctypes.c_double, _p]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads of the oracle's parallel loops from now on; returns the previous count."""
    return int(lib().oracle_set_num_threads(int(n)))


def bf16_round(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_round(_ptr(x), x.size, _ptr(out))
    return out


def quantize(w: np.ndarray, group: int):
    """w [rows, K] fp32 -> (q uint32 [rows, K/8], scale uint16 [rows, K/G], bias uint16)."""
    w = _c(w, np.float32)
    rows, K = w.shape
    assert K % 8 == 0 and K % group == 0
    q = np.empty((rows, K // 8), np.uint32)
    s = np.empty((rows, K // group), np.uint16)
    b = np.empty((rows, K // group), np.uint16)
    lib().oracle_quantize(_ptr(w), rows, K, group, _ptr(q), _ptr(s), _ptr(b))
    return q, s, b


def dequant(q: np.ndarray, s: np.ndarray, b: np.ndarray, K: int, group: int) -> np.ndarray:
    q = _c(q, np.uint32)
    s = _c(s, np.uint16)
    b = _c(b, np.uint16)
    rows = q.shape[0]
    out = np.empty((rows, K), np.float64)
    lib().oracle_dequant(_ptr(q), _ptr(s), _ptr(b), rows, K, group, _ptr(out))
    return out


def router_logits(x_bits: np.ndarray, Wr: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    Wr = _c(Wr, np.float32)
    T, H = x_bits.shape
    E = Wr.shape[0]
    bias = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    lib().oracle_router_logits(_ptr(x_bits), T, H, _ptr(Wr), _ptr(bias), E, _ptr(out))
    return out


def topk(logits: np.ndarray, k: int, renorm: bool = True):
    """Top-k of every row; weights renormalised over the picked (default) or
    the picked softmax probabilities as they are (renorm=False)."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_topk_opt(_ptr(logits), T, E, k, int(renorm), _ptr(idx), _ptr(w))
    return idx, w


def shared_gate(x_bits: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """Per-token weight of a gated shared expert: sigmoid(x . gate)."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    gate = _c(gate, np.float32)
    out = np.empty(T, np.float64)
    lib().oracle_shared_gate(_ptr(x_bits), T, H, _ptr(gate), _ptr(out))
    return out


def route(idx: np.ndarray, E: int, has_shared: bool, BN: int) -> dict:
    idx = _c(idx, np.int32)
    T, k = idx.shape
    G = E + (1 if has_shared else 0)
    counts = np.empty(G, np.int32)
    offsets = np.empty(G + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    max_tiles = (T * k + T) // BN + G + 1
    tg = np.empty(max_tiles, np.int32)
    tr = np.empty(max_tiles, np.int32)
    tn = np.empty(max_tiles, np.int32)
    n = lib().oracle_route(_ptr(idx), T, k, E, int(has_shared), BN, _ptr(counts), _ptr(offsets),
                           _ptr(perm), _ptr(inv), _ptr(tg), _ptr(tr), _ptr(tn), max_tiles)
    assert n >= 0
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv,
                tile_group=tg[:n].copy(), tile_row=tr[:n].copy(), tile_rows=tn[:n].copy())


class QWeights:
    """Oracle-side int4 weights of one layer: stacked over experts (index E = shared)."""

    def __init__(self, q, s, b, rows, K, group):
        self.q, self.s, self.b = q, s, b
        self.rows, self.K, self.group = rows, K, group


def quantize_stack(w: np.ndarray, group: int) -> QWeights:
    """w [n_exp, rows, K] fp32 -> packed stack with the same leading dims."""
    n, rows, K = w.shape
    q, s, b = quantize(w.reshape(n * rows, K), group)
    return QWeights(q.reshape(n, rows, K // 8), s.reshape(n, rows, K // group),
                    b.reshape(n, rows, K // group), rows, K, group)


def moe_layer(x_bits: np.ndarray, Wr: np.ndarray, bias: Optional[np.ndarray], gate: QWeights,
              up: QWeights, down: QWeights, E: int, k: int, has_shared: bool,
              tokens: Optional[np.ndarray] = None, renorm: bool = True,
              shared_gate_w: Optional[np.ndarray] = None) -> dict:
    """Full layer for the listed tokens (all by default); y is fp64 [n, H].
    Routing variants: renorm=False keeps the picked softmax probabilities;
    shared_gate_w ([H] fp32) gates the shared expert per token."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    I = gate.rows
    G = gate.group
    Wr = _c(Wr, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    n = tokens.shape[0]
    logits = np.empty((n, E), np.float32)
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    y = np.empty((n, H), np.float64)
    arrays = [gate.q, gate.s, gate.b, up.q, up.s, up.b, down.q, down.s, down.b]
    arrays = [_c(a, a.dtype) for a in arrays]
    sw = np.empty(n, np.float64)
    sg = None if shared_gate_w is None else _c(shared_gate_w, np.float32)
    lib().oracle_moe_layer_opt(_ptr(x_bits), T, H, I, E, k, G, int(has_shared), int(renorm), _ptr(Wr),
                               _ptr(bias), _ptr(sg), *[_ptr(a) for a in arrays], _ptr(tokens), n,
                               _ptr(logits), _ptr(idx), _ptr(w), _ptr(y), _ptr(sw))
    return dict(logits=logits, idx=idx, w=w, y=y, tokens=tokens, shared_w=sw)


def residual_rmsnorm(a_bits: np.ndarray, r_bits: np.ndarray, norm_w: np.ndarray, eps: float):
    """Residual add and RMS norm before the layer: (h, x) as bf16 bit patterns."""
    a_bits = _c(a_bits, np.uint16)
    r_bits = _c(r_bits, np.uint16)
    T, H = a_bits.shape
    assert r_bits.shape == (T, H)
    norm_w = _c(norm_w, np.float32)
    h = np.empty((T, H), np.uint16)
    x = np.empty((T, H), np.uint16)
    lib().oracle_residual_rmsnorm(_ptr(a_bits), _ptr(r_bits), T, H, _ptr(norm_w), float(eps), _ptr(h), _ptr(x))
    return h, x


def residual_out(h_bits: np.ndarray, y: np.ndarray) -> np.ndarray:
    """The residual add after the layer: bf16(h + y), y fp64, as bf16 bits."""
    h_bits = _c(h_bits, np.uint16)
    y = _c(y, np.float64)
    assert y.shape == h_bits.shape
    out = np.empty(h_bits.shape, np.uint16)
    lib().oracle_residual_out(_ptr(h_bits), _ptr(y), h_bits.size, _ptr(out))
    return out


def moe_block(a_bits, r_bits, norm_w, eps, Wr, bias, gate: QWeights, up: QWeights, down: QWeights, E: int, k: int,
              has_shared: bool, **kw) -> dict:
    """The layer with the steps either side of it: h = a + r, x = RMSNorm(h) w,
    out = bf16(h + MoE(x)); returns the layer's dict plus h, x and out (bits)."""
    h, x = residual_rmsnorm(a_bits, r_bits, norm_w, eps)
    r = moe_layer(x, Wr, bias, gate, up, down, E, k, has_shared, **kw)
    tok = r["tokens"]
    r.update(h=h, x=x, out=residual_out(h[tok], r["y"]))
    return r


def experts_given_routing(x_bits, gate: QWeights, up: QWeights, down: QWeights, E, has_shared,
                          idx: np.ndarray, w: np.ndarray, shared_w: Optional[np.ndarray] = None) -> np.ndarray:
    """Experts and combine under a given routing (idx [T, k], w [T, k]); the
    shared expert weighs 1, or shared_w [T] per token."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    k = idx.shape[1]
    sw = None if shared_w is None else _c(shared_w, np.float64)
    assert sw is None or sw.shape == (T,)
    y = np.empty((T, H), np.float64)
    arrays = [_c(a, a.dtype) for a in [gate.q, gate.s, gate.b, up.q, up.s, up.b, down.q, down.s, down.b]]
    lib().oracle_experts_given_routing(_ptr(x_bits), T, H, gate.rows, E, k, gate.group, int(has_shared),
                                       *[_ptr(a) for a in arrays], _ptr(idx), _ptr(w), _ptr(sw), _ptr(y))
    return y


def dispatch_combine_identity(x_bits, E, has_shared, idx, w) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    y = np.empty((T, H), np.float64)
    lib().oracle_dispatch_combine_identity(_ptr(x_bits), T, H, E, idx.shape[1], int(has_shared),
                                           _ptr(idx), _ptr(w), _ptr(y))
    return y


def gqa_attention(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, L: int, scale: float) -> np.ndarray:
    """Decode attention of one token (second workload): q [Hq, D], k / v
    [Hkv, L_cap, D] bf16 bit patterns, the first L positions attended;
    query head h uses key-value head h // (Hq // Hkv).  Returns fp64 [Hq, D]."""
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    v_bits = _c(v_bits, np.uint16)
    Hq, D = q_bits.shape
    Hkv, L_cap, D2 = k_bits.shape
    assert D2 == D and v_bits.shape == k_bits.shape and Hq % Hkv == 0 and 1 <= L <= L_cap
    o = np.empty((Hq, D), np.float64)
    lib().oracle_gqa_attention(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), Hq, Hkv, D, L, L_cap, float(scale), _ptr(o))
    return o
