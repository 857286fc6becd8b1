"""CPU oracle for the BRA forward (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package. It wraps the double-precision C implementation in
`bra_oracle.c` through ctypes; arrays are numpy float64 (inputs are widened
exactly from float32 / bfloat16 values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bra_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        sig = {
            "oracle_region_means": [P, I, I, I, I, I, P],
            "oracle_affinity": [P, P, I, I, I, I, I, P],
            "oracle_topk": [P, I, I, I, P],
            "oracle_route": [P, P, I, I, I, I, I, I, P, P],
            "oracle_routed_attention": [P, P, P, P, I, I, I, I, I, I, I, P, I],
            "oracle_query_probs": [P, P, P, P, I, I, I, I, I, I, I, I, I, I, I, P, P, P],
            "oracle_lepe": [P, I, I, I, I, P, P, I, P],
            "oracle_attend": [P, P, P, P, I, I, I, I, I, I, I, P, P, I, P, I],
            "oracle_forward": [P, P, P, I, I, I, I, I, I, I, P, P, I, P, P, I],
            "oracle_qkv_project": [P, I, I, P, P, P, P, P],
            "oracle_layer_norm": [P, I, I, P, P, ctypes.c_double, P],
            "oracle_linear": [P, I, I, P, I, P, P],
            "oracle_gelu": [P, ctypes.c_size_t, P],
            "oracle_attend_backward": [P, P, P, P, I, I, I, I, I, I, I, P, I, P, P, P, P, P,
                                       P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: invalid argument (status {rc})")


def region_means(x, S: int) -> np.ndarray:
    x = _f64(x)
    B, H, W, C = x.shape
    out = np.empty((B, S * S, C))
    _check(_load().oracle_region_means(_p(x), B, H, W, C, S, _p(out)), "region_means")
    return out


def affinity(q, k, S: int) -> np.ndarray:
    q, k = _f64(q), _f64(k)
    B, H, W, C = q.shape
    A = np.empty((B, S * S, S * S))
    _check(_load().oracle_affinity(_p(q), _p(k), B, H, W, C, S, _p(A)), "affinity")
    return A


def topk(A, topk: int) -> np.ndarray:
    """Top-k of each row of A (last axis), largest first, ties to lowest index."""
    A = _f64(A)
    R = A.shape[-1]
    rows = int(np.prod(A.shape[:-1]))
    idx = np.empty(A.shape[:-1] + (topk,), dtype=np.int32)
    _check(_load().oracle_topk(_p(A), rows, R, topk, _p(idx)), "topk")
    return idx


def route(q, k, S: int, topk: int):
    """Returns (idx [B, S*S, topk] int32, affinity [B, S*S, S*S] float64)."""
    q, k = _f64(q), _f64(k)
    B, H, W, C = q.shape
    idx = np.empty((B, S * S, topk), dtype=np.int32)
    A = np.empty((B, S * S, S * S))
    _check(_load().oracle_route(_p(q), _p(k), B, H, W, C, S, topk, _p(idx), _p(A)), "route")
    return idx, A


def routed_attention(q, k, v, idx, heads: int, S: int, threads: int = 1) -> np.ndarray:
    q, k, v, idx = _f64(q), _f64(k), _f64(v), _i32(idx)
    B, H, W, C = q.shape
    out = np.empty_like(q)
    _check(_load().oracle_routed_attention(_p(q), _p(k), _p(v), _p(idx), B, H, W, C,
                                           heads, S, idx.shape[-1], _p(out), threads),
           "routed_attention")
    return out


def query_probs(q, k, v, idx, heads: int, S: int, b: int, y: int, x: int, h: int):
    """(probs [k*n], key token ids y*W+x [k*n], out [d]) of one query."""
    q, k, v, idx = _f64(q), _f64(k), _f64(v), _i32(idx)
    B, H, W, C = q.shape
    topk = idx.shape[-1]
    n = (H // S) * (W // S)
    probs = np.empty(topk * n)
    keys = np.empty(topk * n, dtype=np.int32)
    out = np.empty(C // heads)
    _check(_load().oracle_query_probs(_p(q), _p(k), _p(v), _p(idx), B, H, W, C, heads, S,
                                      topk, b, y, x, h, _p(probs), _p(keys), _p(out)),
           "query_probs")
    return probs, keys, out


def lepe(v, w, bias) -> np.ndarray:
    v, w = _f64(v), _f64(w)
    bias = None if bias is None else _f64(bias)
    B, H, W, C = v.shape
    out = np.empty_like(v)
    _check(_load().oracle_lepe(_p(v), B, H, W, C, _p(w), _p(bias), w.shape[-1], _p(out)),
           "lepe")
    return out


def attend(q, k, v, idx, heads: int, S: int, w, bias, threads: int = 1) -> np.ndarray:
    q, k, v, idx, w = _f64(q), _f64(k), _f64(v), _i32(idx), _f64(w)
    bias = None if bias is None else _f64(bias)
    B, H, W, C = q.shape
    out = np.empty_like(q)
    _check(_load().oracle_attend(_p(q), _p(k), _p(v), _p(idx), B, H, W, C, heads, S,
                                 idx.shape[-1], _p(w), _p(bias), w.shape[-1], _p(out),
                                 threads), "attend")
    return out


def attend_backward(q, k, v, idx, heads: int, S: int, w, dout):
    """Gradients of attend's output (attention + LePE, the routing fixed) for
    the upstream gradient dout: (dq, dk, dv, dw, db)."""
    q, k, v, idx, w, dout = _f64(q), _f64(k), _f64(v), _i32(idx), _f64(w), _f64(dout)
    B, H, W, C = q.shape
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dw = np.empty_like(w)
    db = np.empty(C)
    _check(_load().oracle_attend_backward(_p(q), _p(k), _p(v), _p(idx), B, H, W, C, heads, S,
                                          idx.shape[-1], _p(w), w.shape[-1], _p(dout), _p(dq),
                                          _p(dk), _p(dv), _p(dw), _p(db)), "attend_backward")
    return dq, dk, dv, dw, db


def forward(q, k, v, heads: int, S: int, topk: int, w, bias, threads: int = 1):
    """Returns (out [B, H, W, C] float64, idx [B, S*S, topk] int32)."""
    q, k, v, w = _f64(q), _f64(k), _f64(v), _f64(w)
    bias = None if bias is None else _f64(bias)
    B, H, W, C = q.shape
    out = np.empty_like(q)
    idx = np.empty((B, S * S, topk), dtype=np.int32)
    _check(_load().oracle_forward(_p(q), _p(k), _p(v), B, H, W, C, heads, S, topk,
                                  _p(w), _p(bias), w.shape[-1], _p(idx), _p(out), threads),
           "forward")
    return out, idx


def qkv_project(x, w, bias=None):
    """(q, k, v) = the three C-column blocks of x W^T + bias, per token.
    x [..., C]; w [3C, C]; bias [3C] or None. Returns float64 arrays of x's
    shape."""
    x, w = _f64(x), _f64(w)
    bias = None if bias is None else _f64(bias)
    C = x.shape[-1]
    if w.shape != (3 * C, C):
        raise ValueError("w must be [3C, C]")
    M = int(np.prod(x.shape[:-1]))
    q, k, v = (np.empty_like(x) for _ in range(3))
    _check(_load().oracle_qkv_project(_p(x), M, C, _p(w), _p(bias), _p(q), _p(k), _p(v)),
           "qkv_project")
    return q, k, v


def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """nn.LayerNorm over the last axis (biased variance), float64."""
    x = _f64(x)
    C = x.shape[-1]
    gamma = None if gamma is None else _f64(gamma)
    beta = None if beta is None else _f64(beta)
    y = np.empty_like(x)
    _check(_load().oracle_layer_norm(_p(x), int(np.prod(x.shape[:-1])), C, _p(gamma), _p(beta),
                                     float(eps), _p(y)), "layer_norm")
    return y


def block_attention(x, ln_w, ln_b, w_qkv, b_qkv, heads: int, S: int, topk: int, lepe_w,
                    lepe_b, eps: float = 1e-5, threads: int = 1):
    """The attention branch of the BiFormer block (p3 "BiFormer架构核心思想解析"
    §3.1): y = x + bra(norm1(x)), bra being the projections of p1 §3 followed
    by the routed attention + LePE. Returns (y, idx, the stages: normalised x,
    q, k, v)."""
    x = _f64(x)
    xn = layer_norm(x, ln_w, ln_b, eps)
    q, k, v = qkv_project(xn, w_qkv, b_qkv)
    out, idx = forward(q, k, v, heads, S, topk, lepe_w, lepe_b, threads=threads)
    return x + out, idx, (xn, q, k, v)


def linear(x, w, bias=None) -> np.ndarray:
    """nn.Linear over the last axis: x [..., K], w [N, K], bias [N] or None."""
    x, w = _f64(x), _f64(w)
    bias = None if bias is None else _f64(bias)
    K = x.shape[-1]
    N = w.shape[0]
    if w.shape != (N, K):
        raise ValueError("w must be [N, K]")
    M = int(np.prod(x.shape[:-1]))
    y = np.empty(x.shape[:-1] + (N,))
    _check(_load().oracle_linear(_p(x), M, K, _p(w), N, _p(bias), _p(y)), "linear")
    return y


def gelu(x) -> np.ndarray:
    """nn.GELU, exact (erf) form."""
    x = _f64(x)
    y = np.empty_like(x)
    _check(_load().oracle_gelu(_p(x), x.size, _p(y)), "gelu")
    return y


def block_ffn(x, ln_w, ln_b, w1, b1, conv_w, conv_b, w2, b2, eps: float = 1e-5):
    """The ConvFFN branch of the BiFormer block (p3 "BiFormer架构核心思想解析"
    §3.1 `x = x + self.ffn(self.norm2(x))`; p1 §4 ratio 3): y = x +
    fc2(GELU(dwconv3x3(fc1(norm2(x))))). x [B, H, W, C]; w1 [3C, C]; conv_w
    [3C, 3, 3], conv_b [3C] (the depthwise convolution, zero padding 1, the
    same operation as the LePE's); w2 [C, 3C]. Returns (y, the stages: x_n,
    fc1 output, convolved, activated)."""
    x = _f64(x)
    xn = layer_norm(x, ln_w, ln_b, eps)
    h = linear(xn, w1, b1)
    hc = lepe(h, conv_w, conv_b)
    ha = gelu(hc)
    return x + linear(ha, w2, b2), (xn, h, hc, ha)
