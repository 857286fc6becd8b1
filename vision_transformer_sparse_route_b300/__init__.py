"""Bi-Level Routing Attention (BRA) forward on B300 (sm_103a).

Python binding of the C ABI declared in include/bra.h. It only marshals
arguments: every step of the computation runs in the CUDA kernels of
libbra.so, and importing fails loudly when that library has not been built
(`python -m vision_transformer_sparse_route_b300.build`). Tensors are torch
tensors (torch supplies device memory and streams), contiguous, channels-last
[B, H, W, C], float32 or bfloat16.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["BraError", "qkv_project", "route", "attend", "attend_backward", "attend_tc", "forward", "forward_static", "forward_host",
           "HostPipeline",
           "idx_workspace_bytes", "forward_launches", "device_status", "check_wait_timeout", "library_path",
           "SYMBOLS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libbra.so")

BRA_OK, BRA_ERR_INVALID_ARG, BRA_ERR_UNSUPPORTED, BRA_ERR_CUDA, BRA_ERR_TIMEOUT = range(5)
BRA_F32, BRA_BF16 = 0, 1

# Entry points of include/bra.h with their ctypes signatures.
_P, _I = ctypes.c_void_p, ctypes.c_int
SYMBOLS = {
    "bra_route": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "bra_attend": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P]),
    "bra_attend_tc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P]),
    "bra_forward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P]),
    "bra_forward_static": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P]),
    "bra_qkv_project": (_I, [_P, _P, _P, ctypes.c_longlong, _I, _I, _P, _P, _P, _P]),
    "bra_idx_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "bra_forward_launches": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "bra_device_status": (_I, [_P, _I]),
    "bra_status_string": (ctypes.c_char_p, [_I]),
    "bra_abi_version": (_I, []),
    "bra_check_wait_timeout": (_I, [ctypes.c_uint64, _P]),
    "bra_layer_norm": (_I, [_P, _P, _P, ctypes.c_longlong, _I, ctypes.c_float, _I, _P, _P]),
    "bra_residual_add": (_I, [_P, _P, ctypes.c_longlong, _I, _P, _P]),
    "bra_block_attention_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "bra_linear": (_I, [_P, _P, _P, ctypes.c_longlong, _I, _I, _P, _I, _P, _P]),
    "bra_dwconv_gelu": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "bra_block_ffn_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "bra_block_ffn": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                           _I, _P, _P, _P]),
    "bra_block_attention": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _I, _I, _I, _I, _I, _I,
                                 _I, _P, _P, _I, _I, _P, _P, _P]),
    "bra_attend_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I,
                                 _P, _P, _P, _P, _P, _P]),
}

_lib = None


class BraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m vision_transformer_sparse_route_b300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SYMBOLS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return _load().bra_status_string(status).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return BRA_F32
    if t.dtype == torch.bfloat16:
        return BRA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str) -> None:
    if rc != BRA_OK:
        raise BraError(rc, what)


def _map(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, W, C]")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.shape


def idx_workspace_bytes(B: int, S: int, topk: int) -> int:
    return _load().bra_idx_workspace_bytes(B, S, topk)


def forward_launches(B: int, H: int, W: int, C: int, heads: int, S: int, topk: int,
                     lepe_ks: int, dtype: int = BRA_BF16) -> int:
    """Kernels one bra_forward enqueues for this problem (1 or 2)."""
    n = _load().bra_forward_launches(B, H, W, C, heads, S, topk, lepe_ks, dtype)
    if n < 0:
        raise BraError(-n, "bra_forward_launches")
    return n


def route(q, k, S: int, topk: int, idx=None, affinity=None, stream=None):
    """Top-k region routing; returns idx int32 [B, S*S, topk] (and fills
    `affinity` float32 [B, S*S, S*S] when given)."""
    B, H, W, C = _map(q, "q")
    _map(k, "k")
    if idx is None:
        idx = torch.empty((B, S * S, topk), dtype=torch.int32, device=q.device)
    rc = _load().bra_route(_ptr(q), _ptr(k), B, H, W, C, S, topk, _dtype_code(q),
                           _ptr(idx), _ptr(affinity), _stream(stream))
    _check(rc, "bra_route")
    return idx


def attend(q, k, v, idx, heads: int, S: int, lepe_w, lepe_b=None, out=None, stream=None):
    """Routed attention + LePE given the routing index; returns out."""
    B, H, W, C = _map(q, "q")
    if out is None:
        out = torch.empty_like(q)
    topk = idx.shape[-1]
    rc = _load().bra_attend(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), B, H, W, C, heads, S,
                            topk, _ptr(lepe_w), _ptr(lepe_b), lepe_w.shape[-1],
                            _dtype_code(q), _ptr(out), _stream(stream))
    _check(rc, "bra_attend")
    return out


def attend_backward(q, k, v, idx, heads: int, S: int, lepe_w, dout, stream=None):
    """Gradients of attend's output for the upstream gradient dout, the
    routing fixed: (dq, dk, dv, dlepe_w, dlepe_b), float32."""
    B, H, W, C = _map(q, "q")
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=q.device) for _ in range(3))
    dw = torch.empty(lepe_w.shape, dtype=torch.float32, device=q.device)
    db = torch.empty(C, dtype=torch.float32, device=q.device)
    rc = _load().bra_attend_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), B, H, W, C, heads,
                                     S, idx.shape[-1], _ptr(lepe_w), lepe_w.shape[-1],
                                     _ptr(dout), _dtype_code(q), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(dw), _ptr(db), _stream(stream))
    _check(rc, "bra_attend_backward")
    return dq, dk, dv, dw, db


def qkv_project(x, w, bias=None, q=None, k=None, v=None, stream=None):
    """(q, k, v) = the per-token projections x W^T + bias of a [..., C] bf16
    tensor, with w [3C, C] bf16 and bias [3C] float32 (or None)."""
    if not x.is_contiguous() or not w.is_contiguous():
        raise ValueError("x and w must be contiguous")
    C = x.shape[-1]
    M = x.numel() // C
    q = torch.empty_like(x) if q is None else q
    k = torch.empty_like(x) if k is None else k
    v = torch.empty_like(x) if v is None else v
    rc = _load().bra_qkv_project(_ptr(x), _ptr(w), _ptr(bias), M, C, _dtype_code(x), _ptr(q),
                                 _ptr(k), _ptr(v), _stream(stream))
    _check(rc, "bra_qkv_project")
    return q, k, v


def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5, out=None, stream=None):
    """nn.LayerNorm over the last axis of a bf16 tensor (gamma, beta float32
    [C] or None); out may be x."""
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    C = x.shape[-1]
    out = torch.empty_like(x) if out is None else out
    rc = _load().bra_layer_norm(_ptr(x), _ptr(gamma), _ptr(beta), x.numel() // C, C, eps,
                                _dtype_code(x), _ptr(out), _stream(stream))
    _check(rc, "bra_layer_norm")
    return out


def residual_add(x, r, out=None, stream=None):
    """x + r (bf16, one rounding); out may be x or r."""
    if not (x.is_contiguous() and r.is_contiguous()) or x.shape != r.shape:
        raise ValueError("x and r must be contiguous and of one shape")
    out = torch.empty_like(x) if out is None else out
    rc = _load().bra_residual_add(_ptr(x), _ptr(r), x.numel(), _dtype_code(x), _ptr(out),
                                  _stream(stream))
    _check(rc, "bra_residual_add")
    return out


def block_attention(x, ln_w, ln_b, w_qkv, b_qkv, heads: int, S: int, topk: int, lepe_w,
                    lepe_b=None, eps: float = 1e-5, out=None, workspace=None, stream=None):
    """The attention branch of the BiFormer block: x + bra(norm1(x)), with the
    Q/K/V projections (w_qkv [3C, C] bf16, b_qkv [3C] float32) inside bra.
    Returns out [B, H, W, C] bf16."""
    B, H, W, C = _map(x, "x")
    lib = _load()
    if workspace is None:
        n = lib.bra_block_attention_workspace_bytes(B, H, W, C, S, topk)
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    out = torch.empty_like(x) if out is None else out
    rc = lib.bra_block_attention(_ptr(x), _ptr(ln_w), _ptr(ln_b), eps, _ptr(w_qkv), _ptr(b_qkv),
                                 B, H, W, C, heads, S, topk, _ptr(lepe_w), _ptr(lepe_b),
                                 lepe_w.shape[-1], _dtype_code(x), _ptr(workspace), _ptr(out),
                                 _stream(stream))
    _check(rc, "bra_block_attention")
    return out


def linear(x, w, bias=None, residual=None, out=None, stream=None):
    """x W^T + bias (+ residual) over the last axis: x [..., K] bf16, w [N, K]
    bf16, bias [N] float32 or None, residual [..., N] bf16 or None."""
    if not x.is_contiguous() or not w.is_contiguous():
        raise ValueError("x and w must be contiguous")
    K, N = x.shape[-1], w.shape[0]
    M = x.numel() // K
    out = torch.empty(x.shape[:-1] + (N,), dtype=x.dtype, device=x.device) if out is None \
        else out
    rc = _load().bra_linear(_ptr(x), _ptr(w), _ptr(bias), M, K, N, _ptr(residual),
                            _dtype_code(x), _ptr(out), _stream(stream))
    _check(rc, "bra_linear")
    return out


def dwconv_gelu(h, w, bias=None, out=None, stream=None):
    """GELU(depthwise 3x3 conv of h [B, H, W, Ch] bf16 with w [Ch, 3, 3] and
    bias [Ch] float32, zero padding 1)."""
    B, H, W, Ch = _map(h, "h")
    out = torch.empty_like(h) if out is None else out
    rc = _load().bra_dwconv_gelu(_ptr(h), _ptr(w), _ptr(bias), B, H, W, Ch, _dtype_code(h),
                                 _ptr(out), _stream(stream))
    _check(rc, "bra_dwconv_gelu")
    return out


def block_ffn(x, ln_w, ln_b, w1, b1, conv_w, conv_b, w2, b2, eps: float = 1e-5, out=None,
              workspace=None, stream=None):
    """The ConvFFN branch of the BiFormer block: x + fc2(GELU(dwconv3x3(fc1(
    norm2(x))))); w1 [3C, C], w2 [C, 3C] bf16, conv_w [3C, 3, 3] and the
    biases float32."""
    B, H, W, C = _map(x, "x")
    lib = _load()
    if workspace is None:
        workspace = torch.empty(lib.bra_block_ffn_workspace_bytes(B, H, W, C), dtype=torch.uint8,
                                device=x.device)
    out = torch.empty_like(x) if out is None else out
    rc = lib.bra_block_ffn(_ptr(x), _ptr(ln_w), _ptr(ln_b), eps, _ptr(w1), _ptr(b1),
                           _ptr(conv_w), _ptr(conv_b), _ptr(w2), _ptr(b2), B, H, W, C,
                           _dtype_code(x), _ptr(workspace), _ptr(out), _stream(stream))
    _check(rc, "bra_block_ffn")
    return out


def attend_tc(q, k, v, idx, heads: int, S: int, lepe_w, lepe_b=None, out=None, stream=None):
    """bra_attend on the tcgen05 tensor cores (8 x 8 regions, C = 64, topk <= 4)."""
    B, H, W, C = _map(q, "q")
    if out is None:
        out = torch.empty_like(q)
    topk = idx.shape[-1]
    rc = _load().bra_attend_tc(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), B, H, W, C, heads, S,
                               topk, _ptr(lepe_w), _ptr(lepe_b), lepe_w.shape[-1],
                               _dtype_code(q), _ptr(out), _stream(stream))
    _check(rc, "bra_attend_tc")
    return out


def forward(q, k, v, heads: int, S: int, topk: int, lepe_w, lepe_b=None, out=None,
            idx=None, stream=None):
    """The whole BRA forward on device tensors; returns (out, idx)."""
    B, H, W, C = _map(q, "q")
    if out is None:
        out = torch.empty_like(q)
    if idx is None:
        idx = torch.empty((B, S * S, topk), dtype=torch.int32, device=q.device)
    rc = _load().bra_forward(_ptr(q), _ptr(k), _ptr(v), B, H, W, C, heads, S, topk,
                             _ptr(lepe_w), _ptr(lepe_b), lepe_w.shape[-1], _dtype_code(q),
                             _ptr(idx), _ptr(out), _stream(stream))
    _check(rc, "bra_forward")
    return out, idx


# Routing-index entries the library's built-in array holds (include/bra.h).
STATIC_IDX_MAX_ENTRIES = 1 << 18


def forward_static(q, k, v, heads: int, S: int, topk: int, lepe_w, lepe_b=None, out=None,
                   stream=None):
    """The whole BRA forward without a routing-index workspace, for callers
    that may not allocate device memory: the index lives in an array inside
    the library, shared by every call on the device (calls that overlap on the
    GPU race on it). Returns out; B * S*S * topk must not exceed
    STATIC_IDX_MAX_ENTRIES. The first call on a device looks the array up and
    should come before any stream capture."""
    B, H, W, C = _map(q, "q")
    if out is None:
        out = torch.empty_like(q)
    rc = _load().bra_forward_static(_ptr(q), _ptr(k), _ptr(v), B, H, W, C, heads, S, topk,
                                    _ptr(lepe_w), _ptr(lepe_b), lepe_w.shape[-1],
                                    _dtype_code(q), _ptr(out), _stream(stream))
    _check(rc, "bra_forward_static")
    return out


class HostBuffers:
    """Device staging buffers for forward_host, reused across calls."""

    def __init__(self, shape, dtype, S: int, topk: int, device):
        self.q, self.k, self.v, self.out = (torch.empty(shape, dtype=dtype, device=device)
                                            for _ in range(4))
        self.idx = torch.empty((shape[0], S * S, topk), dtype=torch.int32, device=device)


def forward_host(q, k, v, heads: int, S: int, topk: int, lepe_w, lepe_b, out,
                 buffers: HostBuffers, stream=None):
    """BRA forward on host tensors (pinned for asynchronous copies): copies
    q, k, v to the device buffers, runs bra_forward and copies out back, all
    on `stream`. lepe_w / lepe_b are device tensors."""
    s = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.stream(s):
        buffers.q.copy_(q, non_blocking=True)
        buffers.k.copy_(k, non_blocking=True)
        buffers.v.copy_(v, non_blocking=True)
        forward(buffers.q, buffers.k, buffers.v, heads, S, topk, lepe_w, lepe_b,
                out=buffers.out, idx=buffers.idx, stream=s)
        out.copy_(buffers.out, non_blocking=True)
    return out


class HostPipeline:
    """BRA forwards on host tensors with copies and compute overlapped.

    Each `submit` copies one batch's q, k, v (pinned host tensors) to a device
    buffer set on a copy-in stream, runs bra_forward on a compute stream once
    they have landed, and copies out back on a copy-out stream. With `depth`
    buffer sets, batch i's compute overlaps batch i+1's copy-in and batch
    i-1's copy-out (the two copy directions use separate copy engines).
    Submissions return at once; `synchronize` waits for all of them. The host
    tensors passed to a submission must not change until it has completed.
    """

    def __init__(self, shape, dtype, S: int, topk: int, device, depth: int = 2):
        self.slots = [HostBuffers(shape, dtype, S, topk, device) for _ in range(depth)]
        self.copy_in = torch.cuda.Stream(device=device)
        self.compute = torch.cuda.Stream(device=device)
        self.copy_out = torch.cuda.Stream(device=device)
        self._free = [None] * depth  # copy-out of the slot's last batch done
        self._n = 0

    def submit(self, q, k, v, heads: int, S: int, topk: int, lepe_w, lepe_b, out):
        slot = self._n % len(self.slots)
        buf = self.slots[slot]
        if self._free[slot] is not None:
            self.copy_in.wait_event(self._free[slot])
        with torch.cuda.stream(self.copy_in):
            buf.q.copy_(q, non_blocking=True)
            buf.k.copy_(k, non_blocking=True)
            buf.v.copy_(v, non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(self.copy_in)
        self.compute.wait_event(landed)
        forward(buf.q, buf.k, buf.v, heads, S, topk, lepe_w, lepe_b, out=buf.out,
                idx=buf.idx, stream=self.compute)
        done = torch.cuda.Event()
        done.record(self.compute)
        self.copy_out.wait_event(done)
        with torch.cuda.stream(self.copy_out):
            out.copy_(buf.out, non_blocking=True)
            freed = torch.cuda.Event()
            freed.record(self.copy_out)
        self._free[slot] = freed
        self._n += 1
        return out

    def synchronize(self):
        self.copy_out.synchronize()


def check_wait_timeout(limit_ns: int = 2_000_000, stream=None) -> None:
    """Enqueues a kernel whose bounded wait must give up after limit_ns; the
    next device_status() reports BRA_ERR_TIMEOUT (see include/bra.h)."""
    _check(_load().bra_check_wait_timeout(limit_ns, _stream(stream)), "bra_check_wait_timeout")


def device_status(stream=None, clear: bool = True) -> int:
    """Synchronises the stream and returns the device status word as a
    status code (see include/bra.h)."""
    return _load().bra_device_status(_stream(stream), 1 if clear else 0)
