"""The attention branch of the BiFormer block around BRA (page "BiFormer架构
核心思想解析" §3.1: x = x + bra(norm1(x))): the LayerNorm and residual-add
kernels against the oracle, and bra_block_attention checked step by step,
each step against the oracle on the GPU's own inputs to that step."""
import numpy as np
import pytest
import torch

import bra_synth
import oracle
import vision_transformer_sparse_route_b300 as bra
from bra_synth import Workload
from parity import TOL, routing_report

pytestmark = pytest.mark.gpu


def bf16(a, device) -> torch.Tensor:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(device)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def ln_bound(ref: np.ndarray) -> np.ndarray:
    # one bf16 rounding of the output (half an ulp: 2^-9 relative) plus the
    # float32 statistics
    return 2.0 ** -8 * np.abs(ref) + 1e-4


def linear_bound(ref: np.ndarray) -> np.ndarray:
    # one bf16 rounding of the output (half an ulp, 2^-9 relative; twice
    # that as the bound) plus the float32 accumulation of at most 384
    # products of unit-size terms
    return 2.0 ** -8 * np.abs(ref) + 1e-3


@pytest.mark.parametrize("C", [64, 128, 256])
def test_layer_norm_matches_oracle(C, cuda_device):
    rng = np.random.default_rng(C)
    x = bf16(rng.standard_normal((3, 37, C)) * 2 + 0.5, cuda_device)  # 111 tokens: ragged
    g = rng.standard_normal(C).astype(np.float32)
    b = (0.5 * rng.standard_normal(C)).astype(np.float32)
    gt, bt = torch.from_numpy(g).to(cuda_device), torch.from_numpy(b).to(cuda_device)
    y = bra.layer_norm(x, gt, bt)
    ref = oracle.layer_norm(f64(x), g, b)
    assert np.all(np.abs(f64(y) - ref) <= ln_bound(ref))
    # no scale and shift; in place gives the same
    y0 = bra.layer_norm(x)
    ref0 = oracle.layer_norm(f64(x))
    assert np.all(np.abs(f64(y0) - ref0) <= ln_bound(ref0))
    xi = x.clone()
    bra.layer_norm(xi, gt, bt, out=xi)
    assert torch.equal(xi, y)


def test_layer_norm_rejects_other_shapes(cuda_device):
    x = torch.zeros((4, 96), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(bra.BraError):
        bra.layer_norm(x)
    with pytest.raises(bra.BraError):
        bra.layer_norm(torch.zeros((4, 64), device=cuda_device))


def test_residual_add_is_one_rounding(cuda_device):
    rng = np.random.default_rng(9)
    x = bf16(rng.standard_normal((5, 7, 64)) * 3, cuda_device)
    r = bf16(rng.standard_normal((5, 7, 64)), cuda_device)
    ref = (x.float() + r.float()).to(torch.bfloat16)  # torch's round-to-nearest-even
    assert torch.equal(bra.residual_add(x, r), ref)
    rr = r.clone()
    bra.residual_add(x, rr, out=rr)
    assert torch.equal(rr, ref)


BLOCK_SHAPES = [
    Workload("blk_n64_top2", 2, 16, 16, 64, 2, 2, 2, 5, "bf16"),
    Workload("blk_stage2_like", 1, 28, 28, 128, 4, 7, 4, 3, "bf16"),
    Workload("blk_stage3_like", 2, 14, 14, 256, 8, 7, 16, 5, "bf16"),
    bra_synth.WORKLOADS["stage1_bf16"].replace(B=2),
]


@pytest.mark.parametrize("wl", BLOCK_SHAPES, ids=lambda w: w.name)
def test_block_attention_step_by_step(wl, cuda_device):
    rng = np.random.default_rng(11)
    C = wl.C
    inp = bra_synth.make_inputs(wl, seed=5)
    x = bf16(inp.q, cuda_device)  # the synthetic map stands in for the block input
    ln_w = (1 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    ln_b = (0.1 * rng.standard_normal(C)).astype(np.float32)
    w_qkv = bf16(rng.standard_normal((3 * C, C)) / np.sqrt(C), cuda_device)
    b_qkv = (0.02 * rng.standard_normal(3 * C)).astype(np.float32)
    lw = torch.from_numpy(inp.lepe_w).to(cuda_device)
    lb = torch.from_numpy(inp.lepe_b).to(cuda_device)
    lnw, lnb = torch.from_numpy(ln_w).to(cuda_device), torch.from_numpy(ln_b).to(cuda_device)
    bq = torch.from_numpy(b_qkv).to(cuda_device)

    y = bra.block_attention(x, lnw, lnb, w_qkv, bq, wl.heads, wl.S, wl.topk, lw, lb)
    # the same four steps one by one give the same bits
    xn = bra.layer_norm(x, lnw, lnb)
    q, k, v = bra.qkv_project(xn, w_qkv, bq)
    out, idx = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, lw, lb)
    y2 = bra.residual_add(x, out)
    assert bra.device_status() == bra.BRA_OK
    assert torch.equal(y, y2)

    # each step against the oracle on that step's GPU inputs
    ref = oracle.layer_norm(f64(x), ln_w, ln_b)
    assert np.all(np.abs(f64(xn) - ref) <= ln_bound(ref))
    qr, kr, vr = oracle.qkv_project(f64(xn), f64(w_qkv), b_qkv)
    for got, want in ((q, qr), (k, kr), (v, vr)):
        assert np.abs(f64(got) - want).max() <= TOL["bf16"]
    q64, k64, v64 = f64(q), f64(k), f64(v)
    idx_o, A_o = oracle.route(q64, k64, wl.S, wl.topk)
    n_set, n_ord, n_skip, bad = routing_report(idx.cpu().numpy(), A_o, idx_o, wl.topk)
    assert not bad
    att = oracle.attend(q64, k64, v64, idx.cpu().numpy(), wl.heads, wl.S, inp.lepe_w,
                        inp.lepe_b)
    assert np.abs(f64(out) - att).max() <= TOL["bf16"]
    assert torch.equal(y2, (x.float() + out.float()).to(torch.bfloat16))


@pytest.mark.parametrize("M,K,N,with_res", [(300, 64, 192, False), (257, 192, 64, True),
                                            (130, 384, 64, True), (200, 128, 384, False),
                                            (129, 384, 128, True)])
def test_linear_matches_oracle(M, K, N, with_res, cuda_device):
    rng = np.random.default_rng(M + K + N)
    x = bf16(rng.standard_normal((M, K)), cuda_device)
    w = bf16(rng.standard_normal((N, K)) / np.sqrt(K), cuda_device)
    b = (0.1 * rng.standard_normal(N)).astype(np.float32)
    res = bf16(rng.standard_normal((M, N)) * 2, cuda_device) if with_res else None
    y = bra.linear(x, w, torch.from_numpy(b).to(cuda_device), residual=res)
    ref = oracle.linear(f64(x), f64(w), b) + (f64(res) if with_res else 0)
    assert np.all(np.abs(f64(y) - ref) <= linear_bound(ref))
    if with_res:  # in place on the residual
        r2 = res.clone()
        bra.linear(x, w, torch.from_numpy(b).to(cuda_device), residual=r2, out=r2)
        assert torch.equal(r2, y)


@pytest.mark.parametrize("Ch,H,W", [(192, 7, 9), (384, 17, 8), (264, 9, 20), (192, 56, 56)])
def test_dwconv_gelu_matches_oracle(Ch, H, W, cuda_device):
    # 192: one TMA box of the input tile; 384: two boxes; 264: the unstaged
    # kernel (above 256 channels and not a multiple of 16); ragged maps
    rng = np.random.default_rng(21 + Ch)
    h = bf16(rng.standard_normal((2, H, W, Ch)), cuda_device)
    w = (rng.standard_normal((Ch, 3, 3)) / 3).astype(np.float32)
    b = (0.1 * rng.standard_normal(Ch)).astype(np.float32)
    y = bra.dwconv_gelu(h, torch.from_numpy(w).to(cuda_device), torch.from_numpy(b).to(cuda_device))
    ref = oracle.gelu(oracle.lepe(f64(h), w, b))
    assert np.all(np.abs(f64(y) - ref) <= ln_bound(ref))


FFN_SHAPES = [Workload("ffn_c64", 2, 16, 16, 64, 2, 2, 2, 5, "bf16"),
              Workload("ffn_c128_ragged", 1, 14, 10, 128, 4, 2, 2, 5, "bf16")]


@pytest.mark.parametrize("wl", FFN_SHAPES, ids=lambda w: w.name)
def test_block_ffn_step_by_step(wl, cuda_device):
    rng = np.random.default_rng(31)
    C = wl.C
    x = bf16(bra_synth.make_inputs(wl, seed=6).q, cuda_device)
    ln_w = (1 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    ln_b = (0.1 * rng.standard_normal(C)).astype(np.float32)
    w1 = bf16(rng.standard_normal((3 * C, C)) / np.sqrt(C), cuda_device)
    b1 = (0.02 * rng.standard_normal(3 * C)).astype(np.float32)
    cw = (rng.standard_normal((3 * C, 3, 3)) / 3).astype(np.float32)
    cb = (0.02 * rng.standard_normal(3 * C)).astype(np.float32)
    w2 = bf16(rng.standard_normal((C, 3 * C)) / np.sqrt(3 * C), cuda_device)
    b2 = (0.02 * rng.standard_normal(C)).astype(np.float32)
    d = lambda a: torch.from_numpy(a).to(cuda_device)  # noqa: E731
    y = bra.block_ffn(x, d(ln_w), d(ln_b), w1, d(b1), d(cw), d(cb), w2, d(b2))
    # the four steps one by one give the same bits
    xn = bra.layer_norm(x, d(ln_w), d(ln_b))
    h = bra.linear(xn, w1, d(b1))
    ha = bra.dwconv_gelu(h, d(cw), d(cb))
    y2 = bra.linear(ha, w2, d(b2), residual=x)
    assert bra.device_status() == bra.BRA_OK
    assert torch.equal(y, y2)
    # each step against the oracle on that step's GPU input
    ref = oracle.layer_norm(f64(x), ln_w, ln_b)
    assert np.all(np.abs(f64(xn) - ref) <= ln_bound(ref))
    ref = oracle.linear(f64(xn), f64(w1), b1)
    assert np.all(np.abs(f64(h) - ref) <= linear_bound(ref))
    ref = oracle.gelu(oracle.lepe(f64(h), cw, cb))
    assert np.all(np.abs(f64(ha) - ref) <= ln_bound(ref))
    ref = f64(x) + oracle.linear(f64(ha), f64(w2), b2)
    assert np.all(np.abs(f64(y2) - ref) <= linear_bound(ref))


def test_block_ffn_rejects_wide_channels(cuda_device):
    C = 256
    x = torch.zeros((1, 8, 8, C), dtype=torch.bfloat16, device=cuda_device)
    z = lambda *s: torch.zeros(s, device=cuda_device)  # noqa: E731
    wb = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device=cuda_device)  # noqa: E731
    with pytest.raises(bra.BraError):
        bra.block_ffn(x, None, None, wb(3 * C, C), None, z(3 * C, 3, 3), None, wb(C, 3 * C),
                      None)
