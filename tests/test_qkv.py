"""bra_qkv_project (the q_proj / k_proj / v_proj linear maps in front of BRA,
on the tcgen05 tensor cores) against the oracle's double-precision
projection, element by element."""
import numpy as np
import pytest
import torch

import bra_synth
import oracle
import vision_transformer_sparse_route_b300 as bra
from parity import TOL

pytestmark = pytest.mark.gpu


def run(M, C, seed, with_bias, device, rows=None):
    x, w, b = bra_synth.make_projection_inputs(M, C, seed)
    xd = torch.from_numpy(x).to(torch.bfloat16).to(device)
    wd = torch.from_numpy(w).to(torch.bfloat16).to(device)
    bd = torch.from_numpy(b).to(device) if with_bias else None
    q, k, v = bra.qkv_project(xd, wd, bd)
    assert bra.device_status() == bra.BRA_OK
    sel = slice(None) if rows is None else rows
    ref = oracle.qkv_project(x[sel], w, b if with_bias else None)
    errs = [float(np.abs(t.float().cpu().numpy()[sel] - r).max()) for t, r in zip((q, k, v), ref)]
    return max(errs)


@pytest.mark.parametrize("M,C,bias", [(128, 64, True), (300, 64, True), (1000, 128, True),
                                      (257, 256, True), (130, 64, False), (4096, 256, False)],
                         ids=["one_tile", "ragged_c64", "c128_resident", "c256_streamed",
                              "no_bias", "c256_many_tiles"])
def test_projection_matches_oracle(M, C, bias, cuda_device):
    assert run(M, C, 1, bias, cuda_device) <= TOL["bf16"]


def test_projection_full_stage1_size_sampled(cuda_device):
    """64 images of 56 x 56 tokens, 64 channels (the stage-1 map): 3000
    sampled tokens compared with the oracle."""
    M, C = 64 * 56 * 56, 64
    rows = np.sort(np.random.default_rng(0).choice(M, 3000, replace=False))
    assert run(M, C, 2, True, cuda_device, rows=rows) <= TOL["bf16"]


def test_projection_feeds_the_forward(cuda_device):
    """x -> (q, k, v) -> bra_forward: the same result as the forward on the
    oracle's projections rounded to bf16 (one-bf16-ulp differences in q, k, v
    allowed for by the tolerance)."""
    wl = bra_synth.WORKLOADS["stage3_bf16"].replace(B=2)
    M, C = wl.B * wl.H * wl.W, wl.C
    x, w, b = bra_synth.make_projection_inputs(M, C, 3)
    xd = torch.from_numpy(x).to(torch.bfloat16).to(cuda_device).reshape(wl.B, wl.H, wl.W, C)
    q, k, v = bra.qkv_project(xd, torch.from_numpy(w).to(torch.bfloat16).to(cuda_device),
                              torch.from_numpy(b).to(cuda_device))
    rq, rk, rv = (bra_synth.round_bf16(t.astype(np.float32)).reshape(q.shape)
                  for t in oracle.qkv_project(x, w, b))
    assert float(np.abs(q.float().cpu().numpy() - rq).max()) <= 2 ** -7 * np.abs(rq).max()
    lw = torch.zeros((C, 5, 5), device=cuda_device)
    out, idx = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, lw, None)
    ref = oracle.attend(q.float().cpu().numpy(), k.float().cpu().numpy(),
                        v.float().cpu().numpy(), idx.cpu().numpy(), wl.heads, wl.S,
                        np.zeros((C, 5, 5)), None)
    assert float(np.abs(out.float().cpu().numpy() - ref).max()) <= TOL["bf16"]


def test_projection_rejects_unsupported_channels(cuda_device):
    x = torch.zeros((10, 96), dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros((288, 96), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(bra.BraError) as e:
        bra.qkv_project(x, w)
    assert e.value.status == bra.BRA_ERR_UNSUPPORTED
