"""The backward of attend (routed attention + LePE, the routing fixed) on the
GPU against the oracle's backward, element by element, on the GPU's own
inputs (the bf16-rounded q, k, v and dout) and the GPU's own routing.

Tolerance: the kernels work in float32 (fast exp, sums of at most a few
hundred products, atomic adds in any order), so each gradient is compared
within 2e-4 of its own largest magnitude plus 1e-3 of the element (about a
hundred float32 roundings of the largest term); a dropped term, a wrong sign
or a transposed tap is of the size of the gradient itself."""
import numpy as np
import pytest
import torch

import bra_synth
import oracle
import vision_transformer_sparse_route_b300 as bra
from bra_synth import Workload
from parity import device_inputs

pytestmark = pytest.mark.gpu


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def close(got: torch.Tensor, ref: np.ndarray) -> bool:
    g = f64(got)
    bound = 2e-4 * max(1.0, float(np.abs(ref).max())) + 1e-3 * np.abs(ref)
    return bool(np.all(np.abs(g - ref) <= bound))


def check(wl: Workload, device, seed: int = 3):
    x = bra_synth.make_inputs(wl, seed=seed)
    q, k, v, w, _ = device_inputs(wl, x, device)
    rng = np.random.default_rng(seed)
    dout_np = rng.standard_normal((wl.B, wl.H, wl.W, wl.C)).astype(np.float32)
    dout = torch.from_numpy(dout_np).to(q.dtype).to(device)
    idx = bra.route(q, k, wl.S, wl.topk)
    dq, dk, dv, dw, db = bra.attend_backward(q, k, v, idx, wl.heads, wl.S, w, dout)
    assert bra.device_status() == bra.BRA_OK
    refs = oracle.attend_backward(f64(q), f64(k), f64(v), idx.cpu().numpy(), wl.heads, wl.S,
                                  x.lepe_w, f64(dout))
    for name, got, ref in zip(("dq", "dk", "dv", "dw", "db"), (dq, dk, dv, dw, db), refs):
        assert close(got, ref), (wl.name, name, float(np.abs(f64(got) - ref).max()),
                                 float(np.abs(ref).max()))


SHAPES = [
    Workload("bwd_n64_top2", 2, 16, 16, 64, 2, 2, 2, 5, "bf16"),
    Workload("bwd_ragged_n15", 1, 12, 20, 128, 4, 4, 3, 3, "bf16"),
    Workload("bwd_n4_top16", 2, 14, 14, 256, 8, 7, 16, 5, "bf16"),
    Workload("bwd_ks7_f32", 1, 12, 12, 64, 2, 3, 3, 7, "f32"),
    Workload("bwd_d64_f32", 1, 8, 8, 128, 2, 2, 2, 1, "f32"),
    Workload("bwd_one_region", 2, 8, 8, 64, 2, 1, 1, 5, "bf16"),
]


@pytest.mark.parametrize("wl", SHAPES, ids=lambda w: w.name)
def test_attend_backward_matches_oracle(wl, cuda_device):
    check(wl, cuda_device)


@pytest.mark.parametrize("name,B", [("stage1_bf16", 1), ("stage2_bf16", 1), ("stage3_bf16", 2),
                                    ("seg512_bf16", 1), ("tiny_f32", 1)])
def test_attend_backward_on_the_workload_shapes(name, B, cuda_device):
    check(bra_synth.WORKLOADS[name].replace(B=B), cuda_device)


def test_attend_backward_rejects_wide_heads(cuda_device):
    wl = Workload("wide", 1, 8, 8, 256, 2, 2, 2, 5, "bf16")  # d = 128
    x = bra_synth.make_inputs(wl, seed=1)
    q, k, v, w, _ = device_inputs(wl, x, cuda_device)
    idx = bra.route(q, k, wl.S, wl.topk)
    with pytest.raises(bra.BraError):
        bra.attend_backward(q, k, v, idx, wl.heads, wl.S, w, q)


def test_attend_backward_out_of_range_index_flags_and_spares_other_regions(cuda_device):
    """An out-of-range routing entry (in the last query region) sets the
    status word and leaves every gradient finite; dq of a region whose own
    routing is valid still equals the oracle's."""
    wl = Workload("bwd_bad", 1, 8, 8, 64, 2, 2, 2, 3, "bf16")
    x = bra_synth.make_inputs(wl, seed=4)
    q, k, v, w, _ = device_inputs(wl, x, cuda_device)
    R = wl.S * wl.S
    good = np.stack([np.arange(R), (np.arange(R) + 1) % R], axis=1)[None].astype(np.int32)
    bad = good.copy()
    bad[0, R - 1, 1] = R + 3
    dout = torch.from_numpy(np.random.default_rng(4).standard_normal(q.shape).astype(np.float32))
    dout = dout.to(torch.bfloat16).to(cuda_device)
    bra.device_status(clear=True)
    grads = bra.attend_backward(q, k, v, torch.from_numpy(bad).to(cuda_device), wl.heads, wl.S,
                                w, dout)
    assert bra.device_status(clear=True) == bra.BRA_ERR_INVALID_ARG
    assert bra.device_status(clear=True) == bra.BRA_OK
    for g in grads:
        assert torch.isfinite(g).all()
    refs = oracle.attend_backward(f64(q), f64(k), f64(v), good, wl.heads, wl.S, x.lepe_w,
                                  f64(dout))
    hr = wl.H // wl.S
    got_dq, ref_dq = grads[0][:, :hr, :hr], refs[0][:, :hr, :hr]  # region 0
    assert close(got_dq, ref_dq)
