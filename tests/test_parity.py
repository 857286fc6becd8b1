"""CUDA path vs the oracle, element by element, through the C ABI.

Small shapes span several tiles, ragged regions (slots padded to 8 rows),
LePE borders, one region (dense attention), all regions routed and large
region grids; the full-size workloads run at the sizes the benchmark times,
with every output compared against the oracle. Maps whose regions hold fewer
than 16 tokens and whose 64-channel chunk fits in shared memory take the
image-resident attend kernel (the image_* and n4 / ragged_n15 shapes); the
others take the region kernel.
"""
import json
import os

import numpy as np
import pytest
import torch

import bra_synth
import oracle
import vision_transformer_sparse_route_b300 as bra
from bra_synth import Workload
from parity import TOL, device_inputs, run_and_compare

pytestmark = pytest.mark.gpu

SMALL = [
    Workload("n64_bf16", 3, 16, 16, 64, 2, 2, 2, 5, "bf16"),
    Workload("ragged_n15_bf16", 2, 12, 20, 128, 4, 4, 3, 5, "bf16"),
    Workload("n4_bf16", 2, 14, 14, 256, 8, 7, 16, 5, "bf16"),
    Workload("one_region_bf16", 2, 8, 8, 64, 2, 1, 1, 5, "bf16"),
    Workload("all_routed_bf16", 1, 16, 16, 64, 2, 2, 4, 3, "bf16"),
    Workload("ks7_bf16", 2, 16, 16, 64, 2, 4, 2, 7, "bf16"),
    Workload("ks1_bf16", 2, 16, 16, 64, 2, 4, 2, 1, "bf16"),
    Workload("wide_region_bf16", 1, 4, 64, 64, 2, 2, 1, 5, "bf16"),
    Workload("tall_region_bf16", 1, 40, 8, 64, 2, 4, 3, 5, "bf16"),
    Workload("grid32_bf16", 1, 64, 64, 64, 2, 32, 2, 5, "bf16"),
    Workload("n16_c128_bf16", 3, 28, 28, 128, 4, 7, 4, 5, "bf16"),
    Workload("n64_top3_many_units_bf16", 1, 128, 128, 64, 2, 16, 3, 5, "bf16"),
    Workload("ragged_n15_region_bf16", 1, 36, 60, 64, 2, 12, 3, 5, "bf16"),
    Workload("topk40_serial_copies_bf16", 1, 32, 32, 64, 2, 8, 40, 5, "bf16"),
    Workload("image_ks3_bf16", 3, 12, 12, 64, 2, 4, 5, 3, "bf16"),
    Workload("image_ks7_bf16", 2, 14, 14, 128, 4, 7, 4, 7, "bf16"),
    Workload("image_ks1_128keys_bf16", 2, 8, 16, 64, 2, 4, 16, 1, "bf16"),
    Workload("image_wide_c256_bf16", 1, 6, 15, 256, 8, 3, 7, 5, "bf16"),
    Workload("small_f32", 2, 12, 12, 64, 2, 3, 3, 5, "f32"),
    Workload("ragged_f32", 1, 15, 10, 32, 1, 5, 4, 3, "f32"),
    Workload("d64_f32", 1, 8, 8, 128, 2, 2, 2, 5, "f32"),
    Workload("one_region_f32", 1, 6, 6, 64, 2, 1, 1, 5, "f32"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_shapes_match_oracle(wl, cuda_device):
    res = run_and_compare(wl, cuda_device, seed=7)
    assert res["rows_set"] + res["rows_near_tie"] == res["rows"]


@pytest.mark.parametrize("name", list(bra_synth.WORKLOADS))
def test_full_workloads_match_oracle(name, cuda_device):
    wl = bra_synth.WORKLOADS[name]
    res = run_and_compare(wl, cuda_device, seed=0)
    print(name, res)
    record = os.environ.get("BRA_PARITY_RECORD")
    if record:  # a JSON line per workload: the measured errors against the oracle
        with open(record, "a") as f:
            f.write(json.dumps({"workload": name, "seed": 0, "tolerance": TOL[wl.dtype],
                                **res}) + "\n")
    # with these value distributions near-ties are rare
    assert res["rows_near_tie"] <= max(2, res["rows"] // 1000)


def test_attend_with_oracle_routing(cuda_device):
    """bra_attend on the oracle's own routing (decoupled from bra_route)."""
    wl = bra_synth.WORKLOADS["stage2_bf16"].replace(B=4)
    x = bra_synth.make_inputs(wl, seed=3)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    idx_o, _ = oracle.route(x.q, x.k, wl.S, wl.topk)
    out = bra.attend(q, k, v, torch.from_numpy(idx_o).to(cuda_device), wl.heads, wl.S, w, b)
    ref = oracle.attend(x.q, x.k, x.v, idx_o, wl.heads, wl.S, x.lepe_w, x.lepe_b)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL["bf16"]


def test_no_bias_and_repeated_routing(cuda_device):
    """lepe_b = NULL; an index list that repeats a region counts its keys twice."""
    wl = Workload("rep", 1, 16, 16, 64, 2, 2, 3, 5, "bf16")
    x = bra_synth.make_inputs(wl, seed=5)
    q, k, v, w, _ = device_inputs(wl, x, cuda_device)
    idx = np.array([[[0, 0, 1], [1, 2, 1], [3, 3, 3], [2, 0, 1]]], dtype=np.int32)
    out = bra.attend(q, k, v, torch.from_numpy(idx).to(cuda_device), wl.heads, wl.S, w, None)
    ref = oracle.attend(x.q, x.k, x.v, idx, wl.heads, wl.S, x.lepe_w, None)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["bf16"]


@pytest.mark.parametrize("dtype,H,S", [("bf16", 16, 2), ("f32", 16, 2), ("bf16", 14, 7)],
                         ids=["bf16_region", "f32", "bf16_image"])
def test_out_of_range_index_reads_zeros_and_flags(dtype, H, S, cuda_device):
    wl = Workload("bad", 1, H, H, 64, 2, S, 2, 3, dtype)
    x = bra_synth.make_inputs(wl, seed=2)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    R = S * S
    good = np.stack([np.arange(R), (np.arange(R) + 1) % R], axis=1)[None].astype(np.int32)
    idx = good.copy()
    idx[0, 1:, 1] = np.where(np.arange(1, R) % 2, R + np.arange(1, R), -np.arange(1, R))
    bra.device_status(clear=True)
    out = bra.attend(q, k, v, torch.from_numpy(idx).to(cuda_device), wl.heads, wl.S, w, b)
    assert bra.device_status(clear=True) == bra.BRA_ERR_INVALID_ARG
    assert bra.device_status(clear=True) == bra.BRA_OK
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    # region 0, whose routing is valid, is unaffected
    ref = oracle.attend(x.q, x.k, x.v, good, wl.heads, wl.S, x.lepe_w, x.lepe_b)
    hr = H // S
    assert np.abs(got[:, :hr, :hr] - ref[:, :hr, :hr]).max() <= TOL[dtype]


def test_empty_batch_is_a_no_op(cuda_device):
    q = torch.empty((0, 14, 14, 64), dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros((64, 5, 5), device=cuda_device)
    out, idx = bra.forward(q, q.clone(), q.clone(), 2, 7, 4, w, None)
    assert out.shape == q.shape and idx.shape == (0, 49, 4)


def test_unsupported_shape_raises(cuda_device):
    q = torch.zeros((1, 8, 8, 64), dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros((64, 5, 5), device=cuda_device)
    with pytest.raises(bra.BraError) as e:
        bra.forward(q, q.clone(), q.clone(), 1, 2, 1, w, None)  # d = 64 in bf16
    assert e.value.status == bra.BRA_ERR_UNSUPPORTED


def test_side_stream_and_determinism(cuda_device):
    wl = bra_synth.WORKLOADS["stage3_bf16"].replace(B=2)
    x = bra_synth.make_inputs(wl, seed=11)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, i1 = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b, stream=s)
    s.synchronize()
    o2, i2 = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(o1, o2)


def test_host_pipeline_matches_forward(cuda_device):
    """Overlapped host batches give exactly the device forward's results."""
    wl = bra_synth.WORKLOADS["stage2_bf16"].replace(B=2)
    batches = [bra_synth.make_inputs(wl, seed=s) for s in (31, 32, 33)]
    w = torch.from_numpy(batches[0].lepe_w).to(cuda_device)
    b = torch.from_numpy(batches[0].lepe_b).to(cuda_device)
    host = [[torch.from_numpy(a).to(torch.bfloat16).pin_memory() for a in (x.q, x.k, x.v)]
            for x in batches]
    outs = [torch.empty_like(h[0]).pin_memory() for h in host]
    pipe = bra.HostPipeline(host[0][0].shape, torch.bfloat16, wl.S, wl.topk, cuda_device)
    for h, o in zip(host, outs):
        pipe.submit(*h, wl.heads, wl.S, wl.topk, w, b, o)
    pipe.synchronize()
    for h, o in zip(host, outs):
        ref, _ = bra.forward(*(t.to(cuda_device) for t in h), wl.heads, wl.S, wl.topk, w, b)
        assert torch.equal(o, ref.cpu())


@pytest.mark.parametrize("B", [64, 2])
def test_one_launch_forward_equals_two_kernel_forward(B, cuda_device):
    """The stage-3 shape runs as one kernel (routing inside, clusters of C/64
    CTAs); the routing kernel followed by the attend kernel gives the same
    routing and output bit for bit."""
    wl = bra_synth.WORKLOADS["stage3_bf16"].replace(B=B)
    assert bra.forward_launches(B, wl.H, wl.W, wl.C, wl.heads, wl.S, wl.topk, wl.ks) == 1
    x = bra_synth.make_inputs(wl, seed=17)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    out_one, idx_one = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b)
    idx_two = bra.route(q, k, wl.S, wl.topk)
    out_two = bra.attend(q, k, v, idx_two, wl.heads, wl.S, w, b)
    assert bra.device_status() == bra.BRA_OK
    assert torch.equal(idx_one, idx_two)
    assert torch.equal(out_one, out_two)


TC_SHAPES = [
    Workload("tc_n64_top2", 3, 16, 16, 64, 2, 2, 2, 5, "bf16"),
    Workload("tc_top4_ks3", 1, 16, 16, 64, 2, 2, 4, 3, "bf16"),
    Workload("tc_top3_many_units", 1, 128, 128, 64, 2, 16, 3, 5, "bf16"),
    Workload("tc_one_region_ks1", 2, 8, 8, 64, 2, 1, 1, 1, "bf16"),
]


@pytest.mark.parametrize("wl", TC_SHAPES + [bra_synth.WORKLOADS["stage1_bf16"],
                                            bra_synth.WORKLOADS["seg512_bf16"]],
                         ids=lambda w: w.name)
def test_tensor_memory_attend_matches_oracle(wl, cuda_device):
    """bra_attend_tc (tcgen05.mma, accumulators in tensor memory) against the
    oracle on the routing of bra_route, element by element."""
    x = bra_synth.make_inputs(wl, seed=9)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    idx = bra.route(q, k, wl.S, wl.topk)
    out = bra.attend_tc(q, k, v, idx, wl.heads, wl.S, w, b)
    assert bra.device_status() == bra.BRA_OK
    ref = oracle.attend(x.q, x.k, x.v, idx.cpu().numpy(), wl.heads, wl.S, x.lepe_w, x.lepe_b,
                        threads=8)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL["bf16"], err


def test_tensor_memory_attend_rejects_other_shapes(cuda_device):
    q = torch.zeros((1, 28, 28, 128), dtype=torch.bfloat16, device=cuda_device)
    idx = torch.zeros((1, 49, 4), dtype=torch.int32, device=cuda_device)
    w = torch.zeros((128, 5, 5), device=cuda_device)
    with pytest.raises(bra.BraError) as e:
        bra.attend_tc(q, q.clone(), q.clone(), idx, 4, 7, w)
    assert e.value.status == bra.BRA_ERR_UNSUPPORTED
