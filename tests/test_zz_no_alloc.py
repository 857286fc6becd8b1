"""bra_forward_static: the forward for callers that may not allocate device
memory (they are handed only their input and output buffers, e.g. a plugin
inside an engine that owns the device memory budget). Its routing index lives
in an array inside the library instead of a caller workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import bra_synth
import vision_transformer_sparse_route_b300 as bra
from parity import TOL, device_inputs


def test_static_forward_rejects_sizes_beyond_its_array():
    lib = bra._load()
    fake = [ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(5)]
    # 64 images x 256 regions x 16 routed = 262144 + 1 entries > 1 << 18
    rc = lib.bra_forward_static(fake[0], fake[1], fake[2], 65, 128, 128, 64, 2, 16, 16,
                                fake[3], None, 5, 1, fake[4], None)
    assert rc == bra.BRA_ERR_UNSUPPORTED
    assert bra.STATIC_IDX_MAX_ENTRIES == 1 << 18


@pytest.mark.gpu
def test_static_forward_matches_forward_twice(cuda_device):
    # two different problems in a row: the second call must not see the
    # first call's routing index
    for name, B, seed in [("stage3_bf16", 3, 21), ("stage2_bf16", 2, 22)]:
        wl = bra_synth.WORKLOADS[name].replace(B=B)
        x = bra_synth.make_inputs(wl, seed=seed)
        q, k, v, w, b = device_inputs(wl, x, cuda_device)
        ref, _ = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b)
        got = bra.forward_static(q, k, v, wl.heads, wl.S, wl.topk, w, b)
        assert bra.device_status() == bra.BRA_OK
        err = (got.float() - ref.float()).abs().max().item()
        assert err <= TOL[wl.dtype], (name, err)
    # the float32 path too, on the caller's stream
    wl = bra_synth.WORKLOADS["tiny_f32"]
    x = bra_synth.make_inputs(wl, seed=23)
    q, k, v, w, b = device_inputs(wl, x, cuda_device)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ref, _ = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b, stream=s)
        got = bra.forward_static(q, k, v, wl.heads, wl.S, wl.topk, w, b, stream=s)
    s.synchronize()
    assert float(np.abs(got.cpu().numpy() - ref.cpu().numpy()).max()) <= TOL["f32"]
