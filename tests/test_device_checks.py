"""Device-side behaviour that the random workloads reach only by chance:
exact affinity ties (ties go to the lowest region index, on every top-k
path of the routing kernel), and the bounded wait that gives up and reports
a timeout instead of trapping."""
import numpy as np
import pytest
import torch

import vision_transformer_sparse_route_b300 as bra

pytestmark = pytest.mark.gpu


def tied_inputs(B, H, W, C, S, dtype, pattern):
    """q = 1 everywhere; k per region: 'flat' -> 1 everywhere (every
    affinity row constant), 'two' -> 1 in even regions and 0.5 in odd ones
    (two values per row, each shared by many regions). All values and all
    affinities are exact in float32 and bfloat16."""
    q = np.ones((B, H, W, C), np.float32)
    k = np.ones((B, H, W, C), np.float32)
    if pattern == "two":
        hr, wr = H // S, W // S
        for r in range(S * S):
            if r % 2:
                y0, x0 = (r // S) * hr, (r % S) * wr
                k[:, y0:y0 + hr, x0:x0 + wr, :] = 0.5
    t = lambda a: torch.from_numpy(a).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    return t(q), t(k)


def expected_idx(R, topk, pattern):
    order = list(range(R)) if pattern == "flat" else \
        list(range(0, R, 2)) + list(range(1, R, 2))
    return np.array(order[:topk], np.int32)


# (B, H, W, C, S, topk, dtype): the rank path (at most 64 regions, topk > 4),
# the shuffle arg-max path (topk <= 4, or more than 64 regions), 256 regions
# (eight values a lane) and the float32 route
CASES = [
    (3, 14, 14, 256, 7, 16, "bf16"),
    (2, 14, 14, 64, 7, 5, "bf16"),
    (2, 56, 56, 64, 7, 1, "bf16"),
    (2, 28, 28, 128, 7, 4, "bf16"),
    (1, 128, 128, 64, 16, 4, "bf16"),
    (1, 64, 64, 64, 16, 9, "bf16"),
    (1, 14, 14, 64, 7, 4, "f32"),
    (1, 16, 16, 32, 8, 12, "f32"),
]


@pytest.mark.parametrize("pattern", ["flat", "two"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_%dx%d_C%d_S%d_k%d_%s" % c)
def test_exact_ties_go_to_the_lowest_region(case, pattern, cuda_device):
    B, H, W, C, S, topk, dtype = case
    q, k = tied_inputs(B, H, W, C, S, dtype, pattern)
    q, k = q.to(cuda_device), k.to(cuda_device)
    idx = bra.route(q, k, S, topk)
    assert bra.device_status() == bra.BRA_OK
    want = expected_idx(S * S, topk, pattern)
    got = idx.cpu().numpy()
    assert (got == want[None, None, :]).all(), got[0, :3]


@pytest.mark.parametrize("pattern", ["flat", "two"])
def test_forward_routes_ties_like_route(pattern, cuda_device):
    """The forward's own routing (the index it leaves in the workspace)
    breaks exact ties the same way."""
    B, H, W, C, S, topk, dtype = 2, 14, 14, 256, 7, 16, "bf16"
    q, k = tied_inputs(B, H, W, C, S, dtype, pattern)
    q, k = q.to(cuda_device), k.to(cuda_device)
    v = torch.randn(q.shape, device=cuda_device).to(q.dtype)
    w = torch.zeros((C, 5, 5), device=cuda_device)
    _, idx = bra.forward(q, k, v, 8, S, topk, w, None)
    assert bra.device_status() == bra.BRA_OK
    want = expected_idx(S * S, topk, pattern)
    assert (idx.cpu().numpy() == want[None, None, :]).all()


def test_bounded_wait_gives_up_and_reports_timeout(cuda_device):
    bra.device_status(clear=True)
    bra.check_wait_timeout(2_000_000)  # 2 ms
    assert bra.device_status(clear=True) == bra.BRA_ERR_TIMEOUT
    assert bra.device_status(clear=True) == bra.BRA_OK
    # the context is still usable and later kernels wait normally again
    q = torch.ones((1, 16, 16, 64), dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros((64, 5, 5), device=cuda_device)
    out, _ = bra.forward(q, q.clone(), q.clone(), 2, 2, 2, w, None)
    assert bra.device_status() == bra.BRA_OK
    assert torch.allclose(out.float(), torch.ones_like(out, dtype=torch.float32))
