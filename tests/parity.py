"""Helpers that compare the CUDA path (through the C ABI) with the oracle on
the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import bra_synth
import oracle
import vision_transformer_sparse_route_b300 as bra

# Tolerances stated for this method: routing bit-exact where the oracle's
# k-th vs (k+1)-th affinity gap exceeds 1e-4; outputs within max-abs 1e-4
# (float32 path) or 2e-2 (bf16 inputs, float32 accumulation).
GAP = 1e-4
TOL = {"f32": 1e-4, "bf16": 2e-2}
THREADS = max(1, min(32, os.cpu_count() or 1))


def to_device(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.to(device)


def device_inputs(wl: bra_synth.Workload, x: bra_synth.Inputs, device):
    q, k, v = (to_device(a, wl.dtype, device) for a in (x.q, x.k, x.v))
    w = torch.from_numpy(x.lepe_w).to(device)
    b = torch.from_numpy(x.lepe_b).to(device)
    return q, k, v, w, b


def routing_report(idx_gpu: np.ndarray, A_oracle: np.ndarray, idx_oracle: np.ndarray,
                   topk: int):
    """Checks the routing against the oracle under the gap rule. Returns
    (rows checked as sets, rows checked in order, rows skipped, mismatches)."""
    R = A_oracle.shape[-1]
    A = A_oracle.reshape(-1, R)
    gi = idx_gpu.reshape(-1, topk)
    oi = idx_oracle.reshape(-1, topk)
    srt = -np.sort(-A, axis=1)
    n_set = n_ord = n_skip = 0
    bad = []
    for r in range(A.shape[0]):
        if topk < R:
            gap = srt[r, topk - 1] - srt[r, topk]
            if gap <= GAP:
                n_skip += 1
                continue
        n_set += 1
        if set(gi[r].tolist()) != set(oi[r].tolist()):
            bad.append(r)
            continue
        lead = srt[r, :min(topk + 1, R)]
        if np.all(lead[:-1] - lead[1:] > GAP) if len(lead) > 1 else True:
            n_ord += 1
            if not np.array_equal(gi[r], oi[r]):
                bad.append(r)
    return n_set, n_ord, n_skip, bad


def run_and_compare(wl: bra_synth.Workload, device, seed: int = 0, x=None,
                    check_affinity: bool = True):
    """Runs route + attend + forward on the GPU and checks them against the
    oracle. Returns a dict of the measured errors."""
    if x is None:
        x = bra_synth.make_inputs(wl, seed=seed)
    q, k, v, w, b = device_inputs(wl, x, device)
    R = wl.R
    aff = torch.empty((wl.B, R, R), dtype=torch.float32, device=device)
    idx = bra.route(q, k, wl.S, wl.topk, affinity=aff)
    out, idx_fwd = bra.forward(q, k, v, wl.heads, wl.S, wl.topk, w, b)
    assert bra.device_status() == bra.BRA_OK
    idx_g = idx.cpu().numpy()
    np.testing.assert_array_equal(idx_fwd.cpu().numpy(), idx_g)
    aff_g = aff.cpu().numpy().astype(np.float64)

    idx_o, A_o = oracle.route(x.q, x.k, wl.S, wl.topk)
    # the kernel's own selection, redone by the oracle's top-k on the
    # kernel's float32 affinity: identical on every row
    np.testing.assert_array_equal(oracle.topk(aff_g, wl.topk), idx_g)
    n_set, n_ord, n_skip, bad = routing_report(idx_g, A_o, idx_o, wl.topk)
    assert not bad, f"routing differs from the oracle on rows {bad[:10]}"
    res = dict(rows=wl.B * R, rows_set=n_set, rows_ordered=n_ord, rows_near_tie=n_skip)
    if check_affinity:
        # float32 means, then a float32 dot product: |err| <= (C + 2n + 4) u sum_c |q|_c |k|_c
        # (means of |x| bound both the means and their rounding errors)
        qm = oracle.region_means(np.abs(x.q), wl.S)
        km = oracle.region_means(np.abs(x.k), wl.S)
        bound = (wl.C + 2 * wl.n + 4) * 2.0 ** -24 * np.einsum(
            "bic,bjc->bij", qm, km) + 1e-30
        err = np.abs(aff_g - A_o)
        assert np.all(err <= bound), f"affinity error {err.max()} over bound"
        res["affinity_max_err"] = float(err.max())

    ref = oracle.attend(x.q, x.k, x.v, idx_g, wl.heads, wl.S, x.lepe_w, x.lepe_b,
                        threads=THREADS)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    res["out_max_err"] = float(err.max())
    assert err.max() <= TOL[wl.dtype], f"max abs error {err.max()} > {TOL[wl.dtype]}"
    return res
