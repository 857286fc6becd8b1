"""Pins for the CPU oracle: closed forms, special cases that reduce to library
routines, invariants and a hand-derived worked example.

None of these re-types the oracle's code: each check computes the expected
value another way (numpy / torch CPU library routines in float64, closed
forms, or constructions whose answer follows from the mathematics).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import bra_synth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def region_tokens_per_page(H, W, S):
    """Token ids y*W+x of each region, built the way the BRA write-up
    partitions the map: reshape (S, H/S, S, W/S) then swap the two middle
    axes, giving [S^2, HW/S^2] (page "CVPR2023：BiFormer中的双层路由注意力机制解析",
    section 3)."""
    ids = np.arange(H * W).reshape(S, H // S, S, W // S)
    return ids.transpose(0, 2, 1, 3).reshape(S * S, (H // S) * (W // S))


def rand_map(B, H, W, C, scale=1.0):
    return RNG.standard_normal((B, H, W, C)) * scale


def sdpa_heads(q, k, v, heads, mask=None):
    """Multi-head softmax(QK^T/sqrt(d))V over token sequences with torch
    (float64, CPU). q,k,v: [B, N, C]; mask: [B, N, N] bool (True = attend)."""
    B, N, C = q.shape
    d = C // heads
    t = lambda a: torch.from_numpy(a).reshape(B, N, heads, d).transpose(1, 2)
    m = None if mask is None else torch.from_numpy(mask)[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=m)
    return o.transpose(1, 2).reshape(B, N, C).numpy()


# --------------------------------------------------------------------------
# Region means
# --------------------------------------------------------------------------

def test_region_means_closed_form_zero_noise():
    wl = bra_synth.Workload("t", 2, 12, 8, 16, 2, 4, 2, 3, "f32")
    x = bra_synth.make_inputs(wl, seed=3, noise_std=0.0)
    means = oracle.region_means(x.q, wl.S)
    # with no per-token noise every token of a region holds the region offset
    regs = region_tokens_per_page(wl.H, wl.W, wl.S)
    flat = x.q.reshape(wl.B, wl.H * wl.W, wl.C).astype(np.float64)
    for r in range(wl.R):
        np.testing.assert_array_equal(means[:, r], flat[:, regs[r, 0]])
        np.testing.assert_array_equal(means[:, r], flat[:, regs[r, -1]])


def test_region_means_library_mean_over_page_partition():
    B, H, W, C, S = 2, 12, 9, 5, 3
    x = rand_map(B, H, W, C)
    regs = region_tokens_per_page(H, W, S)
    ref = x.reshape(B, H * W, C)[:, regs].mean(axis=2)
    np.testing.assert_allclose(oracle.region_means(x, S), ref, rtol=0, atol=1e-13)
    # the mean of the region means is the mean of all tokens (equal sizes)
    np.testing.assert_allclose(oracle.region_means(x, S).mean(axis=1),
                               x.reshape(B, -1, C).mean(axis=1), atol=1e-13)


# --------------------------------------------------------------------------
# Affinity and top-k routing
# --------------------------------------------------------------------------

def test_affinity_closed_form_one_hot_offsets():
    """Region offsets a_i e_{pi(i)} for q and b_j e_{sigma(j)} for k give
    A[i, j] = a_i b_j [pi(i) == sigma(j)] exactly."""
    B, S, hr, wr = 1, 3, 2, 2
    H, W, R = S * hr, S * wr, S * S
    C = R
    pi, sigma = RNG.permutation(R), RNG.permutation(R)
    a, b = RNG.integers(1, 9, R).astype(float), RNG.integers(1, 9, R).astype(float)
    regs = region_tokens_per_page(H, W, S)
    q = np.zeros((B, H * W, C))
    k = np.zeros((B, H * W, C))
    for r in range(R):
        q[0, regs[r], pi[r]] = a[r]
        k[0, regs[r], sigma[r]] = b[r]
    A = oracle.affinity(q.reshape(B, H, W, C), k.reshape(B, H, W, C), S)
    expect = np.where(pi[:, None] == sigma[None, :], a[:, None] * b[None, :], 0.0)
    np.testing.assert_array_equal(A[0], expect)
    idx, _ = oracle.route(q.reshape(B, H, W, C), k.reshape(B, H, W, C), S, 3)
    # first pick is the one matching column; the rest are zero ties -> lowest j
    for i in range(R):
        j0 = int(np.nonzero(sigma == pi[i])[0][0])
        rest = [j for j in range(R) if j != j0][:2]
        assert list(idx[0, i]) == [j0] + rest


def test_topk_matches_stable_argsort_with_ties():
    for R, k in [(5, 1), (9, 4), (49, 16), (256, 4), (64, 64)]:
        A = RNG.integers(-3, 4, size=(7, R)).astype(float)  # many ties
        ref = np.argsort(-A, axis=-1, kind="stable")[:, :k]
        np.testing.assert_array_equal(oracle.topk(A, k), ref)
        A = RNG.standard_normal((7, R))
        ref = np.argsort(-A, axis=-1, kind="stable")[:, :k]
        np.testing.assert_array_equal(oracle.topk(A, k), ref)


def test_topk_constant_row_takes_lowest_indices():
    A = np.full((3, 10), 2.5)
    np.testing.assert_array_equal(oracle.topk(A, 4), np.tile(np.arange(4), (3, 1)))


def test_topk_brute_force_sets_tiny():
    """The chosen set maximises the sum of affinities over all k-subsets."""
    import itertools
    for _ in range(20):
        R, k = 6, 3
        A = RNG.standard_normal((1, R))
        best = max(itertools.combinations(range(R), k), key=lambda s: A[0, list(s)].sum())
        assert set(oracle.topk(A, k)[0]) == set(best)


def test_self_route_by_cauchy_schwarz():
    """q = k with equal-norm, pairwise non-parallel region offsets and no
    token noise: A[i, i] = |o|^2 > o_i . o_j, so every region routes to itself
    first."""
    B, S, hr, wr, C = 2, 4, 2, 3, 8
    H, W, R = S * hr, S * wr, S * S
    o = RNG.standard_normal((B, R, C))
    o /= np.linalg.norm(o, axis=-1, keepdims=True)
    regs = region_tokens_per_page(H, W, S)
    x = np.zeros((B, H * W, C))
    for r in range(R):
        x[:, regs[r]] = o[:, r][:, None]
    x = x.reshape(B, H, W, C)
    idx, A = oracle.route(x, x, S, 1)
    np.testing.assert_array_equal(idx[..., 0], np.tile(np.arange(R), (B, 1)))


# --------------------------------------------------------------------------
# Routed attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("heads", [1, 2, 4])
def test_single_region_is_dense_attention(heads):
    B, H, W, C = 2, 6, 5, 16
    q, k, v = (rand_map(B, H, W, C) for _ in range(3))
    idx = np.zeros((B, 1, 1), dtype=np.int32)
    out = oracle.routed_attention(q, k, v, idx, heads, S=1)
    ref = sdpa_heads(*(a.reshape(B, H * W, C) for a in (q, k, v)), heads)
    np.testing.assert_allclose(out.reshape(B, H * W, C), ref, atol=1e-12)


def test_all_regions_routed_is_dense_attention():
    B, S, H, W, C, heads = 2, 3, 6, 9, 8, 2
    q, k, v = (rand_map(B, H, W, C) for _ in range(3))
    for _ in range(2):  # any order of the S^2 regions
        idx = np.stack([np.stack([RNG.permutation(S * S) for _ in range(S * S)])
                        for _ in range(B)]).astype(np.int32)
        out = oracle.routed_attention(q, k, v, idx, heads, S)
        ref = sdpa_heads(*(a.reshape(B, H * W, C) for a in (q, k, v)), heads)
        np.testing.assert_allclose(out.reshape(B, H * W, C), ref, atol=1e-12)
    # and through the full routing with topk = S^2
    out, _ = oracle.forward(q, k, v, heads, S, S * S, np.zeros((C, 1, 1)), None)
    np.testing.assert_allclose(out.reshape(B, H * W, C), ref, atol=1e-12)


def test_routed_equals_masked_dense_attention():
    B, S, H, W, C, heads, topk = 2, 4, 8, 12, 16, 4, 3
    q, k, v = (rand_map(B, H, W, C) for _ in range(3))
    idx = np.stack([np.stack([RNG.choice(S * S, topk, replace=False) for _ in range(S * S)])
                    for _ in range(B)]).astype(np.int32)
    regs = region_tokens_per_page(H, W, S)
    tok_region = np.empty(H * W, dtype=int)
    for r in range(S * S):
        tok_region[regs[r]] = r
    mask = np.zeros((B, H * W, H * W), dtype=bool)
    for b in range(B):
        for t in range(H * W):
            mask[b, t] = np.isin(tok_region, idx[b, tok_region[t]])
    ref = sdpa_heads(*(a.reshape(B, H * W, C) for a in (q, k, v)), heads, mask)
    out = oracle.routed_attention(q, k, v, idx, heads, S)
    np.testing.assert_allclose(out.reshape(B, H * W, C), ref, atol=1e-12)


def test_window_attention_when_each_region_routes_to_itself():
    """topk = 1 with self routing is non-overlapping window attention, the
    local-window formula softmax(QK^T/sqrt(d_k))V inside each window (page
    "Biformer注意力机制的原理及数学公式推导", local window attention)."""
    B, S, hr, wr, C, heads = 1, 3, 4, 2, 8, 2
    H, W = S * hr, S * wr
    q, k, v = (rand_map(B, H, W, C) for _ in range(3))
    idx = np.arange(S * S, dtype=np.int32).reshape(1, S * S, 1).repeat(B, 0)
    out = oracle.routed_attention(q, k, v, idx, heads, S)
    win = lambda a: a.reshape(B, S, hr, S, wr, C).transpose(0, 1, 3, 2, 4, 5).reshape(
        B * S * S, hr * wr, C)
    ref = sdpa_heads(win(q), win(k), win(v), heads)
    ref = ref.reshape(B, S, S, hr, wr, C).transpose(0, 1, 3, 2, 4, 5).reshape(B, H, W, C)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_softmax_rows_sum_to_one_and_order_invariance():
    wl = bra_synth.WORKLOADS["tiny_f32"]
    x = bra_synth.make_inputs(wl)
    idx, _ = oracle.route(x.q, x.k, wl.S, wl.topk)
    for (b, y, xx, h) in [(0, 0, 0, 0), (0, 13, 13, 1), (0, 5, 8, 0), (0, 7, 2, 1)]:
        p, keys, _ = oracle.query_probs(x.q, x.k, x.v, idx, wl.heads, wl.S, b, y, xx, h)
        assert p.shape == (wl.topk * wl.n,)
        assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()
        assert len(set(keys.tolist())) == len(keys)  # distinct routed regions
    perm = idx[..., ::-1].copy()
    a = oracle.routed_attention(x.q, x.k, x.v, idx, wl.heads, wl.S)
    c = oracle.routed_attention(x.q, x.k, x.v, perm, wl.heads, wl.S)
    np.testing.assert_allclose(a, c, atol=1e-12)


def test_heads_are_independent_channel_blocks():
    B, S, H, W, C, heads, topk = 1, 2, 4, 6, 12, 3, 2
    q, k, v = (rand_map(B, H, W, C) for _ in range(3))
    idx = np.stack([np.stack([RNG.choice(S * S, topk, replace=False) for _ in range(S * S)])
                    for _ in range(B)]).astype(np.int32)
    full = oracle.routed_attention(q, k, v, idx, heads, S)
    d = C // heads
    for h in range(heads):
        sl = slice(h * d, (h + 1) * d)
        part = oracle.routed_attention(q[..., sl], k[..., sl], v[..., sl], idx, 1, S)
        np.testing.assert_allclose(full[..., sl], part, atol=1e-13)


# --------------------------------------------------------------------------
# LePE
# --------------------------------------------------------------------------

@pytest.mark.parametrize("ks", [1, 3, 5, 7])
def test_lepe_is_depthwise_conv2d(ks):
    B, H, W, C = 2, 9, 7, 6
    v = rand_map(B, H, W, C)
    w = RNG.standard_normal((C, ks, ks))
    bias = RNG.standard_normal(C)
    ref = torch.nn.functional.conv2d(torch.from_numpy(v).permute(0, 3, 1, 2),
                                     torch.from_numpy(w)[:, None], torch.from_numpy(bias),
                                     padding=ks // 2, groups=C).permute(0, 2, 3, 1).numpy()
    np.testing.assert_allclose(oracle.lepe(v, w, bias), ref, atol=1e-12)


def test_lepe_delta_kernel_is_identity():
    v = rand_map(1, 5, 6, 4)
    w = np.zeros((4, 5, 5))
    w[:, 2, 2] = 1.0
    np.testing.assert_array_equal(oracle.lepe(v, w, None), v)


def test_attend_is_attention_plus_lepe():
    wl = bra_synth.WORKLOADS["tiny_f32"]
    x = bra_synth.make_inputs(wl)
    idx, _ = oracle.route(x.q, x.k, wl.S, wl.topk)
    total = oracle.attend(x.q, x.k, x.v, idx, wl.heads, wl.S, x.lepe_w, x.lepe_b)
    parts = (oracle.routed_attention(x.q, x.k, x.v, idx, wl.heads, wl.S)
             + oracle.lepe(x.v, x.lepe_w, x.lepe_b))
    np.testing.assert_allclose(total, parts, atol=1e-14)
    out, idx2 = oracle.forward(x.q, x.k, x.v, wl.heads, wl.S, wl.topk, x.lepe_w, x.lepe_b,
                               threads=3)
    np.testing.assert_array_equal(idx, idx2)
    np.testing.assert_allclose(out, total, atol=1e-14)


# --------------------------------------------------------------------------
# Worked example derived by hand
# --------------------------------------------------------------------------

def test_hand_worked_example():
    """2x2 map, S = 2 (one token per region), C = 2, one head, top-2, 1x1 LePE.

    Region r is token (r // 2, r % 2). Affinity rows (q_i . k_j):
      q0=(1,0): [1, 0,-1, 0] -> [0, 1]  (tie 0 between j=1 and j=3 -> 1)
      q1=(0,1): [0, 2, 0, 0] -> [1, 0]
      q2=(1,1): [1, 2,-1, 0] -> [1, 0]
      q3=(2,0): [2, 0,-2, 0] -> [0, 1]
    With s = 1/sqrt(2) and sig(z) = 1/(1+e^-z), the softmax over the two
    routed keys gives out0 = (sig(s), 1-sig(s)), out1 = (1-sig(2s), sig(2s)),
    out2 = (1-sig(s), sig(s)), out3 = (sig(2s), 1-sig(2s)). Region 2's value
    (2, 2) is routed by nobody and must not appear. LePE with w = (0.5, -2),
    bias = (0.25, 1) adds (0.5 v0 + 0.25, -2 v1 + 1) per token.
    """
    q = np.array([[1, 0], [0, 1], [1, 1], [2, 0]], float).reshape(1, 2, 2, 2)
    k = np.array([[1, 0], [0, 2], [-1, 0], [0, 0]], float).reshape(1, 2, 2, 2)
    v = np.array([[1, 0], [0, 1], [2, 2], [0, -1]], float).reshape(1, 2, 2, 2)
    w = np.array([0.5, -2.0]).reshape(2, 1, 1)
    bias = np.array([0.25, 1.0])
    out, idx = oracle.forward(q, k, v, 1, 2, 2, w, bias)
    np.testing.assert_array_equal(idx[0], [[0, 1], [1, 0], [1, 0], [0, 1]])
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    s = 1.0 / math.sqrt(2.0)
    attn = np.array([[sig(s), 1 - sig(s)], [1 - sig(2 * s), sig(2 * s)],
                     [1 - sig(s), sig(s)], [sig(2 * s), 1 - sig(2 * s)]])
    vv = v.reshape(4, 2)
    lepe = np.stack([0.5 * vv[:, 0] + 0.25, -2.0 * vv[:, 1] + 1.0], axis=1)
    np.testing.assert_allclose(out.reshape(4, 2), attn + lepe, atol=1e-15)


# --------------------------------------------------------------------------
# Facts the pages print
# --------------------------------------------------------------------------

def test_shapes_match_page_annotations():
    with open(os.path.join(GOLDEN, "p1_shape_annotations.json")) as f:
        g = json.load(f)
    e = g["example"]
    H, W, C, S, k = e["H"], e["W"], e["C"], e["S"], e["topk"]
    env = {"S^2": S * S, "HW/S^2": H * W // (S * S), "C": C, "k": k,
           "k*HW/S^2": k * H * W // (S * S)}
    shp = {n: tuple(env[s] for s in dims) for n, dims in g["shapes"].items()}
    x = np.ones((1, H, W, C))
    assert region_tokens_per_page(H, W, S).shape == shp["partitioned_tokens"][:2]
    assert oracle.region_means(x, S)[0].shape == shp["region_query_mean"]
    idx, A = oracle.route(x, x, S, k)
    assert A[0].shape == shp["region_affinity"]
    assert idx[0].shape == shp["routing_index"]
    p, _, _ = oracle.query_probs(x, x, x, idx, 2, S, 0, 0, 0, 0)
    assert p.shape == (shp["gathered_keys"][1],)


def test_workloads_follow_page_stage_settings():
    with open(os.path.join(GOLDEN, "p1_stage_routing.json")) as f:
        g = json.load(f)
    W = bra_synth.WORKLOADS
    # ImageNet-224 stage maps: stride 4 -> 56, 8 -> 28, 16 -> 14
    for name, stage in [("stage1_bf16", "stage1"), ("stage2_bf16", "stage2"),
                        ("stage3_bf16", "stage3")]:
        assert W[name].topk == g["stage_topk"][stage]
        assert W[name].H == 224 // g["stage_stride"][stage]
        assert W[name].S == g["region_grid_S"]["classification"]
    assert W["seg512_bf16"].S == g["region_grid_S"]["segmentation"]
    assert W["seg512_bf16"].H == 512 // g["stage_stride"]["stage1"]


def test_oracle_rejects_bad_arguments():
    x = np.ones((1, 6, 6, 4))
    with pytest.raises(ValueError):
        oracle.region_means(x, 4)  # 6 % 4 != 0
    with pytest.raises(ValueError):
        oracle.route(x, x, 3, 10)  # topk > S^2
    with pytest.raises(ValueError):
        oracle.lepe(x, np.ones((4, 2, 2)), None)  # even kernel


# ---------------------------------------------------------------- projections
def test_qkv_projection_equals_a_library_matmul():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 6, 4, 16))
    w = rng.standard_normal((48, 16))
    b = rng.standard_normal(48)
    q, k, v = oracle.qkv_project(x, w, b)
    full = np.einsum("bhwc,oc->bhwo", x, w) + b  # numpy's contraction, independently
    np.testing.assert_allclose(q, full[..., :16], rtol=0, atol=1e-12)
    np.testing.assert_allclose(k, full[..., 16:32], rtol=0, atol=1e-12)
    np.testing.assert_allclose(v, full[..., 32:], rtol=0, atol=1e-12)


def test_qkv_projection_special_cases():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5, 8))
    eye = np.eye(8)
    # stacked multiples of the identity: q = x, k = 2x, v = -x exactly
    q, k, v = oracle.qkv_project(x, np.concatenate([eye, 2 * eye, -eye]), None)
    assert np.array_equal(q, x) and np.array_equal(k, 2 * x) and np.array_equal(v, -x)
    # zero weight: every token gets the bias
    b = rng.standard_normal(24)
    q, k, v = oracle.qkv_project(x, np.zeros((24, 8)), b)
    assert np.array_equal(q, np.broadcast_to(b[:8], x.shape))
    assert np.array_equal(v, np.broadcast_to(b[16:], x.shape))
    # a permutation weight moves channels
    perm = np.eye(8)[::-1]
    q, _, _ = oracle.qkv_project(x, np.concatenate([perm, eye, eye]), None)
    assert np.array_equal(q, x[..., ::-1])


# ------------------------------------------------------- block (LayerNorm)
def test_layer_norm_equals_the_library_routine():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 3, 5, 24)) * 3 + 1.5
    g, b = rng.standard_normal(24), rng.standard_normal(24)
    y = oracle.layer_norm(x, g, b)
    t = torch.nn.functional.layer_norm(torch.from_numpy(x), (24,), torch.from_numpy(g),
                                       torch.from_numpy(b), 1e-5).numpy()
    np.testing.assert_allclose(y, t, rtol=0, atol=1e-12)


def test_layer_norm_invariants():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((40, 16))
    y = oracle.layer_norm(x, eps=0.0)
    # without scale and shift every token has mean 0 and (biased) variance 1
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-14)
    np.testing.assert_allclose((y * y).mean(-1), 1, atol=1e-13)
    # a positive scale and a shift of a token change nothing
    np.testing.assert_allclose(oracle.layer_norm(3.5 * x - 2.0, eps=0.0), y, atol=1e-13)
    # the affine part is applied after the normalisation
    g, b = rng.standard_normal(16), rng.standard_normal(16)
    np.testing.assert_allclose(oracle.layer_norm(x, g, b, eps=0.0), y * g + b, atol=1e-13)
    # a constant token: variance 0, so the output is the shift alone
    c = np.full((1, 16), 7.0)
    np.testing.assert_array_equal(oracle.layer_norm(c, g, b), b[None, :])


def test_block_attention_composes_the_stages():
    """y = x + bra(norm1(x)): with a zero LePE and zero projection weights
    and bias, q = k = v = 0, every logit is 0, the attention averages v = 0,
    so y = x exactly; and in general it is x plus the forward of the
    projected normalised tokens."""
    rng = np.random.default_rng(7)
    B, H, W, C, heads, S, topk, ks = 2, 8, 8, 16, 2, 2, 2, 3
    x = rng.standard_normal((B, H, W, C))
    ln_w, ln_b = rng.standard_normal(C), rng.standard_normal(C)
    zw, zb = np.zeros((C, ks, ks)), np.zeros(C)
    y, _, _ = oracle.block_attention(x, ln_w, ln_b, np.zeros((3 * C, C)), None, heads, S, topk,
                                     zw, zb)
    np.testing.assert_array_equal(y, x)
    w_qkv, b_qkv = rng.standard_normal((3 * C, C)) / 4, rng.standard_normal(3 * C)
    lw, lb = rng.standard_normal((C, ks, ks)) * 0.1, rng.standard_normal(C) * 0.1
    y, idx, (xn, q, k, v) = oracle.block_attention(x, ln_w, ln_b, w_qkv, b_qkv, heads, S, topk,
                                                   lw, lb)
    tn = torch.nn.functional.layer_norm(torch.from_numpy(x), (C,), torch.from_numpy(ln_w),
                                        torch.from_numpy(ln_b), 1e-5).numpy()
    full = tn @ w_qkv.T + b_qkv
    np.testing.assert_allclose(q, full[..., :C], atol=1e-12)
    np.testing.assert_allclose(v, full[..., 2 * C:], atol=1e-12)
    out, idx2 = oracle.forward(q, k, v, heads, S, topk, lw, lb)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(y - x, out, atol=1e-12)


# ------------------------------------------------------- block (ConvFFN)
def test_linear_and_gelu_equal_library_routines():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 4, 10))
    w, b = rng.standard_normal((7, 10)), rng.standard_normal(7)
    np.testing.assert_allclose(oracle.linear(x, w, b), np.einsum("abk,nk->abn", x, w) + b,
                               rtol=0, atol=1e-12)
    t = torch.from_numpy(x * 3)
    np.testing.assert_allclose(oracle.gelu(x * 3), torch.nn.functional.gelu(t).numpy(),
                               rtol=0, atol=1e-12)
    # GELU(x) - GELU(-x) = x (erf is odd), GELU(0) = 0, GELU(x) -> x for large x
    g = oracle.gelu(x) - oracle.gelu(-x)
    np.testing.assert_allclose(g, x, atol=1e-14)
    assert oracle.gelu(np.zeros(3)).tolist() == [0.0, 0.0, 0.0]
    np.testing.assert_allclose(oracle.gelu(np.array([40.0])), [40.0], rtol=0, atol=1e-12)


def test_block_ffn_composes_the_stages():
    """y = x + fc2(GELU(dwconv(fc1(norm2(x))))): zero fc2 weight and bias give
    y = x exactly; in general the stages equal torch's layer_norm, linear,
    depthwise conv2d and gelu applied in that order."""
    rng = np.random.default_rng(13)
    B, H, W, C = 2, 6, 5, 8
    x = rng.standard_normal((B, H, W, C))
    ln_w, ln_b = rng.standard_normal(C), rng.standard_normal(C)
    w1, b1 = rng.standard_normal((3 * C, C)) / 3, rng.standard_normal(3 * C)
    cw, cb = rng.standard_normal((3 * C, 3, 3)) / 3, rng.standard_normal(3 * C)
    w2, b2 = rng.standard_normal((C, 3 * C)) / 5, rng.standard_normal(C)
    y, _ = oracle.block_ffn(x, ln_w, ln_b, w1, b1, cw, cb, np.zeros((C, 3 * C)), None)
    np.testing.assert_array_equal(y, x)
    y, (xn, h, hc, ha) = oracle.block_ffn(x, ln_w, ln_b, w1, b1, cw, cb, w2, b2)
    F = torch.nn.functional
    tx = torch.from_numpy(x)
    tn = F.layer_norm(tx, (C,), torch.from_numpy(ln_w), torch.from_numpy(ln_b), 1e-5)
    th = F.linear(tn, torch.from_numpy(w1), torch.from_numpy(b1))
    tc = F.conv2d(th.permute(0, 3, 1, 2), torch.from_numpy(cw)[:, None], torch.from_numpy(cb),
                  padding=1, groups=3 * C).permute(0, 2, 3, 1)
    ty = tx + F.linear(F.gelu(tc), torch.from_numpy(w2), torch.from_numpy(b2))
    np.testing.assert_allclose(hc, tc.numpy(), atol=1e-12)
    np.testing.assert_allclose(y, ty.numpy(), atol=1e-12)


# ---- the backward of attend (routing held fixed) ----------------------------

def _torch_attend(q, k, v, idx, heads, S, w, bias):
    """attend written with torch tensor ops (region reshape, gather of the
    routed regions, one softmax per query over all routed keys, depthwise
    conv2d for the LePE): an implementation independent of the oracle's loops,
    differentiated by torch autograd in float64."""
    B, H, W, C = q.shape
    hr, wr, R, d = H // S, W // S, S * S, C // heads
    n, topk = hr * wr, idx.shape[-1]

    def regions(x):  # [B, R, n, C], regions and their tokens row-major
        return x.reshape(B, S, hr, S, wr, C).permute(0, 1, 3, 2, 4, 5).reshape(B, R, n, C)

    qr, kr, vr = regions(q), regions(k), regions(v)
    ib = torch.from_numpy(np.asarray(idx, np.int64))
    bi = torch.arange(B)[:, None, None]
    kg = kr[bi, ib].reshape(B, R, topk * n, heads, d).permute(0, 3, 1, 2, 4)
    vg = vr[bi, ib].reshape(B, R, topk * n, heads, d).permute(0, 3, 1, 2, 4)
    qh = qr.reshape(B, R, n, heads, d).permute(0, 3, 1, 2, 4)
    att = torch.softmax(qh @ kg.transpose(-1, -2) / math.sqrt(d), dim=-1)
    o = (att @ vg).permute(0, 2, 3, 1, 4).reshape(B, S, S, hr, wr, C)
    o = o.permute(0, 1, 3, 2, 4, 5).reshape(B, H, W, C)
    lepe = torch.nn.functional.conv2d(v.permute(0, 3, 1, 2), w[:, None], bias,
                                      padding=w.shape[-1] // 2, groups=C)
    return o + lepe.permute(0, 2, 3, 1)


@pytest.mark.parametrize("B,H,W,C,heads,S,topk,ks", [
    (2, 8, 8, 8, 2, 2, 2, 3),     # 4 regions of 16 tokens, top-2
    (1, 6, 9, 12, 3, 3, 4, 5),    # ragged 2 x 3 regions, 3 heads of 4
    (1, 4, 4, 4, 1, 4, 16, 1),    # one-token regions, every region routed
])
def test_attend_backward_matches_torch_autograd(B, H, W, C, heads, S, topk, ks):
    rng = np.random.default_rng(B * 100 + H + C + ks)
    q, k, v = (rng.standard_normal((B, H, W, C)) for _ in range(3))
    w = rng.standard_normal((C, ks, ks)) * 0.3
    bias = rng.standard_normal(C) * 0.1
    dout = rng.standard_normal((B, H, W, C))
    idx, _ = oracle.route(q, k, S, topk)
    dq, dk, dv, dw, db = oracle.attend_backward(q, k, v, idx, heads, S, w, dout)
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v, w, bias)]
    out = _torch_attend(*t[:3], idx, heads, S, t[3], t[4])
    assert np.allclose(out.detach().numpy(), oracle.attend(q, k, v, idx, heads, S, w, bias),
                       atol=1e-12)
    out.backward(torch.from_numpy(dout))
    for got, ref in zip((dq, dk, dv, dw, db), t):
        np.testing.assert_allclose(got, ref.grad.numpy(), rtol=0, atol=1e-11)


def test_attend_backward_is_the_derivative_of_attend():
    """Central differences of L = sum(dout * attend(...)) along random
    directions equal the oracle's gradients dotted with those directions."""
    rng = np.random.default_rng(7)
    B, H, W, C, heads, S, topk, ks = 1, 6, 6, 4, 2, 3, 3, 3
    q, k, v = (rng.standard_normal((B, H, W, C)) for _ in range(3))
    w, bias = rng.standard_normal((C, ks, ks)) * 0.3, rng.standard_normal(C) * 0.1
    dout = rng.standard_normal((B, H, W, C))
    idx, _ = oracle.route(q, k, S, topk)  # held fixed, as in the backward
    grads = oracle.attend_backward(q, k, v, idx, heads, S, w, dout)
    params = [q, k, v, w, bias]
    L = lambda p: float(np.sum(dout * oracle.attend(*p[:3], idx, heads, S, p[3], p[4])))  # noqa: E731
    for trial in range(4):
        dirs = [rng.standard_normal(p.shape) for p in params]
        eps = 1e-5
        plus = [p + eps * d for p, d in zip(params, dirs)]
        minus = [p - eps * d for p, d in zip(params, dirs)]
        fd = (L(plus) - L(minus)) / (2 * eps)
        an = sum(float(np.sum(g * d)) for g, d in zip(grads, dirs))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (trial, fd, an)
