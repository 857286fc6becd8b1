"""The seeded input generator (bra_synth), pinned to its published
definitions: SplitMix64 (Steele, Lea and Flood, OOPSLA 2014; the outputs of
Vigna's public reference implementation), round-to-nearest-even bfloat16
(checked against torch's own conversion), the Box-Muller transform (moments),
and the batch-slicing property the multi-rank bench relies on."""
import numpy as np
import pytest
import torch

import bra_synth


def test_splitmix64_reference_outputs():
    # the first outputs of the reference generator started from state 0
    z = bra_synth.splitmix64(0, 0, 3)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_is_counter_based():
    # output i depends only on (seed, i): a window equals the same slice of a longer run
    full = bra_synth.splitmix64(12345, 0, 64)
    assert np.array_equal(bra_synth.splitmix64(12345, 17, 20), full[17:37])


def test_round_bf16_ties_to_even_and_matches_torch():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)  # bf16 spacing above 1
    x = np.array([one + ulp / 2,           # tie: to even (1.0)
                  one + 3 * ulp / 2,       # tie: to even (1 + 2 ulp)
                  one + ulp / 2 + 2 ** -20,  # above the tie: up
                  -(one + ulp / 2),        # sign symmetric
                  3.0e38, 1e-40, 0.0, -0.0], dtype=np.float32)
    got = bra_synth.round_bf16(x)
    assert got[0] == one and got[1] == one + 2 * ulp and got[2] == one + ulp
    assert got[3] == -one
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    rng = np.random.default_rng(3)
    y = (rng.standard_normal(100000) * 10.0 ** rng.integers(-20, 20, 100000)).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bra_synth.round_bf16(y).view(np.uint32), ref.view(np.uint32))


def test_box_muller_normals_have_unit_moments():
    n = bra_synth.normals(7, 400000)
    assert abs(n.mean()) < 0.01
    assert abs(n.std() - 1.0) < 0.01
    # fourth moment of a standard normal is 3
    assert abs((n ** 4).mean() - 3.0) < 0.05
    # pairs (cos, sin) of one radius are uncorrelated
    assert abs(np.corrcoef(n[0::2], n[1::2])[0, 1]) < 0.01


@pytest.mark.parametrize("start", [0, 1, 3])
def test_batch_slices_equal_the_full_draw(start):
    wl = bra_synth.Workload("s", 5, 6, 6, 8, 2, 3, 2, 3, "bf16")
    full = bra_synth.make_inputs(wl, seed=4)
    part = bra_synth.make_inputs(wl, seed=4, batch=slice(start, start + 2))
    for a, b in zip((full.q, full.k, full.v), (part.q, part.k, part.v)):
        assert np.array_equal(a[start:start + 2], b)
    assert np.array_equal(full.lepe_w, part.lepe_w)
    # bf16 workloads hold exactly representable bf16 values
    assert np.array_equal(bra_synth.round_bf16(full.q), full.q)
