"""The output-tolerance metric of the GPU tests, pinned on the CPU: a correct
rounding of the fp64 value costs nothing beyond the format, a rounding to the
other neighbour costs only its excess over half an ulp, an error of a few
units in the last place is counted, and one bad head is caught although the
norm over its whole sequence would hide it."""
import numpy as np
import torch

from harness import HEAD_BLOCK_MIN, out_errors, ulp_of


def test_ulp_of_bf16_matches_the_spacing():
    ref = np.array([1.0, 1.5, 0.75, -3.0, 2.0 ** -10])
    np.testing.assert_array_equal(ulp_of(ref, torch.bfloat16), np.array([2 ** -7, 2 ** -7, 2 ** -8, 2 ** -6, 2 ** -17]))
    assert ulp_of(np.array([0.0]), torch.bfloat16)[0] == 0.0


def test_correct_rounding_costs_nothing_beyond_the_format():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((16, 4, 128)) * 0.3          # 2,048 elements a head
    t = torch.from_numpy(ref).to(torch.bfloat16)
    plain, fmt = out_errors(t, ref, [0, 16])
    assert fmt == 0.0 and 5e-4 < plain < 2e-3


def test_a_flip_costs_its_distance_past_the_midpoint():
    # a value 0.1 ulp above the midpoint of two bf16 neighbours, rounded down:
    # 0.6 ulp away, so 0.1 ulp beyond half an ulp
    base = np.float64(1.0)
    u = 2.0 ** -7
    ref = np.full((16, 1, 128), 0.5)
    ref[0, 0, 0] = base + 0.6 * u
    o = torch.from_numpy(ref).to(torch.bfloat16)
    o[0, 0, 0] = torch.tensor(base, dtype=torch.bfloat16)  # the other neighbour
    plain, fmt = out_errors(o, ref, [0, 16])
    np.testing.assert_allclose(fmt, 0.1 * u / np.linalg.norm(ref), rtol=1e-9)


def test_errors_of_a_few_ulps_are_counted():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((2, 4, 128)) * 0.3
    bad = ref * (1 + 0.03)                        # ~4 ulps on every element
    plain, fmt = out_errors(torch.from_numpy(bad).to(torch.bfloat16), ref, [0, 1, 2])
    assert fmt > 1e-2 and plain > 2.5e-2
    # fp32 outputs: the format is ~1e-7, so fmt tracks the plain error
    o32 = torch.from_numpy(ref * (1 + 1e-4)).float()
    p32, f32 = out_errors(o32, ref, [0, 1, 2])
    assert abs(f32 - p32) < 1e-6 and 9e-5 < p32 < 1.1e-4


def test_one_bad_head_among_32_fails_the_per_head_bound():
    """A 5e-3 error on one of 32 heads is diluted to ~0.9e-3 by a norm over the
    whole sequence; per head it shows in full."""
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((64, 32, 128))                # 8,192 elements a head
    o = ref.copy()
    o[:, 7] *= 1 + 5e-3
    plain, _ = out_errors(torch.from_numpy(o), ref, [0, 64])
    np.testing.assert_allclose(plain, 5e-3, rtol=1e-6)
    whole = np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert whole < 1e-3


def test_short_blocks_take_the_norm_over_the_whole_sequence():
    """One decode token per sequence: 128 elements a head, below the per-head
    minimum, so the sequence's heads are taken together."""
    assert 128 < HEAD_BLOCK_MIN
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((3, 32, 128))
    o = ref.copy()
    o[1, 5] *= 1 + 5e-3
    plain, _ = out_errors(torch.from_numpy(o), ref, [0, 1, 2, 3])
    np.testing.assert_allclose(plain, np.linalg.norm(o[1] - ref[1]) / np.linalg.norm(ref[1]), rtol=1e-9)
    assert plain < 1e-3
