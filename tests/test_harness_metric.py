"""The output-tolerance metric of the GPU tests, pinned on the CPU: a correct
rounding of the fp64 value (either bf16 neighbour) costs nothing beyond the
format, an error of a few units in the last place is counted, and the plain
metric sees the rounding itself."""
import numpy as np
import torch

from harness import out_errors, ulp_of


def _bf16_neighbours(ref):
    t = torch.from_numpy(ref).to(torch.bfloat16)
    lo = torch.nextafter(t.float(), torch.tensor(-np.inf)).to(torch.bfloat16)
    return t, lo


def test_ulp_of_bf16_matches_the_spacing():
    ref = np.array([1.0, 1.5, 0.75, -3.0, 2.0 ** -10])
    np.testing.assert_array_equal(ulp_of(ref, torch.bfloat16), np.array([2 ** -7, 2 ** -7, 2 ** -8, 2 ** -6, 2 ** -17]))
    assert ulp_of(np.array([0.0]), torch.bfloat16)[0] == 0.0


def test_correct_rounding_and_flips_cost_nothing_beyond_the_format():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((1, 4, 128)) * 0.3
    t = torch.from_numpy(ref).to(torch.bfloat16)
    plain, fmt = out_errors(t, ref, [0, 1])
    assert fmt == 0.0 and 5e-4 < plain < 4e-3
    # the other bf16 neighbour of the largest element (a legitimate flip)
    flat = t.clone().view(-1)
    i = int(np.argmax(np.abs(ref)))
    up = torch.tensor(ref.reshape(-1)[i], dtype=torch.float64)
    nb = (flat[i].double() + torch.sign(up - flat[i].double()) * float(ulp_of(np.array([ref.reshape(-1)[i]]), torch.bfloat16)[0]))
    flat[i] = nb.to(torch.bfloat16)
    assert out_errors(flat.view(t.shape), ref, [0, 1])[1] == 0.0


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
