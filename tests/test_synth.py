"""The seeded input generator: published SplitMix64 outputs, rounding, ranges."""

import numpy as np
import pytest
import torch

from synth import configs, gen


def test_splitmix64_published_seed0_outputs():
    # First three outputs of SplitMix64 seeded with 0, as published with the
    # generator's reference implementation.
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [gen.splitmix64_int(0, i) for i in range(3)] == expect
    assert [int(x) for x in gen.stream_bits(0, np.arange(3))] == expect


def test_vectorised_matches_integer_form():
    for key in (0, 1, 0xDEADBEEF, (1 << 64) - 1, gen.tensor_key(1238, 63, 12)):
        idx = np.array([0, 1, 2, 1000, 123456789, (1 << 40) + 7], dtype=np.uint64)
        assert [int(x) for x in gen.stream_bits(key, idx)] == [gen.splitmix64_int(key, int(i)) for i in idx]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 1e-3,
                        rng.uniform(-1, 1, 100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, -1.0, 2.0 ** -130, 3.0e38], dtype=np.float32)])
    ours = gen.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("dist", [gen.UNIFORM, gen.NORMAL, gen.OUTLIER, gen.INTEGER])
def test_distributions(dist):
    bits = gen.bf16_values(gen.tensor_key(7, 1, 2), np.arange(200000, dtype=np.uint64), dist)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.isfinite(x).all()
    if dist == gen.UNIFORM:
        assert x.min() >= -1 and x.max() <= 1 and abs(x.mean()) < 0.01
    elif dist == gen.NORMAL:
        assert abs(x.std() - 1e-3) < 2e-5 and abs(x.mean()) < 2e-5
    elif dist == gen.OUTLIER:
        frac = (np.abs(x) > 4e-3).mean()   # no plain value exceeds ~3.47 sigma
        assert 0.07 < frac < 0.10
    else:
        assert np.array_equal(x, np.round(x)) and x.min() == -128 and x.max() == 128


def test_workload_shapes():
    w = configs.get(2)
    assert w.N == 8 and w.M * w.L == w.N and w.total_grad_elems() == 855_654_400
    w = configs.get(3)
    assert w.P == 391 and w.total_grad_elems() == 623_120_384
    w = configs.get(4)
    assert w.P == 13 and w.N == 64 and w.total_grad_elems() == 351_288_320
    w = configs.get(5)
    assert w.P == 257 and w.N == 48
    assert all(1 <= r <= 5000 and 1 <= c <= 4096 for r, c in w.shapes)
    assert sum(1 for r, c in w.shapes if r % 48) > 200            # most carry padding
    assert sum(1 for r, c in w.shapes if c % 2) >= 120            # many odd widths
    assert 2 * w.N * w.total_grad_elems() <= 48 << 30
    w = configs.get(1)
    assert [s[0] // w.N for s in w.shapes] == [2, 1, 3]
