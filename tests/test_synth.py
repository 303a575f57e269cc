"""The seeded input generator: determinism, counter addressing, distribution, bf16 rounding."""
import numpy as np
import torch

import fpsynth


def test_deterministic_and_counter_based():
    a = fpsynth.normal(7, 1, 1000)
    b = fpsynth.normal(7, 1, 1000)
    assert np.array_equal(a, b)
    # element i depends only on (seed, stream, i): a window equals the slice
    c = fpsynth.normal(7, 1, 100, start=450)
    assert np.array_equal(c, a[450:550])
    # chunking does not change the stream
    d = fpsynth.normal(7, 1, 1000, chunk=33)
    assert np.array_equal(a, d)
    assert not np.array_equal(a, fpsynth.normal(8, 1, 1000))
    assert not np.array_equal(a, fpsynth.normal(7, 2, 1000))


def test_moments():
    z = fpsynth.normal(3, 1, 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.05  # Gaussian kurtosis


def test_bf16_rounding_matches_torch():
    z = (fpsynth.normal(5, 1, 100_000) * 3).astype(np.float32)
    z[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # ties to even
    ours = fpsynth.f32_to_bf16_bits(z)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = fpsynth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(z).to(torch.bfloat16).float().numpy())


def test_workload_shapes():
    w = fpsynth.WORKLOADS["walrus_bf16"]
    assert (w.Bb, w.T, w.M, w.N) == (4, 6144, 24576, 5376)
    assert fpsynth.WORKLOADS["llm_qkv_rope_bf16"].N == 12288
    assert fpsynth.WORKLOADS["unet_qkv_fp32"].M == 8192
    assert fpsynth.WORKLOADS["tiny_fp32"].N == 160
    inp = fpsynth.make_inputs(fpsynth.WORKLOADS["tiny_fp32"])
    assert inp["x"].shape == (1, 32, 8, 8, 1) and inp["x"].dtype == np.float32
    assert inp["W"].shape == (32, 160) and inp["b"].shape == (160,)
    # weight variance 1/C
    assert abs(inp["W"].var() * 32 - 1.0) < 0.1
