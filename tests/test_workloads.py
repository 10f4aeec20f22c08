"""The seeded input generator (CPU only)."""
import math

import numpy as np
import torch

from selective_state_space_diagonal_b300 import workloads as wl


def test_splitmix64_reference_outputs():
    # SplitMix64 started from state 0 yields these first three outputs (Steele, Lea and
    # Flood's generator as published; the draw at counter i is the output after i+1 steps).
    got = wl.draws(np.uint64(0), np.arange(3, dtype=np.uint64))
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_thread_independent():
    w = wl.WORKLOADS["euler_f32_tiny"].with_shape(B=2, L=300, D=24, N=8, mode=1)
    a = wl.generate(w, threads=1)
    b = wl.generate(w, threads=8)
    for k in ("x", "delta", "A", "Bc", "Cc", "theta", "lam", "Dskip"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-8, 3, 100000)).astype(np.float32)
    mine = wl.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    back = wl.bf16_bits_to_f32(mine)
    assert np.array_equal(back, torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_distributions():
    w = wl.WORKLOADS["trap_bf16_batch"].with_shape(B=2, L=512, D=64, N=16)
    inp = wl.generate(w)
    f = wl.widen(inp)
    assert abs(f["x"].mean()) < 0.02 and abs(f["x"].std() - 1.0) < 0.02
    assert abs(f["Bc"].real.std() - 0.5) < 0.02 and abs(f["Cc"].imag.std() - 0.5) < 0.02
    assert f["delta"].min() >= 1e-3 * 0.99 and f["delta"].max() <= 1e-1 * 1.01
    lg = np.log(f["delta"])
    assert abs(lg.mean() - 0.5 * (math.log(1e-3) + math.log(1e-1))) < 0.05
    assert f["theta"].min() >= -math.pi * 1.001 and f["theta"].max() <= math.pi * 1.001
    assert 0.0 < f["lam"].min() and f["lam"].max() < 1.0 and abs(f["lam"].mean() - 0.5) < 0.03
    assert f["A"].max() <= -1.0 + 1e-6 and f["A"].min() >= -16.0 - 1e-5
    w3 = wl.WORKLOADS["euler_bf16_long"].with_shape(L=64, D=8)
    A3 = wl.generate(w3).A
    assert np.array_equal(A3, np.tile(-(np.arange(16) + 1) / 16.0, (8, 1)).astype(np.float32))
    assert wl.generate(w3).lam is None


def test_min_bytes():
    expect = {"euler_f32_tiny": 9.07e4, "euler_f32_mamba1": 3.91e7, "trap_bf16_mamba3": 2.74e8,
              "euler_bf16_long": 1.095e9, "trap_bf16_batch": 2.71e9}
    for name, v in expect.items():
        assert abs(wl.WORKLOADS[name].min_bytes() / v - 1.0) < 0.01, name
