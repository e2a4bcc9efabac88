"""The seeded input generators shared by the oracle and the CUDA path:
deterministic, counter-based (values do not depend on the thread count or on
how much is drawn after them), and the bf16 storage rounding is IEEE
round-to-nearest-even.  CPU only."""
import numpy as np
import pytest
import torch

import workloads as W


def test_same_seed_same_values_and_roles_differ():
    a = W.normal(3, W.TID["a"], (1000,))
    assert np.array_equal(a, W.normal(3, W.TID["a"], (1000,)))
    assert not np.array_equal(a, W.normal(3, W.TID["b"], (1000,)))
    assert not np.array_equal(a, W.normal(4, W.TID["a"], (1000,)))


def test_values_do_not_depend_on_the_amount_drawn():
    n = W.BLOCK + 1000  # two blocks
    big = W.normal(5, 1, (n,))
    assert np.array_equal(big[:1000], W.normal(5, 1, (1000,)))
    assert np.array_equal(W.uniform(5, 2, (n,), 0.1, 1.0)[:777], W.uniform(5, 2, (777,), 0.1, 1.0))


def test_values_do_not_depend_on_the_thread_count(monkeypatch):
    n = 2 * W.BLOCK + 5
    many = W.sigmoid_of_normal(6, 1, (n,), 2.0, 1.0)
    monkeypatch.setattr(W, "_threads", lambda: 1)
    assert np.array_equal(many, W.sigmoid_of_normal(6, 1, (n,), 2.0, 1.0))


def test_distributions_and_ranges():
    z = W.normal(7, 1, (200000,), mean=1.0, std=0.5).astype(np.float64)
    assert abs(z.mean() - 1.0) < 0.01 and abs(z.std() - 0.5) < 0.01
    u = W.uniform(7, 2, (200000,), 0.9, 1.0)
    assert u.min() >= 0.9 and u.max() <= 1.0
    s = W.sigmoid_of_normal(7, 3, (1000,))
    assert s.min() > 0.0 and s.max() < 1.0


def test_bf16_rounding_is_nearest_even():
    r = np.random.default_rng(8)
    x = np.concatenate([
        r.standard_normal(100000).astype(np.float32),
        np.float32([0.0, -0.0, 1.0, -2.5, 3.4e38, -3.4e38, 1e-40, np.inf, -np.inf]),
        # exact ties: the low 16 bits are 0x8000, rounding to the even neighbour
        (np.uint32([0x3F808000, 0x3F818000, 0xBF808000]).view(np.float32)),
    ])
    got = W.f32_to_bf16(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert np.array_equal(W.to_f64(got, "bf16"), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_bf16_rounding_keeps_nan():
    x = np.uint32([0x7F800001, 0xFF800001, 0x7FC00000, 0x7FFFFFFF]).view(np.float32)
    got = W.bf16_to_f32(W.f32_to_bf16(x))
    assert np.isnan(got).all()
    assert np.signbit(got).tolist() == [False, True, False, False]
