"""Pins of the fused MLA write oracle (oracle/mla_write_ref.py): bf16 rounding,
RMSNorm and RoPE against closed forms, invariants and a library rounding routine."""
import numpy as np
import torch

from oracle import mla_write_ref as mw
from oracle.paged_ref import bf16_bits_to_f64


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(71)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    # Exact halfway cases: lower 16 bits 0x8000.
    ties = ((rng.integers(0x3000, 0x4F00, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mw.round_to_bf16_bits(x.astype(np.float64)), want)


def test_bf16_rounding_ties_to_even_by_hand():
    one = 1.0
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even neighbour is 1.
    assert bf16_bits_to_f64(mw.round_to_bf16_bits(np.array([one + 2 ** -8])))[0] == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert bf16_bits_to_f64(mw.round_to_bf16_bits(np.array([one + 3 * 2 ** -8])))[0] == 1 + 2 ** -6
    assert bf16_bits_to_f64(mw.round_to_bf16_bits(np.array([one + 2 ** -8 + 2 ** -30])))[0] == 1 + 2 ** -7


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(72)
    g = rng.standard_normal(512)
    c = np.full((1, 512), -3.5)
    np.testing.assert_allclose(mw.rmsnorm(c, g, 0.0)[0], -g, rtol=1e-15)
    x = rng.standard_normal((4, 512))
    np.testing.assert_allclose(mw.rmsnorm(7.25 * x, g, 0.0), mw.rmsnorm(x, g, 0.0), rtol=1e-13)
    y = mw.rmsnorm(x, np.ones(512), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-13)
    # eps enters under the root: a zero row stays zero, a tiny row is damped.
    assert np.all(mw.rmsnorm(np.zeros((1, 512)), g, 1e-6) == 0)
    t = np.full((1, 512), 1e-3)
    np.testing.assert_allclose(mw.rmsnorm(t, np.ones(512), 1e-6)[0], 1e-3 / np.sqrt(1e-6 + 1e-6))


def test_rope_pairs_i_with_i_plus_half():
    d = 64
    e0 = np.zeros((1, d))
    e0[0, 0] = 1.0
    cos, sin = np.zeros((1, d)), np.ones((1, d))  # angle pi/2 everywhere
    out = mw.rope_rotate_half(e0, cos, sin)[0]
    assert out[32] == 1.0 and np.count_nonzero(out) == 1
    e32 = np.zeros((1, d))
    e32[0, 32] = 1.0
    out = mw.rope_rotate_half(e32, cos, sin)[0]
    assert out[0] == -1.0 and np.count_nonzero(out) == 1
    x = np.random.default_rng(73).standard_normal((3, d))
    np.testing.assert_array_equal(mw.rope_rotate_half(x, np.ones((3, d)), np.zeros((3, d))), x)


def test_rope_is_a_rotation_per_pair_and_composes():
    rng = np.random.default_rng(74)
    d = 64
    x = rng.standard_normal((5, d))
    th1 = rng.uniform(-4, 4, (5, d // 2))
    th2 = rng.uniform(-4, 4, (5, d // 2))

    def cs(th):
        full = np.concatenate([th, th], axis=1)
        return np.cos(full), np.sin(full)

    y = mw.rope_rotate_half(x, *cs(th1))
    np.testing.assert_allclose(y[:, :32] ** 2 + y[:, 32:] ** 2, x[:, :32] ** 2 + x[:, 32:] ** 2, rtol=1e-12)
    np.testing.assert_allclose(mw.rope_rotate_half(y, *cs(th2)), mw.rope_rotate_half(x, *cs(th1 + th2)),
                               atol=1e-12)
