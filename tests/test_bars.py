"""The bf16 parity bar (tests/bars.py) against torch's own bf16 rounding."""

from __future__ import annotations

import numpy as np
import torch

from tests.bars import O_MAX, bf16_half_spacing, o_bar


def _bf16_neighbours(x: np.ndarray):
    """(bf16(x), the next bf16 value away from zero), via the bit patterns."""
    b = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().astype(np.int32)
    up = torch.from_numpy((bits + 1).astype(np.int16)).view(torch.bfloat16)
    return b.double().numpy(), up.double().numpy()


def test_half_spacing_is_half_the_gap_between_bf16_neighbours():
    g = np.random.default_rng(0)
    # float32 values, which torch rounds to bf16 in one step
    x = np.ldexp(g.uniform(1.0, 2.0, 4000), g.integers(-12, 12, 4000)).astype(np.float32)
    r, up = _bf16_neighbours(x)
    # r and its neighbour are in the same binade unless r is the binade's top
    same = np.frexp(up)[1] == np.frexp(r)[1]
    np.testing.assert_array_equal(bf16_half_spacing(r)[same], (up - r)[same] / 2)
    # rounding moves no value by more than the half-spacing of the result
    assert (np.abs(r - x) <= bf16_half_spacing(r)).all()


def test_bar_is_flat_below_8_and_adds_the_half_spacing_from_8():
    assert bf16_half_spacing(7.99) == 2.0 ** -6 and bf16_half_spacing(8.0) == 2.0 ** -5
    assert o_bar(np.array([7.9]), np.array([7.95]))[0] == O_MAX
    assert o_bar(np.array([7.99]), np.array([8.01]))[0] == O_MAX + 2.0 ** -5
    assert o_bar(np.array([-20.0]), np.array([-19.0]))[0] == O_MAX + 2.0 ** -4
    assert o_bar(np.array([0.0]), np.array([0.0]))[0] == O_MAX
