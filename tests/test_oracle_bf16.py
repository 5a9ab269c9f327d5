"""Pins for the oracle's fp32 -> bf16 round-to-nearest-even (deg/zero.py, gather_params).

Pinned against torch's own float -> bfloat16 conversion (a library routine, independent of
the oracle) over a structured sweep of bit patterns, and against hand-worked ties.
"""
import numpy as np
import torch

from oracle.bf16 import bf16_bits_to_f32, f32_to_bf16_bits


def torch_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_hand_ties_and_specials():
    f = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8), 0.0, -0.0,
                  np.inf, -np.inf], dtype=np.float32)
    b = f32_to_bf16_bits(f)
    # 1+2^-8 is a tie between 1 (even) and 1+2^-7 -> 1; 1+3*2^-8 ties to 1+2^-6 (even)
    assert b.tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80, 0x0000, 0x8000, 0x7F80, 0xFF80]
    # the largest finite fp32 rounds past the largest bf16: RNE gives infinity
    assert f32_to_bf16_bits(np.array([np.finfo(np.float32).max], np.float32))[0] == 0x7F80
    nan = np.array([0x7FC00001, 0xFF800001, 0x7F800001], dtype=np.uint32).view(np.float32)
    out = f32_to_bf16_bits(nan)
    assert np.all((out & 0x7F80) == 0x7F80) and np.all((out & 0x007F) != 0)
    assert (out[1] & 0x8000) == 0x8000


def test_against_torch_structured_sweep():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x3FFF, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF, 0x1234, 0xC000],
                    dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).reshape(-1)
    rng = np.random.default_rng(7)
    pats = np.concatenate([pats, rng.integers(0, 1 << 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)])
    x = pats.view(np.float32)
    mine = f32_to_bf16_bits(x)
    ref = torch_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(np.isnan(bf16_bits_to_f32(mine[nan])))


def test_widening_is_exact():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f32(b)
    back = f32_to_bf16_bits(f)
    ok = ~np.isnan(f)
    assert np.array_equal(back[ok], b[ok])
