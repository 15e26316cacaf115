"""Pins of the oracle's bfloat16 rounding and 8-bit pixel quantisation (oracle.round_bf16,
oracle.quantize_u8), checked against values worked out by hand, a library routine on the cases
it covers, and closed-form properties; every plausible mistake planted in a copy of the
quantiser below fails at least one of them.

Reading of the 8-bit output (the pages name 8-bit frames, "How Synthesia optimizes generative AI
video inference on Amazon EC2 G7e instances", but not the mapping): the bf16 output v of a decoder
whose outputs lie in [-1, 1] maps to clamp(round_half_even(fp32(fp32(v + 1) * 127.5)), 0, 255).
"""
import math

import numpy as np
import pytest
import torch

import oracle

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127

# (y, round_bf16(y)), worked out by hand from the 8-significant-bit grid
ROUND_PINS = [
    (0.5 + 2 ** -9, 0.5),                 # tie between 0.5 (even) and 0.50390625: down
    (0.5 + 3 * 2 ** -9, 0.5078125),       # tie between 0.50390625 and 0.5078125 (even): up
    (1 + 2 ** -8, 1.0),                   # tie at the bottom of [1, 2): even is 1.0
    (1 + 3 * 2 ** -8, 1.015625),          # tie between 1.0078125 and 1.015625 (even): up
    (1 + 2 ** -8 + 2 ** -20, 1.0078125),  # just above a tie: up
    (-(1 + 3 * 2 ** -8), -1.015625),      # the sign does not change the magnitude's rounding
    (0.1, 0.10009765625),                 # 0.1 = 1.6 * 2^-4 -> 205/128 * 2^-4
    (1.5 * 2 ** -133, 2 ** -132),         # subnormal tie (spacing 2^-133): to even 2 * 2^-133
    (2 ** -140, 0.0),                     # below half the smallest subnormal
    (3.39e38, BF16_MAX),                  # below the overflow threshold (2 - 2^-8) * 2^127
    (3.4e38, math.inf),                   # above it
    (0.0, 0.0),
]

# (y, quantize_u8(y)), worked out by hand
QUANT_PINS = [
    (-1.0, 0),            # t = 0
    (1.0, 255),           # t = 255
    (0.0, 128),           # t = 127.5, tie to even 128
    (-2.0, 0),            # t = -127.5: clamped
    (3.0, 255),           # t = 510: clamped
    (-0.5, 64),           # t = 63.75
    (0.5, 191),           # t = 191.25
    (-2 ** -30, 128),     # fp32(1 - 2^-30) = 1, t = 127.5 -> 128 (float64 arithmetic would give 127)
    (0.5 + 2 ** -9, 191),  # v = 0.5 (bf16 tie to even), t = 191.25
    (0.501957, 192),      # v = 0.50390625 (bf16 rounds up across the pixel boundary 0.50196...)
    (-1 + 1 / 255, 0),    # v = -255/256, t = 0.498046875
]


def pin_failures(quant, rnd=oracle.round_bf16):
    """The pins a (possibly mutated) quantiser / rounding pair fails."""
    bad = []
    for y, exp in ROUND_PINS:
        got = float(rnd(np.array([y]))[0])
        if not (got == exp or (math.isinf(exp) and got == exp)):
            bad.append(("round_bf16", y, got, exp))
    for y, exp in QUANT_PINS:
        got = int(quant(np.array([y]))[0])
        if got != exp:
            bad.append(("quantize_u8", y, got, exp))
    # closed-form properties on a fine grid: monotone, ends pinned, within half a level (plus
    # the bf16 step) of the linear map on [-1, 1]
    y = np.linspace(-1.5, 1.5, 30001)
    q = quant(y).astype(np.int64)
    if np.any(np.diff(q) < 0):
        bad.append(("monotone",))
    inside = np.abs(y) <= 1
    lin = (y[inside] + 1) * 127.5
    if np.max(np.abs(q[inside] - lin)) > 0.5 + 127.5 * 2 ** -8 + 1e-9:
        bad.append(("linear map",))
    return bad


def test_round_bf16_and_quantize_u8_meet_their_pins():
    assert pin_failures(oracle.quantize_u8) == []


def test_round_bf16_equals_the_library_conversion_on_float32_inputs():
    """torch's float32 -> bfloat16 conversion rounds to nearest even: on float32 inputs the two
    agree (a library special case of the definition)."""
    rng = np.random.default_rng(3)
    mant = rng.uniform(1.0, 2.0, 200000)
    expo = rng.integers(-130, 127, 200000)
    v = (np.ldexp(mant, expo) * rng.choice([-1, 1], 200000)).astype(np.float32)
    # exact ties and their neighbours: the 16 low bits of the float32 pattern at 0x8000 +- 1 under
    # random finite upper halves (sign, exponent 1..254, 7 mantissa bits)
    hi = rng.integers(0x0080, 0x7F80, 20000, dtype=np.uint32) | (rng.integers(0, 2, 20000, dtype=np.uint32) << 15)
    base = hi << np.uint32(16)
    ties = np.concatenate([base | np.uint32(0x8000), base | np.uint32(0x7FFF), base | np.uint32(0x8001)])
    v = np.concatenate([v, ties.view(np.float32)])
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(v.astype(np.float64)), lib)


# plausible mistakes, each planted in a copy of the quantiser; every one must fail a pin
def _m_no_bf16(y):
    t = (np.asarray(y, np.float64).astype(np.float32) + np.float32(1)) * np.float32(127.5)
    return np.clip(np.rint(t), 0, 255).astype(np.uint8)


def _m_float64_math(y):
    t = (oracle.round_bf16(y) + 1.0) * 127.5
    return np.clip(np.rint(t), 0, 255).astype(np.uint8)


def _m_scale_128(y):
    t = (oracle.round_bf16(y).astype(np.float32) + np.float32(1)) * np.float32(128.0)
    return np.clip(np.rint(t), 0, 255).astype(np.uint8)


def _m_no_clamp(y):
    t = (oracle.round_bf16(y).astype(np.float32) + np.float32(1)) * np.float32(127.5)
    return np.rint(t).astype(np.int64).astype(np.uint8)


def _m_truncate(y):
    t = (oracle.round_bf16(y).astype(np.float32) + np.float32(1)) * np.float32(127.5)
    return np.clip(np.trunc(t), 0, 255).astype(np.uint8)


def _m_wrong_offset(y):
    t = (oracle.round_bf16(y).astype(np.float32) - np.float32(1)) * np.float32(127.5)
    return np.clip(np.rint(t), 0, 255).astype(np.uint8)


def _r_half_up(y):
    y = np.asarray(y, np.float64)
    _, e = np.frexp(y)
    s = np.maximum(e, -125) - 8
    return np.ldexp(np.sign(y) * np.floor(np.abs(np.ldexp(y, -s)) + 0.5), s)


def _r_truncate(y):
    y = np.asarray(y, np.float64)
    _, e = np.frexp(y)
    s = np.maximum(e, -125) - 8
    return np.ldexp(np.trunc(np.ldexp(y, -s)), s)


def _r_no_subnormals(y):
    y = np.asarray(y, np.float64)
    _, e = np.frexp(y)
    s = e - 8
    return np.ldexp(np.rint(np.ldexp(y, -s)), s)


def _quant_with(rnd):
    def q(y):
        t = (rnd(y).astype(np.float32) + np.float32(1)) * np.float32(127.5)
        return np.clip(np.rint(t), 0, 255).astype(np.uint8)
    return q


MUTANTS = {
    "no bf16 rounding": (_m_no_bf16, oracle.round_bf16),
    "float64 arithmetic": (_m_float64_math, oracle.round_bf16),
    "scale 128": (_m_scale_128, oracle.round_bf16),
    "no clamp": (_m_no_clamp, oracle.round_bf16),
    "truncation instead of rounding": (_m_truncate, oracle.round_bf16),
    "offset -1": (_m_wrong_offset, oracle.round_bf16),
    "bf16 ties away from zero": (_quant_with(_r_half_up), _r_half_up),
    "bf16 truncation": (_quant_with(_r_truncate), _r_truncate),
    "bf16 without subnormals": (_quant_with(_r_no_subnormals), _r_no_subnormals),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name):
    quant, rnd = MUTANTS[name]
    assert pin_failures(quant, rnd), name
