"""Pins of the oracle's E4M3 codec and MXFP8 block rule against things other than itself.

Page "Efficient MoE training for biological foundation models", Key technical approaches,
item 2: 8-bit values with one scale per block of 32 consecutive values.  The element format is
E4M3 and the scale rule the OCP-MX one (reading stated in the oracle's header).
"""
import math
import os
import re

import numpy as np
import pytest
import torch

from tests import _independent as ind

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.txt")


def test_decode_all_codes_match_torch_float8(oracle):
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = ind.torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero kept
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_decode_landmarks(oracle):
    d = oracle.e4m3_decode(np.array([0x7E, 0x01, 0x08, 0x38, 0x07, 0x77, 0xFE], dtype=np.uint8))
    assert d.tolist() == [448.0, 2.0 ** -9, 2.0 ** -6, 1.0, 7 * 2.0 ** -9, 240.0, -448.0]


def test_encode_decode_roundtrip_every_finite_code(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def _bf16_like_values():
    """Every 8-significant-bit magnitude m*2^e (the values a bf16 element takes after any
    power-of-two block scale), both signs, from far below the subnormal range up past the
    saturation point."""
    m = np.arange(128, 256, dtype=np.float64)
    e = np.arange(-170, 3)
    mag = (m[None, :] * np.ldexp(1.0, e)[:, None]).reshape(-1)
    return np.concatenate([mag, -mag, [0.0, -0.0]])


def test_encode_matches_bruteforce_search_exhaustive_bf16(oracle):
    t = _bf16_like_values()
    assert np.array_equal(oracle.e4m3_encode(t), ind.nearest_code(t))


def test_encode_matches_bruteforce_on_midpoints_and_fp32(oracle):
    pos = ind.torch_e4m3_values()[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    # midpoints, one float32 ulp either side, and random float32 values with full 24-bit mantissas
    f32 = mids.astype(np.float32)
    near = np.concatenate([mids, np.nextafter(f32, np.float32(np.inf)).astype(np.float64),
                           np.nextafter(f32, np.float32(-np.inf)).astype(np.float64)])
    rng = np.random.default_rng(7)
    rnd = (rng.uniform(1, 2, 200000) * np.ldexp(1.0, rng.integers(-14, 10, 200000))).astype(np.float32)
    t = np.concatenate([near, -near, rnd.astype(np.float64), -rnd.astype(np.float64),
                        [448.0, 449.0, 463.99, 464.0, 480.0, 511.9, 1e30]])
    assert np.array_equal(oracle.e4m3_encode(t), ind.nearest_code(t))


def test_encode_agrees_with_torch_cast_after_clamp(oracle):
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(100000) * np.ldexp(1.0, rng.integers(-12, 9, 100000))).astype(np.float32)
    clamped = torch.from_numpy(v).clamp(-448, 448)
    ref = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v.astype(np.float64)), ref)


def _eval(expr: str) -> float:
    if not re.fullmatch(r"[0-9.+\-*()p2 ]+", expr):
        raise ValueError(expr)
    return float(eval(expr, {"__builtins__": {}}, {"p2": lambda k: math.ldexp(1.0, k)}))


def _golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "values": [0.0] * 32, "codes": [0] * 32}
            cases.append(cur)
        elif key == "values":
            for tok in rest.split():
                p, v = tok.split(":", 1)
                cur["values"][int(p)] = _eval(v)
        elif key == "sf":
            cur["sf"] = int(rest, 16)
        elif key == "codes":
            for tok in rest.split():
                p, c = tok.split(":", 1)
                cur["codes"][int(p)] = int(c, 16)
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_blocks(oracle, case):
    codes, sf = oracle.quantize_block(np.array(case["values"]))
    assert sf == case["sf"], f"E8M0 byte {sf:#04x} != {case['sf']:#04x}"
    assert codes.tolist() == case["codes"], [hex(c) for c in codes]


def test_golden_file_has_cases():
    assert len(_golden_cases()) >= 10


def test_scaled_amax_lands_in_top_binade(oracle):
    """floor(log2 amax) - 8 is the unique s with amax * 2^-s in [256, 512) (unclamped)."""
    rng = np.random.default_rng(3)
    for _ in range(2000):
        v = rng.standard_normal(32) * math.ldexp(1.0, int(rng.integers(-100, 100)))
        _, sf = oracle.quantize_block(v)
        scaled = np.abs(v).max() * math.ldexp(1.0, -(sf - 127))
        assert 256.0 <= scaled < 512.0


def test_lossless_powers_of_two(oracle):
    """With block max 2^a, every 2^b for a-17 <= b <= a is an E4M3 value after scaling (from 2^8
    down to the smallest subnormal 2^-9) and comes back exactly; 2^(a-18) is a tie with 0."""
    for a in (-100, -3, 0, 5, 60):
        bs = list(range(a - 17, a + 1))
        v = np.array([math.ldexp(1.0, b) for b in bs] + [-math.ldexp(1.0, a - 5)] +
                     [math.ldexp(1.0, a - 18)] + [0.0] * (32 - len(bs) - 2))
        codes, sf = oracle.quantize_block(v)
        back = ind.torch_e4m3_values()[codes] * math.ldexp(1.0, sf - 127)
        assert np.array_equal(back[:len(bs) + 1], v[:len(bs) + 1])
        assert back[len(bs) + 1] == 0.0


def test_three_bit_mantissas_are_lossless(oracle):
    rng = np.random.default_rng(5)
    for _ in range(200):
        a = int(rng.integers(-60, 60))
        m = rng.integers(8, 16, 32) / 8.0                    # 1.xxx with 3 fraction bits
        b = rng.integers(a - 14, a + 1, 32)                  # normal range under the block scale
        m = np.where(b == a, np.minimum(m, 1.75), m)         # above 1.75*2^a the top binade saturates
        v = m * np.ldexp(1.0, b) * rng.choice([-1.0, 1.0], 32)
        v[0] = math.ldexp(1.75, a)                           # pins amax's binade to a
        codes, sf = oracle.quantize_block(v)
        assert sf - 127 == a - 8
        back = ind.torch_e4m3_values()[codes] * math.ldexp(1.0, sf - 127)
        assert np.array_equal(back, v)


def test_sign_symmetry_and_power_of_two_equivariance(oracle):
    rng = np.random.default_rng(9)
    for _ in range(500):
        v = rng.standard_normal(32) * math.ldexp(1.0, int(rng.integers(-40, 40)))
        c0, s0 = oracle.quantize_block(v)
        c1, s1 = oracle.quantize_block(-v)
        assert s1 == s0 and np.array_equal(c1, c0 ^ 0x80)
        k = int(rng.integers(-30, 30))
        c2, s2 = oracle.quantize_block(v * math.ldexp(1.0, k))
        assert s2 == s0 + k and np.array_equal(c2, c0)
