"""Pins the fp8 (e4m3) rounding that the fp8-cache tests take as their expected
bytes (a torch cast) to the format's own definition: 1 sign bit, 4 exponent bits
with bias 7, 3 mantissa bits, subnormals below 2^-6, largest finite value 448,
and round to nearest with ties to the even code."""

import numpy as np
import torch


def _e4m3_values():
    """Value of every finite code 0..255 (codes 0x7F and 0xFF are NaN)."""
    vals = {}
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 0xF, code & 0x7
        if e == 0xF and m == 0x7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = -mag if s else mag
    return vals


def _round_to_e4m3(x: float) -> int:
    """Nearest finite code, ties to the code with an even mantissa (sign kept for zero)."""
    vals = _e4m3_values()
    pos = sorted((v, c) for c, v in vals.items() if c < 0x80)
    mag = min(abs(x), 448.0)
    best = min(pos, key=lambda vc: (abs(vc[0] - mag), vc[1] & 1))
    code = best[1]
    return code | (0x80 if x < 0 or (x == 0 and np.signbit(x)) else 0)


def test_format_table():
    v = _e4m3_values()
    assert len(v) == 254 and max(v.values()) == 448.0 and min(x for x in v.values() if x > 0) == 2.0 ** -9
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0 and v[0x08] == 2.0 ** -6


def test_torch_cast_is_round_to_nearest_even_e4m3():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(3000, generator=g) * 40, torch.randn(1000, generator=g) * 0.01,
                   torch.tensor([0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875,
                                 17.0, 19.0, 440.0, 432.0])])
    x = x.clamp(-448, 448)
    got = x.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    want = [_round_to_e4m3(float(t)) for t in x]
    assert got == want
