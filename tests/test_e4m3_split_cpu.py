"""The two-term e4m3 form of q that the FP8-cache kernels' score MMAs take.

Over an FP8 cache (head_dim 128) the kernels compute S on the e4m3 key codes as
they are, against q written as two e4m3 terms per element: a row (prefill) or
head (decode) of q is scaled by 2^(8 - ex), ex the binary exponent of its
largest magnitude, so that every element x lies below 256; the first term is
the e4m3 rounding of x and the second the e4m3 rounding of the remainder.

The claim checked here, with PyTorch's float8_e4m3fn rounding (round to nearest
even, the rounding of cvt.rn.satfinite.e4m3x2.f32) as the reference: for every
bf16 value (8 significant bits) the remainder is a multiple of x's last bit no
larger than 8 of them, hence an e4m3 value, and the two terms sum to x exactly
unless the remainder falls under e4m3's smallest subnormal (2^-9); then the
error is at most half of it, 2^-10 in the scaled unit.
"""
import numpy as np
import pytest
import torch


def _split(x: torch.Tensor):
    t1 = x.to(torch.float8_e4m3fn).to(torch.float32)
    t2 = (x - t1).to(torch.float8_e4m3fn).to(torch.float32)
    return t1, t2


def _all_bf16_in(lo_exp: int, hi_exp: int) -> torch.Tensor:
    """Every bf16 value with binary exponent in [lo_exp, hi_exp), both signs."""
    vals = []
    for e in range(lo_exp, hi_exp):
        m = torch.arange(128, dtype=torch.float32)
        vals.append((1.0 + m / 128.0) * 2.0 ** e)
    v = torch.cat(vals)
    v = v.to(torch.bfloat16).to(torch.float32)
    return torch.cat([v, -v])


def test_two_terms_are_exact_above_the_floor():
    """Every bf16 magnitude from 2^-2 up to the scaled row maximum (< 256)."""
    x = _all_bf16_in(-2, 8)
    t1, t2 = _split(x)
    assert torch.equal(t1 + t2, x)


def test_below_the_floor_error_is_at_most_half_a_subnormal_step():
    x = _all_bf16_in(-16, -2)
    t1, t2 = _split(x)
    err = (t1 + t2 - x).abs()
    assert float(err.max()) <= 2.0 ** -10
    # and the first term alone would be far coarser: the second term does work here
    assert float((t1 - x).abs().max()) > 2.0 ** -8


def test_row_scaling_keeps_every_element_below_256():
    """Scaling by 2^(8 - ex) (frexp's exponent of the largest magnitude) puts the
    largest element in [128, 256), so no term saturates at e4m3's 448."""
    rng = np.random.default_rng(5)
    for scale in [1e-3, 0.7, 1.0, 3.0, 200.0, 6.0e4]:
        q = torch.from_numpy(rng.standard_normal((64, 128)).astype(np.float32) * scale)
        q = q.to(torch.bfloat16).to(torch.float32)
        m = q.abs().amax(dim=1)
        ex = torch.frexp(m).exponent
        f = torch.ldexp(torch.ones_like(m), 8 - ex)
        xs = q * f[:, None]
        assert float(xs.abs().max()) < 256.0 and float(xs.abs().amax(dim=1).min()) >= 128.0
        t1, t2 = _split(xs)
        rec = (t1 + t2) / f[:, None]
        # relative to each row's largest magnitude the representation error is
        # below 2^-17 (2^-10 of the scaled unit over a row maximum of at least 128)
        rel = ((rec - q).abs() / m[:, None]).max()
        assert float(rel) <= 2.0 ** -17, float(rel)
        # and every element of at least 2^-9 of its row's largest comes back exactly
        # (scaled, it is at least 2^-9 x 128 = 2^-2, where the terms are exact)
        big = q.abs() >= m[:, None] * 2.0 ** -9
        assert torch.equal(rec[big], q[big])


@pytest.mark.parametrize("v", [1.0, 1.9921875, 255.0, 0.25, 127.5])
def test_hand_worked_values(v):
    """1.9921875 = 1 + 127/128 rounds up to 2 (remainder -1/128, an e4m3
    subnormal multiple); 255 = 256 - 1 rounds to 256 (remainder -1)."""
    x = torch.tensor([v], dtype=torch.float32)
    t1, t2 = _split(x)
    assert float(t1 + t2) == v
