"""The rotary-angle method the kernels use, replayed step by step in float32 on the host: the
inverse frequency as a float pair (hi, lo), the position times it carried with its fma-recovered
rounding error, and a Cody-Waite reduction by 2*pi with a two-part constant.  The reduced angle
must give cos/sin within 5e-7 of float64 over positions up to 2^24 for every frequency of the
workloads' RoPE tables, and the first reduction product must cancel exactly."""
import math

import numpy as np

F = np.float32
C1 = F(2 * math.pi)                       # float(2 pi)
C2 = F(2 * math.pi - float(C1))           # the remainder of 2 pi
INV_2PI = F(1 / (2 * math.pi))


def fma32(a, b, c):
    """float32 fused multiply-add: exact product and sum, one rounding (float64 holds the
    product of two float32 values exactly, and the sum of the magnitudes here exactly too)."""
    return F(np.float64(a) * np.float64(b) + np.float64(c))


def reduce_angle(p, ih, il):
    pf = F(p)
    hi = F(pf * ih)
    lo = F(fma32(pf, ih, -hi) + F(pf * il))
    k = F(np.rint(F(hi * INV_2PI)))
    r = fma32(-k, C1, hi)
    r = F(fma32(-k, C2, r) + lo)
    return r, k, hi


def inv_table(base, D, two_d=False):
    width = D // 2 if two_d else D
    return [base ** (-2.0 * j / width) for j in range(width // 2)]


def test_first_reduction_step_is_exact():
    rng = np.random.default_rng(1)
    for inv in inv_table(1e6, 128) + inv_table(1.11588e7, 128):
        ih = F(inv)
        for p in rng.integers(0, 1 << 24, 300):
            hi = F(F(p) * ih)
            k = F(np.rint(F(hi * INV_2PI)))
            exact = np.float64(hi) - np.float64(k) * np.float64(C1)
            assert np.float64(fma32(-k, C1, hi)) == exact


def test_cos_sin_match_float64():
    rng = np.random.default_rng(0)
    positions = list(rng.integers(0, 1 << 24, 400)) + [0, 1, 2, 511, 767, 32767, 33792, (1 << 24) - 1]
    worst = 0.0
    for base, D, two_d in ((1e6, 128, False), (1.11588e7, 128, False), (1e6, 72, True), (1e6, 64, False)):
        for inv in inv_table(base, D, two_d):
            ih = F(inv)
            il = F(inv - float(ih))
            for p in positions:
                r, _, _ = reduce_angle(int(p), ih, il)
                exact = math.remainder(int(p) * inv, 2 * math.pi)
                err = abs(math.cos(float(r)) - math.cos(exact)) + abs(math.sin(float(r)) - math.sin(exact))
                worst = max(worst, err)
    assert worst <= 5e-7, worst


def test_reduced_angle_is_small():
    """k comes from a float estimate of hi / (2 pi), so near a half-turn boundary it can be off by
    one for large positions: the reduced angle stays within 2 pi (float sin/cos stay on their
    short-argument path), and within pi + 1e-3 while p * inv < 2^17."""
    for inv in inv_table(1e6, 128) + inv_table(1.11588e7, 128):
        ih = F(inv)
        il = F(inv - float(ih))
        for p in list(range(0, 1 << 24, 99991)) + [(1 << 24) - 1]:
            r, _, hi = reduce_angle(p, ih, il)
            assert abs(float(r)) <= 2 * math.pi
            if abs(float(hi)) < (1 << 17):
                assert abs(float(r)) <= math.pi + 1e-3
