"""The pre-attention kernel's rotation angles, method checked on the CPU.

The kernel forms sin and cos of pos * f in float32 (below position 2^24):
pos * f as ph + pl from f split into two floats, a Cody-Waite reduction by
pi / 2 held in three floats, a second reduction step for the quadrant's
rounding above 2^22, then the Taylor series of sin (through x^9) and cos
(through x^8) on [-pi/4, pi/4] and the quadrant's symmetry. This test
restates those float32 steps (each FMA as an exact double product plus one
rounding to float32) and bounds their error against fp64 sin and cos of
pos * f, where f is the double frequency the host computes: the kernel's
error budget in the parity bar (2^-20 of |y_d| + |y_partner| for all of its
fp32 error) leaves room for about 2^-21 here. The constants below are the
method's; the GPU tests check the kernel itself against the fp64 oracle.
"""
import numpy as np
import pytest

F32 = np.float32
P1, P2, P3 = F32(1.5707963705062866), F32(-4.3711388286737929e-8), F32(-1.7151245100058819e-15)
TWO_OVER_PI = F32(0.63661974668502808)


def fma(a, b, c):
    """float32 fma: the product of two floats is exact in a double."""
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)
            ).astype(F32)


def sincos_quadrant(x, qd):
    x2 = (x * x).astype(F32)
    sp = fma(x2, F32(1 / 362880), F32(-1 / 5040))
    sp = fma(x2, sp, F32(1 / 120))
    sp = fma(x2, sp, F32(-1 / 6))
    sx = fma((x * x2).astype(F32), sp, x)
    cp = fma(x2, F32(1 / 40320), F32(-1 / 720))
    cp = fma(x2, cp, F32(1 / 24))
    cp = fma(x2, cp, F32(-0.5))
    cx = fma(x2, cp, F32(1))
    s0 = np.where(qd & 1, cx, sx)
    c0 = np.where(qd & 1, sx, cx)
    return np.where(qd & 2, -s0, s0), np.where((qd + 1) & 2, -c0, c0)


def angle_sincos(pos, f):
    """(sin, cos, reduced x) of pos * f for integer positions below 2^24."""
    fh = f.astype(F32)
    fl = (f - fh.astype(np.float64)).astype(F32)
    pf = pos.astype(F32)
    ph = (pf * fh).astype(F32)
    pl = fma(pf, fl, fma(pf, fh, -ph))
    n1 = np.rint((ph * TWO_OVER_PI).astype(F32)).astype(F32)
    x = (fma(-n1, P3, fma(-n1, P2, fma(-n1, P1, ph))) + pl).astype(F32)
    n2 = np.rint((x * TWO_OVER_PI).astype(F32)).astype(F32)
    x = fma(-n2, P2, fma(-n2, P1, x))
    qd = n1.astype(np.int64) + n2.astype(np.int64)
    s, c = sincos_quadrant(x, qd)
    return s, c, x


def test_three_float_half_pi_split():
    """Each part is the float nearest to what the earlier ones leave of pi / 2
    (50-digit arithmetic), so P1 + P2 + P3 is within half a float unit of P3
    of pi / 2; 2 / pi is the float nearest to it."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    half_pi = mpmath.pi / 2
    rest = half_pi
    for part in (P1, P2, P3):
        assert part == F32(float(rest)), part
        rest = rest - mpmath.mpf(float(part))
    assert abs(rest) <= abs(mpmath.mpf(float(P3))) * 2.0 ** -24
    assert TWO_OVER_PI == F32(float(2 / mpmath.pi))


def test_angles_within_budget():
    rng = np.random.default_rng(7)
    pos = np.concatenate([
        np.arange(0, 4096),                                   # the first pages
        rng.integers(4096, 1 << 22, 3000),                    # one reduction step
        rng.integers(1 << 22, 1 << 24, 3000),                 # the second step acts here
        np.arange((1 << 24) - 256, 1 << 24),                  # the top of the float path
    ]).astype(np.int64)
    worst = 0.0
    for hd, theta in ((256, 1e4), (512, 1e6)):
        i = np.arange(hd // 2)
        f = np.exp(-2.0 * i / hd * np.log(theta))
        P, Fq = np.meshgrid(pos, f, indexing="ij")
        s, c, x = angle_sincos(P.ravel(), Fq.ravel())
        assert np.abs(x).max() <= np.pi / 4 + 1e-6, "remainder outside [-pi/4, pi/4]"
        a = P.ravel().astype(np.float64) * Fq.ravel()
        err = max(np.abs(s - np.sin(a)).max(), np.abs(c - np.cos(a)).max())
        worst = max(worst, float(err))
    assert worst < 2.5e-7, worst


def test_one_reduction_step_is_not_enough_above_2_22():
    """Without the second step the quadrant is sometimes off near 2^24: the
    remainder then leaves [-pi/4, pi/4], where the polynomials do not hold
    (this is why the kernel takes the second step)."""
    pos = np.arange((1 << 24) - 20000, 1 << 24, dtype=np.int64)
    f = np.exp(-2.0 * np.arange(128) / 256 * np.log(1e4))
    P, Fq = np.meshgrid(pos, f, indexing="ij")
    fh = Fq.ravel().astype(F32)
    fl = (Fq.ravel() - fh.astype(np.float64)).astype(F32)
    pf = P.ravel().astype(F32)
    ph = (pf * fh).astype(F32)
    pl = fma(pf, fl, fma(pf, fh, -ph))
    n1 = np.rint((ph * TWO_OVER_PI).astype(F32)).astype(F32)
    x = (fma(-n1, P3, fma(-n1, P2, fma(-n1, P1, ph))) + pl).astype(F32)
    assert np.abs(x).max() > np.pi / 4 + 0.1
