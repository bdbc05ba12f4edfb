"""The append kernels compute x / s as Markstein's correction of the
reciprocal product (P. Markstein, IBM J. Res. Develop. 34, 1990): y = RN(1/s),
q0 = RN(x y), r = RN(x - q0 s) (exact), q = RN(q0 + r y), with the sign of q0
put on q (so that -0 stays -0). They take that path for a scale in
[2^-80, 2^100] and a group of finite inputs whose largest |x| y stays below
2^100; the IEEE division elsewhere. Two facts make that exact for the e4m3
codes the oracle computes from RN(x / s): where the code depends on the
quotient's last bit (|x / s| in [2^-12, 2^10]) the corrected quotient equals
RN(x / s), checked in exact arithmetic on every finite bf16 x for a sample of
scales (powers of two and their neighbours, log-uniform, amax/448); and
everywhere on the fast path the code of the corrected quotient equals the
code of RN(x / s), checked over every finite bf16 x for scales across the
whole accepted range. CPU only: these pin the identities the GPU path relies
on, not the GPU."""
from fractions import Fraction

import numpy as np


def _rn32_sum(a64, b64):
    """RN32(a + b) for float64 a, b whose exact sum may need more than 53 bits."""
    s = a64 + b64
    bb = s - a64
    err = (a64 - (s - bb)) + (b64 - bb)          # a + b == s + err exactly (TwoSum)
    r = s.astype(np.float32)
    r64 = r.astype(np.float64)
    up = np.nextafter(r, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(r, np.float32(-np.inf)).astype(np.float64)
    tie = ((s - r64) * 2 == (up - r64)) | ((s - r64) * 2 == (dn - r64))
    for i in np.nonzero(tie & (err != 0))[0]:
        v = Fraction(float(s[i])) + Fraction(float(err[i]))
        lo, hi = (float(dn[i]), float(r64[i])) if v < Fraction(float(r64[i])) else (float(r64[i]), float(up[i]))
        r[i] = np.float32(lo if v < (Fraction(lo) + Fraction(hi)) / 2 else hi)
    return r


def test_markstein_quotient_equals_ieee_division_where_used():
    rng = np.random.default_rng(7)
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x)]
    x64 = x.astype(np.float64)
    p2 = np.float32(2.0) ** np.arange(-16, 8, dtype=np.float32)
    scales = np.concatenate([
        (10.0 ** rng.uniform(-4, 2, 60)).astype(np.float32), p2,
        np.nextafter(p2, np.float32(np.inf)), np.nextafter(p2, np.float32(0)),
        (rng.uniform(0.001, 10, 40) / 448).astype(np.float32),
    ])
    checked = 0
    with np.errstate(all="ignore"):
        for s in scales:
            s = np.float32(s)
            y = np.float32(1.0) / s                                    # RN(1 / s)
            q0 = x * y                                                 # RN(x y)
            r = (x64 - q0.astype(np.float64) * np.float64(s)).astype(np.float32)  # exact residual
            q = _rn32_sum(r.astype(np.float64) * np.float64(y), q0.astype(np.float64))
            used = (np.abs(x) >= np.float32(2.0 ** -100)) & (np.abs(q0) >= np.float32(2.0 ** -12)) & \
                   (np.abs(q0) <= np.float32(2.0 ** 10))
            assert np.array_equal(q[used], (x / s)[used]), float(s)
            checked += int(used.sum())
    assert checked > 500_000


def _corrected(x, s):
    """The kernels' fast path for the values x (float32) and the scale s."""
    x64 = x.astype(np.float64)
    y = np.float32(1.0) / s                                        # RN(1 / s)
    q0 = x * y                                                     # RN(x y)
    r = (x64 - q0.astype(np.float64) * np.float64(s)).astype(np.float32)  # RN(x - q0 s)
    q = _rn32_sum(r.astype(np.float64) * np.float64(y), q0.astype(np.float64))
    return np.copysign(q, q0), y


def test_corrected_quotient_gives_the_oracles_codes_on_the_whole_fast_path():
    from oracle.append_ref import e4m3_encode
    rng = np.random.default_rng(11)
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x)]                                          # every finite bf16, both zeros included
    p2 = np.float32(2.0) ** np.arange(-80, 101, 9, dtype=np.float32)
    scales = np.concatenate([p2, np.nextafter(p2, np.float32(np.inf)),
                             np.float32(2.0) ** rng.uniform(-80, 100, 24).astype(np.float32),
                             np.float32([2.0 ** -80, 2.0 ** 100, 0.0137, 1.0 / 448, 3.0 ** 60])])
    checked = 0
    with np.errstate(all="ignore"):
        for s in scales:
            s = np.float32(s)
            q, y = _corrected(x, s)
            fast = np.abs(x).astype(np.float64) * abs(float(y)) < 2.0 ** 100
            got, want = e4m3_encode(q[fast]), e4m3_encode((x / s)[fast])
            assert np.array_equal(got, want), (float(s), x[fast][got != want][:4])
            checked += int(fast.sum())
    assert checked > 3_000_000
