"""The group quantiser's fast path against the definition it replaces.

The CUDA quantiser (the W_c3 epilogue and the decode-time write) takes each code
q = floor(RN(RN(d / delta) + 1/2)), d = z - min, from x = d * RN(1/delta): one FMA adds
1.5 * 2^23 so that round(x) lands in the low mantissa bits, a second FMA gives
r = x - round(x), and the whole group is recomputed with the division when any |r| comes
within 2^-17 of 1/2.  This test restates those float32 steps with exact emulation (a
float32 FMA is the float64 sum of the exact product, rounded once to float32) and checks,
on random groups and on groups built to sit on or next to the decision points, that every
group the fast path accepts gets the codes of the definition, and that the ties go to the
division.  It runs on the CPU and uses neither the oracle nor the CUDA library."""
import numpy as np
import pytest

F32 = np.float32
MAGIC = F32(12582912.0)          # 1.5 * 2^23
LIMIT = F32(0.5) - F32(2.0 ** -17)


def fma32(a, b, c):
    # a * b is exact in float64 for float32 operands.  For r (|a b + c| <= 16 with c an
    # integer) the float64 sum is exact too, so the one rounding to float32 is the FMA's.
    # For t (c = 1.5 * 2^23) the float64 sum may round first; that can change the float32
    # result only within about 2^-29 of a half-integer, where |r| is near 1/2 and the fast
    # path declines the group whatever t is.
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F32)


def definition(v, bits):
    qmax = (1 << bits) - 1
    lo, hi = v.min(), v.max()
    if hi == lo:
        return np.zeros(v.shape, np.int64), F32(0)
    dl = F32(F32(hi - lo) / F32(qmax))
    u = F32(F32(F32(v - lo) / dl) + F32(0.5))
    return np.clip(np.floor(u).astype(np.int64), 0, qmax), dl


def fast_path(v, bits):
    """(codes, accepted): the codes the fast path forms and whether it keeps them."""
    qmax = (1 << bits) - 1
    lo, hi = v.min(), v.max()
    dl = F32(F32(hi - lo) / F32(qmax))
    rdl = F32(F32(1.0) / dl)
    d = F32(v - lo)
    rd = np.full_like(d, rdl)
    t = fma32(d, rd, np.full_like(d, MAGIC))
    nq = F32(MAGIC - t)
    r = fma32(d, rd, nq)
    q = (t.view(np.uint32) & np.uint32(qmax)).astype(np.int64)
    return q, bool(dl >= F32(2.0 ** -100) and np.abs(r).max() <= LIMIT)


@pytest.mark.parametrize("bits", [4, 2])
def test_random_groups_match_the_definition(bits):
    rng = np.random.default_rng(bits)
    accepted = 0
    for scale in (1e-3, 0.3, 1.0, 37.0):
        for _ in range(4000):
            v = (rng.normal(size=32) * scale + rng.normal() * scale).astype(F32)
            want, _ = definition(v, bits)
            got, ok = fast_path(v, bits)
            if ok:
                accepted += 1
                assert np.array_equal(got, want)
    assert accepted > 15000          # the division is the rare path


@pytest.mark.parametrize("bits", [4, 2])
def test_groups_on_and_next_to_the_decision_points(bits):
    # coordinates whose quotient d/delta is a half-integer or within a few units of the
    # last place of one: the fast path must either reproduce the definition or hand the
    # group to the division, and an exact half-integer must always go to the division
    rng = np.random.default_rng(10 + bits)
    qmax = (1 << bits) - 1
    handed_over = 0
    for _ in range(3000):
        lo = F32(rng.normal())
        span = F32(abs(rng.normal()) + 0.25)
        v = (lo + rng.random(32).astype(F32) * span).astype(F32)
        v[0], v[1] = lo, F32(lo + span)
        dl = F32(F32(v.max() - v.min()) / F32(qmax))
        k = rng.integers(0, qmax)
        target = (k + 0.5) * np.float64(dl) + np.float64(v.min())
        v[2] = F32(target)
        v[3] = np.nextafter(F32(target), F32(np.inf))
        v[4] = np.nextafter(F32(target), F32(-np.inf))
        want, _ = definition(v, bits)
        got, ok = fast_path(v, bits)
        if ok:
            assert np.array_equal(got, want)
        else:
            handed_over += 1
    assert handed_over > 0


def test_exact_half_integer_goes_to_the_division():
    # d / delta = 0.5 exactly: q = floor(1.0) = 1, and the fast path declines the group
    v = np.zeros(32, F32)
    v[1] = F32(15.0)                  # delta = 1 for INT4
    v[2] = F32(0.5)
    want, dl = definition(v, 4)
    assert dl == F32(1.0) and want[2] == 1
    _, ok = fast_path(v, 4)
    assert not ok
