"""The GPU quantiser divides a weight by its block scale without a general
fp32 division: an e4m3 scale s is d * 2^e with d an odd integer <= 15, so
RN(v / s) = RN(v / d) * 2^-e, and RN(v / d) comes from the correctly rounded
reciprocal r = RN(1/d) by one fused multiply-add correction (Markstein's
division refinement: q0 = RN(v r), rem = RN(v - q0 d), q1 = RN(q0 + rem r)).

These tests check that method on the CPU, emulated step by step with exact
arithmetic, against the correctly rounded quotient computed with integers:
for every fp32 significand (all 2^23 values of v in [1, 2); other binades
scale exactly) and every odd d.  Also: the (d, e) split reproduces every
finite nonzero e4m3 value.  (The oracle divides with plain fp32 `/`; the GPU
parity tests compare the kernel's codes with it bit for bit.)"""
import numpy as np
import pytest

import oracle


def _rn32_quotient(f, d):
    """RN_fp32((2^23 + f) / 2^23 / d) for int64 f in [0, 2^23), exactly."""
    N = (np.int64(1 << 23) + f) << np.int64(30)          # v * 2^53, < 2^54
    Q, R = N // d, N % d                                 # v / d = (Q + R/d) * 2^-53
    bl = (50 + (Q >= (1 << 50)).astype(np.int64) + (Q >= (1 << 51)).astype(np.int64) +
          (Q >= (1 << 52)).astype(np.int64))             # bit length (Q >= 2^49)
    sh = bl - 24
    hi = Q >> sh
    lo = Q - (hi << sh)
    twice = 2 * (lo * d + R)                             # compare lo + R/d with 2^(sh-1)
    half = (np.int64(1) << sh) * d
    up = (twice > half) | ((twice == half) & ((hi & 1) == 1))
    hi = hi + up
    return hi.astype(np.float64) * np.exp2((sh - 53).astype(np.float64))


def _method(f, d):
    """The kernel's steps, each rounding emulated exactly."""
    v = (np.float64(1 << 23) + f.astype(np.float64)) / float(1 << 23)
    r = np.float64(np.float32(1.0) / np.float32(d))      # RN(1/d)
    q0 = (v * r).astype(np.float32).astype(np.float64)   # v*r exact in fp64 (48 bits)
    rem = (v - q0 * d).astype(np.float32).astype(np.float64)   # exact in fp64, then RN32
    t = rem * r                                          # exact in fp64 (48 bits)
    # RN32(q0 + t): the nearest of q0 and its fp32 neighbours, ties to the even
    # significand; each distance (q0 - c) + t is exact in fp64
    q0f = q0.astype(np.float32)
    cands = [np.nextafter(q0f, np.float32(-np.inf)), q0f, np.nextafter(q0f, np.float32(np.inf))]
    best = None
    for c in cands:
        c64 = c.astype(np.float64)
        dist = np.abs((q0 - c64) + t)
        even = (c.view(np.uint32) & 1) == 0
        if best is None:
            best, best_d, best_even = c64, dist, even
        else:
            take = (dist < best_d) | ((dist == best_d) & even & ~best_even)
            best = np.where(take, c64, best)
            best_d = np.where(take, dist, best_d)
            best_even = np.where(take, even, best_even)
    return best


@pytest.mark.parametrize("d", [3, 5, 7, 9, 11, 13, 15])
def test_refined_reciprocal_division_is_correctly_rounded(d):
    chunk = 1 << 21
    for start in range(0, 1 << 23, chunk):
        f = np.arange(start, start + chunk, dtype=np.int64)
        got = _method(f, d)
        want = _rn32_quotient(f, d)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (d, int(f[bad[0]]), got[bad[0]], want[bad[0]])


def test_the_correction_step_is_needed():
    # without the FMA correction (q = RN(v * RN(1/d))) the quotient is often
    # one ulp off: a kernel that skipped the step would fail the check above
    f = np.arange(0, 1 << 20, dtype=np.int64)
    for d in (3, 11, 13):
        v = (np.float64(1 << 23) + f.astype(np.float64)) / float(1 << 23)
        r = np.float64(np.float32(1.0) / np.float32(d))
        q0 = (v * r).astype(np.float32).astype(np.float64)
        assert np.count_nonzero(q0 != _rn32_quotient(f, d)) > 1000


def test_scale_split_reproduces_every_e4m3_value():
    # s = d * 2^e with d odd in [1, 15], for every finite nonzero e4m3 byte
    for b in range(1, 0x7F):
        E, m = (b >> 3) & 15, b & 7
        sig, ex = (8 + m, E - 10) if E else (m, -9)
        t = (sig & -sig).bit_length() - 1
        d, e = sig >> t, ex + t
        assert d % 2 == 1 and 1 <= d <= 15 and -9 <= e <= 8
        assert d * 2.0 ** e == oracle.e4m3(b)
