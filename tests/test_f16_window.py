"""The f16 path of the few-row kernel (M <= 8) converts each activation row to
f16 after scaling it by 2^a, a chosen from the row's running maximum |x| so
that max * 2^a < 2^15 (a = min(126, max(-126, 141 - e_max)), e_max the
biased bf16 exponent of the maximum, running over the stages seen so far).
A stage whose row holds a nonzero value with biased exponent e < 110 - a is
flagged and multiplied in bf16 instead.  The converter finds the smallest
nonzero magnitude with 16-bit integer lanes: per 32-bit word of |x| bits,
(w + 0x7FFF7FFF) & 0x7FFF7FFF gives h - 1 for a magnitude h > 0 and 0x7FFF
for h = 0, min.u16x2 keeps the lane minima, and the flag is
min < (110 - a) * 128 - 1.

These tests run those integer steps on the CPU (numpy) and check:
  * the lane minimum is the smallest nonzero magnitude less one (0x7FFF for
    an all-zero row), on random, sparse, all-zero and signed rows;
  * over every finite bf16 magnitude and every exponent a the converter can
    choose: a value that is not flagged converts to f16 exactly, and is not
    beyond f16's range when it is at most the row maximum;
  * the threshold is tight: for every a, some value one binade below it
    does not convert exactly (so the flag cannot be dropped a binade lower).
(The GPU tests check the kernel's results against the oracle on rows that
span more than the window.)"""
import numpy as np


def _min_u16x2(a, b):
    lo = np.minimum(a & 0xFFFF, b & 0xFFFF)
    hi = np.minimum(a >> 16, b >> 16)
    return (hi << 16) | lo


def _kernel_min_nonzero_less1(words):
    """words: uint64 [rows, n] (32-bit words of bf16 pairs) -> [rows]."""
    acc = np.full(words.shape[0], 0x7FFF7FFF, np.uint64)
    for i in range(words.shape[1]):
        a = words[:, i] & 0x7FFF7FFF
        acc = _min_u16x2(acc, ((a + 0x7FFF7FFF) & 0xFFFFFFFF) & 0x7FFF7FFF)
    return np.minimum(acc & 0xFFFF, acc >> 16)


def _plain_min_nonzero_less1(words):
    h = np.stack([(words >> (16 * j)) & 0x7FFF for j in range(2)], axis=-1).reshape(
        words.shape[0], -1)
    big = np.where(h == 0, np.uint64(0x8000), h)
    return np.where((h == 0).all(axis=1), 0x7FFF, big.min(axis=1) - 1)


def test_lane_minimum_is_the_smallest_nonzero_magnitude():
    rng = np.random.default_rng(5)
    cases = [rng.integers(0, 2 ** 32, size=(4000, 128), dtype=np.uint64)]
    sparse = rng.integers(0, 2 ** 32, size=(4000, 128), dtype=np.uint64)
    sparse &= np.where(rng.random((4000, 128)) < 0.97, np.uint64(0), np.uint64(0xFFFFFFFF))
    cases.append(sparse)
    cases.append(np.zeros((3, 128), np.uint64))
    cases.append(np.full((3, 128), 0x80008000, np.uint64))            # all -0
    one = np.zeros((64, 128), np.uint64)
    for r in range(64):                                                # one nonzero lane
        one[r, r % 128] = np.uint64(1 + r) << np.uint64(16 * (r % 2))
    cases.append(one)
    for w in cases:
        assert np.array_equal(_kernel_min_nonzero_less1(w), _plain_min_nonzero_less1(w))


def _bf16_to_f64(h):
    return (np.asarray(h, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_unflagged_values_convert_to_f16_exactly():
    h = np.arange(0, 0x7F80, dtype=np.int64)           # every finite magnitude
    x = _bf16_to_f64(h)
    e = h >> 7
    for e_max in range(0, 255):                        # every running maximum's exponent
        a = min(126, max(-126, 141 - e_max))
        row = h[(e <= e_max)]                          # values at most the maximum's binade
        if row.size == 0:
            continue
        flagged = (row - 1 < (110 - a) * 128 - 1) & (row > 0)
        keep = row[~flagged]
        v = _bf16_to_f64(keep) * np.float64(2.0) ** a   # exact in fp64
        f = v.astype(np.float16).astype(np.float64)
        assert np.array_equal(f, v), (e_max, a, keep[f != v][:4])
        assert np.all(v < 2.0 ** 16), e_max             # below f16's largest binade's end


def test_window_threshold_is_tight():
    for a in range(-114, 110):
        e = 109 - a                                    # one binade below the threshold
        if not 1 <= e <= 254:
            continue
        h = np.arange(e << 7, (e + 1) << 7, dtype=np.int64)
        v = _bf16_to_f64(h) * np.float64(2.0) ** a
        assert np.any(v.astype(np.float16).astype(np.float64) != v), a
