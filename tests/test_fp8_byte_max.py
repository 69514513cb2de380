"""The FP8 maximum pass takes the largest e4m3 magnitude of a unit (4 x 16
bytes) with 16-bit integer lanes instead of a byte-wise maximum: per 32-bit
word, max.u16x2 over (word & 0x7F7F7F7F) keeps the largest odd byte as the
high byte of each lane (the low byte only breaks ties), and max.u16x2 over
(word & 0x007F007F) keeps the largest even byte alone in its lane; the unit
maximum is the largest of the four resulting bytes.

These tests run those integer steps on the CPU (numpy) and compare them with
the plain maximum of the 7-bit magnitudes, on random units, units with every
sign bit set, all-zero units and units whose maximum sits in each of the
four byte positions.  (The GPU tests check the quantiser's outputs against
the oracle bit for bit.)"""
import numpy as np


def _max_u16x2(a, b):
    lo = np.maximum(a & 0xFFFF, b & 0xFFFF)
    hi = np.maximum(a >> 16, b >> 16)
    return (hi << 16) | lo


def _kernel_unit_max(words):
    """words: uint64 [units, 16] (each holding a 32-bit word) -> [units]."""
    m_odd = np.zeros(words.shape[0], np.uint64)
    m_even = np.zeros(words.shape[0], np.uint64)
    for i in range(words.shape[1]):
        m_odd = _max_u16x2(m_odd, words[:, i] & 0x7F7F7F7F)
        m_even = _max_u16x2(m_even, words[:, i] & 0x007F007F)
    return np.maximum(np.maximum((m_odd >> 8) & 0xFF, m_odd >> 24),
                      np.maximum(m_even & 0xFF, m_even >> 16))


def _plain_unit_max(words):
    b = np.stack([(words >> (8 * j)) & 0x7F for j in range(4)], axis=-1)
    return b.reshape(words.shape[0], -1).max(axis=1)


def _check(words):
    words = words.astype(np.uint64)
    assert np.array_equal(_kernel_unit_max(words), _plain_unit_max(words))


def test_random_units():
    rng = np.random.default_rng(5)
    _check(rng.integers(0, 1 << 32, size=(200000, 16), dtype=np.uint64))


def test_sign_bits_never_count():
    rng = np.random.default_rng(6)
    w = rng.integers(0, 1 << 32, size=(50000, 16), dtype=np.uint64) | 0x80808080
    _check(w)
    _check(np.full((4, 16), 0x80808080, np.uint64))      # -0 everywhere -> 0
    _check(np.zeros((4, 16), np.uint64))


def test_maximum_in_each_byte_position():
    rng = np.random.default_rng(7)
    base = rng.integers(0, 0x30, size=(4 * 16 * 4, 16, 4), dtype=np.uint64)
    k = 0
    for pos in range(4):
        for word in range(16):
            for val in (0x30, 0x7E, 0x7F, 0xFE):
                base[k, word, pos] = val
                k += 1
    words = sum(base[:, :, j] << (8 * j) for j in range(4))
    _check(words)
