"""Pins for the oracle's counter-based generator (Philox4x32-10, SC'11)."""
import numpy as np
import pytest
from scipy import stats

from conftest import read_golden
from philox_py import philox, philox_vec, accept_uniform, race_exponential_vec


def _kat():
    rows = []
    with open(__import__("os").path.join(__import__("os").path.dirname(__file__), "golden",
                                         "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat())
def test_python_philox_matches_published_kat(row):
    assert list(philox(row[0:4], row[4:6])) == row[6:10]


@pytest.mark.parametrize("row", _kat())
def test_oracle_philox_matches_published_kat(orc, row):
    assert list(orc.philox4x32_10(row[0:4], row[4:6])) == row[6:10]


def test_oracle_philox_matches_python_many_counters(orc):
    rng = np.random.default_rng(7)
    for _ in range(300):
        ctr = rng.integers(0, 2 ** 32, 4, dtype=np.uint64)
        key = rng.integers(0, 2 ** 32, 2, dtype=np.uint64)
        assert list(orc.philox4x32_10(ctr, key)) == list(philox(ctr, key))


def test_accept_uniform_mapping(orc):
    for seed in (0, 1, 12345, 2 ** 40 + 17):
        for b in (0, 3, 255):
            for j in range(8):
                u = orc.accept_uniform(seed, b, j)
                assert u == float(accept_uniform(seed, b, j))
                assert 0.0 <= u < 1.0


def test_race_exponential_mapping(orc):
    v = np.arange(0, 2000, 7)
    for seed, b, j, tag in ((0, 0, 0, 2), (99, 5, 3, 3), (2 ** 33, 1, 1, 2)):
        ref = race_exponential_vec(seed, b, j, v, tag)
        got = np.array([orc.race_exponential(seed, b, j, int(x), tag) for x in v], np.float32)
        # log1p is a libm call: allow 2 ulp between the oracle's libm and numpy's.
        np.testing.assert_array_max_ulp(got, ref, maxulp=2)


def test_philox_output_bytes_uniform():
    n = 1 << 16
    c = np.arange(n, dtype=np.uint64)
    words = philox_vec(c, np.zeros(n), np.zeros(n), np.zeros(n), 1234, 5678)
    by = np.concatenate([w.view(np.uint8) for w in words])
    counts = np.bincount(by, minlength=256)
    chi2 = ((counts - by.size / 256) ** 2 / (by.size / 256)).sum()
    assert stats.chi2.sf(chi2, 255) > 1e-3


def test_race_exponential_is_exp1(orc):
    v = np.arange(20000)
    E = race_exponential_vec(0, 1, 2, v, 2)
    # Kolmogorov-Smirnov against Exp(1) on the numpy restatement, plus a sample of the oracle's.
    assert stats.kstest(E, "expon").pvalue > 1e-3
    got = np.array([orc.race_exponential(0, 1, 2, int(x), 2) for x in v[:500]], np.float32)
    np.testing.assert_array_max_ulp(got, E[:500], maxulp=2)


def test_race_words_are_the_four_words_of_one_counter(orc):
    """Vocabulary entries 4g .. 4g+3 take words 0..3 of counter (b, j, g, tag),
    checked against the known-answer-pinned scalar Philox."""
    from philox_py import race_words_vec
    seed, b, j, tag = 0x0123_4567_89AB, 7, 2, 3
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for v in (0, 1, 2, 3, 4, 5, 6, 7, 1001, 151935):
        want = philox((b, j, v // 4, tag), key)[v % 4]
        assert int(race_words_vec(seed, b, j, [v], tag)[0]) == want
        u = np.float32(want) * np.float32(2.0 ** -32)
        e = np.float32(-np.log1p(-u))
        got = np.float32(orc.race_exponential(seed, b, j, v, tag))
        assert abs(float(got) - float(e)) <= 2 * float(np.spacing(e))
