"""GPU parity of sampling beyond greedy against the oracle (oracle/sampling.py)."""
import numpy as np
import pytest

from oracle import sampling
from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


def _logits(seed, B, V, scale=2.0):
    return (np.random.default_rng(seed).normal(size=(B, V)) * scale).astype(np.float32)


def test_sample_greedy_is_first_argmax(a8w8):
    x = _logits(1, 5, 151936)
    x[2, 7] = x[2].max()                     # a tie: the lower index wins
    got = to_host(a8w8.a8w8_sample(to_dev(x), 0.0, 1.0, 0, 0))
    assert np.array_equal(got, np.argmax(x, axis=1))
    assert got[2] == 7


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 0.9), (1.3, 0.5), (0.5, 0.95), (2.0, 0.2)])
def test_sample_matches_oracle_full_vocab(a8w8, T, top_p):
    x = _logits(2, 4, 151936)
    d = to_dev(x)
    agree, n = 0, 0
    for step in range(5):
        got = to_host(a8w8.a8w8_sample(d, T, top_p, seed=0x1234_5678_9ABC, step=step))
        ref = sampling.sample_rows(x, T, top_p, 0x1234_5678_9ABC, step)
        agree += int((got == ref).sum())
        n += len(ref)
    # the exponentials and masses are two-float on the device and float64 in the
    # oracle; only the float32 Gumbel keys can differ, within ~1e-6: a different
    # token needs the two best keys that close
    assert agree >= n - 1, (agree, n)


def test_sample_deterministic_per_seed_and_step(a8w8):
    d = to_dev(_logits(3, 8, 5000))
    a = to_host(a8w8.a8w8_sample(d, 0.9, 0.9, seed=5, step=11))
    b = to_host(a8w8.a8w8_sample(d, 0.9, 0.9, seed=5, step=11))
    c = to_host(a8w8.a8w8_sample(d, 0.9, 0.9, seed=5, step=12))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_sample_distribution_is_the_softmax(a8w8):
    # 4096 rows of the same logits are independent streams (the row is part of
    # the counter): frequencies against softmax(l / T)
    base = np.array([1.0, 0.0, -1.0, 2.0, 0.5, -3.0], np.float32)
    x = np.tile(base, (4096, 1))
    d = to_dev(x)
    T = 0.8
    p = np.exp(base / T) / np.exp(base / T).sum()
    draws = np.concatenate([to_host(a8w8.a8w8_sample(d, T, 1.0, 77, s)) for s in range(5)])
    n = len(draws)
    freq = np.bincount(draws, minlength=6) / n
    assert (np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / n) + 1e-4).all(), (freq, p)


def test_sample_nucleus_renormalises(a8w8):
    p = np.array([0.5, 0.3, 0.1, 0.05, 0.05])
    x = np.tile(np.log(p).astype(np.float32), (4096, 1))
    d = to_dev(x)
    draws = np.concatenate([to_host(a8w8.a8w8_sample(d, 1.0, 0.75, 3, s)) for s in range(4)])
    n = len(draws)
    freq = np.bincount(draws, minlength=5) / n
    assert freq[2:].sum() == 0
    assert abs(freq[0] - 0.625) < 5 * np.sqrt(0.625 * 0.375 / n)
    # and the oracle draws the same tokens for the same streams
    ref = sampling.sample_rows(x[:64], 1.0, 0.75, 3, 0)
    got = to_host(a8w8.a8w8_sample(to_dev(x[:64]), 1.0, 0.75, 3, 0))
    assert (got == ref).mean() >= 63 / 64
