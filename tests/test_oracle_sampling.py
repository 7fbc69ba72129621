"""Pins for the temperature > 0 drafting oracle (oracle/sampling_ref.py).

What fixes it outside the oracle: the SplitMix64 definition (published
reference outputs), the Gumbel-max theorem (a draw's frequencies equal
softmax(z / T)), the T -> 0 limit (the greedy argmax), and independence of
the rows' streams.  A planted mistake in the oracle fails at least one.
"""
import numpy as np
import pytest

import oracle.sampling_ref as SR
from workload.gen import splitmix64_bits, stream_key as wl_stream_key


def test_generator_is_published_splitmix64():
    # SplitMix64 reference outputs for initial state 1234567
    assert SR.stream_bits(1234567, np.arange(5)).tolist() == [
        6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431, 16408922859458223821]
    # the same key folding and element addressing as the input generators
    for seed, ids in [(0, (1, 0, 0, 1)), (7, (1, 3, 11, 15)), (2 ** 63 + 5, (1, 63, 1000, 2))]:
        assert SR.stream_key(seed, *ids) == wl_stream_key(seed, *ids)
        k = SR.stream_key(seed, *ids)
        idx = np.array([0, 1, 151935, 2 ** 20])
        assert np.array_equal(SR.stream_bits(k, idx), splitmix64_bits(k, idx))


def test_uniforms_inside_unit_interval_and_exact_in_float32():
    u = SR.uniform23(SR.stream_key(3, 1, 0, 0, 1), np.arange(200000))
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    # 23-bit grid, mean 1/2 and variance 1/12 of a uniform
    assert abs(u.mean() - 0.5) < 0.003 and abs(u.var() - 1 / 12) < 0.002
    g = SR.gumbel(SR.stream_key(3, 1, 0, 0, 2), np.arange(200000))
    # standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2 / 6
    assert abs(g.mean() - 0.5772156649) < 0.01 and abs(g.var() - np.pi ** 2 / 6) < 0.03


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
def test_gumbel_max_draws_follow_softmax(T):
    z = np.array([0.3, -1.2, 1.1, 0.0, 0.8, -0.4])
    p = np.exp(z / T - np.max(z / T))
    p /= p.sum()
    n = 30000
    counts = np.zeros(z.size)
    for r in range(n):
        i, _ = SR.sample_row(z, T, SR.stream_key(99, SR.DRAFT, 0, r, 1))
        counts[i] += 1
    f = counts / n
    sd = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(f - p) < 4.5 * sd), (f, p)


def test_small_temperature_is_the_argmax():
    rng = np.random.default_rng(4)
    for _ in range(50):
        z = rng.permutation(np.arange(40) * 0.1)
        i, _ = SR.sample_row(z, 1e-4, SR.stream_key(5, SR.DRAFT, 0, 0, 1))
        assert i == int(np.argmax(z))


def test_rows_requests_rounds_and_seeds_draw_independently():
    z = np.zeros((15, 64))  # every row uniform over 64 ids
    base, _ = SR.sample_drafts(z, 1.0, 11, 0, 0)
    assert len(set(base.tolist())) > 8                       # rows differ
    for other in [SR.sample_drafts(z, 1.0, 11, 1, 0)[0],     # another request
                  SR.sample_drafts(z, 1.0, 11, 0, 1)[0],     # another round
                  SR.sample_drafts(z, 1.0, 12, 0, 0)[0]]:    # another seed
        assert np.mean(other == base) < 0.4


def test_shift_invariance_and_margin():
    z = np.array([2.0, 1.0, 0.5, -3.0, 0.0])
    k = SR.stream_key(1, SR.DRAFT, 2, 3, 4)
    i, m = SR.sample_row(z, 0.8, k)
    j, m2 = SR.sample_row(z + 8.0, 0.8, k)
    assert i == j and abs(m - m2) < 1e-9 and m >= 0.0


# ----------------------------------------------------------------- planted mistakes

def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    cases = {
        # Gumbel with the wrong sign: -(-ln(-ln u))
        "gumbel sign": ("gumbel", lambda key, idx: np.log(-np.log(SR.uniform23(key, idx)))),
        # exponential instead of Gumbel noise
        "exponential noise": ("gumbel", lambda key, idx: -np.log(SR.uniform23(key, idx))),
    }
    for name, (attr, fn) in cases.items():
        with monkeypatch.context() as m:
            m.setattr(SR, attr, fn)
            assert _fails(lambda: test_gumbel_max_draws_follow_softmax(1.0)) or \
                _fails(test_uniforms_inside_unit_interval_and_exact_in_float32), name

    # temperature multiplied instead of divided
    def sample_row_times_T(z, T, key):
        pert = z * T + SR.gumbel(key, np.arange(z.shape[-1]))
        i = int(np.argmax(pert))
        t2 = np.partition(pert, -2)[-2:]
        return i, float(t2[1] - t2[0])
    with monkeypatch.context() as m:
        m.setattr(SR, "sample_row", sample_row_times_T)
        assert _fails(lambda: test_gumbel_max_draws_follow_softmax(0.5))

    # one stream for every row
    def drafts_same_row(z, T, seed, b, rnd):
        out = [SR.sample_row(z[k], T, SR.stream_key(seed, SR.DRAFT, b, rnd, 1)) for k in range(z.shape[0])]
        return np.array([o[0] for o in out]), np.array([o[1] for o in out])
    with monkeypatch.context() as m:
        m.setattr(SR, "sample_drafts", drafts_same_row)
        assert _fails(test_rows_requests_rounds_and_seeds_draw_independently)
