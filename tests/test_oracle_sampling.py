"""Pins of the oracle's target-only sampled verification (oracle/sampling.py).

* Philox4x32-10 against the known-answer vectors published with the generator
  (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011,
  and its reference implementation's test vectors).
* The Gumbel-max pick is a draw from softmax(l / temperature): empirical frequencies over
  many positions against the exact probabilities (chi-square), and the limit
  temperature -> 0 is the argmax.
* Losslessness ([DMTP] §5 target-only verification, [colibri] verify contract):
  speculative rounds with sampled verify picks commit exactly the plain sampled decode
  of the target, naturally and with drafts forced right, wrong, or wrong in one row.
"""
import numpy as np
import pytest

from oracle import OracleModel
from oracle.sampling import gumbel, philox4x32_10, sampled_scores, uniforms
from synth import CONFIGS, make_prompts, make_weights

TINY = CONFIGS["tiny"]
TAU, SEED = 0.8, 20260611


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_known_answers(ctr, key, want):
    out = philox4x32_10(np.array(ctr, dtype=np.uint64).reshape(4, 1),
                        np.array(key, dtype=np.uint64))
    assert tuple(int(x) for x in out[:, 0]) == want


def test_uniforms_open_interval_and_layout():
    u = uniforms(SEED, 3, 1234, 1001)
    assert u.shape == (1001,) and (u > 0).all() and (u < 1).all()
    # word i of block j serves vocabulary index 4 j + i: the first 8 entries come from
    # the first two blocks' words in order
    ctr = np.zeros((4, 2), dtype=np.uint64)
    ctr[0] = [0, 1]
    ctr[1], ctr[2] = 1234, 3
    w = philox4x32_10(ctr, np.array([SEED & 0xFFFFFFFF, SEED >> 32], dtype=np.uint64))
    expect = ((w.T.reshape(-1) >> 8).astype(np.float64) + 0.5) * 2.0 ** -24
    np.testing.assert_array_equal(u[:8], expect)
    # different positions, sequences and seeds give different streams
    assert not np.array_equal(u, uniforms(SEED, 3, 1235, 1001))
    assert not np.array_equal(u, uniforms(SEED, 4, 1234, 1001))
    assert not np.array_equal(u, uniforms(SEED + 1, 3, 1234, 1001))


def test_gumbel_max_draws_from_softmax():
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4])
    p = np.exp(logits / TAU)
    p /= p.sum()
    n = 20000
    picks = np.array([np.argmax(sampled_scores(logits, TAU, SEED, 0, pos)) for pos in range(n)])
    counts = np.bincount(picks, minlength=logits.size)
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < 25.7  # 5 degrees of freedom, p = 1e-4
    # the noise itself: Gumbel(0, 1) has mean = Euler's gamma, variance pi^2 / 6
    g = np.concatenate([gumbel(SEED, 1, pos, 1000) for pos in range(50)])
    assert abs(g.mean() - 0.5772156649) < 0.02
    assert abs(g.var() - np.pi ** 2 / 6) < 0.06


def test_zero_temperature_limit_is_argmax():
    rng = np.random.default_rng(1)
    for pos in range(50):
        logits = rng.normal(size=300)
        assert np.argmax(sampled_scores(logits, 1e-9, SEED, 2, pos)) == np.argmax(logits)


@pytest.fixture(scope="module")
def sampler():
    return OracleModel(TINY, make_weights(TINY, "cpu"), temperature=TAU, sample_seed=SEED)


@pytest.fixture(scope="module")
def prompt():
    return make_prompts(TINY)[0]


@pytest.fixture(scope="module")
def sampled(sampler, prompt):
    return sampler.sampled_decode(prompt, 8 * 8 + 9, b=0)


def test_sampled_decode_differs_from_greedy(sampler, prompt, sampled):
    greedy = OracleModel(TINY, make_weights(TINY, "cpu")).greedy_decode(prompt, len(sampled))
    assert sampled[0] == greedy[0]          # A is an argmax pick
    assert sampled != greedy


def test_sampled_rounds_lossless_natural(sampler, prompt, sampled):
    st = sampler.prefill(prompt, b=0)
    stream = [st.A]
    for _ in range(8):
        stream += sampler.round(st)["committed"]
    assert stream == sampled[:len(stream)]


@pytest.mark.parametrize("wrong_row", [None, 0, 3, 6])
def test_sampled_rounds_lossless_forced(sampler, prompt, sampled, wrong_row):
    st = sampler.prefill(prompt, b=0)
    stream = [st.A]
    for _ in range(6):
        k = len(stream) - 1               # stream index of the pending token
        d = list(sampled[k + 1:k + 8])
        if wrong_row is not None:
            d[wrong_row] = (d[wrong_row] + 1) % (TINY.vocab - 1)
        rec = sampler.round(st, forced=d)
        assert rec["n"] == (7 if wrong_row is None else wrong_row)
        stream += rec["committed"]
    assert stream == sampled[:len(stream)]
