"""The native draft-head token list (include/dmtp_vocab.h, host code in libdmtp.so)
against the oracle (oracle/shortlist.py): the same seeded streams of request starts and
picks give the same counts, list and statistics after every call; bad ids are refused
with the list unchanged. No GPU."""
import numpy as np
import pytest

from mtp_block_draft_gb300 import DmtpError, DmtpVocabList
from oracle.shortlist import VocabList


def _same(native, ref):
    np.testing.assert_array_equal(native.counts(), ref.counts)
    np.testing.assert_array_equal(native.ids(), ref.ids())
    np.testing.assert_array_equal(native.mask(), ref.members)
    st = native.stats()
    assert st["listed"] == int(ref.members.sum()) and st["counted"] == ref.counted
    assert (st["rebuilds"], st["appended"], st["picks"], st["picks_in"]) == \
        (ref.rebuilds, ref.appended, ref.picks, ref.picks_in)


@pytest.mark.parametrize("seed,V,size", [(0, 50, 8), (1, 300, 40), (2, 1000, 64),
                                         (3, 40, 60), (4, 151936, 16000)])
def test_native_list_matches_oracle(seed, V, size):
    rng = np.random.default_rng(seed)
    native, ref = DmtpVocabList(V, size), VocabList(V, size)
    _same(native, ref)
    # skewed ids (a few frequent tokens), long enough for several halvings
    weights = 1.0 / np.arange(1, V + 1) ** 1.1
    weights /= weights.sum()
    steps = 30 if V > 10000 else 60
    for i in range(steps):
        if rng.random() < 0.25:
            prompt = rng.choice(V, size=int(rng.integers(0, 400)), p=weights)
            new = bool(rng.random() < 0.6)
            native.begin_request(prompt, new)
            ref.begin_request(prompt, new)
        else:
            toks = rng.choice(V, size=int(rng.integers(1, 9)), p=weights)
            if rng.random() < 0.3:
                toks[0] = rng.integers(0, V)          # a rare token
            native.picked(toks)
            ref.picked(toks)
        if V <= 10000 or i % 10 == 9:
            _same(native, ref)
    _same(native, ref)
    native.close()


def test_default_size_and_refusals():
    native = DmtpVocabList(30000)                     # size 0: the page's 16000
    ref = VocabList(30000)
    rng = np.random.default_rng(7)
    p = rng.integers(0, 30000, 5000)
    native.begin_request(p)
    ref.begin_request(p)
    _same(native, ref)
    before = (native.counts(), native.ids(), native.stats())
    for bad in ([30000], [-1], [5, 30001]):
        with pytest.raises(DmtpError):
            native.picked(bad)
        with pytest.raises(DmtpError):
            native.begin_request(bad)
    after = (native.counts(), native.ids(), native.stats())
    np.testing.assert_array_equal(before[0], after[0])
    np.testing.assert_array_equal(before[1], after[1])
    assert before[2] == after[2]
    for bad_v, bad_size in ((0, 10), (10, -1)):
        with pytest.raises(DmtpError):
            DmtpVocabList(bad_v, bad_size)
