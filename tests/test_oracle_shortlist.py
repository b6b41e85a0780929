"""Pins of the draft heads' frequent-token shortlist oracle (oracle/shortlist.py) on hand
counts (colibri speculative-decoding doc, the list a draft head scores):

* counting and halving: 1023 counted tokens leave the counts, the 1024th halves them
  (floor) and rebuilds the list;
* composition: the `size` highest counts, any count reaching three quarters of the smallest of them,
  and the conversation's tokens; membership does not depend on how equal counts order;
* no counts yet: the whole vocabulary;
* a picked token missing from the list joins at once and is counted;
* restricted argmax: the lowest listed id of the largest listed logit.
"""
import numpy as np
import pytest

from oracle.shortlist import HALVE_EVERY, VocabList, restricted_argmax


def _hand_counts(size=3):
    v = VocabList(20, size)
    # conversation A: counts 5 x8, 2 x6, 7 x6, 9 x5, 11 x4, 3 x1
    v.begin_request([5] * 8 + [2] * 6 + [7] * 6 + [9] * 5 + [11] * 4 + [3])
    v.begin_request([0])                      # a new conversation: {0}
    return v


def test_halving_every_1024_counted_tokens():
    v = VocabList(10, 3)
    v.begin_request([1] * (HALVE_EVERY - 1))
    assert v.counts[1] == 1023 and v.counted == 1023 and v.rebuilds == 1
    v.picked([1])
    assert v.counts[1] == 512 and v.counted == 0 and v.rebuilds == 2
    v.picked([2, 2, 2])
    assert v.counts[2] == 3 and v.counted == 3
    v.begin_request([3] * 1021 + [4] * 5)     # the halving lands inside the prompt
    assert v.counts[1] == 256 and v.counts[2] == 1 and v.counts[3] == 510
    assert v.counts[4] == 5 and v.counted == 5 and v.rebuilds == 4


@pytest.mark.parametrize("size", [2, 3])
def test_list_composition(size):
    v = _hand_counts(size)
    assert v.counts[0] == 1
    # size 3: top 5 (8), 2 (6), 7 (6), last 6: counts >= 4.5 qualify (9 with 5); size 2:
    # top 5, 2 (7 ties with 2 but orders after it), last 6: the same set
    assert v.ids().tolist() == [0, 2, 5, 7, 9]


def test_no_counts_means_the_whole_vocabulary():
    v = VocabList(20, 3)
    assert v.ids().tolist() == list(range(20))
    v.begin_request([4])                      # one counted token: the third count is 0
    assert v.ids().tolist() == list(range(20))
    v.begin_request([4, 6, 8], new_conversation=True)
    assert v.ids().tolist() == [4, 6, 8]      # counts 2, 1, 1: last 1, 3/4 rule keeps 1s


def test_picked_tokens_join_at_once_and_count():
    v = _hand_counts()
    v.picked([13, 5, 13])
    assert v.ids().tolist() == [0, 2, 5, 7, 9, 13]
    assert v.appended == 1 and v.picks == 3 and v.picks_in == 2
    assert v.counts[13] == 2 and 13 in v.conv
    v.begin_request([1], new_conversation=True)   # rebuild: 13 (count 2) no longer listed
    assert v.ids().tolist() == [1, 2, 5, 7, 9]


def test_restricted_argmax_and_range_checks():
    members = np.zeros(8, dtype=bool)
    members[[1, 4, 6]] = True
    logits = np.array([9.0, 2.0, 0.5, 7.0, 2.0, -1.0, 1.0, 3.0])
    assert restricted_argmax(logits, members) == 1            # tie 1 / 4: the lower id
    members[:] = True
    assert restricted_argmax(logits, members) == 0
    v = VocabList(8, 2)
    for bad in ([8], [-1]):
        with pytest.raises(ValueError):
            v.picked(bad)
        with pytest.raises(ValueError):
            v.begin_request(bad)


# ---- the DMTP round with the draft heads on the list -------------------------------------
from oracle import OracleModel                                      # noqa: E402
from synth import CONFIGS, make_prompts, make_weights               # noqa: E402

TINY = CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny():
    return OracleModel(TINY, make_weights(TINY, "cpu", fusion_std=0.02))


def test_full_list_is_the_plain_round(tiny):
    prompt = make_prompts(TINY)[0]
    s1, s2 = tiny.prefill(prompt), tiny.prefill(prompt)
    every = np.ones(TINY.vocab, dtype=bool)
    for _ in range(4):
        r1 = tiny.round(s1)
        r2 = tiny.round(s2, draft_list=every)
        assert r1["drafts"] == r2["drafts"] and r1["g"] == r2["g"]
        assert r1["committed"] == r2["committed"]


def test_short_list_stays_lossless_and_drafts_from_the_list(tiny):
    """The list kept as the page says (prompt counted at request start, picks counted and
    joined), 32 of 512 tokens: drafts come from the list, the stream is greedy decoding."""
    prompt = make_prompts(TINY)[0]
    greedy = tiny.greedy_decode(prompt, 10 * 8 + 9)
    vl = VocabList(TINY.vocab, 32)
    vl.begin_request(prompt)
    st = tiny.prefill(prompt)
    vl.picked([st.A])
    stream = [st.A]
    moved = 0
    for _ in range(10):
        members = vl.members.copy()
        rec = tiny.round(st, draft_list=members)
        assert all(members[t] for t in rec["drafts"])
        full_t1 = int(np.argmax(rec["t1_logits"]))
        moved += int(not members[full_t1])
        assert rec["T1"] == restricted_argmax(rec["t1_logits"], members)
        for s_ in range(6):
            assert rec["drafts"][s_ + 1] == restricted_argmax(rec["draft_logits"][s_], members)
        stream += rec["committed"]
        vl.picked(rec["committed"])
    assert stream == greedy[:len(stream)]
    assert moved > 0                       # the list did change some T1 picks
