"""Pins of the oracle's variable-depth round (OracleModel.round(depth=...)) and of the
draft heads' confidence (oracle/gate.py head_confidence), no GPU:

* head_confidence: 1/V for equal scores, 1 when every other score is more than 20 below,
  1 / (1 + e^-20) at the window's edge, the plain softmax maximum when all scores lie
  within the window;
* a verify of k drafts is the first k + 1 rows of the 8-row verify (causal rows), and the
  accepted count is the 8-row count capped at k: picks, commits and watermarks agree;
* depth 0 is a plain decode step;
* losslessness with the depth chosen every round by the gate (per-step form, fed with the
  heads' confidences and the settled verifies), drafts forced right and wrong: the
  committed stream is still plain greedy decoding (colibri doc: the output matches plain
  decoding, only the number of forwards changes);
* Gated DeltaNet: a shorter verify installs the snapshot after row n as before.
"""
import math

import numpy as np
import pytest
import scipy.special

from oracle import OracleModel
from oracle.gate import DepthGate, head_confidence
from synth import CONFIGS, make_prompts, make_weights

TINY = CONFIGS["tiny"]
HYB = TINY.replace(name="tiny_hybrid", n_layers=4, layer_kinds=(1, 1, 1, 0),
                   gdn_heads=4, gdn_dk=16, gdn_dv=16)


@pytest.fixture(scope="module")
def tiny():
    return OracleModel(TINY, make_weights(TINY, "cpu", fusion_std=0.02))


@pytest.fixture(scope="module")
def prompt():
    return make_prompts(TINY)[0]


@pytest.fixture(scope="module")
def greedy(tiny, prompt):
    return tiny.greedy_decode(prompt, 12 * 8 + 9)


def test_head_confidence_closed_forms():
    assert head_confidence(np.zeros(512)) == pytest.approx(1 / 512, rel=1e-15)
    assert head_confidence([3.0, -17.5, -40.0]) == 1.0
    assert head_confidence([0.0, -20.0, -25.0]) == pytest.approx(1 / (1 + math.exp(-20)),
                                                                  rel=1e-15)
    rng = np.random.default_rng(0)
    for _ in range(20):
        l = rng.normal(0, 3, 300)                     # every score within 20 of the best
        assert l.max() - l.min() < 40
        l = np.clip(l, l.max() - 19.9, None)
        assert head_confidence(l) == pytest.approx(scipy.special.softmax(l).max(), rel=1e-12)


def _forced(greedy, st, prompt_len, wrong):
    off = st.a - prompt_len
    d = list(greedy[off + 1: off + 8])
    if wrong < 7:
        d[wrong] = (d[wrong] + 1) % (TINY.vocab - 1)
    return d


def test_depth_k_is_the_capped_eight_row_round(tiny, prompt, greedy):
    st = tiny.prefill(prompt)
    for r, wrong in enumerate([7, 3, 0, 5, 7, 1]):
        d = _forced(greedy, st, len(prompt), wrong)
        full = tiny.round(st.clone(), forced=d)
        for k in range(8):
            s_k = st.clone()
            rec = tiny.round(s_k, forced=d, depth=k)
            assert rec["depth"] == k and len(rec["g"]) == k + 1
            assert rec["g"] == full["g"][:k + 1]
            np.testing.assert_array_equal(rec["verify_logits"], full["verify_logits"][:k + 1])
            assert rec["n"] == min(full["n"], k)
            assert rec["committed"] == d[:rec["n"]] + [full["g"][rec["n"]]]
            assert s_k.a == st.a + rec["n"] + 1 and rec["kv_len"] == s_k.a
        tiny.round(st, forced=d)


def test_depth_zero_is_a_plain_step(tiny, prompt, greedy):
    st = tiny.prefill(prompt)
    stream = [st.A]
    for _ in range(5):
        rec = tiny.round(st, depth=0)
        assert rec["n"] == 0 and len(rec["committed"]) == 1
        stream += rec["committed"]
    assert stream == greedy[:len(stream)]


@pytest.mark.parametrize("form", ["averages", "per_step"])
def test_lossless_with_gate_chosen_depth(tiny, prompt, greedy, form):
    """The averaged form varies the depth as verifies settle; the per-step form sees the
    untrained heads' low confidence (near 1/V), declines until its probe, then learns
    from the probe's verify."""
    gate = DepthGate(7)
    for n in range(1, 9):
        gate.forward(n, 1.0 + 0.08 * (n - 1))
    st = tiny.prefill(prompt)
    stream = [st.A]
    depths = []
    pattern = [7, 2, 7, 7, 4, 0, 7, 6, 7, 1, 7, 7]
    for r in range(20):
        d = _forced(greedy, st, len(prompt), pattern[r % len(pattern)])
        chosen = {}

        def choose(drafts, conf):
            assert len(drafts) == 7 and len(conf) == 7
            assert all(0.0 < p <= 1.0 for p in conf)
            chosen["conf"] = conf
            return gate.pick(7)[0] if form == "averages" else gate.pick_p(conf)[0]

        rec = tiny.round(st, forced=d, depth=choose)
        k = rec["depth"]
        depths.append(k)
        gate.forward(k + 1, 1.0 + 0.08 * k)
        if k:
            n = rec["n"]
            judged = n if n == k else n + 1
            gate.result(judged, n, chosen["conf"][:judged])
        stream += rec["committed"]
    assert stream == greedy[:len(stream)]
    if form == "averages":
        assert len(set(depths)) > 1 and min(depths) >= 1
    else:
        # declined until the probe of the 16th pick; its accepted draft lifts the lowest
        # probability bin, after which the gate drafts
        assert depths[:15] == [0] * 15 and depths[15] == 1 and max(depths[16:]) >= 1


def test_hybrid_shorter_verify_installs_the_row_snapshot():
    hyb = OracleModel(HYB, make_weights(HYB, "cpu"))
    prompt = make_prompts(HYB)[0][:40]
    greedy = hyb.greedy_decode(prompt, 50)
    st = hyb.prefill(prompt)
    stream = [st.A]
    for r, (wrong, k) in enumerate([(7, 3), (1, 5), (7, 0), (4, 7), (7, 6)]):
        off = st.a - len(prompt)
        d = list(greedy[off + 1: off + 8])
        if wrong < 7:
            d[wrong] = (d[wrong] + 1) % (HYB.vocab - 1)
        pre = st.clone()
        rec = hyb.round(st, forced=d, depth=k)
        assert rec["n"] == min(wrong, k) and rec["snap_slot"] == rec["n"]
        rp = pre.clone()
        for s_, t in enumerate(([pre.A] + d)[:rec["n"] + 1]):
            hyb.target_rows(rp, [t], pre.a + s_, head=False)
        for l, kind in enumerate(HYB.layer_kinds):
            if kind:
                np.testing.assert_array_equal(st.gdn_S[l], rp.gdn_S[l])
        stream += rec["committed"]
    assert stream == greedy[:len(stream)]


def test_depth_out_of_range_is_refused(tiny, prompt):
    st = tiny.prefill(prompt)
    for bad in (-1, 8, lambda drafts, conf: 9):
        with pytest.raises(ValueError):
            tiny.round(st.clone(), depth=bad)
