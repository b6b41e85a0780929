"""Pins of the draft-depth gate oracle (oracle/gate.py) against closed forms and brute
force (colibri speculative-decoding doc, the gate's value(k) paragraph):

* constant acceptance a and a linear forward cost T(n) = T(1)(1 + (n - 1) rho): E(k) is
  the geometric sum (1 - a^(k+1)) / (1 - a), value(k) = E(k) / (1 + k rho), and the pick
  is the brute-force argmax over k (smaller k on ties), declined when no value exceeds 1;
* rho = 0 drafts as deep as proposed; a = 0 declines except the probe of every 16th pick;
* the exponential average: m accepted verifies move a_1 from a0 to 1 - (1 - a0)(15/16)^m;
* a verify judges the accepted drafts and the first rejected one, nothing past it;
* the plain step after 64 multi-row forwards, reset by a plain forward;
* rho recovered exactly from linear timings; the per-draft cost d enters as (k - 1) d / T(1);
* the per-step bins: edges, the two-verify prior at the bin centre, pricing the verify only.
"""
import math

import pytest

from oracle.gate import DepthGate


def _linear_gate(a, rho, K=7, measured=(1, 3)):
    g = DepthGate(K, priors=[a] * K)
    for n in measured:
        g.forward(n, 2.0 * (1.0 + (n - 1) * rho))      # T(1) = 2 s
    return g


@pytest.mark.parametrize("a,rho", [(0.7, 0.05), (0.9, 0.3), (0.5, 0.5), (0.95, 0.01),
                                    (0.3, 0.2), (0.8, 1.5)])
def test_geometric_acceptance_linear_cost(a, rho):
    g = _linear_gate(a, rho)
    assert g.rho() == pytest.approx(rho, abs=1e-12)
    closed = [(1 - a ** (k + 1)) / (1 - a) / (1 + k * rho) for k in range(1, 8)]
    for k in range(1, 8):
        assert g.value(k) == pytest.approx(closed[k - 1], rel=1e-12)
    for proposed in range(0, 8):
        best, best_v = 0, 1.0
        for k in range(1, proposed + 1):
            if closed[k - 1] > best_v + 1e-15:
                best, best_v = k, closed[k - 1]
        k, v = g.pick(proposed)
        assert k == best
        assert v == pytest.approx(best_v, rel=1e-12)


def test_flat_cost_drafts_as_deep_as_proposed():
    g = _linear_gate(0.4, 0.0)
    for proposed in range(1, 8):
        assert g.pick(proposed)[0] == proposed
    assert g.pick(9)[0] == 7                              # capped at max_drafts


def test_zero_acceptance_declines_but_probes():
    g = _linear_gate(0.0, 0.1)
    ks = [g.pick(7)[0] for _ in range(48)]
    assert ks == [1 if (i + 1) % 16 == 0 else 0 for i in range(48)]


def test_probe_is_one_deeper_than_the_best():
    g = _linear_gate(0.9, 0.3)
    best = g.pick(7)[0]
    assert 1 <= best < 7
    ks = [g.pick(7)[0] for _ in range(15)]               # picks 2..16
    assert ks[:-1] == [best] * 14 and ks[-1] == best + 1


def test_running_average_closed_form():
    g = DepthGate(1, priors=[0.8])
    for m in range(1, 40):
        g.result(1, 1)
        assert g.a[0] == pytest.approx(1 - 0.2 * (15 / 16) ** m, rel=1e-13)
    g = DepthGate(1, priors=[0.8])
    for m in range(1, 40):
        g.result(1, 0)
        assert g.a[0] == pytest.approx(0.8 * (15 / 16) ** m, rel=1e-13)


def test_default_priors_and_judged_drafts_only():
    g = DepthGate(7)
    assert g.a == [0.8, 0.6, 0.5, 0.5, 0.5, 0.5, 0.5]
    g.result(3, 2)                                        # drafts 1, 2 accepted, 3 rejected
    assert g.a[0] == pytest.approx(0.8 + 0.2 / 16)
    assert g.a[1] == pytest.approx(0.6 + 0.4 / 16)
    assert g.a[2] == pytest.approx(0.5 - 0.5 / 16)
    assert g.a[3:] == [0.5] * 4
    g.result(7, 7)                                        # all seven accepted
    assert all(x > y for x, y in zip(g.a[3:], [0.5] * 4))
    for bad in ((3, 1), (2, 3), (8, 7), (-1, 0)):
        with pytest.raises(ValueError):
            g.result(*bad)


def test_plain_step_after_64_forwards():
    g = _linear_gate(0.9, 0.05)
    g.forward(1, 2.0)
    for i in range(63):
        g.forward(8, 2.5)
        assert g.pick(7)[0] > 0 or (g.picks % 16 == 0)
    g.forward(8, 2.5)                                     # the 64th without a plain step
    assert g.pick(7) == (0, 1.0)
    assert g.pick(7) == (0, 1.0)                          # still owed
    g.forward(1, 2.0)
    assert g.pick(7)[0] > 0


def test_rho_default_and_fit():
    g = DepthGate(7)
    assert g.rho() == 0.5                                 # nothing measured
    g.forward(4, 3.0)
    assert g.rho() == 0.5                                 # T(1) unmeasured
    assert g.t_rel(4) == pytest.approx(2.5)
    g.forward(1, 1.0)
    assert g.rho() == pytest.approx(2.0 / 3.0)            # (3/1 - 1) / (4 - 1)
    g2 = DepthGate(7)
    g2.forward(1, 1.0)
    assert g2.rho() == 0.5                                # no multi-row forward yet
    # exact least squares through the origin of two points: (1, 0.2), (3, 0.9)
    g2.forward(2, 1.2)
    g2.forward(4, 1.9)
    assert g2.rho() == pytest.approx((1 * 0.2 + 3 * 0.9) / (1 + 9))
    assert g2.t_rel(3) == pytest.approx(1 + 2 * g2.rho())   # unmeasured row count
    assert g2.t_rel(4) == pytest.approx(1.9)                # measured


def test_timings_average():
    g = DepthGate(7)
    g.forward(1, 1.0)
    g.forward(1, 3.0)
    assert g.T[1] == pytest.approx(1.0 + 2.0 / 16)
    g.draft_cost(0.5)
    g.draft_cost(0.1)
    assert g.d == pytest.approx(0.5 - 0.4 / 16)


def test_draft_cost_enters_per_extra_draft():
    g = _linear_gate(0.8, 0.1, measured=(1, 2, 3, 4, 5, 6, 7, 8))
    base = [g.value(k) for k in range(1, 8)]
    g.draft_cost(0.3)                                     # T(1) = 2 s: 0.15 T(1) per draft
    for k in range(1, 8):
        e = (1 - 0.8 ** (k + 1)) / 0.2
        assert g.value(k) == pytest.approx(e / (1 + 0.1 * k + 0.15 * (k - 1)), rel=1e-12)
    assert g.value(1) == pytest.approx(base[0])           # the first draft is free of d
    assert all(g.value(k) < base[k - 1] for k in range(2, 8))


def test_bins():
    g = DepthGate(7)
    assert [g.bin_of(p) for p in (0.0, 0.0999, 0.1, 0.55, 0.9, 0.999, 1.0)] == \
        [0, 0, 1, 5, 9, 9, 9]
    assert [g.bin_estimate(b) for b in range(10)] == pytest.approx(
        [(b + 0.5) / 10 for b in range(10)])
    # three verifies of drafts at p = 0.93 (bin 9): two accepted all, one rejected draft 2
    g.result(2, 2, p=[0.93, 0.91])
    g.result(2, 2, p=[0.95, 0.97])
    g.result(2, 1, p=[0.92, 0.96])
    assert g.bin_judged[9] == 6 and g.bin_accepted[9] == 5
    assert g.bin_estimate(9) == pytest.approx((2 * 0.95 + 5) / (2 + 6))
    assert g.bin_judged[:9] == [0] * 9


def test_pick_p_prices_only_the_verify():
    g = _linear_gate(0.5, 0.1, measured=(1, 2))
    g.draft_cost(1.0)                                     # would dominate if counted
    sure, doubtful = [0.97] * 7, [0.05] * 7
    k, v = g.pick_p(sure)
    e = 1.0
    run = 1.0
    best, best_v = 0, 1.0
    for kk in range(1, 8):
        run *= 0.95
        e += run
        if e / (1 + 0.1 * kk) > best_v:
            best, best_v = kk, e / (1 + 0.1 * kk)
    assert (k, v) == (best, pytest.approx(best_v))
    assert k == 7
    assert g.pick_p(doubtful)[0] == 0
    mixed = [0.97, 0.97, 0.05, 0.97, 0.97, 0.97, 0.97]   # the third draft is doubtful
    assert g.pick_p(mixed)[0] == 2


def test_value_of_a_plain_step_is_one():
    g = _linear_gate(0.0, 0.0)
    assert g.value(0) == 1.0 and g.value_p([0.5], 0) == 1.0
    assert math.isclose(g.value(3), 1.0)                  # a = 0, flat cost: E = 1
    assert g.pick(7)[0] == 0                              # not above a plain step
