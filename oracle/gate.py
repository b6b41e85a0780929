"""Draft-depth gate (TEST INFRASTRUCTURE ONLY: imported by tests/ alone).

colibri speculative-decoding doc, the draft-depth gate (the value(k) paragraph) and its
per-step refinement (the paragraph on each step's own drafts), in this module's words:

* a_j estimates how often draft j survives verification given that every earlier draft
  of the same verify did; the estimates begin at 0.8, 0.6 and 0.5 (an MTP head's
  starting values) and move as a running mean over roughly the last 16 verifies.
* T(n) is the observed duration of an n-row forward; d is the observed extra time one
  more draft costs its source beyond the first draft.
* E(k) = 1 + a_1 + a_1 a_2 + ... + a_1 ... a_k is the expected count of committed
  tokens when k drafts are checked at once; cost(k) = (T(k+1) + (k - 1) d) / T(1) expresses its time in plain
  decode steps; value(k) = E(k) / cost(k). The gate verifies the depth of highest value,
  and falls back to a plain step (worth exactly 1) unless that value is above 1.
* Row counts with no observation are priced by the line T(1) (1 + (n - 1) rho), whose
  slope rho is fitted to the observed multi-row forwards once T(1) is known (0.5 before).
* To keep estimates alive the gate goes one draft past its choice on every 16th
  decision, and to keep T(1) observed it forces a plain step once 64 forwards in a row
  had several rows.
* A settled verify reports how many drafts were judged: the accepted ones plus the first
  rejected one, if any; later drafts carry no information about a_j.
* Per-step form: a source that can rate every draft of the current step with a probability
  p_j lets the gate replace a_j by the acceptance it has observed for drafts rated alike
  (ten equal bins of p, each seeded with its own centre as if two verifies had shown it
  and updated by every verify), and since those drafts are already written only their
  verify is priced: cost(k) = T(k+1) / T(1).

Readings where the page leaves a step open (the native gate takes the same ones):
  1. "an average over about 16 verifies" is an exponential average of weight 1/16 per
     judged draft; measured times T(n) and d are averaged the same way (the first
     measurement sets them).
  2. rho is the least-squares slope through the origin of T(n)/T(1) - 1 against n - 1
     over the measured n >= 2.
  3. While T(1) is unmeasured, cost(k) = 1 + k rho and d is not counted (it has no unit
     of T(1) yet).
  4. Equal values go to the smaller k. A probe (every 16th pick, counted from the first)
     takes min(proposed, best + 1), best being 0 when the gate declines; the forced plain
     step takes precedence over a probe.
  5. Bin i of p holds p in [i/10, (i+1)/10) (p = 1 in bin 9) and starts at its centre
     (i + 1/2)/10: estimate = (2 centre + accepted) / (2 + judged) over the drafts of
     that bin.
  6. One source (the DMTP block: T1 from MTP, T2..T7 from the drafter), so the a_j
     priors are the MTP head's.
"""
from __future__ import annotations

import numpy as np

DEFAULT_PRIORS = (0.8, 0.6, 0.5)
AVG_WEIGHT = 1.0 / 16.0
PROBE_EVERY = 16
PLAIN_EVERY = 64
RHO0 = 0.5
N_BINS = 10


def head_confidence(logits, window: float = 20.0) -> float:
    """The probability a draft head gives its own (argmax) pick, normalised over the
    scores no more than `window` below the best (the per-step paragraph's estimate for
    MTP heads),
    1 / sum over {v : l_v >= l_max - window} of exp(l_v - l_max)."""
    l = np.asarray(logits, dtype=np.float64)
    m = float(l.max())
    near = l[l >= m - window]
    return float(1.0 / np.sum(np.exp(near - m)))


class DepthGate:
    def __init__(self, max_drafts: int, priors=None):
        if max_drafts < 1:
            raise ValueError("max_drafts >= 1")
        self.K = max_drafts
        if priors is None:
            priors = [DEFAULT_PRIORS[min(j, len(DEFAULT_PRIORS) - 1)] for j in range(max_drafts)]
        self.a = [float(x) for x in priors]            # a_1 .. a_K
        self.T = {}                                     # rows -> measured seconds
        self.d = None                                   # seconds per draft past the first
        self.picks = 0
        self.since_plain = 0                            # forwards since the last plain step
        self.bin_judged = [0] * N_BINS
        self.bin_accepted = [0] * N_BINS

    # -- measured quantities ------------------------------------------------------------
    @staticmethod
    def _avg(old, x):
        return x if old is None else old + (x - old) * AVG_WEIGHT

    def forward(self, rows: int, seconds: float):
        if rows < 1 or not seconds > 0:
            raise ValueError("rows >= 1, seconds > 0")
        self.T[rows] = self._avg(self.T.get(rows), float(seconds))
        self.since_plain = 0 if rows == 1 else self.since_plain + 1

    def draft_cost(self, seconds: float):
        if not seconds >= 0:
            raise ValueError("seconds >= 0")
        self.d = self._avg(self.d, float(seconds))

    def result(self, judged: int, accepted: int, p=None):
        if not (0 <= accepted <= judged <= self.K and judged <= accepted + 1):
            raise ValueError("0 <= accepted <= judged <= accepted + 1, judged <= max_drafts")
        for j in range(judged):
            x = 1.0 if j < accepted else 0.0
            self.a[j] = self._avg(self.a[j], x)
            if p is not None:
                b = self.bin_of(p[j])
                self.bin_judged[b] += 1
                self.bin_accepted[b] += int(j < accepted)

    # -- model ------------------------------------------------------------------------------
    def rho(self) -> float:
        if 1 not in self.T:
            return RHO0
        rows = sorted(n for n in self.T if n >= 2)       # increasing row count
        if not rows:
            return RHO0
        sxy = sxx = 0.0                                  # plain left-to-right sums
        for n in rows:
            x, y = float(n - 1), self.T[n] / self.T[1] - 1.0
            sxy += x * y
            sxx += x * x
        return sxy / sxx

    def t_rel(self, n: int) -> float:
        """T(n) / T(1): measured where both are, else 1 + (n - 1) rho."""
        if 1 in self.T and n in self.T:
            return self.T[n] / self.T[1]
        return 1.0 + (n - 1) * self.rho()

    def cost(self, k: int, count_drafting: bool = True) -> float:
        c = self.t_rel(k + 1)
        if count_drafting and k >= 1 and self.d is not None and 1 in self.T:
            c += (k - 1) * self.d / self.T[1]
        return c

    @staticmethod
    def expected_tokens(acc) -> float:
        """E(k) = 1 + a_1 + a_1 a_2 + ... for the given a_1 .. a_k."""
        e, run = 1.0, 1.0
        for x in acc:
            run *= x
            e += run
        return e

    def value(self, k: int) -> float:
        if k == 0:
            return 1.0
        return self.expected_tokens(self.a[:k]) / self.cost(k)

    @staticmethod
    def bin_of(p: float) -> int:
        return min(N_BINS - 1, max(0, int(np.floor(float(p) * N_BINS))))

    def bin_estimate(self, b: int) -> float:
        centre = (b + 0.5) / N_BINS
        return (2.0 * centre + self.bin_accepted[b]) / (2.0 + self.bin_judged[b])

    def value_p(self, p, k: int) -> float:
        if k == 0:
            return 1.0
        acc = [self.bin_estimate(self.bin_of(x)) for x in p[:k]]
        return self.expected_tokens(acc) / self.cost(k, count_drafting=False)

    # -- decisions ----------------------------------------------------------------------------
    def _decide(self, proposed: int, values):
        """values[k - 1] = value(k) for k = 1..proposed; returns (k, value of k)."""
        self.picks += 1
        if self.since_plain >= PLAIN_EVERY or proposed == 0:
            return 0, 1.0
        best, best_v = 0, 1.0
        for k in range(1, proposed + 1):
            if values[k - 1] > best_v:
                best, best_v = k, values[k - 1]
        if self.picks % PROBE_EVERY == 0:
            k = min(proposed, best + 1)
            return k, (values[k - 1] if k else 1.0)
        return best, best_v

    def pick(self, proposed: int):
        proposed = min(int(proposed), self.K)
        if proposed < 0:
            raise ValueError("proposed >= 0")
        return self._decide(proposed, [self.value(k) for k in range(1, proposed + 1)])

    def pick_p(self, p):
        p = [float(x) for x in p][:self.K]
        return self._decide(len(p), [self.value_p(p, k) for k in range(1, len(p) + 1)])
