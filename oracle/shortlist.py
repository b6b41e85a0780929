"""Frequent-token shortlist for the draft heads (TEST INFRASTRUCTURE ONLY).

colibri speculative-decoding doc, the paragraph on the token list a draft head scores
in place of the full vocabulary, in this module's words:

* Listed tokens: the `size` most frequent ones (16000 unless set), any other token whose
  frequency reaches three quarters of the smallest frequency among those, and any token
  that occurs in the conversation being served.
* Frequencies: each prompt token and each committed pick raises its token's count by
  one; after every 1024 counted tokens all counts are halved.
* Upkeep: the list is recomputed at the start of each request and after each halving; a
  pick that is not listed is added immediately.
* Verification scores the full vocabulary, so the committed tokens are unaffected; a
  token left off the list can only cost a draft.

Readings where the page leaves a step open (the native list takes the same ones):
  1. Counts are integers; halving is floor division by 2; the 1024th counted token since
     the last halving triggers it (the counter then restarts).
  2. The `size` most frequent tokens are ranked by count, then by id (lower first); the
     three-quarters rule compares 4 count >= 3 count_last exactly. When fewer than `size` tokens
     have a positive count, the last count is 0 and every token qualifies (no counts:
     the whole vocabulary).
  3. A request start joins the prompt's tokens to the conversation (after clearing it
     when a new conversation begins), counts them in order (a halving in between rebuilds
     the list then), and rebuilds the list.
  4. A picked token is counted, joins the conversation, and joins the list if missing.
  5. One list serves a whole batch: its conversation is the union of the batch's prompts
     and picks.
"""
from __future__ import annotations

import numpy as np

DEFAULT_SIZE = 16000
HALVE_EVERY = 1024


class VocabList:
    def __init__(self, vocab: int, size: int = DEFAULT_SIZE):
        if vocab < 1 or size < 1:
            raise ValueError("vocab >= 1, size >= 1")
        self.V, self.size = int(vocab), int(size)
        self.counts = np.zeros(self.V, dtype=np.int64)
        self.counted = 0                       # tokens counted since the last halving
        self.conv: set[int] = set()
        self.members = np.ones(self.V, dtype=bool)   # before any request: every token
        self.rebuilds = 0
        self.appended = 0
        self.picks = 0
        self.picks_in = 0

    def _check(self, tokens):
        t = np.asarray(tokens, dtype=np.int64).reshape(-1)
        if t.size and (t.min() < 0 or t.max() >= self.V):
            raise ValueError("token id out of range")
        return t

    def _count(self, t: int):
        self.counts[t] += 1
        self.counted += 1
        if self.counted == HALVE_EVERY:
            self.counts //= 2
            self.counted = 0
            self.rebuild()

    def rebuild(self):
        order = np.lexsort((np.arange(self.V), -self.counts))   # count desc, then id asc
        top = order[:min(self.size, self.V)]
        last = int(self.counts[top[-1]])
        members = np.zeros(self.V, dtype=bool)
        members[top] = True
        members |= 4 * self.counts >= 3 * last
        for t in self.conv:
            members[t] = True
        self.members = members
        self.rebuilds += 1

    def begin_request(self, prompt, new_conversation: bool = True):
        t = self._check(prompt)
        if new_conversation:
            self.conv = set()
        self.conv.update(int(x) for x in t)
        for x in t:
            self._count(int(x))
        self.rebuild()

    def picked(self, tokens):
        for x in self._check(tokens):
            x = int(x)
            self.picks += 1
            self.picks_in += int(self.members[x])
            self._count(x)
            self.conv.add(x)
            if not self.members[x]:
                self.members[x] = True
                self.appended += 1

    def ids(self) -> np.ndarray:
        return np.flatnonzero(self.members).astype(np.int32)


def restricted_argmax(logits, members) -> int:
    """The lowest id of the largest logit among the listed tokens."""
    l = np.asarray(logits, dtype=np.float64)
    ids = np.flatnonzero(members)
    return int(ids[np.argmax(l[ids])])
