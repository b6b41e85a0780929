"""Planted mistakes in the oracle (on the CPU) are caught by its pins: each case patches
one plausible slip into an oracle function (a dropped term, a wrong sign or order, a
swapped operand, a wrong constant) and requires the pin that guards it to fail. The
oracle itself is untouched outside each case (monkeypatch undoes the patch)."""
import numpy as np
import pytest

import test_oracle_depth as D
import test_oracle_fp8 as F
import test_oracle_gate as G
import test_oracle_primitives as P
import test_oracle_round as R
import test_oracle_sampling as S
from oracle import dmtp_oracle as O
from oracle import fp8 as fp8_mod
from oracle import gate as gate_mod
from oracle import sampling as sampling_mod


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


def test_primitives_pins_catch_slips(monkeypatch):
    rms = O.rms_norm
    monkeypatch.setattr(O, "rms_norm", lambda x, g, eps: rms(x, g, 0.0))       # eps dropped
    _fails(P.test_rms_norm_matches_torch)
    monkeypatch.setattr(O, "rms_norm", lambda x, g, eps: rms(x, np.ones_like(g), eps))
    _fails(P.test_rms_norm_matches_torch)                                        # gain dropped
    monkeypatch.undo()

    rope = O.rope
    monkeypatch.setattr(O, "rope", lambda x, pos, theta: rope(x, -np.asarray(pos), theta))
    _fails(P.test_rope_closed_forms)                                             # wrong sign
    monkeypatch.setattr(O, "rope", lambda x, pos, theta: rope(x, pos, theta / 10))
    _fails(P.test_rope_closed_forms)                                             # wrong base
    monkeypatch.undo()

    att = O.attend_rows

    def unscaled(q, K, V, hi, lo=0):                                             # no 1/sqrt(hd)
        return att(q * np.sqrt(q.shape[-1]), K, V, hi, lo)
    monkeypatch.setattr(O, "attend_rows", unscaled)
    _fails(P.test_attention_matches_torch_sdpa, 4, 2)
    monkeypatch.undo()

    step = O.gdn_step
    monkeypatch.setattr(O, "gdn_step", lambda S_, q, k, v, a, b: step(S_, q, k, -v, a, b))
    _fails(P.test_gdn_closed_forms)                                              # sign of v k^T
    monkeypatch.setattr(O, "gdn_step", lambda S_, q, k, v, a, b: step(S_, k, q, v, a, b))
    _fails(P.test_gdn_closed_forms)                                              # q, k swapped


def test_round_pins_catch_slips(monkeypatch):
    tiny, prompt = R._model(), R.make_prompts(R.TINY)[0]

    def swapped_slots(self, A, T1, delta):                                       # anchors swapped
        E = self.W["emb"]
        return np.stack([E[T1] + delta, E[A]] + [E[self.cfg.mask_id]] * 6)
    monkeypatch.setattr(O.OracleModel, "drafter_slots", swapped_slots)
    _fails(R.test_w_zero_reduction, tiny, prompt)
    monkeypatch.undo()

    def swapped_concat(self, T1, h_mtp):                                         # concat order
        W = self.W
        z = np.concatenate([O.rms_norm(h_mtp, W["fuse.norm_m"], self.eps),
                            O.rms_norm(W["emb"][T1], W["fuse.norm_e"], self.eps)])
        return W["fuse.w"] @ z
    monkeypatch.setattr(O.OracleModel, "fusion_delta", swapped_concat)
    _fails(R.test_fusion_concat_order)
    monkeypatch.undo()

    mtp = O.OracleModel.mtp_rows

    def mtp_concat_swapped(self, st, hT_prev, toks, pos0):                      # [e; h] for [h; e]
        W = self.W
        e = W["emb"][np.asarray(toks)]
        u = np.concatenate([O.rms_norm(e, W["mtp.norm_e"], self.eps),
                            O.rms_norm(hT_prev, W["mtp.norm_h"], self.eps)], axis=1)
        x, st.mtp_K, st.mtp_V = self.attn_layer("mtp", u @ W["mtp.proj"].T, st.mtp_K,
                                                st.mtp_V, pos0)
        return x
    monkeypatch.setattr(O.OracleModel, "mtp_rows", mtp_concat_swapped)
    _fails(R.test_mtp_uses_previous_target_hidden, prompt)
    monkeypatch.undo()

    monkeypatch.setattr(O.OracleModel, "mtp_rows",                              # h of position p
                        lambda self, st, h, toks, pos0: mtp(self, st, np.roll(h, -1, axis=0),
                                                            toks, pos0))
    _fails(R.test_mtp_uses_previous_target_hidden, prompt)
    monkeypatch.undo()

    monkeypatch.setattr(O.OracleModel, "mtp_rows",                              # token of p + 1
                        lambda self, st, h, toks, pos0: mtp(self, st, h, np.roll(toks, -1),
                                                            pos0))
    _fails(R.test_mtp_uses_embedding_of_pending_token, prompt)


def test_drafter_pins_catch_slips(monkeypatch):
    tiny, prompt = R._model(), R.make_prompts(R.TINY)[0]
    att = O.attend_rows

    def causal_block(q, K, V, hi, lo=0):                                         # mask in block
        hi = np.asarray(hi)
        if hi.size == 8 and np.all(hi == hi[0]):
            hi = hi - 7 + np.arange(8)
        return att(q, K, V, hi, lo)
    monkeypatch.setattr(O, "attend_rows", causal_block)
    _fails(R.test_drafter_block_is_bidirectional, tiny, prompt)
    monkeypatch.undo()

    real = O.OracleModel.drafter_forward
    for shift in (1, -1):                                                        # window off by one
        def shifted(self, X, st, a, with_head_in=False, _s=shift):
            cfg = self.cfg
            self.cfg = cfg.replace(draft_window=cfg.draft_window + _s)
            try:
                return real(self, X, st, a, with_head_in)
            finally:
                self.cfg = cfg
        monkeypatch.setattr(O.OracleModel, "drafter_forward", shifted)
        _fails(R.test_drafter_window)
        monkeypatch.undo()


def test_state_advance_pin_catches_a6_slips(monkeypatch):
    """The round's state advance (a6): slips that only the rounds make (the prefill's own
    calls start at position 0 or 1) must break state advance == prefill."""
    ctx = O.OracleModel.drafter_ctx_kv
    mtp = O.OracleModel.mtp_rows
    in_round = lambda pos: int(np.asarray(pos).reshape(-1)[0]) > 0

    monkeypatch.setattr(O.OracleModel, "drafter_ctx_kv",                         # taps row + 1
                        lambda self, taps, pos: ctx(self, np.roll(taps, -1, axis=0)
                                                    if in_round(pos) else taps, pos))
    _fails(R.test_state_advance_equals_prefill, "tiny")
    monkeypatch.undo()

    monkeypatch.setattr(O.OracleModel, "drafter_ctx_kv",                         # position + 1
                        lambda self, taps, pos: ctx(self, taps, np.asarray(pos) +
                                                    (1 if in_round(pos) else 0)))
    _fails(R.test_state_advance_equals_prefill, "tiny")
    monkeypatch.undo()

    monkeypatch.setattr(O.OracleModel, "mtp_rows",                               # token of p + 1
                        lambda self, st, h, toks, pos0: mtp(
                            self, st, h, list(toks[1:]) + [toks[-1]] if pos0 > 1 and
                            st.a > 0 and pos0 == st.a + 1 else toks, pos0))
    _fails(R.test_state_advance_equals_prefill, "tiny")
    monkeypatch.undo()

    monkeypatch.setattr(O.OracleModel, "mtp_rows",                               # h of row p
                        lambda self, st, h, toks, pos0: mtp(
                            self, st, np.roll(h, -1, axis=0) if pos0 > 1 and
                            pos0 == st.a + 1 else h, toks, pos0))
    _fails(R.test_state_advance_equals_prefill, "tiny_hybrid")


def test_sampling_pin_catches_a_swapped_key(monkeypatch):
    ph = sampling_mod.philox4x32_10
    monkeypatch.setattr(S, "philox4x32_10", lambda ctr, key: ph(ctr, np.asarray(key)[::-1]))
    _fails(S.test_philox_known_answers, (0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344),
           (0xA4093822, 0x299F31D0), (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))


def test_sampling_pin_catches_a_flipped_noise_sign(monkeypatch):
    gum = sampling_mod.gumbel
    flipped = lambda seed, b, pos, vocab: -gum(seed, b, pos, vocab)            # Gumbel-min
    monkeypatch.setattr(sampling_mod, "gumbel", flipped)
    monkeypatch.setattr(S, "gumbel", flipped)
    _fails(S.test_gumbel_max_draws_from_softmax)


def test_fp8_scale_and_metric_pins_catch_slips(monkeypatch):
    ps = fp8_mod.pow2_scale
    loose = lambda amax: 2.0 * ps(amax)                                           # one power off
    monkeypatch.setattr(fp8_mod, "pow2_scale", loose)
    monkeypatch.setattr(F, "pow2_scale", loose)
    _fails(F.test_pow2_scales_tight_and_exact)
    monkeypatch.undo()

    mal = O.mean_accept_len
    monkeypatch.setattr(O, "mean_accept_len", lambda h: mal(h) - 1.0)            # no bonus token
    _fails(P.test_accept_metrics_hand_histograms)


def test_fp8_pin_catches_ties_away_from_zero(monkeypatch):
    grid = fp8_mod.e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2
    real = fp8_mod.round_e4m3

    def ties_away(x):
        x = np.asarray(x, dtype=np.float64)
        out = real(x)
        a = np.abs(x)
        idx = np.searchsorted(mids, a)
        tie = (idx < mids.size) & (mids[np.minimum(idx, mids.size - 1)] == a)
        return np.where(tie, np.sign(x) * grid[np.minimum(idx + 1, grid.size - 1)], out)
    monkeypatch.setattr(F, "round_e4m3", ties_away)
    _fails(F.test_rounding_matches_torch)


def test_gate_pins_catch_slips(monkeypatch):
    et = gate_mod.DepthGate.expected_tokens
    monkeypatch.setattr(gate_mod.DepthGate, "expected_tokens",
                        staticmethod(lambda acc: et(list(acc)[:-1])))      # last term dropped
    _fails(G.test_geometric_acceptance_linear_cost, 0.9, 0.3)
    monkeypatch.undo()

    cost = gate_mod.DepthGate.cost
    monkeypatch.setattr(gate_mod.DepthGate, "cost",
                        lambda self, k, count_drafting=True: cost(self, k, False))   # d ignored
    _fails(G.test_draft_cost_enters_per_extra_draft)
    monkeypatch.undo()

    monkeypatch.setattr(gate_mod, "PROBE_EVERY", 15)                        # probe period
    _fails(G.test_zero_acceptance_declines_but_probes)
    monkeypatch.undo()

    monkeypatch.setattr(gate_mod, "AVG_WEIGHT", 1.0 / 8.0)                  # average weight
    _fails(G.test_running_average_closed_form)
    monkeypatch.undo()

    res = gate_mod.DepthGate.result

    def judges_all(self, judged, accepted, p=None):                          # past the rejection
        res(self, judged, accepted, p)
        for j in range(judged, self.K):
            self.a[j] = self._avg(self.a[j], 0.0)
    monkeypatch.setattr(gate_mod.DepthGate, "result", judges_all)
    _fails(G.test_default_priors_and_judged_drafts_only)
    monkeypatch.undo()

    monkeypatch.setattr(gate_mod, "PLAIN_EVERY", 65)                        # plain-step period
    _fails(G.test_plain_step_after_64_forwards)


def test_head_confidence_pin_catches_a_narrow_window(monkeypatch):
    hc = gate_mod.head_confidence
    monkeypatch.setattr(D, "head_confidence", lambda l, window=20.0: hc(l, 10.0))
    _fails(D.test_head_confidence_closed_forms)


def test_shortlist_pins_catch_slips(monkeypatch):
    import test_oracle_shortlist as L
    from oracle import shortlist as sl
    monkeypatch.setattr(sl, "HALVE_EVERY", 1000)                             # halving period
    _fails(L.test_halving_every_1024_counted_tokens)
    monkeypatch.undo()

    def half_rule(self):                                                     # 1/2 for 3/4
        order = np.lexsort((np.arange(self.V), -self.counts))
        last = int(self.counts[order[:self.size][-1]])
        members = 2 * self.counts >= last
        members[order[:self.size]] = True
        for t in self.conv:
            members[t] = True
        self.members = members
        self.rebuilds += 1
    monkeypatch.setattr(sl.VocabList, "rebuild", half_rule)
    _fails(L.test_list_composition, 3)
    monkeypatch.undo()

    pk = sl.VocabList.picked

    def no_join(self, tokens):                                               # picks not joined
        before = self.members.copy()
        pk(self, tokens)
        self.members = before
    monkeypatch.setattr(sl.VocabList, "picked", no_join)
    _fails(L.test_picked_tokens_join_at_once_and_count)
