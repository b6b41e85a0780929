"""Parity of the CUDA round (through the C ABI) with the oracle, in lock-step.

Integer fields (drafts, picks, n, committed, kv_len, mtp_len, snapshot slot) must be
bit-exact wherever the oracle's top-1/top-2 gap exceeds 0.05; float fields (T1,
drafter and verify logits, Delta, h_MTP) within max-abs 2e-2. Sizes span several
GEMM tiles (vocab and weight rows with ragged tails), several attention chunks
(contexts > 256 keys with a ragged tail) and per-sequence ragged contexts.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, make_prompts, make_weights

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _lockstep(cfg, rounds, fusion_std=None, seqs=None, prompts=None):
    from lockstep import Lockstep
    w = make_weights(cfg, "cuda", fusion_std=fusion_std)
    prompts = make_prompts(cfg) if prompts is None else prompts
    return Lockstep(cfg, w, prompts, rounds, seqs=seqs)


TINY = CONFIGS["tiny"]
# small-model shape (vocab 32000, d 1024, 8 layers of 16/16 x 64) with a shorter prompt
SMALL_R = CONFIGS["small"].replace(ctx_lo=300, ctx_hi=300)
# B32 shape at reduced width: 256 GEMM rows, GQA 8/2, ragged vocab (5000 = 39*128 + 8)
B32_R = CONFIGS["b32"].replace(name="b32_r", vocab=5000, d_model=256, n_layers=2, n_heads=8,
                               n_kv_heads=2, head_dim=64, ffn=512, ctx_lo=40, ctx_hi=300)
# hybrid target at reduced width: GDN, GDN, GDN, attention
HYB_R = CONFIGS["hybrid"].replace(name="hybrid_r", vocab=3000, d_model=256, n_layers=4,
                                  layer_kinds=(1, 1, 1, 0), n_heads=4, n_kv_heads=2,
                                  head_dim=64, ffn=512, batch=4, ctx_lo=60, ctx_hi=120,
                                  gdn_heads=4, gdn_dk=64, gdn_dv=64)


# target-only sampled verification (DMTP §5): the verify picks are the target's samples
TINY_S = TINY.replace(name="tiny_sampled", temperature=0.8, sample_seed=20260611)
B32_RS = B32_R.replace(name="b32_r_sampled", temperature=1.0, sample_seed=0x5EED_0000_0007)


def test_tiny_natural_16_rounds():
    ls = _lockstep(TINY, 16)
    for _ in range(16):
        ls.step(tol=TOL)
    assert ls.max_err["verify_logits"] < 1e-3   # fp32 storage: far inside the bar
    ls.close()


def test_tiny_with_fusion_weights():
    ls = _lockstep(TINY, 8, fusion_std=0.02)
    for _ in range(8):
        _, recs = ls.step(tol=TOL)
        assert np.abs(recs[0]["delta"]).max() > 0
    ls.close()


def _greedy(ls, b, n):
    return ls.oracle.greedy_decode(ls.prompts[b], n)


@pytest.mark.parametrize("mode", ["all_right", "all_wrong", "alternating", "cycling"])
def test_tiny_forced_modes(mode):
    """The colibri page's forced-draft modes: every accepted length 0..7 is exercised,
    and the committed stream stays the plain greedy stream."""
    ls = _lockstep(TINY, 10)
    greedy = _greedy(ls, 0, 8 * 10 + 9)
    P = len(ls.prompts[0])
    stream = [ls.states[0].A]
    for r in range(10):
        off = ls.states[0].a - P
        d = list(greedy[off + 1: off + 8])
        wrong = {"all_right": [], "all_wrong": list(range(7)),
                 "alternating": [] if r % 2 == 0 else [0], "cycling": [r % 8] if r % 8 < 7 else []}[mode]
        for j in wrong:
            d[j] = (d[j] + 1) % (TINY.vocab - 1)
        o, recs = ls.step(forced=np.array([d], np.int32), tol=TOL)
        assert recs[0]["n"] == (min(wrong) if wrong else 7)
        stream += recs[0]["committed"]
    assert stream == greedy[:len(stream)]
    ls.close()


def test_small_shape_bf16():
    ls = _lockstep(SMALL_R, 4)
    for _ in range(4):
        ls.step(tol=TOL)
    ls.close()


def test_b32_shape_bf16_ragged():
    ls = _lockstep(B32_R, 3)
    for _ in range(3):
        ls.step(tol=TOL)
    ls.close()


@pytest.mark.parametrize("pairs", ["1", "0"])
def test_b32_shape_gemm_kernel_forms(monkeypatch, pairs):
    """Every projection GEMM with a split operand as CTA pairs (one M = 256 MMA over two
    SMs, each CTA loading one half of the token columns), then never: both kernel forms
    in lock-step, whichever the timing picks."""
    monkeypatch.setenv("DMTP_GEMM_PAIRS", pairs)
    ls = _lockstep(B32_R, 2)
    for _ in range(2):
        ls.step(tol=TOL)
    ls.close()


def test_b32_shape_graph_rounds_ints_only():
    """Rounds without float outputs replay the captured CUDA graph."""
    ls = _lockstep(B32_R, 4, seqs=[0, 5, 31])
    for _ in range(4):
        ls.step(floats=False)
    assert ls.gpu.launches_per_round() > 0
    ls.close()


def test_hybrid_shape_snapshot_swap():
    ls = _lockstep(HYB_R, 6)
    greedy = [_greedy(ls, b, 8 * 6 + 9) for b in range(HYB_R.batch)]
    for r in range(6):
        forced = []
        for b in range(HYB_R.batch):
            off = ls.states[b].a - len(ls.prompts[b])
            d = list(greedy[b][off + 1: off + 8])
            j = (r + b) % 8
            if j < 7:
                d[j] = (d[j] + 1) % (HYB_R.vocab - 1)
            forced.append(d)
        o, recs = ls.step(forced=np.array(forced, np.int32), tol=TOL)
        for b in range(HYB_R.batch):
            assert recs[b]["n"] == min((r + b) % 8, 7)
            assert int(o["snap_slot"][b]) == recs[b]["n"]
    ls.close()


def test_round_host_matches_device_outputs():
    from mtp_block_draft_gb300 import DmtpRound, default_max_ctx
    w = make_weights(B32_R, "cuda")
    prompts = make_prompts(B32_R)
    a = DmtpRound(B32_R, w, prompts, default_max_ctx(prompts, 4))
    b = DmtpRound(B32_R, w, prompts, default_max_ctx(prompts, 4))
    for _ in range(3):
        out = a.alloc_out()
        a.round(out)
        committed = np.zeros((B32_R.batch, 8), np.int32)
        n = np.zeros(B32_R.batch, np.int32)
        b.round_host(committed, n)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out["committed"].cpu().numpy(), committed)
        np.testing.assert_array_equal(out["n_accepted"].cpu().numpy(), n)
    a.close()
    b.close()


def _sampled_stream(ls, b, n):
    return ls.oracle.sampled_decode(ls.prompts[b], n, b=b)


def test_tiny_sampled_natural_rounds():
    """Sampled picks (CUDA-core head) in lock-step with the oracle's scores l / T + G,
    and the committed stream equals plain one-token sampled decoding."""
    ls = _lockstep(TINY_S, 12)
    ref = _sampled_stream(ls, 0, 8 * 12 + 9)
    assert ref != _greedy(ls, 0, len(ref))
    stream = [ls.states[0].A]
    for _ in range(12):
        _, recs = ls.step(tol=TOL)
        stream += recs[0]["committed"]
    if not ls.adopted:   # an adopted near tie may branch off the oracle's own decode
        assert stream == ref[:len(stream)]
    ls.close()


def test_tiny_noise_dominated_picks():
    """At temperature 1000 the logits move the scores by < 1e-3: the picks are the argmax
    of the Gumbel noise alone, so the noise's counter, word and sequence layout must
    match the oracle's generator element for element."""
    ls = _lockstep(TINY_S.replace(temperature=1000.0), 4)
    for _ in range(4):
        ls.step(tol=TOL)
    ls.close()


@pytest.mark.parametrize("wrong", [None, 0, 4, 6])
def test_tiny_sampled_forced(wrong):
    """Drafts forced to the sampled stream are all accepted; one wrong draft at row j
    accepts j and commits the target's sample there; the stream stays the sampled one."""
    ls = _lockstep(TINY_S, 8)
    ref = _sampled_stream(ls, 0, 8 * 8 + 9)
    P = len(ls.prompts[0])
    stream = [ls.states[0].A]
    for _ in range(8):
        off = ls.states[0].a - P
        d = list(ref[off + 1: off + 8])
        if wrong is not None:
            d[wrong] = (d[wrong] + 1) % (TINY.vocab - 1)
        _, recs = ls.step(forced=np.array([d], np.int32), tol=TOL)
        assert recs[0]["n"] == (7 if wrong is None else wrong)
        stream += recs[0]["committed"]
    if not ls.adopted:
        assert stream == ref[:len(stream)]
    ls.close()


def test_b32_shape_sampled_tensor_core_head():
    """Sampled picks from the tcgen05 head's epilogue (quad-shared Philox blocks) over
    256 verify rows and a ragged vocabulary, float outputs within 2e-2."""
    ls = _lockstep(B32_RS, 3)
    for _ in range(3):
        ls.step(tol=TOL)
    ls.close()


def test_b32_shape_sampled_graph_rounds():
    """Captured-graph replays of sampled rounds: the noise follows each round's positions."""
    ls = _lockstep(B32_RS, 4, seqs=[0, 9, 31])
    for _ in range(4):
        ls.step(floats=False)
    ls.close()


def test_hybrid_shape_sampled_with_snapshots():
    """Sampled verification on the hybrid target (Gated DeltaNet snapshots): the noise
    follows each sequence's own positions while the rollback swaps snapshot slots."""
    cfg = HYB_R.replace(name="hybrid_r_sampled", temperature=0.9, sample_seed=4242)
    ls = _lockstep(cfg, 4)
    for _ in range(4):
        ls.step(tol=TOL)
    ls.close()


def test_b32_shape_fp8_draft_heads():
    """T1 and drafter heads on the E4M3 head copy (tcgen05 kind::f8f6f4): drafts and their
    logits against the oracle's quantised heads; the verify head stays bf16."""
    ls = _lockstep(B32_R.replace(name="b32_r_fp8", draft_head_fp8=True), 3)
    for _ in range(3):
        ls.step(tol=TOL)
    ls.close()


def test_fp8_draft_heads_forced_stay_lossless():
    """With quantised draft heads, drafts forced to the greedy stream are all accepted and
    the commit is the plain greedy decode (only the drafts may change)."""
    cfg = B32_R.replace(name="b32_r_fp8", draft_head_fp8=True, batch=2)
    ls = _lockstep(cfg, 4)
    greedy = [_greedy(ls, b, 8 * 4 + 9) for b in range(2)]
    streams = [[ls.states[b].A] for b in range(2)]
    for r in range(4):
        forced = []
        for b in range(2):
            off = ls.states[b].a - len(ls.prompts[b])
            d = list(greedy[b][off + 1: off + 8])
            if r % 2:
                d[3] = (d[3] + 1) % (cfg.vocab - 1)
            forced.append(d)
        o, recs = ls.step(forced=np.array(forced, np.int32), tol=TOL)
        for b in range(2):
            assert recs[b]["n"] == (3 if r % 2 else 7)
            streams[b] += recs[b]["committed"]
    for b in range(2):
        if not ls.adopted:
            assert streams[b] == greedy[b][:len(streams[b])]
    ls.close()


def test_b32_shape_sampled_with_fp8_draft_heads():
    """Sampled verification and E4M3 draft heads together: the drafts come from the
    quantised heads, the verify picks from the bf16 head's sampling epilogue."""
    cfg = B32_RS.replace(name="b32_r_sampled_fp8", draft_head_fp8=True)
    ls = _lockstep(cfg, 2, seqs=[0, 17, 31])
    for _ in range(2):
        ls.step(tol=TOL)
    ls.close()


def test_prefill_stats():
    """dmtp_prefill_stats: the prompt tokens dmtp_init prefilled and a positive device time."""
    from mtp_block_draft_gb300 import DmtpRound, default_max_ctx
    prompts = make_prompts(B32_R)
    g = DmtpRound(B32_R, make_weights(B32_R, "cuda"), prompts, default_max_ctx(prompts, 2))
    ms, tok = g.prefill_stats()
    assert tok == sum(len(p) for p in prompts) and ms > 0
    g.close()


def test_temperature_validation():
    from mtp_block_draft_gb300 import DmtpError, DmtpRound
    w = make_weights(TINY, "cuda")
    for t in (-1.0, 1e-6, float("nan"), float("inf")):
        with pytest.raises(DmtpError):
            DmtpRound(TINY.replace(temperature=t), w, make_prompts(TINY), 256)
    with pytest.raises(DmtpError):  # E4M3 draft heads need a bf16 model
        DmtpRound(TINY.replace(draft_head_fp8=True), w, make_prompts(TINY), 256)


def test_device_timeout_poisons_context():
    """The device failure path with nothing faulted: a bounded wait that nothing satisfies
    (dmtp_selftest_timeout, 50 us) gives up and sets the timeout bit; the host then reports
    DMTP_EDEVICE, every later call DMTP_ESTATE, dmtp_free is clean, and a new context on
    the same device runs rounds normally."""
    from mtp_block_draft_gb300 import DmtpError, DmtpRound, default_max_ctx
    w = make_weights(B32_R, "cuda")
    prompts = make_prompts(B32_R)
    g = DmtpRound(B32_R, w, prompts, default_max_ctx(prompts, 4))
    g.round()
    g.read_state()                                   # clean so far
    with pytest.raises(DmtpError) as e:
        g.selftest_timeout(10)                       # limit below 1 us: rejected
    assert e.value.code == -1
    g.selftest_timeout(50_000)
    with pytest.raises(DmtpError) as e:
        g.read_state()
    assert e.value.code == -5                        # DMTP_EDEVICE
    assert e.value.word == 4                         # the timeout bit, nothing else
    for call in (g.round, g.read_state, g.profile_round, lambda: g.selftest_timeout(50_000)):
        with pytest.raises(DmtpError) as e:
            call()
        assert e.value.code == -6                    # DMTP_ESTATE
    g.close()
    torch.cuda.synchronize()
    g2 = DmtpRound(B32_R, w, prompts, default_max_ctx(prompts, 4))
    out = g2.alloc_out(ints=True)
    g2.round(out)
    kv, _, _ = g2.read_state()
    assert (kv > np.array([len(p) for p in prompts])).all()
    g2.close()


# the draft heads over a token list (colibri frequent-token list): a small batch of short
# prompts, so the list (conversation tokens plus the most counted) is a few hundred of
# the 5000 tokens and most verify picks join it as they are committed
B32_RL = B32_R.replace(name="b32_r_list", batch=4, ctx_lo=40, ctx_hi=80, draft_list_cap=5000)


@pytest.mark.parametrize("fp8", [False, True])
def test_draft_heads_over_token_list(fp8):
    """T1 and T2..T7 are the argmax over the listed tokens (dmtp_set_draft_list), the
    verify still scores every token: lock-step against the oracle's round(draft_list=...)
    with the list kept by the native list (dmtp_vocab.h), joined picks appended each
    round; then the list is turned off and the full heads come back."""
    from lockstep import Lockstep
    from mtp_block_draft_gb300 import DmtpError, DmtpVocabList
    cfg = B32_RL.replace(draft_head_fp8=fp8)
    prompts = make_prompts(cfg)
    ls = Lockstep(cfg, make_weights(cfg, "cuda"), prompts, rounds=8)
    vl = DmtpVocabList(cfg.vocab, 100)
    vl.begin_request(np.concatenate(prompts))
    _, A, _ = ls.gpu.read_state()
    vl.picked(A)
    moved, sizes = 0, []
    for _ in range(6):
        ids, mask = vl.ids(), vl.mask()
        sizes.append(len(ids))
        ls.gpu.set_draft_list(ids)
        o, recs = ls.step(tol=TOL, draft_list=mask)
        for b, rec in recs.items():
            assert all(mask[t] for t in rec["drafts"])
            moved += int(not mask[int(np.argmax(rec["t1_logits"]))])
        vl.picked(np.concatenate([o["committed"][b][:o["n_accepted"][b] + 1]
                                  for b in range(cfg.batch)]))
    assert moved > 0 and sizes[0] < cfg.vocab // 4 and sizes[-1] > sizes[0]
    with pytest.raises(DmtpError) as e:
        ls.gpu.set_draft_list([5, 5, 7])          # not strictly increasing
    assert e.value.code == -1
    with pytest.raises(DmtpError):
        ls.gpu.set_draft_list([cfg.vocab])        # out of range
    ls.gpu.set_draft_list([])                    # off: the full heads again
    ls.step(tol=TOL)
    ls.close()
    vl.close()


def test_draft_list_needs_capacity():
    from mtp_block_draft_gb300 import DmtpError, DmtpRound, default_max_ctx
    prompts = make_prompts(B32_R)
    g = DmtpRound(B32_R, make_weights(B32_R, "cuda"), prompts, default_max_ctx(prompts, 2))
    with pytest.raises(DmtpError) as e:
        g.set_draft_list([1, 2, 3])
    assert e.value.code == -1
    g.close()


# verifies of fewer drafts (colibri draft-depth gate): rounds at depths 0..7
DEPTHS = (7, 3, 0, 5, 1, 6, 2, 4, 0, 7)


def _greedy_next(ls, b, n):
    """The next n tokens of plain greedy decoding from the oracle's state of sequence b."""
    st = ls.states[b].clone()
    out, tok, pos = [], st.A, st.a
    for _ in range(n):
        _, _, logits, _ = ls.oracle.target_rows(st, [tok], pos)
        tok, pos = int(np.argmax(logits[0])), pos + 1
        out.append(tok)
    return out


@pytest.mark.parametrize("name", ["tiny", "b32_r", "hybrid_r"])
def test_variable_depth_rounds(name):
    """dmtp_round_depth at every depth 0..7, natural drafts and drafts forced to the greedy
    continuation with one wrong row, in lock-step with the oracle's round(depth=k): at most
    k drafts accepted, the verify over k + 1 rows, a recurrent target's slot n swapped in
    below depth k and the live state kept at n = k."""
    from lockstep import Lockstep
    base = {"tiny": TINY, "b32_r": B32_R.replace(batch=8), "hybrid_r": HYB_R}[name]
    cfg = base.replace(name=base.name + "_depth", variable_depth=True)
    ls = Lockstep(cfg, make_weights(cfg, "cuda"), make_prompts(cfg), rounds=len(DEPTHS))
    seen = set()
    for r, depth in enumerate(DEPTHS):
        forced = None
        if r % 2 == 1:
            forced = np.array([_greedy_next(ls, b, 7) for b in range(cfg.batch)], np.int32)
            w = (3 * r) % 8
            if w < 7:
                forced[:, w] = (forced[:, w] + 1) % (cfg.vocab - 1)
        o, recs = ls.step(forced=forced, depth=depth, tol=TOL)
        for b, rec in recs.items():
            assert rec["n"] <= depth and int(o["n_accepted"][b]) == rec["n"]
            seen.add((depth, rec["n"]))
    assert any(n == d and d > 0 for d, n in seen)     # a full accept below depth 7
    assert any(0 < n < d for d, n in seen)            # a rejection inside a short verify
    ls.close()


def test_depth_needs_variable_depth_context():
    from mtp_block_draft_gb300 import DmtpError, DmtpRound, default_max_ctx
    prompts = make_prompts(B32_R)
    g = DmtpRound(B32_R, make_weights(B32_R, "cuda"), prompts, default_max_ctx(prompts, 2))
    for depth in (3, -1, 8):
        with pytest.raises(DmtpError) as e:
            g.round(depth=depth)
        assert e.value.code == -1
    g.round(depth=7)
    g.close()


@pytest.mark.parametrize("variant", ["bf16", "fp8", "list"])
def test_draft_confidence(variant):
    """The draft heads' confidence of their own picks (draft_confidence; the colibri
    page's per-step estimate: 1 / sum of exp(l - l_max) over the scores within 20 of the
    best), per draft T1..T7, against the oracle's head_confidence: bf16 heads, E4M3 heads,
    and heads over a token list (the sum over the listed tokens)."""
    from lockstep import Lockstep
    cfg = B32_R.replace(name="b32_r_conf", batch=4, ctx_lo=40, ctx_hi=80, draft_confidence=True,
                        draft_head_fp8=variant == "fp8",
                        draft_list_cap=B32_R.vocab if variant == "list" else 0)
    ls = Lockstep(cfg, make_weights(cfg, "cuda"), make_prompts(cfg), rounds=4)
    mask = None
    if variant == "list":
        ids = np.arange(0, cfg.vocab, 7, dtype=np.int32)  # every 7th token
        mask = np.zeros(cfg.vocab, bool)
        mask[ids] = True
        ls.gpu.set_draft_list(ids)
    for _ in range(3):
        o, recs = ls.step(tol=TOL, draft_list=mask)
        assert (o["draft_conf"] > 0).all() and (o["draft_conf"] <= 1).all()
    ls.close()


def test_rounds_are_bitwise_reproducible():
    """With deterministic = 1, two contexts from the same weights and prompts give
    bitwise-identical rounds: every split GEMM sums its K parts in a fixed order, the
    attention merges its partials in CTA order, and the argmax keys break ties by index,
    so nothing depends on which CTA finishes first."""
    from mtp_block_draft_gb300 import DmtpRound, default_max_ctx
    cfg = B32_R.replace(name="b32_r_det", deterministic=True)
    w = make_weights(cfg, "cuda")
    prompts = make_prompts(cfg)
    outs = []
    for _ in range(2):
        g = DmtpRound(cfg, w, prompts, default_max_ctx(prompts, 4))
        rec = []
        for _ in range(3):
            o = g.alloc_out(ints=True, floats=True)
            g.round(o)
            torch.cuda.synchronize()
            rec.append({k: v.cpu().numpy().copy() for k, v in o.items()})
        g.close()
        outs.append(rec)
    for r0, r1 in zip(*outs):
        for k in r0:
            np.testing.assert_array_equal(r0[k], r1[k], err_msg=k)
