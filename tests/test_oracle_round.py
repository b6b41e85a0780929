"""Pins of the oracle's DMTP round on the tiny configuration (no GPU).

What pins what:
* losslessness: the committed stream equals plain greedy decoding, natural and forced;
* accepted length = matched prefix + 1 for a mismatch forced at every row;
* watermarks follow kv_len' = kv_len + n + 1, mtp_len = kv_len + 1;
* W = 0 reduces the drafter input to [E(A), E(T1), E(MASK) x 6]; Δ is linear in W;
* special matrices: fusion W = [I 0] / [0 I], MTP projection [I 0] / [0 I] with an
  identity block, drafter with identity layers;
* block == chain for verify rows; causality; drafter block bidirectionality and window;
* Gated DeltaNet: snapshot swap == replay of the accepted rows; losslessness.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import OracleModel
from oracle import dmtp_oracle as O
from synth import CONFIGS, make_prompts, make_weights

TINY = CONFIGS["tiny"]
HYB = TINY.replace(name="tiny_hybrid", n_layers=4, layer_kinds=(1, 1, 1, 0),
                   gdn_heads=4, gdn_dk=16, gdn_dv=16)


def _model(cfg=TINY, fusion_std=None, **over):
    w = make_weights(cfg, "cpu", fusion_std=fusion_std)
    for k, v in over.items():
        w[k] = v
    return OracleModel(cfg, w)


def _run(model, prompt, rounds, forced_fn=None):
    st = model.prefill(prompt)
    stream = [st.A]
    recs = []
    for r in range(rounds):
        forced = forced_fn(r, st) if forced_fn else None
        rec = model.round(st, forced=forced)
        stream += rec["committed"]
        recs.append(rec)
    return st, stream, recs


@pytest.fixture(scope="module")
def tiny():
    return _model()


@pytest.fixture(scope="module")
def prompt():
    return make_prompts(TINY)[0]


@pytest.fixture(scope="module")
def greedy(tiny, prompt):
    return tiny.greedy_decode(prompt, 16 * 8 + 1)


def test_lossless_natural(tiny, prompt, greedy):
    st, stream, recs = _run(tiny, prompt, 16)
    assert stream == greedy[:len(stream)]
    assert st.tokens == list(prompt) + stream


def test_lossless_with_fusion_weights(prompt, greedy):
    m = _model(fusion_std=0.02)
    _, stream, recs = _run(m, prompt, 8)
    assert stream == greedy[:len(stream)]
    assert any(np.abs(r["delta"]).max() > 0 for r in recs)


def _forced_from_greedy(greedy, prompt_len, wrong_rows):
    """Drafts = the plain-greedy continuation, except rows in wrong_rows(r) get a
    different id."""
    def fn(r, st):
        off = st.a - prompt_len              # stream index of A is 0 -> st.a - P
        d = list(greedy[off + 1: off + 8])
        for j in wrong_rows(r):
            d[j] = (d[j] + 1) % (TINY.vocab - 1)
        return d
    return fn


@pytest.mark.parametrize("mode", ["all_right", "all_wrong", "alternating", "cycling"])
def test_lossless_forced_modes(tiny, prompt, greedy, mode):
    wrong = {"all_right": lambda r: [],
             "all_wrong": lambda r: list(range(7)),
             "alternating": lambda r: [] if r % 2 == 0 else [0],
             "cycling": lambda r: [r % 7]}[mode]
    long_greedy = tiny.greedy_decode(prompt, 8 * 8 + 9)
    fn = _forced_from_greedy(long_greedy, len(prompt), wrong)
    _, stream, recs = _run(tiny, prompt, 8, fn)
    assert stream == long_greedy[:len(stream)]
    for r, rec in enumerate(recs):
        w = wrong(r)
        assert rec["n"] == (min(w) if w else 7)


def test_accept_len_each_row(tiny, prompt):
    long_greedy = tiny.greedy_decode(prompt, 20)
    for r in range(8):
        st = tiny.prefill(prompt)
        d = list(long_greedy[1:8])
        if r < 7:
            d[r] = (d[r] + 3) % (TINY.vocab - 1)
        rec = tiny.round(st, forced=d)
        assert rec["n"] == r
        assert rec["accept_len"] == r + 1
        assert rec["committed"] == long_greedy[1:1 + r] + [long_greedy[1 + r]]
        assert rec["kv_len"] == len(prompt) + r + 1
        assert rec["mtp_len"] == rec["kv_len"] + 1
        assert st.A == long_greedy[1 + r]


def test_watermarks_closed_form(tiny, prompt):
    st = tiny.prefill(prompt)
    kv = len(prompt)
    for r in range(6):
        rec = tiny.round(st)
        kv += rec["n"] + 1
        assert st.a == kv == rec["kv_len"]
        assert st.mtp_K.shape[0] == kv                  # MTP rows for positions 1..kv
        assert st.dft_K[0].shape[0] == kv
        assert all(k.shape[0] == kv for k in st.tgt_K)


def test_w_zero_reduction(tiny, prompt):
    """W = 0 => Δ = 0 and the drafts are those of plain block drafting over
    [E(A), E(T1), E(MASK) x 6] with T1 = argmax of the MTP head."""
    st = tiny.prefill(prompt)
    for _ in range(3):
        pre = st.clone()
        rec = tiny.round(st)
        assert np.all(rec["delta"] == 0)
        E = tiny.W["emb"]
        T1 = int(np.argmax(tiny.t1_head(pre.h_mtp)))
        X = np.stack([E[pre.A], E[T1]] + [E[TINY.mask_id]] * 6)
        np.testing.assert_array_equal(rec["slots"], X)          # [E(A), E(T1), E(MASK) x 6]
        dl = tiny.drafter_forward(X, pre, pre.a)
        np.testing.assert_array_equal(rec["draft_logits"], dl)
        assert rec["drafts"] == [T1] + [int(np.argmax(r)) for r in dl]


def test_fusion_linear_in_w():
    m1 = _model(fusion_std=0.02)
    w2 = make_weights(TINY, "cpu", fusion_std=0.02)
    w2["fuse.w"] = w2["fuse.w"] * 2
    m2 = OracleModel(TINY, w2)
    h = np.random.default_rng(3).standard_normal(TINY.d_model)
    d1, d2 = m1.fusion_delta(17, h), m2.fusion_delta(17, h)
    np.testing.assert_allclose(d2, 2 * d1, rtol=1e-12, atol=1e-15)


def test_fusion_concat_order():
    """Δ = W [RMS_e(e_T1); RMS_m(h)]: W = [I 0] gives RMS(e_T1), W = [0 I] gives RMS(h)."""
    d = TINY.d_model
    I, Z = torch.eye(d), torch.zeros(d, d)
    h = np.random.default_rng(4).standard_normal(d)
    for W, which in [(torch.cat([I, Z], 1), "e"), (torch.cat([Z, I], 1), "m")]:
        m = _model(**{"fuse.w": W})
        got = m.fusion_delta(33, h)
        src = m.W["emb"][33] if which == "e" else h
        ref = Fnn.rms_norm(torch.from_numpy(src), (d,), eps=TINY.rms_eps).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def _identity_mtp_block():
    d = TINY.d_model
    return {"mtp.wo": torch.zeros(d, TINY.q_dim), "mtp.wdown": torch.zeros(d, TINY.ffn)}


def test_mtp_uses_previous_target_hidden(prompt):
    """Projection [I 0] and an identity block make h_MTP = RMS(h^T_{a-1}); the head
    then reproduces the target's own pick at a-1, i.e. T1 == A every round."""
    d = TINY.d_model
    over = _identity_mtp_block()
    over["mtp.proj"] = torch.cat([torch.eye(d), torch.zeros(d, d)], 1)
    m = _model(**over)
    st = m.prefill(prompt)
    for _ in range(5):
        A = st.A
        rec = m.round(st)
        assert rec["T1"] == A


def test_mtp_uses_embedding_of_pending_token(prompt):
    """Projection [0 I] and an identity block: T1 = argmax H E(A) (positive scale)."""
    d = TINY.d_model
    over = _identity_mtp_block()
    over["mtp.proj"] = torch.cat([torch.zeros(d, d), torch.eye(d)], 1)
    m = _model(**over)
    st = m.prefill(prompt)
    for _ in range(5):
        A = st.A
        rec = m.round(st)
        assert rec["T1"] == int(np.argmax(m.W["head"] @ m.W["emb"][A]))


def test_identity_drafter_predicts_mask_continuation(prompt):
    """Identity drafter layers: every MASK slot's pick is argmax H RMS(E(MASK))."""
    over = {}
    for j in range(TINY.draft_layers):
        over[f"D{j}.wo"] = torch.zeros(TINY.d_model, TINY.q_dim)
        over[f"D{j}.wdown"] = torch.zeros(TINY.d_model, TINY.ffn)
    m = _model(**over)
    st = m.prefill(prompt)
    rec = m.round(st)
    want = int(np.argmax(m.W["head"] @ m.W["emb"][TINY.mask_id]))
    assert rec["drafts"][1:] == [want] * 6


def test_block_equals_chain(tiny, prompt):
    """Verify rows (one-row routine) == one causal block forward of 8 rows."""
    st = tiny.prefill(prompt)
    pre = st.clone()
    rec = tiny.round(st)
    rows = [pre.A] + rec["drafts"]
    _, _, block_logits, _ = tiny.target_rows(pre.clone(), rows, pre.a)
    np.testing.assert_allclose(rec["verify_logits"], block_logits, rtol=1e-10, atol=1e-10)


def test_verify_is_causal(tiny, prompt):
    st0 = tiny.prefill(prompt)
    base = [5, 6, 7, 8, 9, 10, 11]
    r1 = tiny.round(st0.clone(), forced=base)
    for s in range(1, 7):
        alt = list(base)
        alt[s] = 100 + s
        r2 = tiny.round(st0.clone(), forced=alt)
        # row s+1 reads T_{s+1} = alt[s]; rows 0..s are unchanged bit for bit
        np.testing.assert_array_equal(r1["verify_logits"][:s + 1], r2["verify_logits"][:s + 1])
        assert np.abs(r1["verify_logits"][s + 1] - r2["verify_logits"][s + 1]).max() > 0


def test_drafter_block_is_bidirectional(tiny, prompt):
    st = tiny.prefill(prompt)
    E = tiny.W["emb"]
    X = np.stack([E[st.A], E[3]] + [E[TINY.mask_id]] * 6)
    X2 = X.copy()
    X2[7] = E[4]
    d1 = tiny.drafter_forward(X, st, st.a)
    d2 = tiny.drafter_forward(X2, st, st.a)
    assert np.abs(d1[0] - d2[0]).max() > 1e-6        # slot 2 sees slot 7


def test_drafter_window():
    cfg = TINY.replace(draft_window=16)
    m = OracleModel(cfg, make_weights(cfg, "cpu"))
    st = m.prefill(make_prompts(cfg)[0])
    a = st.a
    X = np.stack([m.W["emb"][st.A], m.W["emb"][3]] + [m.W["emb"][cfg.mask_id]] * 6)
    base = m.drafter_forward(X, st, a)
    s2 = st.clone()
    for j in range(cfg.draft_layers):
        s2.dft_K[j][:a - 16] += 5.0
        s2.dft_V[j][:a - 16] -= 3.0
    np.testing.assert_array_equal(m.drafter_forward(X, s2, a), base)
    s3 = st.clone()
    s3.dft_V[0][a - 16] += 3.0
    assert np.abs(m.drafter_forward(X, s3, a) - base).max() > 0


def test_prefill_matches_one_row_steps(tiny, prompt):
    a = tiny.prefill(prompt)
    st = tiny.empty_state()
    for p, t in enumerate(prompt):
        tiny.target_rows(st, [t], p, head=False)
    for l in range(TINY.n_layers):
        np.testing.assert_allclose(a.tgt_K[l], st.tgt_K[l], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(a.tgt_V[l], st.tgt_V[l], rtol=1e-11, atol=1e-12)


def _assert_same_state(a, b, tol=1e-10):
    """Two sequence states agree: positions, pending token, every cache and h_MTP."""
    assert a.a == b.a and a.A == b.A
    pairs = [(a.mtp_K, b.mtp_K), (a.mtp_V, b.mtp_V), (a.h_mtp, b.h_mtp)]
    pairs += list(zip(a.dft_K, b.dft_K)) + list(zip(a.dft_V, b.dft_V))
    for x, y in zip(a.tgt_K + a.tgt_V + a.gdn_S, b.tgt_K + b.tgt_V + b.gdn_S):
        assert (x is None) == (y is None)
        if x is not None:
            pairs.append((x, y))
    for x, y in pairs:
        assert x.shape == y.shape
        np.testing.assert_allclose(x, y, rtol=0, atol=tol)


def test_prefill_in_blocks_matches_one_block(tiny, prompt):
    """Prefill in row blocks (any block size) builds the state a single block builds:
    causal rows see only earlier positions, so splitting the rows changes no value."""
    one = tiny.prefill(prompt)
    w = make_weights(TINY, "cpu")
    for chunk in (1, 5, 16):
        _assert_same_state(OracleModel(TINY, w, chunk=chunk).prefill(prompt), one, 1e-12)
    st = tiny.empty_state()
    for p, t in enumerate(prompt):
        tiny.target_rows(st, [t], p, head=False)
    for l in range(TINY.n_layers):
        np.testing.assert_allclose(one.tgt_K[l], st.tgt_K[l], rtol=0, atol=1e-12)


def _advance_rounds(m, prompt, greedy, rounds):
    """Rounds with natural drafts and with drafts forced from the greedy stream with one
    wrong row (every accepted length 0..7 occurs)."""
    st = m.prefill(prompt)
    for r in range(rounds):
        if r % 3 == 0:
            m.round(st)
            continue
        off = st.a - len(prompt)
        d = list(greedy[off + 1: off + 8])
        wrong = (r * 5) % 8
        if wrong < 7:
            d[wrong] = (d[wrong] + 1) % (m.cfg.vocab - 1)
        m.round(st, forced=d)
    return st


@pytest.mark.parametrize("which", ["tiny", "tiny_hybrid"])
def test_state_advance_equals_prefill(which):
    """[DMTP] §6.1 and §6.3: the rounds advance the target KV (or recurrent state), the
    drafter's context K/V, the MTP KV and h_MTP to exactly the state a prefill of the
    prompt followed by the committed stream (the pending token A excluded) builds."""
    cfg = TINY if which == "tiny" else HYB
    m = OracleModel(cfg, make_weights(cfg, "cpu"))
    prompt = make_prompts(cfg)[0][:40]
    greedy = m.greedy_decode(prompt, 12 * 8 + 2)
    st = _advance_rounds(m, prompt, greedy, 12)
    assert st.tokens == list(prompt) + greedy[:len(st.tokens) - len(prompt)]
    ref = m.prefill(st.tokens[:-1])
    _assert_same_state(st, ref)


@pytest.fixture(scope="module")
def hyb():
    return OracleModel(HYB, make_weights(HYB, "cpu"))


def test_hybrid_lossless_and_swap_equals_replay(hyb):
    prompt = make_prompts(HYB)[0][:40]
    greedy = hyb.greedy_decode(prompt, 60)
    st = hyb.prefill(prompt)
    stream = [st.A]
    for r in range(6):
        off = st.a - len(prompt)
        d = list(greedy[off + 1: off + 8])
        wrong = r % 8
        if wrong < 7:
            d[wrong] = (d[wrong] + 1) % (HYB.vocab - 1)
        pre = st.clone()
        rec = hyb.round(st, forced=d)
        assert rec["n"] == min(wrong, 7) and rec["snap_slot"] == rec["n"]
        stream += rec["committed"]
        # replay rows 0..n from the pre-round state: same GDN state, same KV
        rp = pre.clone()
        for s_, t in enumerate(([pre.A] + d)[:rec["n"] + 1]):
            hyb.target_rows(rp, [t], pre.a + s_, head=False)
        for l, kind in enumerate(HYB.layer_kinds):
            if kind:
                np.testing.assert_array_equal(st.gdn_S[l], rp.gdn_S[l])
            else:
                np.testing.assert_array_equal(st.tgt_K[l], rp.tgt_K[l])
    assert stream == greedy[:len(stream)]


def test_bf16_kv_storage_keeps_the_pins(prompt):
    """With K/V stored as bf16 the caches hold bf16 values only, and the committed
    stream still equals plain greedy decoding of the same (bf16-KV) model."""
    w = make_weights(TINY, "cpu")
    m = OracleModel(TINY, w, kv_store="bf16")
    greedy = m.greedy_decode(prompt, 40)
    _, stream, _ = _run(m, prompt, 5)
    assert stream == greedy[:len(stream)]
    st = m.prefill(prompt)
    m.round(st)
    for arr in [st.tgt_K[0], st.tgt_V[1], st.dft_K[0], st.mtp_V]:
        np.testing.assert_array_equal(arr, O.round_bf16(arr))
    # and the rounding is not a no-op: the exact model's caches differ
    st2 = OracleModel(TINY, w).prefill(prompt)
    assert np.abs(st2.tgt_K[0] - st.tgt_K[0][:st2.a]).max() > 0
