"""Pins of the oracle's E4M3 draft-head quantisation (oracle/fp8.py).

* The E4M3 grid against the format's definition (sign, 4-bit exponent with bias 7,
  3-bit mantissa, subnormals, 448 the largest finite value), and round-to-nearest-even
  against torch's float8_e4m3fn conversion on float32 inputs: random values, every
  midpoint between neighbouring grid values (ties) and the subnormal range.
* Power-of-two row scales: tight (max|row| in (224 s, 448 s]) and exact division.
* Special case that reduces to exact arithmetic: rows already on the scaled E4M3 grid
  give the exact logits.
* The lock-step bound (fp8_logit_bounds): inputs perturbed within delta quantise to
  logits inside it, and it is zero for delta = 0.
* Losslessness with quantised draft heads ([DMTP] §6.5: verification unchanged): the
  committed stream is still plain greedy decoding of the target, naturally and with
  forced drafts, while the draft logits do change.
"""
import numpy as np
import pytest
import torch

from oracle import OracleModel
from oracle.fp8 import (E4M3_MAX, e4m3_grid, fp8_logit_bounds, fp8_logits, pow2_scale,
                        quantize_rows, round_e4m3)
from synth import CONFIGS, make_prompts, make_weights

TINY = CONFIGS["tiny"]


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_grid_matches_format_definition():
    g = e4m3_grid()
    assert g.size == 127 and g[0] == 0.0 and g[-1] == E4M3_MAX == 448.0
    assert g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6           # smallest subnormal, normal
    assert np.all(np.diff(g) > 0)
    # every non-negative finite float8_e4m3fn bit pattern decodes to the same set
    codes = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn)
    np.testing.assert_array_equal(codes.to(torch.float64).numpy(), g)


def test_rounding_matches_torch():
    rng = np.random.default_rng(0)
    g = e4m3_grid()
    mids = (g[1:] + g[:-1]) / 2                               # exact ties in float32
    x = np.concatenate([
        rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 5000), mids, -mids, g, -g,
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1000))]).astype(np.float32)
    np.testing.assert_array_equal(round_e4m3(x.astype(np.float64)), _torch_e4m3(x))


def test_pow2_scales_tight_and_exact():
    rng = np.random.default_rng(1)
    for amax in np.concatenate([rng.uniform(1e-6, 1e4, 200), [448.0, 224.0, 448.0 * 2 ** -20,
                                                                1.0, 0.0]]):
        s = pow2_scale(amax)
        assert np.log2(s) == round(np.log2(s))
        if amax > 0:
            assert 224.0 * s < amax <= 448.0 * s
    X = rng.normal(0, 0.02, (8, 256))
    q, s = quantize_rows(X)
    assert np.all(np.abs(q).max(axis=1) <= 448.0)
    # relative error of E4M3 rounding: at most 2^-4 of the value for normals
    err = np.abs(q * s[:, None] - X)
    assert np.all(err <= np.maximum(np.abs(X) * 2.0 ** -4, s[:, None] * 2.0 ** -10))


def test_on_grid_rows_give_exact_logits():
    rng = np.random.default_rng(2)
    g = e4m3_grid()
    # rows whose largest magnitude is 448 * 2^e, other entries E4M3 values times 2^e
    H = rng.choice(np.concatenate([g, -g]), (50, 64)) * 2.0 ** -12
    H[:, 0] = 448.0 * 2.0 ** -12
    Y = rng.choice(np.concatenate([g, -g]), (3, 64)) * 2.0 ** -7
    Y[:, 5] = -448.0 * 2.0 ** -7
    Hq, Hs = quantize_rows(H)
    np.testing.assert_array_equal(fp8_logits(Y, Hq, Hs), Y @ H.T)


def test_logit_bounds_cover_perturbed_inputs():
    """Rows perturbed by at most delta per element quantise to logits within the bound;
    with delta = 0 the bound is zero."""
    rng = np.random.default_rng(3)
    H = rng.normal(0, 0.02, (300, 128))
    Hq, Hs = quantize_rows(H)
    Y = rng.normal(0, 1, (6, 128))
    Y[0, 7] = 448.0 * 2.0 ** -7 * 0.9999        # near a scale boundary
    l0, w0 = fp8_logit_bounds(Y, Hq, Hs, 0.0)
    np.testing.assert_array_equal(w0, 0.0)
    np.testing.assert_array_equal(l0, fp8_logits(Y, Hq, Hs))
    delta = 1e-2
    logits, width = fp8_logit_bounds(Y, Hq, Hs, delta)
    worst = 0.0
    for _ in range(200):
        Yp = Y + rng.uniform(-delta, delta, Y.shape)
        d = np.abs(fp8_logits(Yp, Hq, Hs) - logits)
        assert np.all(d <= width + 1e-12)
        worst = max(worst, float((d / np.maximum(width, 1e-30)).max()))
    assert worst > 0.05     # the bound is not vacuous


@pytest.fixture(scope="module")
def models():
    w = make_weights(TINY.replace(fusion_std=0.02), "cpu")
    return OracleModel(TINY, w), OracleModel(TINY, w, draft_head_fp8=True)


def test_quantised_draft_heads_stay_lossless(models):
    exact, q = models
    prompt = make_prompts(TINY)[0]
    greedy = exact.greedy_decode(prompt, 8 * 8 + 9)
    st = q.prefill(prompt)
    stream = [st.A]
    differs = False
    st_e = exact.prefill(prompt)
    for _ in range(8):
        rec = q.round(st)
        rec_e = exact.round(st_e)
        differs |= not np.array_equal(rec["t1_logits"], rec_e["t1_logits"])
        stream += rec["committed"]
    assert stream == greedy[:len(stream)]
    assert differs
    # forced drafts right and wrong: the quantised heads never reach the commit
    st = q.prefill(prompt)
    stream = [st.A]
    for r in range(5):
        k = len(stream) - 1
        d = list(greedy[k + 1:k + 8])
        if r % 2:
            d[2] = (d[2] + 1) % (TINY.vocab - 1)
        rec = q.round(st, forced=d)
        assert rec["n"] == (2 if r % 2 else 7)
        stream += rec["committed"]
    assert stream == greedy[:len(stream)]
