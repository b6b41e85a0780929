"""Pins of the oracle's model primitives and metrics against library routines,
closed forms and the page's printed acceptance table (no GPU)."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import dmtp_oracle as O

RNG = np.random.default_rng(1234)


def test_rms_norm_matches_torch():
    x = RNG.standard_normal((5, 7, 48))
    g = RNG.standard_normal(48)
    ref = Fnn.rms_norm(torch.from_numpy(x), (48,), weight=torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(O.rms_norm(x, g, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-13)


def test_silu_sigmoid_l2norm_match_torch():
    x = RNG.standard_normal((3, 64)) * 4
    t = torch.from_numpy(x)
    np.testing.assert_allclose(O.silu(x), Fnn.silu(t).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.sigmoid(x), torch.sigmoid(t).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.l2_normalize(x), Fnn.normalize(t, dim=-1).numpy(), rtol=1e-13)


def test_rope_closed_forms():
    # position 0 is the identity
    x = RNG.standard_normal((3, 2, 8))
    np.testing.assert_array_equal(O.rope(x, 0, 1e4), x)
    # hd = 4, base 1e4: pair 0 turns by pos rad, pair 1 by pos * 1e4^(-1/2) = pos/100
    e0 = np.zeros((1, 4)); e0[0, 0] = 1.0
    r = O.rope(e0, 1.0, 1e4)
    np.testing.assert_allclose(r[0], [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    e1 = np.zeros((1, 4)); e1[0, 1] = 1.0
    r = O.rope(e1, 100.0, 1e4)
    np.testing.assert_allclose(r[0], [0, math.cos(1), 0, math.sin(1)], atol=1e-12)


def test_rope_is_complex_rotation_and_relative():
    hd, half = 64, 32
    x = RNG.standard_normal((6, 4, hd))
    pos = np.arange(6) * 37 + 5
    out = O.rope(x, pos, 1e4)
    # as a complex number z_i = x_i + i x_{i+half}, rope multiplies by e^{i pos w_i}
    z = torch.complex(torch.from_numpy(x[..., :half]), torch.from_numpy(x[..., half:]))
    zo = torch.complex(torch.from_numpy(out[..., :half]), torch.from_numpy(out[..., half:]))
    ratio = (zo / z).numpy()
    np.testing.assert_allclose(np.abs(ratio), 1.0, atol=1e-12)   # a pure rotation
    ang = np.angle(ratio)                                         # = pos * w_i (mod 2pi)
    w = np.angle(np.exp(1j * (ang[1] - ang[0]) / 1))              # step of 37 positions
    # the rotation angle is linear in position: angle(pos=5+37k) - angle(pos=5) = 37k w
    for k in range(2, 6):
        d = np.angle(np.exp(1j * (ang[k] - ang[0])))
        np.testing.assert_allclose(np.exp(1j * d), np.exp(1j * k * w), atol=1e-9)
    # dot products depend only on the position difference
    q = RNG.standard_normal((1, 1, hd)); k = RNG.standard_normal((1, 1, hd))
    d1 = np.sum(O.rope(q, 100, 1e4) * O.rope(k, 90, 1e4))
    d2 = np.sum(O.rope(q, 1010, 1e4) * O.rope(k, 1000, 1e4))
    assert abs(d1 - d2) < 1e-10


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 4)])
def test_attention_matches_torch_sdpa(hq, hkv):
    R, T0, hd = 8, 21, 16
    T = T0 + R
    q = RNG.standard_normal((R, hq, hd))
    K = RNG.standard_normal((T, hkv, hd))
    V = RNG.standard_normal((T, hkv, hd))
    hi = T0 + np.arange(R)
    out = O.attend_rows(q, K, V, hi=hi)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]               # [1, hq, R, hd]
    Kt = torch.from_numpy(K).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    Vt = torch.from_numpy(V).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    mask = torch.from_numpy(np.arange(T)[None, :] <= hi[:, None])
    ref = Fnn.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    # a lower bound on visible keys (the drafter window) equals slicing the keys
    out_lo = O.attend_rows(q, K, V, hi=hi, lo=5)
    np.testing.assert_allclose(out_lo, O.attend_rows(q, K[5:], V[5:], hi=hi - 5), atol=1e-13)


def test_gdn_closed_forms():
    H, dk, dv = 3, 8, 6
    S = RNG.standard_normal((H, dv, dk))
    q = O.l2_normalize(RNG.standard_normal((H, dk)))
    k = O.l2_normalize(RNG.standard_normal((H, dk)))
    v = RNG.standard_normal((H, dv))
    al = np.array([0.3, 0.7, 0.9])
    # beta = 0: pure decay
    S1, o1 = O.gdn_step(S, q, k, v, al, np.zeros(H))
    np.testing.assert_allclose(S1, al[:, None, None] * S, atol=1e-14)
    np.testing.assert_allclose(o1, np.einsum("hvk,hk->hv", al[:, None, None] * S, q), atol=1e-14)
    # alpha = beta = 1 with unit k: the delta rule writes v at key k exactly
    S2, _ = O.gdn_step(S, q, k, v, np.ones(H), np.ones(H))
    np.testing.assert_allclose(np.einsum("hvk,hk->hv", S2, k), v, atol=1e-13)
    # general case against the matrix form alpha S (I - beta k k^T) + beta v k^T (torch)
    be = np.array([0.2, 0.5, 0.8])
    S3, o3 = O.gdn_step(S, q, k, v, al, be)
    St, kt, vt, qt = map(torch.from_numpy, (S, k, v, q))
    for h in range(H):
        I = torch.eye(dk, dtype=torch.float64)
        ref = al[h] * St[h] @ (I - be[h] * torch.outer(kt[h], kt[h])) + be[h] * torch.outer(vt[h], kt[h])
        np.testing.assert_allclose(S3[h], ref.numpy(), atol=1e-13)
        np.testing.assert_allclose(o3[h], (ref @ qt[h]).numpy(), atol=1e-13)


def test_argmax_tie_and_gap():
    x = np.array([0.1, 0.5, 0.2, 0.5])
    assert O.argmax_first(x) == 1
    assert O.top2_gap(x) == 0.0
    assert abs(O.top2_gap(np.array([1.0, 0.25, 0.5])) - 0.5) < 1e-15


def test_accept_metrics_hand_histograms():
    assert O.mean_accept_len([10, 0, 0, 0, 0, 0, 0, 0]) == 1.0
    assert O.mean_accept_len([0, 0, 0, 0, 0, 0, 0, 5]) == 8.0
    assert abs(O.mean_accept_len([1, 1, 0, 0, 0, 0, 0, 2]) - (1 + 15 / 4)) < 1e-15
    assert O.first_candidate_acceptance([3, 1, 0, 0, 0, 0, 0, 0]) == 0.25


def _read_golden(name):
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        rows.append((parts[0], [float(p) / 100 for p in parts[1:8]], float(parts[8])))
    return rows


def test_accept_metrics_vs_printed_table():
    """Histogram implied by the page's conditional rates: hist[k] = P(exactly k accepted).
    Its per-verify mean must match the printed mean length loosely (different runs),
    and its first-candidate acceptance must equal the printed T1 rate exactly."""
    for name, p, printed in _read_golden("dmtp_conditional_acceptance.txt"):
        surv = np.cumprod(p)                       # P(L >= k), k = 1..7
        hist = np.empty(8)
        hist[0] = 1 - p[0]
        for k in range(1, 7):
            hist[k] = surv[k - 1] * (1 - p[k])
        hist[7] = surv[6]
        assert abs(hist.sum() - 1) < 1e-12
        assert abs(O.first_candidate_acceptance(hist) - p[0]) < 1e-12
        m = O.mean_accept_len(hist)
        assert abs(m - (1 + surv.sum())) < 1e-12
        assert abs(m - printed) / printed < 0.02, (name, m, printed)
