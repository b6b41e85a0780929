"""GPU check of dmtp_t1_head_noalloc, the first-candidate head for callers that may
not allocate device memory (engines with their own fixed pool, or paths that cannot
afford an allocation's device synchronisation).

It must give what step a1 of dmtp_round gives: run rounds with debug outputs, feed
each round's starting h_MTP to the no-alloc entry point, and compare the picked ids
(exactly, on rows whose top-1 minus top-2 logit gap exceeds the suite's 0.05 near-tie
gate: the round may time another head tile shape, whose rounding can flip a near tie)
and the logits (within the suite's 2e-2) - two calls in a row, so the shared scratch
array is reused. Sizes past the documented maximum are rejected.
This file sorts last so that a run stopping at the first failure has run the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import CONFIGS, make_prompts, make_weights

pytestmark = pytest.mark.gpu

# 32 rows = the maximum rows per call; bf16 model with a ragged vocabulary tail
CFG = CONFIGS["b32"].replace(name="b32_noalloc", vocab=5000, d_model=256, n_layers=2,
                             n_heads=8, n_kv_heads=2, head_dim=64, ffn=512, ctx_lo=40,
                             ctx_hi=120)


def _clear_rows(logits):
    """Rows whose top-1 minus top-2 logit exceeds the near-tie gate (0.05)."""
    top2 = np.sort(logits, axis=1)[:, -2:]
    return (top2[:, 1] - top2[:, 0]) > 0.05


def _call(lib, w, h, rows, ids, logits, stream):
    return lib.dmtp_t1_head_noalloc(
        ctypes.c_void_p(w["head"].data_ptr()), ctypes.c_void_p(w["mtp.final_norm"].data_ptr()),
        ctypes.c_void_p(h.data_ptr()), rows, CFG.vocab, CFG.d_model, CFG.rms_eps,
        ctypes.c_void_p(ids.data_ptr()),
        ctypes.c_void_p(logits.data_ptr()) if logits is not None else None,
        ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_head_matches_round_a1():
    from mtp_block_draft_gb300 import DmtpRound, default_max_ctx, load_library
    lib = load_library()
    w = make_weights(CFG, "cuda")
    prompts = make_prompts(CFG)
    g = DmtpRound(CFG, w, prompts, default_max_ctx(prompts, 4))
    B, V = CFG.batch, CFG.vocab
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = g.alloc_out(ints=True, floats=True)
        g.round(out)
        ids = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        logits = torch.zeros((B, V), dtype=torch.float32, device="cuda")
        assert _call(lib, w, out["h_mtp"], B, ids, logits, stream) == 0
        torch.cuda.synchronize()
        clear = _clear_rows(out["t1_logits"].cpu().numpy())
        assert clear.sum() >= B // 4
        np.testing.assert_array_equal(ids.cpu().numpy()[clear],
                                      out["drafts"][:, 0].cpu().numpy()[clear])
        err = (logits - out["t1_logits"]).abs().max().item()
        assert err <= 2e-2, err
    # without logits, on a subset of rows
    ids = torch.full((5,), -7, dtype=torch.int32, device="cuda")
    assert _call(lib, w, out["h_mtp"], 5, ids, None, stream) == 0
    torch.cuda.synchronize()
    clear = _clear_rows(out["t1_logits"].cpu().numpy())[:5]
    np.testing.assert_array_equal(ids.cpu().numpy()[clear],
                                  out["drafts"][:5, 0].cpu().numpy()[clear])
    g.close()


def test_noalloc_rejects_sizes_past_the_maximum():
    from mtp_block_draft_gb300 import load_library
    lib = load_library()
    w = make_weights(CFG, "cuda")
    h = torch.zeros((64, CFG.d_model), dtype=torch.float32, device="cuda")
    ids = torch.zeros(64, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    assert _call(lib, w, h, 33, ids, None, stream) == -1      # rows > 32
    assert _call(lib, w, h, 0, ids, None, stream) == -1
