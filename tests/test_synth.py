"""The seeded synthetic inputs follow their stated recipe (no GPU): prompt lengths and id
ranges, the copied-span and repeated-chunk structures, determinism, and weights that are
N(0, std) draws stored in the workload's type with unit norm gains."""
import numpy as np
import pytest
import torch

from synth import CONFIGS, make_prompts, make_weights
from synth.gen import weight_specs


@pytest.mark.parametrize("name", list(CONFIGS))
def test_prompt_lengths_ids_and_determinism(name):
    cfg = CONFIGS[name]
    ps = make_prompts(cfg)
    assert len(ps) == cfg.batch
    for p in ps:
        assert p.dtype == np.int32
        assert cfg.ctx_lo <= len(p) <= cfg.ctx_hi
        assert p.min() >= 0 and p.max() <= cfg.vocab - 2         # the MASK id never appears
    again = make_prompts(cfg)
    assert all(np.array_equal(a, b) for a, b in zip(ps, again))


def test_b32_lengths_vary_over_the_range():
    cfg = CONFIGS["b32"]
    lens = np.array([len(p) for p in make_prompts(cfg)])
    assert lens.min() < 1500 and lens.max() > 3000 and len(set(lens)) > 25


def test_small_prompt_ends_with_a_copied_span():
    cfg = CONFIGS["small"]
    (p,) = make_prompts(cfg)
    tail = p[-256:]
    hits = [s for s in range(0, 1536) if np.array_equal(p[s:s + 256], tail)]
    assert hits, "the last 256 ids copy an earlier span"


def test_long_prompts_repeat_earlier_chunks():
    cfg = CONFIGS["long"]
    copies = 0
    for p in make_prompts(cfg):
        ch = p.reshape(-1, 1024)
        for i in range(1, ch.shape[0]):
            copies += any(np.array_equal(ch[i], ch[j]) for j in range(i))
    total = cfg.batch * (cfg.ctx_lo // 1024 - 1)
    assert 0.3 * total < copies < 0.7 * total                     # each with probability 1/2


def test_weights_recipe():
    cfg = CONFIGS["b32"].replace(name="b32_shape", vocab=640, d_model=128, n_layers=2,
                                 n_heads=4, n_kv_heads=2, head_dim=32, ffn=256)
    w = make_weights(cfg, "cpu")
    assert set(w) == {n for n, _, _ in weight_specs(cfg)}
    for name, shape, kind in weight_specs(cfg):
        t = w[name]
        assert tuple(t.shape) == shape and t.dtype == torch.bfloat16
        if kind == "g":
            assert torch.all(t == 1)
        else:
            x = t.float()
            std = cfg.weight_std if kind == "w" else cfg.fusion_std
            if x.numel() > 4000:
                assert abs(x.std().item() - std) < 0.1 * std and abs(x.mean().item()) < 0.1 * std
    w2 = make_weights(cfg, "cpu")
    assert all(torch.equal(w[k], w2[k]) for k in w)
    tiny = make_weights(CONFIGS["tiny"], "cpu")                  # fp32, zero-init fusion W
    assert tiny["emb"].dtype == torch.float32 and torch.all(tiny["fuse.w"] == 0)
    assert torch.all(make_weights(CONFIGS["tiny"], "cpu", fusion_std=0.02)["fuse.w"] != 0)
