"""The five workloads of the DMTP round, as model dimensions and input recipes.

Dimensions and recipes follow the workloads the DMTP blog ("DMTP: A Better First
Token for Block Drafting via MTP") evaluates: a seven-candidate block (§2, §5),
a 4096-position drafter window (§6.2), batch 1 and batch 32 (§6.5, §7), long
inputs (§7, inputs capped at 128K). The pages use trained Qwen3.6 models; these
configs are random-weight stand-ins of Qwen-like shape (vocab 151936, GQA 32/4).

Free constants the pages leave open (gains, eps, RoPE base, tap layers, mask id)
take the plainest values; each is listed with its reason in the design notes.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field


def tap_layers(n_layers: int) -> tuple[int, ...]:
    """Target layers whose residual stream feeds the drafter's context projection.

    The DMTP blog's ablation (§3, "Ablation Design") speaks of five target
    feature streams; we take min(5, L) evenly spread layers, rounding half up:
    round_half_up(i * (L - 1) / (n - 1)).
    """
    n = min(5, n_layers)
    if n == 1:
        return (0,)
    out = []
    for i in range(n):
        num = 2 * i * (n_layers - 1) + (n - 1)  # (2x + 1) // 2 with x = num/(2(n-1))
        out.append(num // (2 * (n - 1)))
    return tuple(out)


@dataclass(frozen=True)
class DmtpConfig:
    name: str
    vocab: int
    d_model: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    draft_layers: int
    batch: int
    # prompt lengths: (lo, hi) inclusive, drawn uniformly per sequence (lo == hi: fixed)
    ctx_lo: int
    ctx_hi: int
    rounds: int
    dtype: str                      # "fp32" or "bf16": weight / KV storage type
    seed: int
    structure: str = "uniform"      # "uniform" | "copy_span" | "repeat_chunks"
    fusion_std: float = 0.02        # std of the fusion matrix W (0.0: the zero-init W)
    weight_std: float = 0.02
    # hybrid target: layer_kinds[l] == 1 marks a Gated DeltaNet layer, 0 attention
    layer_kinds: tuple[int, ...] = ()
    gdn_heads: int = 0
    gdn_dk: int = 0
    gdn_dv: int = 0
    n_slots: int = 8
    draft_window: int = 4096
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    # verification: 0.0 greedy; > 0 the target's picks are samples at this temperature,
    # drawn with the given sampling seed
    temperature: float = 0.0
    sample_seed: int = 0
    # the T1 and drafter heads read an E4M3 copy of the head (bf16 models only)
    draft_head_fp8: bool = False
    # capacity of the draft heads' token list (0: no list; bf16 models only)
    draft_list_cap: int = 0
    # the context can run verifies of fewer drafts (round depth 0..6)
    variable_depth: bool = False
    # the draft heads also report the confidence of their picks
    draft_confidence: bool = False
    # bitwise-reproducible rounds (split GEMMs sum their K parts in a fixed order)
    deterministic: bool = False

    def __post_init__(self):
        if not self.layer_kinds:
            object.__setattr__(self, "layer_kinds", (0,) * self.n_layers)
        assert len(self.layer_kinds) == self.n_layers
        assert self.n_heads % self.n_kv_heads == 0
        assert self.head_dim % 2 == 0

    @property
    def mask_id(self) -> int:
        # The MASK token is a row of the shared embedding; we take the last id.
        return self.vocab - 1

    @property
    def taps(self) -> tuple[int, ...]:
        return tap_layers(self.n_layers)

    @property
    def n_taps(self) -> int:
        return len(self.taps)

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_dim(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    @property
    def has_gdn(self) -> bool:
        return any(self.layer_kinds)

    def replace(self, **kw) -> "DmtpConfig":
        if "n_layers" in kw and "layer_kinds" not in kw:
            kw["layer_kinds"] = ()
        return dataclasses.replace(self, **kw)


def _hybrid_kinds(n_layers: int) -> tuple[int, ...]:
    # layer l is attention when l % 4 == 3, Gated DeltaNet otherwise
    return tuple(0 if (l % 4 == 3) else 1 for l in range(n_layers))


CONFIGS: dict[str, DmtpConfig] = {
    "tiny": DmtpConfig(
        name="tiny", vocab=512, d_model=128, n_layers=2, n_heads=4, n_kv_heads=4,
        head_dim=32, ffn=256, draft_layers=1, batch=1, ctx_lo=64, ctx_hi=64,
        rounds=16, dtype="fp32", seed=0, fusion_std=0.0),
    "small": DmtpConfig(
        name="small", vocab=32000, d_model=1024, n_layers=8, n_heads=16, n_kv_heads=16,
        head_dim=64, ffn=2816, draft_layers=2, batch=1, ctx_lo=2048, ctx_hi=2048,
        rounds=64, dtype="bf16", seed=1, structure="copy_span", fusion_std=0.01),
    "b32": DmtpConfig(
        name="b32", vocab=151936, d_model=2048, n_layers=16, n_heads=32, n_kv_heads=4,
        head_dim=128, ffn=6144, draft_layers=2, batch=32, ctx_lo=512, ctx_hi=4096,
        rounds=32, dtype="bf16", seed=2),
    "long": DmtpConfig(
        name="long", vocab=151936, d_model=2048, n_layers=16, n_heads=32, n_kv_heads=4,
        head_dim=128, ffn=6144, draft_layers=2, batch=4, ctx_lo=32768, ctx_hi=32768,
        rounds=16, dtype="bf16", seed=3, structure="repeat_chunks"),
    "hybrid": DmtpConfig(
        name="hybrid", vocab=151936, d_model=2048, n_layers=48, n_heads=16, n_kv_heads=2,
        head_dim=128, ffn=6144, draft_layers=2, batch=8, ctx_lo=4096, ctx_hi=4096,
        rounds=16, dtype="bf16", seed=4, layer_kinds=_hybrid_kinds(48),
        gdn_heads=32, gdn_dk=128, gdn_dv=128),
}


def config_by_name(name: str) -> DmtpConfig:
    return CONFIGS[name]
