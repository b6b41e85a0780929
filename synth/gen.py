"""Seeded weight and prompt generation (no arithmetic of the method lives here).

Every tensor is drawn from one ``torch.Generator`` seeded with ``cfg.seed`` in the
fixed order of :func:`weight_specs`. Matrices are N(0, std) drawn in fp32 and, for
bf16 configs, rounded once to bf16 (round-to-nearest-even by torch); RMSNorm gains
are ones and consume no draws. Both the oracle and the CUDA library receive these
exact values (the oracle upcasts them).

Weight layout (all matrices row-major, ``[out_features, in_features]``):

* ``emb``, ``head``: ``[V, d]`` shared embedding and (untied) LM head.
* per target layer ``L{l}``: ``attn_norm [d]``, ``wqkv [(hq + 2 hkv) hd, d]``
  (q rows, then k rows, then v rows), ``wo [d, hq hd]``, ``mlp_norm [d]``,
  ``wgu [2F, d]`` (gate rows, then up rows), ``wdown [d, F]``.
  A Gated DeltaNet layer has ``gdn_wqkv [H dk + H dk + H dv, d]``,
  ``gdn_wa [H, d]``, ``gdn_wb [H, d]``, ``gdn_wo [d, H dv]`` instead of the
  attention matrices.
* ``final_norm [d]`` of the target.
* MTP module ``mtp.*``: ``norm_h``, ``norm_e``, ``proj [d, 2d]`` and one decoder
  layer with the target's attention shape, then ``final_norm``.
* fusion ``fuse.*``: ``norm_e``, ``norm_m``, ``w [d, 2d]``.
* block drafter: ``dft.fc [d, n_taps d]``, ``dft.norm_c``, layers ``D{j}.*`` as a
  target attention layer, ``dft.final_norm``.
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import DmtpConfig


def _layer_specs(prefix: str, cfg: DmtpConfig, kind: int):
    d, F = cfg.d_model, cfg.ffn
    out = [(f"{prefix}.attn_norm", (d,), "g")]
    if kind == 0:
        out += [(f"{prefix}.wqkv", (cfg.qkv_dim, d), "w"),
                (f"{prefix}.wo", (d, cfg.q_dim), "w")]
    else:
        H, dk, dv = cfg.gdn_heads, cfg.gdn_dk, cfg.gdn_dv
        out += [(f"{prefix}.gdn_wqkv", (H * (2 * dk + dv), d), "w"),
                (f"{prefix}.gdn_wa", (H, d), "w"),
                (f"{prefix}.gdn_wb", (H, d), "w"),
                (f"{prefix}.gdn_wo", (d, H * dv), "w")]
    out += [(f"{prefix}.mlp_norm", (d,), "g"),
            (f"{prefix}.wgu", (2 * F, d), "w"),
            (f"{prefix}.wdown", (d, F), "w")]
    return out


def weight_specs(cfg: DmtpConfig):
    """Ordered list of (name, shape, kind); kind 'w' = random matrix, 'g' = ones,
    'f' = the fusion matrix W (its own std)."""
    d, V = cfg.d_model, cfg.vocab
    specs = [("emb", (V, d), "w"), ("head", (V, d), "w")]
    for l, kind in enumerate(cfg.layer_kinds):
        specs += _layer_specs(f"L{l}", cfg, kind)
    specs.append(("final_norm", (d,), "g"))
    specs += [("mtp.norm_h", (d,), "g"), ("mtp.norm_e", (d,), "g"),
              ("mtp.proj", (d, 2 * d), "w")]
    specs += _layer_specs("mtp", cfg, 0)
    specs.append(("mtp.final_norm", (d,), "g"))
    specs += [("fuse.norm_e", (d,), "g"), ("fuse.norm_m", (d,), "g"),
              ("fuse.w", (d, 2 * d), "f")]
    specs += [("dft.fc", (d, cfg.n_taps * d), "w"), ("dft.norm_c", (d,), "g")]
    for j in range(cfg.draft_layers):
        specs += _layer_specs(f"D{j}", cfg, 0)
    specs.append(("dft.final_norm", (d,), "g"))
    return specs


def make_weights(cfg: DmtpConfig, device: str | torch.device = "cpu",
                 fusion_std: float | None = None) -> dict[str, torch.Tensor]:
    """Draw all weights for ``cfg``; returns name -> tensor (fp32 or bf16 storage).

    The draws are made on ``device`` (a CUDA generator gives different numbers
    than a CPU one for the same seed; a copy, not a second draw, serves the
    oracle). ``fusion_std`` overrides ``cfg.fusion_std`` (0.0 gives W = 0).
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    store = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
    fstd = cfg.fusion_std if fusion_std is None else fusion_std
    out: dict[str, torch.Tensor] = {}
    for name, shape, kind in weight_specs(cfg):
        if kind == "g":
            out[name] = torch.ones(shape, dtype=store, device=dev)
            continue
        std = cfg.weight_std if kind == "w" else fstd
        t = torch.randn(shape, generator=gen, dtype=torch.float32, device=dev)
        t = t * std
        out[name] = t.to(store)
    return out


def make_prompts(cfg: DmtpConfig, batch: int | None = None) -> list[np.ndarray]:
    """Per-sequence prompt ids (int32), seeded; ids are uniform in [0, V-2]
    (the last id is the MASK token and never appears in a prompt).

    Structures: ``uniform``; ``copy_span`` (a 256-token span copied from a random
    offset in [0, 1536) to the last 256 positions); ``repeat_chunks`` (1024-token
    chunks, each chunk i >= 1 with probability 1/2 a copy of a uniformly chosen
    earlier chunk).
    """
    B = cfg.batch if batch is None else batch
    rng = np.random.Generator(np.random.PCG64(1000 + cfg.seed))
    prompts = []
    for _ in range(B):
        P = int(rng.integers(cfg.ctx_lo, cfg.ctx_hi + 1))
        ids = rng.integers(0, cfg.vocab - 1, size=P, dtype=np.int64)
        if cfg.structure == "copy_span" and P >= 512:
            span = 256
            src = int(rng.integers(0, max(1, min(1536, P - 2 * span))))
            ids[P - span:] = ids[src:src + span]
        elif cfg.structure == "repeat_chunks":
            C = 1024
            nch = P // C
            for i in range(1, nch):
                if rng.random() < 0.5:
                    j = int(rng.integers(0, i))
                    ids[i * C:(i + 1) * C] = ids[j * C:(j + 1) * C]
        prompts.append(ids.astype(np.int32))
    return prompts
