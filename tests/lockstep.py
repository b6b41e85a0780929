"""Lock-step comparison of the CUDA round (through the C ABI) with the oracle.

Both start from the same prompts and weights. Each round the GPU runs first; the
oracle then runs the same round on each sequence, adopting the GPU's pick at any
argmax where the oracle's own top-1 and the GPU's id are within the near-tie gate
(0.05 in logits, or in the scores l / temperature + G under sampled verification) -
so one near tie cannot make the two diverge for the rest of the run. Any pick outside the gate is a mismatch. Integer fields must then agree
exactly; float fields within `tol` max-abs.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import OracleModel
from oracle.fp8 import fp8_logit_bounds

GATE = 0.05
# E4M3 draft heads: the head inputs (normalised hidden rows) of the two sides agree within
# this much per element (the hidden-state bar is 2e-2; measured ~3e-3), which bounds how
# far each side's quantised input, and so each draft logit, can move
FP8_INPUT_DELTA = 1e-2


def to_np(t):
    return t.detach().cpu().numpy()


class Lockstep:
    def __init__(self, cfg, weights_gpu: dict, prompts, rounds: int, seqs=None, max_ctx=None,
                 kv_floor: bool = False):
        """kv_floor: also run the oracle with its K/V caches rounded to bf16 (the GPU's
        storage) on the same picks. Each float field must then be within `tol` of that
        oracle (the kernels' arithmetic), and within `tol` plus the storage floor - the
        distance between the two oracles on this field this round - of the exact oracle
        (what a bf16 cache alone costs against exact K/V)."""
        from mtp_block_draft_gb300 import DmtpRound, default_max_ctx
        self.cfg = cfg
        self.prompts = prompts
        self.seqs = list(range(len(prompts))) if seqs is None else list(seqs)
        self.gpu = DmtpRound(cfg, weights_gpu, prompts,
                             max_ctx or default_max_ctx(prompts, rounds))
        self.oracle = OracleModel(cfg, {k: v.cpu() for k, v in weights_gpu.items()}, gate=GATE,
                                  temperature=cfg.temperature, sample_seed=cfg.sample_seed,
                                  draft_head_fp8=cfg.draft_head_fp8)
        kv, A, _ = self.gpu.read_state()
        self.states = {}
        self.adopted = []
        for b in self.seqs:
            st = self.oracle.prefill(prompts[b], adopt_A=int(A[b]), b=b)
            assert not self.oracle.prefill_log["mismatch"], self.oracle.prefill_log
            self.adopted += self.oracle.prefill_log["adopted"]
            assert st.A == int(A[b]) and st.a == int(kv[b]) == len(prompts[b])
            self.states[b] = st
        self.floor_oracle, self.floor_states = None, {}
        if kv_floor:
            import copy
            self.floor_oracle = copy.copy(self.oracle)  # same weights, bf16 K/V storage
            self.floor_oracle.kv_bf16 = True
            for b in self.seqs:
                self.floor_states[b] = self.floor_oracle.prefill(prompts[b], adopt_A=int(A[b]),
                                                                 b=b)
                assert not self.floor_oracle.prefill_log["mismatch"]
        self.max_err = {}

    def _err(self, name, a, b):
        e = float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))
        self.max_err[name] = max(self.max_err.get(name, 0.0), e)
        return e

    def step(self, forced: np.ndarray | None = None, floats: bool = True, tol: float = 2e-2,
             draft_list: np.ndarray | None = None, depth: int = 7):
        """draft_list: boolean mask [V] of the tokens the draft heads score (the list the
        GPU context was given with set_draft_list); the draft logits are then compared at
        the listed tokens only. depth: drafts the verify carries (dmtp_round_depth): the
        picks past it must be -1 and the verify logits come as B (depth + 1) rows."""
        g = self.gpu
        out = g.alloc_out(ints=True, floats=floats)
        ft = None
        if forced is not None:
            ft = torch.as_tensor(np.asarray(forced, np.int32), device=g.device)
        g.round(out, forced=ft, depth=depth)
        torch.cuda.synchronize()
        o = {k: to_np(v) for k, v in out.items()}
        G = depth + 1
        if floats:  # sequence-major [B][G][V] at the start of the buffer
            V = self.cfg.vocab
            o["verify_logits"] = o["verify_logits"].reshape(-1)[:self.gpu.B * G * V].reshape(
                self.gpu.B, G, V)
        picks_all = o["picks"]
        o["picks"] = picks_all[:, :G]
        recs = {}
        for b in self.seqs:
            adopt = {"g": o["picks"][b]}
            if forced is None:
                adopt["T"] = o["drafts"][b]
            assert all(int(x) == -1 for x in picks_all[b][G:]), (b, picks_all[b])
            rec = self.oracle.round(self.states[b],
                                    forced=None if forced is None else forced[b],
                                    adopt=adopt, want_logits=floats, draft_list=draft_list,
                                    depth=depth)
            frec = None
            if self.floor_oracle is not None:
                frec = self.floor_oracle.round(self.floor_states[b],
                                               forced=None if forced is None else forced[b],
                                               adopt=adopt, want_logits=floats,
                                               draft_list=draft_list, depth=depth)
                assert not frec["log"]["mismatch"], (b, frec["log"]["mismatch"])
            log = rec["log"]
            assert not log["mismatch"], (b, log["mismatch"])
            self.adopted += log["adopted"]
            assert list(o["drafts"][b]) == rec["drafts"], (b, o["drafts"][b], rec["drafts"])
            assert list(o["picks"][b]) == rec["g"], (b, o["picks"][b], rec["g"])
            assert int(o["n_accepted"][b]) == rec["n"]
            assert list(o["committed"][b][:rec["n"] + 1]) == rec["committed"]
            assert all(int(x) == -1 for x in o["committed"][b][rec["n"] + 1:])
            assert int(o["kv_len"][b]) == rec["kv_len"]
            assert int(o["mtp_len"][b]) == rec["mtp_len"]
            assert int(o["snap_slot"][b]) == rec["snap_slot"]
            if floats:
                fp8 = self.cfg.draft_head_fp8
                listed = ((lambda x: x) if draft_list is None else
                          (lambda x: np.asarray(x)[..., draft_list]))
                for name, key in (("t1_logits", "t1_logits"), ("draft_logits", "draft_logits"),
                                  ("verify_logits", "verify_logits"), ("delta", "delta"),
                                  ("h_mtp", "h_mtp_in")):
                    sel = listed if name in ("t1_logits", "draft_logits") else (lambda x: x)
                    if fp8 and name in ("t1_logits", "draft_logits"):
                        # quantised draft heads: within the interval the input difference
                        # allows (oracle/fp8.py), plus the float bar
                        hin = rec["t1_head_in" if name == "t1_logits" else "draft_head_in"]
                        ref, width = fp8_logit_bounds(hin, self.oracle.Hq, self.oracle.Hs,
                                                      FP8_INPUT_DELTA)
                        gpu = np.asarray(o[name][b], np.float64).reshape(ref.shape)
                        ref, width, gpu = sel(ref), sel(width), sel(gpu)
                        excess = float(np.max(np.abs(gpu - ref) - width))
                        self.max_err[name + "_beyond_bound"] = max(
                            self.max_err.get(name + "_beyond_bound", -1e30), excess)
                        self._err(name, gpu, ref)
                        assert excess <= tol, (b, name, excess)
                        continue
                    e = self._err(name, sel(o[name][b]), sel(rec[key]))
                    if frec is None:
                        assert e <= tol, (b, name, e)
                        continue
                    ef = self._err(name + "_vs_bf16kv_oracle", sel(o[name][b]), sel(frec[key]))
                    floor = self._err(name + "_bf16kv_floor", sel(frec[key]), sel(rec[key]))
                    assert ef <= tol, (b, name, "vs the bf16-KV oracle", ef)
                    assert e <= tol + floor, (b, name, e, floor)
            if floats and "draft_conf" in o:
                # confidence 1 / sum exp(l - l_max): logits within tol of the oracle's move
                # each term's exponent by at most 2 tol
                ref = np.asarray(rec["draft_confidence"], np.float64)
                rel = np.abs(np.asarray(o["draft_conf"][b], np.float64) - ref) / ref
                self.max_err["draft_conf_rel"] = max(self.max_err.get("draft_conf_rel", 0.0),
                                                     float(rel.max()))
                assert rel.max() <= np.expm1(2 * tol), (b, "draft_conf", rel.max())
            recs[b] = rec
        return o, recs

    def close(self):
        print(f"[lockstep] {self.cfg.name}: max float error {self.max_err}, "
              f"near-tie adoptions {len(self.adopted)}")
        self.gpu.close()
