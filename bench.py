#!/usr/bin/env python
"""Accepted tokens/s of the batched DMTP round on GB300 (one JSON line on stdout).

A step is one DMTP round (steps a1-a6) over the batch. The default workload is the
B32 serving round: 32 sequences with prompt lengths uniform in [512, 4096], vocab
151936, d_model 2048, a 16-layer GQA target (32/4 heads x 128, ffn 6144), one MTP
block and a 2-layer block drafter, bf16 weights and KV, random weights N(0, 0.02)
and random prompt ids (synthetic stand-ins for the trained models and datasets the
DMTP blog evaluates). Metric: committed tokens per second = B x rounds/s x mean
accepted length (DMTP blog §7, per-verify length 1 + sum k hist[k] / sum hist).

  value      device-timed: CUDA events on the library's stream around K graph
             replays, inputs (weights, KV, state) resident in HBM; every round
             streams ~7 GB (> 129 MB L2), so no flush is needed between rounds.
  e2e        the same metric through the C ABI with host buffers: each step
             enqueues the round and copies committed[B,8] and n[B] back to pinned
             host memory before the next (wall clock).
  roofline   the dominant kernel class of a profiled round (CUDA events around
             each of its launches, on the launching stream), algorithmic bytes /
             measured time against the measured HBM peak.
  cpu_baseline  the float64 NumPy oracle on the host cores, on a bounded sample
             (one sequence of the same batch, a few rounds after its prefill).

--impl reference times that oracle as the reference arm instead.
Multi-GPU: one process per GPU (torchrun), each with its own 32 sequences
(replicas; no collective on the data path), barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import threading
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "accepted tokens/sec per GPU at B32 (rounds/s x mean accept len); % roofline"
UNIT = "tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _traffic(kernel: str, bytes_per_launch: float, impl_bytes_per_launch: float):
    """DRAM bytes per launch of `kernel` from the ncu captures summarised in profiles/ (the
    ratio of DRAM bytes to the bytes the record's basis counts: the method's bytes, or the
    implementation's), or None once the kernel source changed."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None, None
    src = os.path.join(ROOT, rec["source"])
    if hashlib.sha1(open(src, "rb").read()).hexdigest() != rec["sha1"]:
        return None, "kernel changed since the ncu capture"
    basis = rec.get("basis", "method")
    per = impl_bytes_per_launch if basis == "implementation" else bytes_per_launch
    return per * rec["dram_over_algorithmic"], \
        f"ncu DRAM / {basis} bytes {rec['dram_over_algorithmic']} (profiles/{rec['capture']})"


class Clocks:
    """nvidia-smi sampler for the timed region (200 ms period). The samples are read by a
    thread; ready() waits for the first one, so the sampler is running before the timed
    region starts."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.p = None
        self.lines = []
        self.t = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.p.stdout:
            self.lines.append(line)

    def ready(self, timeout: float = 10.0):
        t0 = time.time()
        while self.p is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)
        self.n0 = len(self.lines)  # samples taken before the timed region are not used

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        lines = list(self.lines[getattr(self, "n0", 0):])
        self.p.terminate()
        try:
            self.p.wait(timeout=10)
        except Exception:
            pass
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_config(cfg, rank: int):
    """Each rank serves its own batch (replicas, weak scaling): rank 0 the workload's
    prompts, rank r the same configuration with prompt seed + 1000 r."""
    return cfg if rank == 0 else cfg.replace(seed=cfg.seed + 1000 * rank)


def combine_ranks(ms, tokens, e2e_s, e2e_tokens, world: int, device):
    """Whole-job numbers over the ranks: the slowest rank's times (device-timed and end
    to end), the sum of the committed tokens."""
    if world == 1:
        return float(ms), float(tokens), float(e2e_s), float(e2e_tokens)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, e2e_s], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens), float(e2e_tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t[0]), float(n[0]), float(t[1]), float(n[1])


def oracle_sample(cfg, weights, prompts, rounds: int, limit_s: float = 30.0):
    """Time the oracle on one sequence (the shortest prompt) of the batch: prefill
    untimed, then up to `rounds` rounds or `limit_s` seconds timed."""
    from oracle import OracleModel
    b = int(np.argmin([len(p) for p in prompts]))
    t0 = time.perf_counter()
    om = OracleModel(cfg, {k: v.cpu() for k, v in weights.items()},
                     temperature=cfg.temperature, sample_seed=cfg.sample_seed,
                     draft_head_fp8=cfg.draft_head_fp8)
    st = om.prefill(prompts[b], b=b)
    setup = time.perf_counter() - t0
    tokens, el, done = 0, 0.0, 0
    while done < rounds and el < limit_s:
        t = time.perf_counter()
        rec = om.round(st, want_logits=False)
        el += time.perf_counter() - t
        tokens += rec["accept_len"]
        done += 1
    cores = len(os.sched_getaffinity(0))
    return {"value": tokens / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"sequence {b} of the batch (prompt {len(prompts[b])} tokens), "
                      f"{done} rounds after an untimed prefill ({setup:.0f} s incl. weight "
                      f"upcast), float64 NumPy, BLAS threads = {cores}",
            "rounds": done, "seconds": el}


# DMTP per-verify acceptance lengths of the DMTP blog §7 ("Acceptance Length and End-to-End
# Throughput", trained Qwen3.6 models at temperature 1): used only for a labelled
# projection of the measured rounds/s, never as a measurement.
PAGE_PER_VERIFY = {"Code": 3.795, "Math": 4.056, "MT-Bench": 3.250, "Agent": 4.709,
                   "SWE": 3.173, "Long-horizon": 4.656}


def acceptance(dh):
    """Per-position acceptance from the histogram deltas of the timed rounds: entry n
    counts sequence-rounds that accepted n drafts (accept length n + 1); p_len_ge[k - 1]
    is the cumulative P(accept length >= k) for k = 1..8 (the DMTP blog's cumulative
    acceptance curve); first_candidate = 1 - hist[0] / sum (the DMTP blog's
    first-candidate acceptance, section 8)."""
    dh = np.asarray(dh, dtype=np.int64)
    tot = max(1, int(dh.sum()))
    return {"hist_n_accepted": [int(x) for x in dh],
            "p_len_ge": [float(dh[k - 1:].sum()) / tot for k in range(1, 9)],
            "first_candidate": (1.0 - float(dh[0]) / tot) if dh.sum() else 0.0}


def forced_accept(cfg, weights, prompts, warmup, steps, max_iter=6):
    """Rounds with every draft accepted: the drafts are forced to the target's own greedy
    continuation, then replayed as the forced-draft graph on a fresh context from the same
    prompts and timed. The continuation must be the one the replay itself computes: a
    near tie in the target's logits can resolve differently when the same position is
    computed as row 0 of a one-token round or as row s of an eight-row round (other
    attention splits, other reduction orders). So the plan is refined to a fixed point:
    a first plan comes from rounds whose drafts are forced wrong (each commits exactly
    the next greedy token); each refinement replays the plan on a fresh context and, for
    every sequence whose replay rejected a draft, keeps the committed tokens up to and
    including the correction and continues that sequence with one-token rounds; once a
    replay accepts every draft of every round, a fresh context replays it again, timed.
    The histogram of the timed rounds gives the accept length reached. The contexts are
    deterministic (fixed-order K-part sums), so a replay reproduces its plan bit for bit
    and the timed rounds include that option's cost."""
    import torch
    from mtp_block_draft_gb300 import DmtpRound
    cfg = cfg.replace(deterministic=cfg.dtype == "bf16")
    B, V, R = len(prompts), cfg.vocab, warmup + steps
    need = 8 * R + 1
    max_ctx = max(len(p) for p in prompts) + 8 * (need + 2) + 64
    forced = torch.empty((B, 7), dtype=torch.int32, device="cuda")

    def wrong(st):
        return [(st[-1] + 1 + j) % (V - 1) for j in range(7)]

    def run(plan):
        """Replay `plan` (list per sequence of R rounds of 7 drafts, or None: all wrong);
        returns the committed streams (each at least `need` tokens) and whether every
        round of every sequence accepted all 7 drafts."""
        g = DmtpRound(cfg, weights, prompts, max_ctx)
        _, A, _ = g.read_state()
        streams = [[int(a)] for a in A]
        ok = [plan is not None] * B
        out = g.alloc_out(ints=True, floats=False)
        r = 0
        while min(len(st) for st in streams) < need:
            rows = []
            for b in range(B):
                on_plan = ok[b] and r < R
                rows.append(plan[b][r] if on_plan else wrong(streams[b]))
            forced.copy_(torch.tensor(rows, dtype=torch.int32))
            g.round(out, forced=forced)
            com, n = out["committed"].cpu().numpy(), out["n_accepted"].cpu().numpy()
            for b in range(B):
                streams[b] += [int(t) for t in com[b][:n[b] + 1]]
                if ok[b] and r < R and n[b] < 7:
                    ok[b] = False  # rejected: keep the correction, continue token by token
            r += 1
        g.close()
        del g
        torch.cuda.empty_cache()
        return streams, all(ok)

    def to_plan(streams):
        return [[streams[b][8 * r + 1: 8 * r + 8] for r in range(R)] for b in range(B)]

    streams, _ = run(None)
    iters, converged = 0, False
    while iters < max_iter and not converged:
        iters += 1
        streams, converged = run(to_plan(streams))
    plan = torch.tensor([[to_plan(streams)[b][r] for b in range(B)] for r in range(R)],
                        dtype=torch.int32, device="cuda")
    g2 = DmtpRound(cfg, weights, prompts, max_ctx)
    stream = g2.stream
    for r in range(warmup):
        g2.round(forced=plan[r])
    _, _, h0 = g2.read_state()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for r in range(warmup, R):
        g2.round(forced=plan[r])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    _, _, h1 = g2.read_state()
    g2.close()
    dh = (h1 - h0).astype(np.int64)
    mean_len = float(np.sum((np.arange(8) + 1) * dh)) / max(1, int(dh.sum()))
    rps = steps / (ms / 1e3)
    return {"rounds_per_s": rps, "mean_accept_len": mean_len, "tokens_per_s": B * rps * mean_len,
            "steps": steps, "warmup": warmup, "acceptance": acceptance(dh),
            "plan_refinements": iters, "plan_converged": converged,
            "deterministic": bool(cfg.deterministic),
            "drafts": "forced to the target's own greedy continuation as the replayed rounds "
                      "compute it (every draft accepted)"}


def fp8_draft_heads(cfg, weights, prompts, warmup, steps):
    """The same workload with the T1 and drafter heads on the E4M3 head copy (DMTP blog
    §6.5 drafting-side head quantisation; verification stays bf16): natural rounds, graph
    replayed, timed like the headline."""
    import torch
    from mtp_block_draft_gb300 import DmtpRound
    c8 = cfg.replace(draft_head_fp8=True)
    R = warmup + steps
    g = DmtpRound(c8, weights, prompts, max(len(p) for p in prompts) + 8 * R + 64)
    for _ in range(warmup):
        g.round()
    _, _, h0 = g.read_state()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(g.stream)
    for _ in range(steps):
        g.round()
    e1.record(g.stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    _, _, h1 = g.read_state()
    prof = g.profile_round()
    g.close()
    dh = (h1 - h0).astype(np.int64)
    mean_len = float(np.sum((np.arange(8) + 1) * dh)) / max(1, int(dh.sum()))
    rps = steps / (ms / 1e3)
    return {"rounds_per_s": rps, "ms_per_step": ms / steps, "mean_accept_len": mean_len,
            "tokens_per_s": len(prompts) * rps * mean_len, "steps": steps, "warmup": warmup,
            "lm_head_ms_per_round": class_ms(prof, ms / steps, "lm_head"),
            "note": "T1 and drafter heads read an E4M3 copy of the vocabulary matrix "
                    "(per-row power-of-two scales); the verify head stays bf16"}


def draft_list_round(cfg, weights, prompts, warmup, steps, size=16000):
    """The same workload with the T1 and drafter heads over the colibri page's frequent-
    token list (dmtp_set_draft_list; the verify head still scores every token): the list
    is the native list (dmtp_vocab.h) after the batch's prompts (one list per batch: the
    16000 most counted tokens, the three-quarters rule and every token of the
    conversation) and the pending tokens, set once before the timed rounds (no upkeep
    inside them); natural rounds, graph replayed, timed like the headline."""
    import torch
    from mtp_block_draft_gb300 import DmtpRound, DmtpVocabList
    cl = cfg.replace(draft_list_cap=cfg.vocab)
    R = warmup + steps
    g = DmtpRound(cl, weights, prompts, max(len(p) for p in prompts) + 8 * R + 64)
    vl = DmtpVocabList(cfg.vocab, size)
    vl.begin_request(np.concatenate(prompts))
    _, A, _ = g.read_state()
    vl.picked(A)
    ids = vl.ids()
    rule_listed = int(len(ids))
    vl.close()
    kind = "the page's rule"
    if len(ids) > cfg.vocab // 2:
        # Uniform random prompts: halvings every 1024 counted tokens leave almost every
        # count at 0 or 1, so the rule lists (nearly) every token. Time the page's default
        # list size instead: the `size` most counted prompt tokens (ties to the lower id).
        cnt = np.bincount(np.concatenate(prompts), minlength=cfg.vocab)
        ids = np.sort(np.lexsort((np.arange(cfg.vocab), -cnt))[:size]).astype(np.int32)
        kind = f"the {size} most counted prompt tokens (the page's default list size)"
    g.set_draft_list(ids)
    for _ in range(warmup):
        g.round()
    _, _, h0 = g.read_state()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(g.stream)
    for _ in range(steps):
        g.round()
    e1.record(g.stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    _, _, h1 = g.read_state()
    prof = g.profile_round()
    g.close()
    dh = (h1 - h0).astype(np.int64)
    mean_len = float(np.sum((np.arange(8) + 1) * dh)) / max(1, int(dh.sum()))
    rps = steps / (ms / 1e3)
    return {"listed_tokens": int(len(ids)), "list": kind, "rule_listed": rule_listed,
            "vocab": cfg.vocab, "rounds_per_s": rps,
            "ms_per_step": ms / steps, "mean_accept_len": mean_len,
            "tokens_per_s": len(prompts) * rps * mean_len, "steps": steps, "warmup": warmup,
            "lm_head_ms_per_round": class_ms(prof, ms / steps, "lm_head"),
            "lm_head_GB_per_round": prof["lm_head"]["bytes"] / 1e9,
            "note": "T1 and drafter heads over the listed rows (a compact copy in the "
                    "workspace); the verify head scores the whole vocabulary. With uniform "
                    "random prompts the conversation alone lists most of the batch's prompt "
                    "tokens"}


def depth_rounds(cfg, weights, prompts, warmup=4, steps=30):
    """Round time at each verify depth k = 0..7 (dmtp_round_depth: the verify carries k
    drafts as B (k + 1) rows), graph replays timed with CUDA events, at this batch and at
    batch 1 (the batch's first prompt); then the native draft-depth gate (colibri page)
    fed with T(n) = the round time at depth n - 1 and the page's MTP-head starting
    acceptances picks a depth for each batch."""
    import torch
    from mtp_block_draft_gb300 import DmtpGate, DmtpRound
    cd = cfg.replace(variable_depth=True)
    res = {}
    for label, ps in ((f"B{len(prompts)}", prompts), ("B1", prompts[:1])):
        R = 8 * (warmup + steps) + 8
        g = DmtpRound(cd, weights, ps, max(len(p) for p in ps) + 8 * R + 64)
        ms = []
        for depth in range(8):
            for _ in range(warmup):
                g.round(depth=depth)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(g.stream)
            for _ in range(steps):
                g.round(depth=depth)
            e1.record(g.stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1) / steps)
        g.close()
        del g
        gate = DmtpGate(7)
        for n in range(1, 9):
            gate.forward(n, ms[n - 1] / 1e3)
        k, v = gate.pick(7)
        st = gate.read()
        gate.close()
        res[label] = {"round_ms_by_depth": [round(x, 4) for x in ms],
                      "gate_pick": {"depth": k, "value": v, "rho": st["rho"],
                                    "acceptance_priors": st["a"][:3]}}
    res["note"] = ("T(n) = whole-round time at depth n - 1: the drafting part (MTP head, "
                   "fusion, block drafter) is the same at every depth; the gate runs on the "
                   "page's starting acceptances (trained-model values), not on the random "
                   "weights' near-zero acceptance")
    return res


def hybrid_round(warmup, steps, hbm_gbs):
    """The hybrid workload (B8, 48 layers of which 36 Gated DeltaNet, prompts of 4096):
    natural rounds, graph replayed, timed like the headline; the Gated DeltaNet class
    (state read, 7 snapshots, live write per layer) with its bandwidth against the HBM
    peak. A side measurement, not the headline."""
    import torch
    from mtp_block_draft_gb300 import DmtpRound
    from synth import CONFIGS, make_prompts, make_weights
    cfg = CONFIGS["hybrid"]
    weights = make_weights(cfg, torch.device("cuda", torch.cuda.current_device()))
    prompts = make_prompts(cfg)
    R = warmup + steps
    g = DmtpRound(cfg, weights, prompts, max(len(p) for p in prompts) + 8 * R + 64)
    for _ in range(warmup):
        g.round()
    _, _, h0 = g.read_state()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(g.stream)
    for _ in range(steps):
        g.round()
    e1.record(g.stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    _, _, h1 = g.read_state()
    prof = g.profile_round()
    pf_ms, pf_tokens = g.prefill_stats()
    g.close()
    del weights
    dh = (h1 - h0).astype(np.int64)
    mean_len = float(np.sum((np.arange(8) + 1) * dh)) / max(1, int(dh.sum()))
    rps = steps / (ms / 1e3)
    gdn = dict(prof["gdn"])
    gdn["ms"] = class_ms(prof, ms / steps, "gdn")
    gdn_gbs = gdn["bytes"] / max(1e-12, gdn["ms"] / 1e3) / 1e9
    return {"workload": f"hybrid: B{len(prompts)}, {cfg.n_layers} layers "
                        f"({sum(cfg.layer_kinds)} Gated DeltaNet, H {cfg.gdn_heads}, "
                        f"dk {cfg.gdn_dk}, dv {cfg.gdn_dv}), prompts {cfg.ctx_lo}",
            "rounds_per_s": rps, "ms_per_step": ms / steps, "mean_accept_len": mean_len,
            "tokens_per_s": len(prompts) * rps * mean_len, "steps": steps, "warmup": warmup,
            "gdn": {"ms_per_round": gdn["ms"], "GB_per_round": gdn["bytes"] / 1e9,
                    "launches": int(gdn["launches"]), "GB/s": gdn_gbs,
                    "frac_of_hbm": gdn_gbs / hbm_gbs},
            "prefill_tokens_per_s": pf_tokens / (pf_ms / 1e3) if pf_ms > 0 else None}


def class_ms(prof: dict, timed_round_ms: float, cls: str) -> float:
    """A class's time in one profiled round (dmtp_round_profile), less the event-node cost
    per launch: (profiled round - timed round) / launches, as for the main line."""
    names = ("gemm", "lm_head", "attention", "gdn", "other")
    n = sum(prof[c]["launches"] for c in names)
    cost = max(0.0, prof["round_ms"] - timed_round_ms) / max(1, n)
    return max(0.0, prof[cls]["ms"] - prof[cls]["launches"] * cost)


def workload_name(cfg, B):
    """The workload as both arms name it in config.workload."""
    return (f"{cfg.name}: B{B} DMTP round, vocab {cfg.vocab}, d {cfg.d_model}, "
            f"{cfg.n_layers}-layer GQA {cfg.n_heads}/{cfg.n_kv_heads}x{cfg.head_dim} "
            f"target, ffn {cfg.ffn}, 1 MTP block, {cfg.draft_layers}-layer drafter, "
            f"prompts U[{cfg.ctx_lo},{cfg.ctx_hi}]")


def run_reference(args, cfg):
    import torch
    from synth import make_prompts, make_weights
    rank, world, _ = _dist()
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    weights = make_weights(cfg, dev)
    prompts = make_prompts(cfg)
    from oracle import OracleModel
    b = int(np.argmin([len(p) for p in prompts]))
    om = OracleModel(cfg, {k: v.cpu() for k, v in weights.items()},
                     temperature=cfg.temperature, sample_seed=cfg.sample_seed,
                     draft_head_fp8=cfg.draft_head_fp8)
    del weights
    st = om.prefill(prompts[b], b=b)
    for _ in range(args.warmup):
        om.round(st, want_logits=False)
    tokens, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        tokens += om.round(st, want_logits=False)["accept_len"]
    el = time.perf_counter() - t0
    v = tokens / el
    cores = len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(cfg, len(prompts)), "global_batch": 1,
                       "seq_len": len(prompts[b]), "parallelism": "none",
                       "note": f"one round of one sequence of the B{len(prompts)} batch per "
                               "step (a bounded sample of the workload)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"one round of sequence {b} (prompt {len(prompts[b])}) "
                                       "per step, float64 NumPy"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="b32")
    ap.add_argument("--repeats", type=int, default=5,
                    help="repeats of the timed K-step loop (at least; more while the timed "
                         "region is shorter than ~1 s); the headline is their median")
    ap.add_argument("--max-repeats", type=int, default=40)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--profile-rounds", type=int, default=3)
    ap.add_argument("--cpu-rounds", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forced-steps", type=int, default=16,
                    help="timed rounds of the forced-accept run (0: skip)")
    ap.add_argument("--fp8-steps", type=int, default=100,
                    help="timed rounds of the run with E4M3 draft heads (0: skip)")
    ap.add_argument("--depth-steps", type=int, default=30,
                    help="timed rounds per verify depth 0..7 at B32 and B1 (0: skip)")
    ap.add_argument("--list-steps", type=int, default=100,
                    help="timed rounds of the run with the draft heads over the token list "
                         "(0: skip)")
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="0: greedy verification (the workloads' setting); > 0: target-only "
                         "sampled verification at this temperature")
    ap.add_argument("--sample-seed", type=int, default=1)
    # smaller cases of the same kernels, for profiler captures (not bench workloads)
    ap.add_argument("--hybrid-steps", type=int, default=100,
                    help="side measurement of the hybrid workload (0: off)")
    ap.add_argument("--layers", type=int, default=None, help="override target layers")
    ap.add_argument("--ctx", type=int, nargs=2, default=None, help="override prompt range")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from synth import CONFIGS
    cfg = CONFIGS[args.config]
    if args.layers is not None:
        kinds = tuple(cfg.layer_kinds[:args.layers]) if cfg.has_gdn else ()
        cfg = cfg.replace(name=f"{cfg.name}-L{args.layers}", n_layers=args.layers,
                          layer_kinds=kinds)
    if args.ctx is not None:
        cfg = cfg.replace(name=f"{cfg.name}-ctx{args.ctx[0]}-{args.ctx[1]}", ctx_lo=args.ctx[0],
                          ctx_hi=args.ctx[1])
    if args.temperature > 0:
        cfg = cfg.replace(name=f"{cfg.name}-T{args.temperature:g}", temperature=args.temperature,
                          sample_seed=args.sample_seed)
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    import torch.distributed as dist
    from mtp_block_draft_gb300 import DmtpRound
    from synth import make_prompts, make_weights

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    weights = make_weights(cfg, dev)
    pcfg = rank_config(cfg, rank)
    prompts = make_prompts(pcfg)
    B = len(prompts)
    max_reps = max(args.repeats, min(args.max_repeats, max(args.repeats, 2000 // args.steps)))
    total_rounds = (args.warmup + max_reps * args.steps + args.e2e_steps + args.profile_rounds
                    + 8)
    max_ctx = max(len(p) for p in prompts) + 8 * total_rounds + 32
    g = DmtpRound(cfg, weights, prompts, max_ctx)
    stream = g.stream

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 2:
            e0.record(stream)
        g.round()
    e1.record(stream)
    torch.cuda.synchronize()
    est_ms = max(1e-3, e0.elapsed_time(e1) / 2)  # the last two warm-up rounds
    # Repeats of the K-step loop: at least args.repeats, and enough that the timed region
    # lasts about a second, so the 200 ms clock sampler sees it (K = 20 rounds of 3 ms are
    # shorter than one sample); the headline is the median repeat.
    reps = int(min(max_reps, max(args.repeats, np.ceil(1000.0 / (args.steps * est_ms)))))
    if world > 1:  # every rank runs the same number of repeats
        r = torch.tensor([reps], dtype=torch.int64, device=dev)
        dist.all_reduce(r, op=dist.ReduceOp.MAX)
        reps = int(r.item())
    _, _, h0 = g.read_state()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.ready()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    # the profiler start/stop marks let an external profiler skip the prefill
    torch.cuda.cudart().cudaProfilerStart()
    ev[0].record(stream)
    for r in range(reps):
        for _ in range(args.steps):
            g.round()
        ev[r + 1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    rep_ms = [ev[r].elapsed_time(ev[r + 1]) for r in range(reps)]
    ms = float(statistics.median(rep_ms))  # K steps
    _, _, h1 = g.read_state()
    dh = (h1 - h0).astype(np.int64)
    seq_rounds = int(dh.sum())  # one histogram entry per sequence per round
    mean_len = float(np.sum((np.arange(8) + 1) * dh)) / max(1, seq_rounds)
    tokens = B * args.steps * mean_len  # committed tokens of K steps at the mean length

    # e2e through the C ABI with host outputs (pinned), wall clock
    committed = torch.empty((B, 8), dtype=torch.int32, pin_memory=True).numpy()
    nacc = torch.empty((B,), dtype=torch.int32, pin_memory=True).numpy()
    torch.cuda.synchronize()
    e2e_tokens, t0 = 0, time.perf_counter()
    for _ in range(args.e2e_steps):
        g.round_host(committed, nacc)
        e2e_tokens += int(np.sum(nacc.astype(np.int64) + 1))
    e2e_s = time.perf_counter() - t0
    ms_all, tok_all, e2e_s_all, e2e_tok_all = combine_ranks(ms, tokens, e2e_s, e2e_tokens,
                                                             world, dev)
    value = tok_all / (ms_all / 1e3)
    e2e_val = e2e_tok_all / e2e_s_all

    # per-kernel-class profile of real rounds: each round a captured graph with event nodes
    # between its launches (dmtp_round_profile), so class times add up to the round
    hbm, tc_burst, tc_sus, peak_src = _peaks()
    prof = [g.profile_round() for _ in range(args.profile_rounds)]
    classes = ("gemm", "lm_head", "attention", "gdn", "other")
    agg = {c: {k: sum(p[c][k] for p in prof) / len(prof)
               for k in ("ms", "bytes", "impl_bytes", "flops", "launches")}
           for c in classes}
    # Each event node between launches costs a few microseconds of its own (the profiled
    # graph runs longer than the timed one). That cost, the same for every launch, is
    # (profiled round - timed round) / launches; it is taken off each launch, so the
    # classes add up to the timed round. The raw event times are reported beside.
    prof_round_ms = sum(p["round_ms"] for p in prof) / len(prof)
    n_launch = sum(agg[c]["launches"] for c in classes)
    ev_cost = max(0.0, prof_round_ms - ms / args.steps) / max(1.0, n_launch)
    for c in classes:
        agg[c]["ms_events"] = agg[c]["ms"]
        agg[c]["ms"] = max(0.0, agg[c]["ms"] - agg[c]["launches"] * ev_cost)
    dom = max(classes, key=lambda c: agg[c]["ms"] if c != "other" else -1)
    a = agg[dom]
    launches = max(1.0, a["launches"])
    per_launch_s = a["ms"] / 1e3 / launches
    gbs = a["bytes"] / launches / per_launch_s / 1e9
    tfs = a["flops"] / launches / per_launch_s / 1e12
    t_mem = a["bytes"] / (hbm * 1e9)
    t_tc = a["flops"] / (tc_sus * 1e12)
    if t_tc > t_mem:
        roof = {"bound": "tensor", "achieved": tfs, "peak": tc_sus, "unit": "TFLOP/s",
                "frac": tfs / tc_sus}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}
    traffic, tsrc = _traffic(dom, a["bytes"] / launches, a["impl_bytes"] / launches)
    roof.update({"kernel": dom, "traffic": traffic, "traffic_source": tsrc,
                 "peak_source": f"{peak_src} (MEASURED_PEAKS.json)"
                 if peak_src == "measured" else "fallback (profiling recipe)",
                 "per_launch_bytes": a["bytes"] / launches,
                 "per_launch_impl_bytes": a["impl_bytes"] / launches,
                 "timing": ("graph replay with event nodes between launches"
                            if all(p["graph"] for p in prof) else
                            "eager round, events between launches") +
                           f", less {ev_cost * 1e3:.2f} us of event cost per launch",
                 "achieved_with_event_cost": a["bytes"] / launches /
                 (a["ms_events"] / 1e3 / launches) / 1e9})
    breakdown = {c: {"ms_per_round": round(agg[c]["ms"], 4),
                     "ms_per_round_with_event_cost": round(agg[c]["ms_events"], 4),
                     "GB_per_round": round(agg[c]["bytes"] / 1e9, 4),
                     "impl_GB_per_round": round(agg[c]["impl_bytes"] / 1e9, 4),
                     "TFLOP_per_round": round(agg[c]["flops"] / 1e12, 4),
                     "launches": int(agg[c]["launches"]),
                     "GB/s": round(agg[c]["bytes"] / max(1e-12, agg[c]["ms"] / 1e3) / 1e9, 1),
                     "frac_of_hbm": round(agg[c]["bytes"] / max(1e-12, agg[c]["ms"] / 1e3)
                                          / 1e9 / hbm, 4)}
                 for c in classes}
    breakdown["gemm"]["frac_of_tensor_sustained"] = round(
        agg["gemm"]["flops"] / max(1e-12, agg["gemm"]["ms"] / 1e3) / 1e12 / tc_sus, 4)
    breakdown["event_cost_us_per_launch"] = round(ev_cost * 1e3, 3)
    alg_bytes = sum(agg[c]["bytes"] for c in classes)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all / args.steps,
            "repeats": {"n": reps, "statistic": "median",
                        "ms_per_step": [round(x / args.steps, 5) for x in rep_ms]},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random weights N(0,0.02) and uniform prompt ids)",
            "config": {"workload": workload_name(cfg, B),
                       "verify": ("greedy" if cfg.temperature == 0 else
                                  f"sampled, temperature {cfg.temperature:g}"),
                       "global_batch": B * world, "seq_len": int(np.mean([len(p) for p in prompts])),
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (~7 GB of weights+KV streamed per round)",
                       "mean_accept_len": mean_len, "rounds_per_s": args.steps / (ms / 1e3)},
            "clocks": clk,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": B * 8 * 4 + B * 4},
            "gpu_launches": g.launches_per_round() * args.steps * reps,
            "gpu_launches_note": f"launches in the timed region: {reps} repeats of "
                                 f"{args.steps} rounds",
            "acceptance": acceptance(dh),
            "roofline": roof,
            "round_roofline": {"algorithmic_GB": alg_bytes / 1e9,
                               "t_roof_ms": alg_bytes / (hbm * 1e9) * 1e3,
                               "profiled_round_ms": prof_round_ms,
                               "frac_of_timed": (alg_bytes / (hbm * 1e9) * 1e3) / (ms / args.steps)},
            "kernels": breakdown}
    pf_ms, pf_tok = g.prefill_stats()
    line["prefill"] = {"tokens": pf_tok, "ms": pf_ms,
                       "tokens_per_s": pf_tok / (pf_ms / 1e3) if pf_ms > 0 else None,
                       "note": "dmtp_init's prefill of the batch's prompts (target, drafter "
                               "context, MTP rows), device time; the round's kernels, 8 "
                               "positions per sequence per step"}
    rps_nat = args.steps / (ms / 1e3)
    line["projection"] = {
        "note": "B x measured rounds/s x the DMTP blog's per-verify acceptance lengths "
                "(trained models); a projection, not a measurement",
        "tokens_per_s": {k: B * rps_nat * v for k, v in PAGE_PER_VERIFY.items()}}
    g.close()
    del g
    if args.forced_steps > 0 and world == 1:
        line["forced_accept"] = forced_accept(cfg, weights, prompts, 4, args.forced_steps)
    if args.fp8_steps > 0 and world == 1 and cfg.dtype == "bf16" and cfg.d_model % 128 == 0:
        line["fp8_draft_heads"] = fp8_draft_heads(cfg, weights, prompts, 16, args.fp8_steps)
    if args.depth_steps > 0 and world == 1:
        line["depth"] = depth_rounds(cfg, weights, prompts, 4, args.depth_steps)
    if args.list_steps > 0 and world == 1 and cfg.dtype == "bf16":
        line["draft_list"] = draft_list_round(cfg, weights, prompts, 16, args.list_steps)
    if args.hybrid_steps > 0 and world == 1 and args.config == "b32" and args.layers is None:
        try:
            line["hybrid"] = hybrid_round(5, args.hybrid_steps, hbm)
        except Exception as e:  # a side field never takes the headline line down
            line["hybrid"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(cfg, weights, prompts, args.cpu_rounds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
