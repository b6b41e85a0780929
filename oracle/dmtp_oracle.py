"""Float64 NumPy restatement of the DMTP round (TEST INFRASTRUCTURE ONLY).

Sources (cited by page title and section):

* [DMTP] "DMTP: A Better First Token for Block Drafting via MTP" (technical blog):
  §2 division of labour, §3 the residual Δ equation and the dual-anchor slots,
  §5 inference order and target-only prefix acceptance, §6.1 state advancement,
  §6.2 visibility rules, §6.3 KV lifetime, §7 per-verify acceptance length.
* [DFvsMTP] "DFlash vs MTP: Two Paths to Breaking the Autoregressive Decoding
  Bottleneck": "MTP: Sequential Prediction Heads" (the h' = M[RMSNorm; RMSNorm]
  equation), "DFlash: Block Diffusion as a Draft Model" (block-diagonal mask,
  KV injection).
* [colibri] colibri speculative-decoding page: the verify contract, "Undoing rows
  on a model with recurrent state" (per-row copies, swap by pointer), "Every verify
  row gets a decode step's bits".
* [mlxcel] mlxcel manual "MTP and DFlash": the block-versus-chain exactness probe,
  per-row accepts in batched rounds, the replay rollback used here only as a check.

Readings where the pages are silent (also listed in the design notes): the target
hidden that feeds MTP is taken after the target's final norm; h_MTP is the MTP
block output before its final norm; norm gains are ones, eps 1e-6, RoPE base 1e4
(rotate-half pairs (i, i + hd/2)); argmax ties go to the lowest id; the MASK token
is id V-1; drafter slot s (2..7) predicts the token at its own position a+s; the
drafter context K/V at position p is RoPE(Wk c_p, p), Wv c_p with
c_p = RMS(W_fc [taps at p]); Gated DeltaNet uses L2-normalised q, k, sigmoid gates,
no short convolution and no output scale.

Storage: weights arrive already in the model's storage type (bf16 values upcast).
Every intermediate result, the K/V caches and the Gated DeltaNet state included, is
computed and kept in float64: the oracle states the round's arithmetic, not a storage
format. (``kv_store="bf16"`` rounds stored keys and values to bf16 instead; it serves
only as a side check that the pins survive a bf16 cache.)
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

import numpy as np

from .fp8 import fp8_logits, quantize_rows
from .sampling import sampled_scores

F64 = np.float64


# --------------------------------------------------------------------------------------
# Model primitives (textbook definitions; pinned against torch fp64 routines)
# --------------------------------------------------------------------------------------

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half convention, at absolute positions.

    x: [..., heads, hd]; pos: scalar, or array with x's leading shape (one
    position per row). Pair (i, i + hd/2) rotates by pos * theta^(-2i/hd).
    """
    hd = x.shape[-1]
    half = hd // 2
    freq = theta ** (-(np.arange(half, dtype=F64) * 2.0) / hd)
    ang = np.asarray(pos, dtype=F64)[..., None, None] * freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def attend_rows(q: np.ndarray, K: np.ndarray, V: np.ndarray, hi: np.ndarray,
                lo: int = 0) -> np.ndarray:
    """Softmax attention with grouped KV heads.

    q: [R, hq, hd]; K, V: [T, hkv, hd]; row r sees keys lo..hi[r] (inclusive).
    Query head h reads KV head h // (hq / hkv). Scores are scaled by 1/sqrt(hd).
    """
    R, hq, hd = q.shape
    T, hkv, _ = K.shape
    grp = hq // hkv
    out = np.empty_like(q)
    idx = np.arange(T)
    for h in range(hq):
        kh = h // grp
        s = (q[:, h, :] @ K[:, kh, :].T) / np.sqrt(hd)          # [R, T]
        vis = (idx[None, :] >= lo) & (idx[None, :] <= hi[:, None])
        s = np.where(vis, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, kh, :]
    return out


def gdn_step(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray,
             alpha: np.ndarray, beta: np.ndarray):
    """One Gated DeltaNet row for all heads.

    S: [H, dv, dk]; q, k: [H, dk] (already L2-normalised); v: [H, dv]; alpha, beta: [H].
    S <- alpha * S (I - beta k k^T) + beta v k^T ; o = S q.
    Returns (S_new, o [H, dv]).
    """
    Sk = np.einsum("hvk,hk->hv", S, k)
    S_new = (alpha[:, None, None] * S
             - (alpha * beta)[:, None, None] * Sk[:, :, None] * k[:, None, :]
             + beta[:, None, None] * v[:, :, None] * k[:, None, :])
    o = np.einsum("hvk,hk->hv", S_new, q)
    return S_new, o


def l2_normalize(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even, torch's conversion), back as float64."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def argmax_first(logits: np.ndarray) -> int:
    """Greedy pick; exactly equal maxima resolve to the lowest id (np.argmax)."""
    return int(np.argmax(logits))


def top2_gap(logits: np.ndarray) -> float:
    i = int(np.argmax(logits))
    m = logits[i]
    rest = np.concatenate([logits[:i], logits[i + 1:]])
    return float(m - rest.max()) if rest.size else float("inf")


# --------------------------------------------------------------------------------------
# Metrics ([DMTP] §7 per-verify length; §8 first-candidate acceptance)
# --------------------------------------------------------------------------------------

def mean_accept_len(hist) -> float:
    """Per-verify mean acceptance length 1 + sum_k k*hist[k] / sum_k hist[k]
    ([DMTP] §7, "Acceptance Length and End-to-End Throughput")."""
    hist = np.asarray(hist, dtype=F64)
    return 1.0 + float(np.sum(np.arange(hist.size) * hist) / np.sum(hist))


def first_candidate_acceptance(hist) -> float:
    """1 - hist[0] / sum_k hist[k] ([DMTP] §8, "First-Candidate T1 Acceptance")."""
    hist = np.asarray(hist, dtype=F64)
    return 1.0 - float(hist[0] / np.sum(hist))


# --------------------------------------------------------------------------------------
# Per-sequence state
# --------------------------------------------------------------------------------------

@dataclass
class SeqState:
    """State of one sequence between rounds.

    a: target kv_len (positions 0..a-1 processed by the target);
    A: the pending token x_a, emitted by the target but not processed by it;
    tgt_K/tgt_V[l]: [a, hkv, hd] for attention layers (None for GDN layers);
    gdn_S[l]: [H, dv, dk] recurrent state for GDN layers (None for attention);
    dft_K/dft_V[j]: drafter context K/V for positions 0..a-1, per drafter layer;
    mtp_K/mtp_V: MTP private KV for positions 1..a (array row p-1);
    h_mtp: the MTP block output at position a, the hidden state that predicts T1.
    tokens: prompt + every emitted token (ends with A).
    b: the sequence's index in its batch (keys the sampling noise).
    """
    a: int
    A: int
    tgt_K: list
    tgt_V: list
    gdn_S: list
    dft_K: list
    dft_V: list
    mtp_K: np.ndarray
    mtp_V: np.ndarray
    h_mtp: np.ndarray
    tokens: list = field(default_factory=list)
    b: int = 0

    def clone(self) -> "SeqState":
        return copy.deepcopy(self)


# --------------------------------------------------------------------------------------
# The model
# --------------------------------------------------------------------------------------

class OracleModel:
    """Target + MTP module + fusion + block drafter, float64, from synth weights."""

    def __init__(self, cfg, weights: dict, gate: float = 0.05, kv_store: str | None = None,
                 temperature: float = 0.0, sample_seed: int = 0,
                 draft_head_fp8: bool = False, chunk: int = 1024):
        """kv_store: "fp32" (default: keys and values kept exactly, in float64) or
        "bf16" (stored keys and values rounded to bf16 when written; a side check only).
        temperature > 0: the verify picks are target samples (sampling.py) with the given
        sampling seed; 0: argmax picks. draft_head_fp8: the T1 and drafter heads score
        with the E4M3-quantised head (fp8.py); the verify head stays exact. chunk: prompt
        rows per block of the prefill (bounds the [rows, keys] score matrices)."""
        self.cfg = cfg
        self.temperature, self.sample_seed = float(temperature), int(sample_seed)
        self.W = {k: v.detach().to("cpu").double().numpy() if hasattr(v, "detach")
                  else np.asarray(v, dtype=F64) for k, v in weights.items()}
        self.gate = gate
        if kv_store not in (None, "fp32", "bf16"):
            raise ValueError("kv_store: 'fp32' or 'bf16'")
        self.kv_bf16 = kv_store == "bf16"
        self.draft_fp8 = bool(draft_head_fp8)
        if int(chunk) < 1:
            raise ValueError("chunk >= 1")
        self.chunk = int(chunk)
        if self.draft_fp8:
            self.Hq, self.Hs = quantize_rows(self.W["head"])
        c = cfg
        self.eps, self.theta = c.rms_eps, c.rope_theta
        self.hq, self.hkv, self.hd = c.n_heads, c.n_kv_heads, c.head_dim
        self.qd, self.kvd = c.q_dim, c.kv_dim

    # ---- building blocks ------------------------------------------------------------

    def _mlp(self, pfx: str, x: np.ndarray) -> np.ndarray:
        """SwiGLU: W_down (silu(W_gate h) * W_up h) with h = RMSNorm(x)."""
        W, F = self.W, self.cfg.ffn
        h = rms_norm(x, W[f"{pfx}.mlp_norm"], self.eps)
        gu = h @ W[f"{pfx}.wgu"].T
        return (silu(gu[:, :F]) * gu[:, F:]) @ W[f"{pfx}.wdown"].T

    def _qkv(self, pfx: str, x: np.ndarray, pos: np.ndarray):
        W = self.W
        h = rms_norm(x, W[f"{pfx}.attn_norm"], self.eps)
        qkv = h @ W[f"{pfx}.wqkv"].T
        R = x.shape[0]
        q = qkv[:, :self.qd].reshape(R, self.hq, self.hd)
        k = qkv[:, self.qd:self.qd + self.kvd].reshape(R, self.hkv, self.hd)
        v = qkv[:, self.qd + self.kvd:].reshape(R, self.hkv, self.hd)
        return rope(q, pos, self.theta), self._store(rope(k, pos, self.theta)), self._store(v)

    def _store(self, kv: np.ndarray) -> np.ndarray:
        return round_bf16(kv) if self.kv_bf16 else kv

    def attn_layer(self, pfx: str, x: np.ndarray, K: np.ndarray, V: np.ndarray,
                   pos0: int, key0: int = 0):
        """Pre-norm causal decoder layer over R rows at positions pos0..pos0+R-1.

        K, V hold the cached keys for positions key0..pos0-1 (row i <-> position
        key0 + i). Row r attends to every cached key and to rows <= r.
        Returns (x_out, K_all, V_all) with the R new keys appended.
        """
        R = x.shape[0]
        pos = pos0 + np.arange(R)
        q, k, v = self._qkv(pfx, x, pos)
        K2 = np.concatenate([K, k], axis=0)
        V2 = np.concatenate([V, v], axis=0)
        T0 = K.shape[0]
        o = attend_rows(q, K2, V2, hi=T0 + np.arange(R))
        x = x + o.reshape(R, -1) @ self.W[f"{pfx}.wo"].T
        x = x + self._mlp(pfx, x)
        return x, K2, V2

    def gdn_layer(self, pfx: str, x: np.ndarray, S: np.ndarray):
        """Gated DeltaNet layer over R rows, one recurrence step per row.

        Returns (x_out, S_final, [S after row r for each r]). The per-row states
        are the snapshot slots of [colibri] "Undoing rows on a model with
        recurrent state".
        """
        W, c = self.W, self.cfg
        H, dk, dv = c.gdn_heads, c.gdn_dk, c.gdn_dv
        R = x.shape[0]
        h = rms_norm(x, W[f"{pfx}.attn_norm"], self.eps)
        qkv = h @ W[f"{pfx}.gdn_wqkv"].T
        q = l2_normalize(qkv[:, :H * dk].reshape(R, H, dk))
        k = l2_normalize(qkv[:, H * dk:2 * H * dk].reshape(R, H, dk))
        v = qkv[:, 2 * H * dk:].reshape(R, H, dv)
        al = sigmoid(h @ W[f"{pfx}.gdn_wa"].T)
        be = sigmoid(h @ W[f"{pfx}.gdn_wb"].T)
        outs, snaps = [], []
        for r in range(R):
            S, o = gdn_step(S, q[r], k[r], v[r], al[r], be[r])
            outs.append(o.reshape(-1))
            snaps.append(S.copy())
        x = x + np.stack(outs) @ W[f"{pfx}.gdn_wo"].T
        x = x + self._mlp(pfx, x)
        return x, S, snaps

    # ---- target ---------------------------------------------------------------------

    def target_rows(self, st: SeqState, toks, pos0: int, collect_snaps: bool = False,
                    head: bool = True):
        """Target forward over R rows (tokens toks at positions pos0..), in place on
        st's caches (attention K/V appended, GDN state advanced).

        Returns (final-normed hidden [R, d], taps [R, n_taps, d], logits [R, V] or
        None without the head, GDN snapshots {layer: [S after row r]}).
        """
        W, c = self.W, self.cfg
        x = W["emb"][np.asarray(toks)]
        taps, snaps = [], {}
        for l, kind in enumerate(c.layer_kinds):
            if kind == 0:
                x, st.tgt_K[l], st.tgt_V[l] = self.attn_layer(
                    f"L{l}", x, st.tgt_K[l], st.tgt_V[l], pos0)
            else:
                x, st.gdn_S[l], sn = self.gdn_layer(f"L{l}", x, st.gdn_S[l])
                if collect_snaps:
                    snaps[l] = sn
            if l in c.taps:
                taps.append(x.copy())
        hT = rms_norm(x, W["final_norm"], self.eps)
        logits = hT @ W["head"].T if head else None
        return hT, np.stack(taps, axis=1), logits, snaps

    # ---- drafter context (KV injection) ---------------------------------------------

    def drafter_ctx_kv(self, taps: np.ndarray, pos: np.ndarray):
        """Drafter context K/V per drafter layer from target taps.

        [DFvsMTP] "KV injection": target hidden features from a few target layers
        are projected and injected into every draft layer's K/V. Here
        c_p = RMS(W_fc [tap_0; ...; tap_{n-1}]), K_j = RoPE(Wk_j c_p, p), V_j = Wv_j c_p.
        taps: [R, n_taps, d]; pos: [R].
        """
        W = self.W
        R = taps.shape[0]
        c = rms_norm(taps.reshape(R, -1) @ W["dft.fc"].T, W["dft.norm_c"], self.eps)
        out = []
        for j in range(self.cfg.draft_layers):
            w = W[f"D{j}.wqkv"]
            k = (c @ w[self.qd:self.qd + self.kvd].T).reshape(R, self.hkv, self.hd)
            v = (c @ w[self.qd + self.kvd:].T).reshape(R, self.hkv, self.hd)
            out.append((self._store(rope(k, pos, self.theta)), self._store(v)))
        return out

    # ---- MTP module -----------------------------------------------------------------

    def mtp_rows(self, st: SeqState, hT_prev: np.ndarray, toks, pos0: int):
        """MTP module over rows at positions pos0..pos0+R-1 (in place on st.mtp_K/V).

        [DFvsMTP] "MTP: Sequential Prediction Heads": h' = M [RMSNorm(h); RMSNorm(Emb(t))],
        then the module's own transformer block with its causal KV ([DMTP] §6.3:
        MTP keeps a private KV cache). hT_prev[r] is the target's final-normed
        hidden at position pos0 + r - 1 and toks[r] the token at pos0 + r.
        Returns the block outputs [R, d] (before the MTP final norm).
        """
        W = self.W
        e = W["emb"][np.asarray(toks)]
        u = np.concatenate([rms_norm(hT_prev, W["mtp.norm_h"], self.eps),
                            rms_norm(e, W["mtp.norm_e"], self.eps)], axis=1)
        x = u @ W["mtp.proj"].T
        x, st.mtp_K, st.mtp_V = self.attn_layer("mtp", x, st.mtp_K, st.mtp_V, pos0)
        return x

    def draft_head(self, Y: np.ndarray) -> np.ndarray:
        """Draft logits H Y^T of normalised rows Y: exact, or with the E4M3 head copy
        ([DMTP] §6.5 drafting-side head quantization; fp8.py)."""
        if self.draft_fp8:
            return fp8_logits(Y, self.Hq, self.Hs)
        return Y @ self.W["head"].T

    def t1_head(self, h_mtp: np.ndarray) -> np.ndarray:
        """Logits of the first candidate: H RMS_f(h_MTP) ([DMTP] §5 step 1, §6.5)."""
        W = self.W
        return self.draft_head(rms_norm(h_mtp[None], W["mtp.final_norm"], self.eps))[0]

    # ---- fusion and block drafter -----------------------------------------------------

    def fusion_delta(self, T1: int, h_mtp: np.ndarray) -> np.ndarray:
        """Δ = W [RMS_e(e_T1); RMS_m(h_MTP)] ([DMTP] §3, the Δ equation)."""
        W = self.W
        e = W["emb"][T1]
        z = np.concatenate([rms_norm(e, W["fuse.norm_e"], self.eps),
                            rms_norm(h_mtp, W["fuse.norm_m"], self.eps)])
        return W["fuse.w"] @ z

    def drafter_slots(self, A: int, T1: int, delta: np.ndarray) -> np.ndarray:
        """The eight dual-anchor slots [E(A), E(T1) + Δ, E(MASK) x 6] ([DMTP] §3)."""
        E = self.W["emb"]
        return np.stack([E[A], E[T1] + delta] + [E[self.cfg.mask_id]] * 6)

    def drafter_forward(self, X: np.ndarray, st: SeqState, a: int, with_head_in: bool = False):
        """One parallel block forward over the 8 slots at positions a..a+7.

        Every slot attends to the context K/V at positions max(0, a - window)..a-1
        ([DMTP] §6.2: a 4096-position window ending just before the anchor) and to all 8
        block slots with no mask inside the block ([DFvsMTP], block-diagonal mask).
        Returns drafter logits [6, V] for slots 2..7 (each predicts the token at its
        own position), and with ``with_head_in`` also the normalised rows the head reads.
        """
        W, c = self.W, self.cfg
        lo = max(0, a - c.draft_window)
        pos = a + np.arange(8)
        for j in range(c.draft_layers):
            pfx = f"D{j}"
            q, k, v = self._qkv(pfx, X, pos)
            K = np.concatenate([st.dft_K[j][lo:a], k], axis=0)
            V = np.concatenate([st.dft_V[j][lo:a], v], axis=0)
            o = attend_rows(q, K, V, hi=np.full(8, K.shape[0] - 1))
            X = X + o.reshape(8, -1) @ W[f"{pfx}.wo"].T
            X = X + self._mlp(pfx, X)
        hn = rms_norm(X[2:8], W["dft.final_norm"], self.eps)
        return (self.draft_head(hn), hn) if with_head_in else self.draft_head(hn)

    # ---- prefill ----------------------------------------------------------------------

    def empty_state(self) -> SeqState:
        c = self.cfg
        z = lambda: np.zeros((0, self.hkv, self.hd), dtype=F64)
        return SeqState(
            a=0, A=-1,
            tgt_K=[z() if k == 0 else None for k in c.layer_kinds],
            tgt_V=[z() if k == 0 else None for k in c.layer_kinds],
            gdn_S=[None if k == 0 else np.zeros((c.gdn_heads, c.gdn_dv, c.gdn_dk), F64)
                   for k in c.layer_kinds],
            dft_K=[z() for _ in range(c.draft_layers)],
            dft_V=[z() for _ in range(c.draft_layers)],
            mtp_K=z(), mtp_V=z(), h_mtp=np.zeros(c.d_model, F64))

    def prefill(self, prompt, adopt_A=None, b: int = 0) -> SeqState:
        """Initialise all three models' states from a prompt ([DMTP] §6.1).

        Target over x_0..x_{P-1}; A = argmax H h^T_{P-1}; drafter context K/V for
        positions 0..P-1; MTP rows p = 1..P (token x_p, hidden h^T_{p-1}, with
        x_P = A), so that h_MTP (the block output at P) predicts x_{P+1}.
        ``adopt_A``: another implementation's pick for A, taken when it lies within the
        near-tie gate of the maximum (see ``round``). A is an argmax pick at any
        temperature (reading: sampling starts with the round's verify picks). ``b``: the
        sequence's index in its batch.
        """
        prompt = [int(t) for t in prompt]
        P = len(prompt)
        st = self.empty_state()
        st.b = int(b)
        # Rows go through in blocks of at most `chunk`: a row attends causally, so a block
        # sees exactly the keys of the blocks before it and its own earlier rows; only the
        # size of the score matrices changes.
        C = self.chunk
        hT, taps = [], []
        for c0 in range(0, P, C):
            h, t, _, _ = self.target_rows(st, prompt[c0:c0 + C], c0, head=False)
            hT.append(h)
            taps.append(t)
        hT, taps = np.concatenate(hT), np.concatenate(taps)
        log = {"gaps": {}, "adopted": [], "mismatch": []}
        A = self._pick(hT[P - 1] @ self.W["head"].T, adopt_A, log, "A")
        self.prefill_log = log
        for j, (k, v) in enumerate(self.drafter_ctx_kv(taps, np.arange(P))):
            st.dft_K[j], st.dft_V[j] = k, v
        mtok = prompt[1:] + [A]
        for c0 in range(0, P, C):
            out = self.mtp_rows(st, hT[c0:c0 + C], mtok[c0:c0 + C], 1 + c0)
        st.h_mtp = out[-1].copy()
        st.a, st.A = P, A
        st.tokens = prompt + [A]
        return st

    # ---- plain greedy decoding (the losslessness reference) ------------------------------

    def greedy_decode(self, prompt, n_new: int) -> list[int]:
        """Plain one-token-per-forward greedy decoding of the target: x_P, x_{P+1}, ...

        [colibri] verify contract: with the same arithmetic, speculative output equals
        plain decoding. Each step is a one-row target forward (target_rows with R=1),
        the same routine the verify below runs row by row.
        """
        st = self.prefill(prompt)
        out = [st.A]
        tok, pos = st.A, st.a
        while len(out) < n_new:
            _, _, logits, _ = self.target_rows(st, [tok], pos)
            tok, pos = argmax_first(logits[0]), pos + 1
            out.append(tok)
        return out[:n_new]

    def sampled_decode(self, prompt, n_new: int, b: int = 0) -> list[int]:
        """Plain one-token-per-forward decoding with the target's samples: the token at
        position p is argmax(l / temperature + G(b, p)) of the one-row forward at p - 1
        (sampling.py); A, the first token after the prompt, is the argmax pick. The
        losslessness reference of sampled verification ([DMTP] §5 target-only
        verification, [colibri] verify contract)."""
        st = self.prefill(prompt, b=b)
        out = [st.A]
        tok, pos = st.A, st.a
        while len(out) < n_new:
            _, _, logits, _ = self.target_rows(st, [tok], pos)
            tok = argmax_first(sampled_scores(logits[0], self.temperature, self.sample_seed,
                                              b, pos + 1))
            pos += 1
            out.append(tok)
        return out[:n_new]

    # ---- one DMTP round ------------------------------------------------------------------

    def _pick(self, logits, adopt, log, where):
        top = argmax_first(logits)
        gap = top2_gap(logits)
        log["gaps"][where] = gap
        if adopt is None or int(adopt) == top:
            return top
        adopt = int(adopt)
        if logits[adopt] >= logits[top] - self.gate:
            log["adopted"].append((where, top, adopt, float(logits[top] - logits[adopt])))
            return adopt
        log["mismatch"].append((where, top, adopt, float(logits[top] - logits[adopt])))
        return top

    def round(self, st: SeqState, forced=None, adopt=None, want_logits: bool = True,
              depth=7, draft_list=None):
        """One DMTP round on one sequence, in place on ``st``.

        Steps ([DMTP] §5 and §6.1):
          a1 T1 = argmax H RMS_f(h_MTP), h_MTP as the previous round left it;
          a2 Δ and the slots [E(A), E(T1)+Δ, E(MASK) x 6];
          a3 one block-drafter forward -> T2..T7;
          a4 target verify of rows [A, T1..T7] at positions a..a+7, each row by the
             one-row decode routine ([colibri]: every verify row gets a decode step's
             bits) -> g_0..g_7 (argmax picks, or at temperature > 0 the target's
             samples for positions a+1..a+8, sampling.py);
          a5 n = longest prefix with T_j = g_{j-1}; commit T_1..T_n and g_n; the target
             KV keeps a+n+1 positions; a GDN state takes the snapshot after row n;
          a6 drafter context K/V for positions a..a+n from the verify taps; MTP rows at
             positions a+1..a+n+1 (token x_p, hidden h^T_{p-1}); h_MTP <- output at
             a+n+1.

        ``forced``: 7 ids overriding T1..T7 (T1 is replaced right after a1, so the
        fusion and drafter see it; T2..T7 after a3). ``adopt``: dict with optional
        'T1', 'T' (7 ids) and 'g' (8 ids) from another implementation; at any argmax
        where that id is within ``gate`` of the maximum it is taken instead (near-tie
        lock-step). ``depth``: how many drafts the verify carries (0..7; 7 is the DMTP
        round), or a callable (drafts, confidences) -> depth called after a3 with each
        probability each draft head gives its own pick (gate.head_confidence): the verify is
        then rows [A, T1..T_depth] and at most depth drafts are accepted (colibri doc: a
        verify of k drafts is one forward of k + 1 rows). ``draft_list``: None, or a
        boolean mask [V] of the tokens the draft heads score (shortlist.VocabList.members,
        colibri doc's frequent-token list): T1..T7 are then the argmax over the listed
        tokens, while the verify still scores every token. Returns a record of every
        intermediate.
        """
        c, W = self.cfg, self.W
        adopt = adopt or {}
        log = {"gaps": {}, "adopted": [], "mismatch": []}
        rec = {"a": st.a, "A": st.A, "log": log}
        a, A = st.a, st.A
        h_mtp = st.h_mtp.copy()
        rec["h_mtp_in"] = h_mtp

        # a1
        t1_logits = self.t1_head(h_mtp)
        rec["t1_head_in"] = rms_norm(h_mtp[None], W["mtp.final_norm"], self.eps)
        listed = ((lambda l: l) if draft_list is None else
                  (lambda l: np.where(draft_list, l, -np.inf)))
        ad = adopt.get("T")
        T1 = self._pick(listed(t1_logits), ad[0] if ad is not None else adopt.get("T1"), log,
                        "T1")
        if forced is not None:
            T1 = int(forced[0])
        # a2
        delta = self.fusion_delta(T1, h_mtp)
        X = self.drafter_slots(A, T1, delta)
        # a3
        dlog, rec["draft_head_in"] = self.drafter_forward(X, st, a, with_head_in=True)
        drafts = [T1]
        for s in range(6):
            drafts.append(self._pick(listed(dlog[s]), ad[s + 1] if ad is not None else None,
                                     log, f"T{s + 2}"))
        if forced is not None:
            drafts = [T1] + [int(t) for t in forced[1:7]]
        if callable(depth) or want_logits:
            # each head's probability of its own pick over the scores it makes (the listed
            # tokens when a list is set), within the window of its best
            from .gate import head_confidence
            conf = [head_confidence(listed(t1_logits))] + [head_confidence(listed(dlog[s]))
                                                          for s in range(6)]
            rec["draft_confidence"] = conf
        if callable(depth):
            depth = depth(list(drafts), conf)
        depth = int(depth)
        if not 0 <= depth <= 7:
            raise ValueError("depth in 0..7")
        rec["depth"] = depth
        # a4: each row by the one-row routine on a working copy of the caches
        work = st.clone()
        rows = [A] + drafts
        hT_rows, tap_rows, vlog, g, vsc = [], [], [], [], []
        snaps = {}
        adg = adopt.get("g")
        for s in range(depth + 1):
            hT, taps, logits, sn = self.target_rows(work, [rows[s]], a + s, collect_snaps=True)
            hT_rows.append(hT[0]); tap_rows.append(taps[0]); vlog.append(logits[0])
            for l, lst in sn.items():
                snaps.setdefault(l, []).append(lst[0])
            sc = logits[0]
            if self.temperature > 0:  # the target's sample for position a + s + 1
                sc = sampled_scores(logits[0], self.temperature, self.sample_seed, st.b,
                                    a + s + 1)
                vsc.append(sc)
            g.append(self._pick(sc, adg[s] if adg is not None else None, log, f"g{s}"))
        # a5
        n = 0
        while n < depth and drafts[n] == g[n]:
            n += 1
        committed = drafts[:n] + [g[n]]
        keep = a + n + 1
        for l, kind in enumerate(c.layer_kinds):
            if kind == 0:
                st.tgt_K[l] = work.tgt_K[l][:keep]
                st.tgt_V[l] = work.tgt_V[l][:keep]
            else:
                st.gdn_S[l] = snaps[l][n]
        # a6
        hT_rows = np.stack(hT_rows)
        tap_rows = np.stack(tap_rows)
        for j, (k, v) in enumerate(self.drafter_ctx_kv(tap_rows[:n + 1], a + np.arange(n + 1))):
            st.dft_K[j] = np.concatenate([st.dft_K[j][:a], k])
            st.dft_V[j] = np.concatenate([st.dft_V[j][:a], v])
        out = self.mtp_rows(st, hT_rows[:n + 1], committed, a + 1)
        st.h_mtp = out[n].copy()
        st.a, st.A = keep, g[n]
        st.tokens = st.tokens + committed

        rec.update(T1=T1, delta=delta, slots=X, drafts=drafts, g=g, n=n,
                   committed=committed, accept_len=n + 1, kv_len=st.a, mtp_len=st.a + 1,
                   snap_slot=(n if c.has_gdn else -1), h_mtp_out=st.h_mtp.copy(),
                   hT_rows=hT_rows)
        if want_logits:
            rec.update(t1_logits=t1_logits, draft_logits=dlog, verify_logits=np.stack(vlog))
            if vsc:
                rec["verify_scores"] = np.stack(vsc)
        return rec
