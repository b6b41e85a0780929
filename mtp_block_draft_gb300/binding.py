"""ctypes binding of libdmtp.so: the C ABI of include/dmtp.h with the same names.

Argument marshalling only. Every step of the round runs in the library's CUDA
kernels; PyTorch supplies device memory (weights, workspace, outputs) and the
stream. Importing works without a GPU; loading the library requires that it has
been built (``__graft_entry__.build()`` or ``python -m mtp_block_draft_gb300.build``)
and raises otherwise - there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdmtp.so")

DMTP_MAX_LAYERS = 64
DMTP_MAX_DRAFT_LAYERS = 8
DMTP_MAX_TAPS = 8

ERRORS = {0: "DMTP_OK", -1: "DMTP_EINVAL", -2: "DMTP_ENOMEM", -3: "DMTP_ECAPACITY",
          -4: "DMTP_ECUDA", -5: "DMTP_EDEVICE", -6: "DMTP_ESTATE"}

# every symbol the headers under include/ declare
EXPORTS = ("dmtp_workspace_size", "dmtp_init", "dmtp_round", "dmtp_round_host",
           "dmtp_read_state", "dmtp_round_launches", "dmtp_round_profile", "dmtp_free",
           "dmtp_strerror", "dmtp_t1_head_noalloc", "dmtp_prefill_stats",
           "dmtp_selftest_timeout", "dmtp_set_draft_list", "dmtp_round_depth",
           "dmtp_error_word",
           "dmtp_gate_create", "dmtp_gate_forward", "dmtp_gate_draft_cost",
           "dmtp_gate_result", "dmtp_gate_pick", "dmtp_gate_pick_p", "dmtp_gate_read",
           "dmtp_gate_free", "dmtp_vocab_create", "dmtp_vocab_begin_request",
           "dmtp_vocab_picked", "dmtp_vocab_ids", "dmtp_vocab_mask", "dmtp_vocab_counts",
           "dmtp_vocab_stats_read", "dmtp_vocab_free")

DMTP_GATE_MAX_DRAFTS = 32
DMTP_GATE_MAX_ROWS = 64
DMTP_GATE_BINS = 10

PROFILE_CLASSES = ("gemm", "lm_head", "attention", "gdn", "other")


class dmtp_config(C.Structure):
    _fields_ = [("vocab", C.c_int), ("d_model", C.c_int), ("n_layers", C.c_int),
                ("n_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
                ("ffn", C.c_int), ("gdn_heads", C.c_int), ("gdn_dk", C.c_int),
                ("gdn_dv", C.c_int), ("layer_kind", C.c_uint8 * DMTP_MAX_LAYERS),
                ("draft_layers", C.c_int), ("draft_window", C.c_int), ("n_taps", C.c_int),
                ("tap_layers", C.c_int * DMTP_MAX_TAPS), ("mask_id", C.c_int),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("max_ctx", C.c_int),
                ("max_batch", C.c_int), ("dtype", C.c_int), ("temperature", C.c_float),
                ("sample_seed", C.c_uint64), ("draft_head_fp8", C.c_int),
                ("draft_list_cap", C.c_int), ("variable_depth", C.c_int),
                ("draft_confidence", C.c_int), ("deterministic", C.c_int)]


_LAYER_FIELDS = ("attn_norm", "wqkv", "wo", "gdn_wqkv", "gdn_wa", "gdn_wb", "gdn_wo",
                 "mlp_norm", "wgu", "wdown")


class dmtp_layer_weights(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in _LAYER_FIELDS]


class dmtp_weights(C.Structure):
    _fields_ = [("emb", C.c_void_p), ("head", C.c_void_p), ("final_norm", C.c_void_p),
                ("layers", dmtp_layer_weights * DMTP_MAX_LAYERS),
                ("mtp_norm_h", C.c_void_p), ("mtp_norm_e", C.c_void_p), ("mtp_proj", C.c_void_p),
                ("mtp", dmtp_layer_weights), ("mtp_final_norm", C.c_void_p),
                ("fuse_norm_e", C.c_void_p), ("fuse_norm_m", C.c_void_p), ("fuse_w", C.c_void_p),
                ("dft_fc", C.c_void_p), ("dft_norm_c", C.c_void_p),
                ("dft", dmtp_layer_weights * DMTP_MAX_DRAFT_LAYERS),
                ("dft_final_norm", C.c_void_p)]


_OUT_INT = ("committed", "n_accepted", "drafts", "picks", "kv_len", "mtp_len", "snap_slot")
_OUT_FLOAT = ("t1_logits", "draft_logits", "verify_logits", "delta", "h_mtp", "draft_conf")


class dmtp_round_out(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in _OUT_INT + _OUT_FLOAT]


class dmtp_gate_stats(C.Structure):
    _fields_ = [("max_drafts", C.c_int), ("a", C.c_double * DMTP_GATE_MAX_DRAFTS),
                ("t", C.c_double * (DMTP_GATE_MAX_ROWS + 1)), ("d", C.c_double),
                ("d_measured", C.c_int), ("rho", C.c_double), ("picks", C.c_longlong),
                ("since_plain", C.c_longlong), ("bin_judged", C.c_longlong * DMTP_GATE_BINS),
                ("bin_accepted", C.c_longlong * DMTP_GATE_BINS)]


class dmtp_vocab_stats(C.Structure):
    _fields_ = [("vocab", C.c_int), ("listed", C.c_int), ("counted", C.c_int),
                ("rebuilds", C.c_int64), ("appended", C.c_int64), ("picks", C.c_int64),
                ("picks_in", C.c_int64)]


class dmtp_profile(C.Structure):
    _fields_ = [("ms", C.c_double * 8), ("bytes", C.c_double * 8), ("flops", C.c_double * 8),
                ("impl_bytes", C.c_double * 8), ("launches", C.c_int * 8),
                ("round_ms", C.c_double), ("graph", C.c_int)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libdmtp.so and declare the prototypes; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run __graft_entry__.build() first")
    lib = C.CDLL(path)
    P = C.c_void_p
    lib.dmtp_workspace_size.argtypes = [C.POINTER(dmtp_config), C.c_int, C.POINTER(C.c_size_t)]
    lib.dmtp_workspace_size.restype = C.c_int
    lib.dmtp_init.argtypes = [C.POINTER(dmtp_config), C.POINTER(dmtp_weights), P, C.c_size_t,
                              P, P, C.c_int, P, C.POINTER(P)]
    lib.dmtp_init.restype = C.c_int
    lib.dmtp_round.argtypes = [P, C.POINTER(dmtp_round_out), P]
    lib.dmtp_round.restype = C.c_int
    lib.dmtp_round_depth.argtypes = [P, C.POINTER(dmtp_round_out), P, C.c_int]
    lib.dmtp_round_depth.restype = C.c_int
    lib.dmtp_round_host.argtypes = [P, P, P]
    lib.dmtp_round_host.restype = C.c_int
    lib.dmtp_read_state.argtypes = [P, P, P, P]
    lib.dmtp_read_state.restype = C.c_int
    lib.dmtp_round_launches.argtypes = [P]
    lib.dmtp_round_launches.restype = C.c_int
    lib.dmtp_prefill_stats.argtypes = [P, C.POINTER(C.c_double), C.POINTER(C.c_int64)]
    lib.dmtp_prefill_stats.restype = C.c_int
    lib.dmtp_round_profile.argtypes = [P, C.POINTER(dmtp_profile)]
    lib.dmtp_round_profile.restype = C.c_int
    lib.dmtp_set_draft_list.argtypes = [P, P, C.c_int]
    lib.dmtp_set_draft_list.restype = C.c_int
    lib.dmtp_selftest_timeout.argtypes = [P, C.c_uint64]
    lib.dmtp_selftest_timeout.restype = C.c_int
    lib.dmtp_error_word.argtypes = [P]
    lib.dmtp_error_word.restype = C.c_uint32
    lib.dmtp_free.argtypes = [P]
    lib.dmtp_free.restype = None
    lib.dmtp_t1_head_noalloc.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, C.c_float, P, P, P]
    lib.dmtp_t1_head_noalloc.restype = C.c_int
    lib.dmtp_strerror.argtypes = [C.c_int]
    lib.dmtp_strerror.restype = C.c_char_p
    D = C.POINTER(C.c_double)
    lib.dmtp_gate_create.argtypes = [C.c_int, D, C.POINTER(P)]
    lib.dmtp_gate_forward.argtypes = [P, C.c_int, C.c_double]
    lib.dmtp_gate_draft_cost.argtypes = [P, C.c_double]
    lib.dmtp_gate_result.argtypes = [P, C.c_int, C.c_int, D]
    lib.dmtp_gate_pick.argtypes = [P, C.c_int, C.POINTER(C.c_int), D]
    lib.dmtp_gate_pick_p.argtypes = [P, C.c_int, D, C.POINTER(C.c_int), D]
    lib.dmtp_gate_read.argtypes = [P, C.POINTER(dmtp_gate_stats)]
    for f in ("create", "forward", "draft_cost", "result", "pick", "pick_p", "read"):
        getattr(lib, "dmtp_gate_" + f).restype = C.c_int
    lib.dmtp_gate_free.argtypes = [P]
    lib.dmtp_gate_free.restype = None
    lib.dmtp_vocab_create.argtypes = [C.c_int, C.c_int, C.POINTER(P)]
    lib.dmtp_vocab_begin_request.argtypes = [P, P, C.c_int64, C.c_int]
    lib.dmtp_vocab_picked.argtypes = [P, P, C.c_int64]
    lib.dmtp_vocab_ids.argtypes = [P, P, C.POINTER(C.c_int)]
    lib.dmtp_vocab_mask.argtypes = [P, P]
    lib.dmtp_vocab_counts.argtypes = [P, P]
    lib.dmtp_vocab_stats_read.argtypes = [P, C.POINTER(dmtp_vocab_stats)]
    for f in ("create", "begin_request", "picked", "ids", "mask", "counts", "stats_read"):
        getattr(lib, "dmtp_vocab_" + f).restype = C.c_int
    lib.dmtp_vocab_free.argtypes = [P]
    lib.dmtp_vocab_free.restype = None
    _lib = lib
    return lib


class DmtpError(RuntimeError):
    def __init__(self, code: int, what: str, word: int = 0):
        msg = load_library().dmtp_strerror(code).decode()
        extra = f"; device error word 0x{word:x}" if word else ""
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({msg}{extra})")
        self.code = code
        self.word = word


def _check(code: int, what: str, ctx=None):
    if code != 0:
        word = int(load_library().dmtp_error_word(ctx)) if ctx else 0
        raise DmtpError(code, what, word)


def make_config(cfg, max_ctx: int, max_batch: int | None = None) -> dmtp_config:
    """dmtp_config from a synth.DmtpConfig."""
    c = dmtp_config()
    c.vocab, c.d_model, c.n_layers = cfg.vocab, cfg.d_model, cfg.n_layers
    c.n_heads, c.n_kv_heads, c.head_dim, c.ffn = (cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                                                  cfg.ffn)
    c.gdn_heads, c.gdn_dk, c.gdn_dv = cfg.gdn_heads, cfg.gdn_dk, cfg.gdn_dv
    for l, k in enumerate(cfg.layer_kinds):
        c.layer_kind[l] = k
    c.draft_layers, c.draft_window = cfg.draft_layers, cfg.draft_window
    c.n_taps = cfg.n_taps
    for i, t in enumerate(cfg.taps):
        c.tap_layers[i] = t
    c.mask_id = cfg.mask_id
    c.rms_eps, c.rope_theta = cfg.rms_eps, cfg.rope_theta
    c.max_ctx = max_ctx
    c.max_batch = cfg.batch if max_batch is None else max_batch
    c.dtype = 0 if cfg.dtype == "fp32" else 1
    c.temperature = cfg.temperature
    c.sample_seed = cfg.sample_seed
    c.draft_head_fp8 = 1 if cfg.draft_head_fp8 else 0
    c.draft_list_cap = int(getattr(cfg, "draft_list_cap", 0))
    c.variable_depth = 1 if getattr(cfg, "variable_depth", False) else 0
    c.draft_confidence = 1 if getattr(cfg, "draft_confidence", False) else 0
    c.deterministic = 1 if getattr(cfg, "deterministic", False) else 0
    return c


def _ptr(t) -> int:
    return t.data_ptr()


def make_weights(cfg, w: dict) -> dmtp_weights:
    """dmtp_weights of device pointers from the synth weight dict (tensors on CUDA)."""
    s = dmtp_weights()
    s.emb, s.head, s.final_norm = _ptr(w["emb"]), _ptr(w["head"]), _ptr(w["final_norm"])

    def fill(dst, pfx):
        for f in _LAYER_FIELDS:
            k = f"{pfx}.{f}"
            setattr(dst, f, _ptr(w[k]) if k in w else None)

    for l in range(cfg.n_layers):
        fill(s.layers[l], f"L{l}")
    s.mtp_norm_h, s.mtp_norm_e, s.mtp_proj = (_ptr(w["mtp.norm_h"]), _ptr(w["mtp.norm_e"]),
                                              _ptr(w["mtp.proj"]))
    fill(s.mtp, "mtp")
    s.mtp_final_norm = _ptr(w["mtp.final_norm"])
    s.fuse_norm_e, s.fuse_norm_m, s.fuse_w = (_ptr(w["fuse.norm_e"]), _ptr(w["fuse.norm_m"]),
                                              _ptr(w["fuse.w"]))
    s.dft_fc, s.dft_norm_c = _ptr(w["dft.fc"]), _ptr(w["dft.norm_c"])
    for j in range(cfg.draft_layers):
        fill(s.dft[j], f"D{j}")
    s.dft_final_norm = _ptr(w["dft.final_norm"])
    return s


def default_max_ctx(prompts, rounds: int) -> int:
    return max(len(p) for p in prompts) + 8 * (rounds + 4) + 32


class DmtpRound:
    """One context of the round library: dmtp_init on construction (prefill),
    dmtp_round per call, dmtp_free on close()."""

    def __init__(self, cfg, weights: dict, prompts, max_ctx: int, stream=None):
        import torch
        self.lib = load_library()
        self.cfg = cfg
        self.B = len(prompts)
        self.weights = weights  # keep the tensors alive
        self.ccfg = make_config(cfg, max_ctx, max_batch=self.B)
        self.cw = make_weights(cfg, weights)
        nbytes = C.c_size_t()
        _check(self.lib.dmtp_workspace_size(C.byref(self.ccfg), self.B, C.byref(nbytes)),
               "dmtp_workspace_size")
        dev = weights["emb"].device
        self.workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        ids = np.ascontiguousarray(np.concatenate([np.asarray(p, np.int32) for p in prompts]))
        lens = np.ascontiguousarray(np.array([len(p) for p in prompts], np.int32))
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        ctx = C.c_void_p()
        _check(self.lib.dmtp_init(C.byref(self.ccfg), C.byref(self.cw),
                                  C.c_void_p(self.workspace.data_ptr()), nbytes.value,
                                  ids.ctypes.data_as(C.c_void_p), lens.ctypes.data_as(C.c_void_p),
                                  self.B, C.c_void_p(self.stream.cuda_stream), C.byref(ctx)),
               "dmtp_init")
        self.ctx = ctx
        self.device = dev

    # ---- rounds ----------------------------------------------------------------------
    def round(self, out: dict | None = None, forced=None, depth: int = 7):
        """Enqueue one round. out: name -> preallocated CUDA tensor (fields of
        dmtp_round_out); forced: CUDA int32 [B, 7] or None; depth: drafts the verify
        carries (dmtp_round_depth; 7 is dmtp_round)."""
        o = dmtp_round_out()
        if out:
            for k, t in out.items():
                setattr(o, k, t.data_ptr())
        f = C.c_void_p(forced.data_ptr()) if forced is not None else None
        if depth == 7:
            _check(self.lib.dmtp_round(self.ctx, C.byref(o), f), "dmtp_round", self.ctx)
        else:
            _check(self.lib.dmtp_round_depth(self.ctx, C.byref(o), f, int(depth)),
                   "dmtp_round_depth", self.ctx)

    def alloc_out(self, ints=True, floats=False):
        import torch
        B, V, d = self.B, self.cfg.vocab, self.cfg.d_model
        dev = self.device
        shapes = {"committed": (B, 8), "n_accepted": (B,), "drafts": (B, 7), "picks": (B, 8),
                  "kv_len": (B,), "mtp_len": (B,), "snap_slot": (B,)}
        out = {}
        if ints:
            for k, s in shapes.items():
                out[k] = torch.empty(s, dtype=torch.int32, device=dev)
        if floats:
            fs = {"t1_logits": (B, V), "draft_logits": (B, 6, V), "verify_logits": (B, 8, V),
                  "delta": (B, d), "h_mtp": (B, d)}
            if getattr(self.cfg, "draft_confidence", False):
                fs["draft_conf"] = (B, 7)
            for k, s in fs.items():
                out[k] = torch.empty(s, dtype=torch.float32, device=dev)
        return out

    def round_host(self, committed: np.ndarray | None = None, n_acc: np.ndarray | None = None):
        """One round with host outputs (pinned or pageable numpy int32 arrays)."""
        cp = committed.ctypes.data_as(C.c_void_p) if committed is not None else None
        npt = n_acc.ctypes.data_as(C.c_void_p) if n_acc is not None else None
        _check(self.lib.dmtp_round_host(self.ctx, cp, npt), "dmtp_round_host", self.ctx)

    def read_state(self):
        kv = np.zeros(self.B, np.int32)
        A = np.zeros(self.B, np.int32)
        hist = np.zeros(8, np.uint64)
        _check(self.lib.dmtp_read_state(self.ctx, kv.ctypes.data_as(C.c_void_p),
                                        A.ctypes.data_as(C.c_void_p),
                                        hist.ctypes.data_as(C.c_void_p)), "dmtp_read_state",
               self.ctx)
        return kv, A, hist

    def profile_round(self) -> dict:
        """One real round with CUDA events around every launch: per kernel class the
        summed device ms, algorithmic bytes and flops, and the launch count."""
        p = dmtp_profile()
        _check(self.lib.dmtp_round_profile(self.ctx, C.byref(p)), "dmtp_round_profile")
        out = {"round_ms": p.round_ms, "graph": bool(p.graph)}
        for i, name in enumerate(PROFILE_CLASSES):
            out[name] = {"ms": p.ms[i], "bytes": p.bytes[i], "flops": p.flops[i],
                         "impl_bytes": p.impl_bytes[i], "launches": p.launches[i]}
        return out

    def prefill_stats(self) -> tuple[float, int]:
        """(device ms, prompt tokens) of the prefill dmtp_init ran."""
        ms = C.c_double()
        tok = C.c_int64()
        _check(self.lib.dmtp_prefill_stats(self.ctx, C.byref(ms), C.byref(tok)),
               "dmtp_prefill_stats")
        return ms.value, tok.value

    def set_draft_list(self, ids):
        """dmtp_set_draft_list: the draft heads score only these (strictly increasing)
        token ids from the next round on; an empty list turns it off."""
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(-1))
        _check(self.lib.dmtp_set_draft_list(self.ctx, a.ctypes.data if a.size else None,
                                            int(a.size)), "dmtp_set_draft_list")

    def selftest_timeout(self, limit_ns: int):
        """dmtp_selftest_timeout: a bounded device wait that gives up after limit_ns."""
        _check(self.lib.dmtp_selftest_timeout(self.ctx, int(limit_ns)), "dmtp_selftest_timeout")

    def launches_per_round(self) -> int:
        return int(self.lib.dmtp_round_launches(self.ctx))

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.dmtp_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _doubles(xs):
    if xs is None:
        return None
    xs = [float(x) for x in xs]
    return (C.c_double * max(1, len(xs)))(*xs)


class DmtpGate:
    """The draft-depth gate of include/dmtp_gate.h (host-only; argument marshalling)."""

    def __init__(self, max_drafts: int, priors=None):
        self.lib = load_library()
        self.g = C.c_void_p()
        _check(self.lib.dmtp_gate_create(int(max_drafts), _doubles(priors), C.byref(self.g)),
               "dmtp_gate_create")

    def forward(self, rows: int, seconds: float):
        _check(self.lib.dmtp_gate_forward(self.g, int(rows), float(seconds)), "dmtp_gate_forward")

    def draft_cost(self, seconds: float):
        _check(self.lib.dmtp_gate_draft_cost(self.g, float(seconds)), "dmtp_gate_draft_cost")

    def result(self, judged: int, accepted: int, p=None):
        _check(self.lib.dmtp_gate_result(self.g, int(judged), int(accepted), _doubles(p)),
               "dmtp_gate_result")

    def pick(self, proposed: int):
        k, v = C.c_int(), C.c_double()
        _check(self.lib.dmtp_gate_pick(self.g, int(proposed), C.byref(k), C.byref(v)),
               "dmtp_gate_pick")
        return k.value, v.value

    def pick_p(self, p):
        k, v = C.c_int(), C.c_double()
        _check(self.lib.dmtp_gate_pick_p(self.g, len(p), _doubles(p), C.byref(k), C.byref(v)),
               "dmtp_gate_pick_p")
        return k.value, v.value

    def read(self) -> dict:
        st = dmtp_gate_stats()
        _check(self.lib.dmtp_gate_read(self.g, C.byref(st)), "dmtp_gate_read")
        K = st.max_drafts
        return {"a": list(st.a[:K]), "t": {n: st.t[n] for n in range(1, DMTP_GATE_MAX_ROWS + 1)
                                          if st.t[n] > 0},
                "d": st.d if st.d_measured else None, "rho": st.rho, "picks": st.picks,
                "since_plain": st.since_plain, "bin_judged": list(st.bin_judged),
                "bin_accepted": list(st.bin_accepted)}

    def close(self):
        if self.g:
            self.lib.dmtp_gate_free(self.g)
            self.g = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DmtpVocabList:
    """The draft heads' frequent-token list of include/dmtp_vocab.h (host-only;
    argument marshalling)."""

    def __init__(self, vocab: int, size: int = 0):
        self.lib = load_library()
        self.vocab = int(vocab)
        self.v = C.c_void_p()
        _check(self.lib.dmtp_vocab_create(self.vocab, int(size), C.byref(self.v)),
               "dmtp_vocab_create")

    @staticmethod
    def _ids(tokens):
        a = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64).reshape(-1))
        if a.size and (a.min() < -2**31 or a.max() >= 2**31):
            raise DmtpError(-1, "token id")
        a = a.astype(np.int32)
        return a, (a.ctypes.data if a.size else None)

    def begin_request(self, prompt, new_conversation: bool = True):
        a, ptr = self._ids(prompt)
        _check(self.lib.dmtp_vocab_begin_request(self.v, ptr, a.size, int(new_conversation)),
               "dmtp_vocab_begin_request")

    def picked(self, tokens):
        a, ptr = self._ids(tokens)
        _check(self.lib.dmtp_vocab_picked(self.v, ptr, a.size), "dmtp_vocab_picked")

    def ids(self) -> np.ndarray:
        out = np.empty(self.vocab, dtype=np.int32)
        n = C.c_int()
        _check(self.lib.dmtp_vocab_ids(self.v, out.ctypes.data, C.byref(n)), "dmtp_vocab_ids")
        return out[:n.value].copy()

    def mask(self) -> np.ndarray:
        out = np.empty(self.vocab, dtype=np.uint8)
        _check(self.lib.dmtp_vocab_mask(self.v, out.ctypes.data), "dmtp_vocab_mask")
        return out.astype(bool)

    def counts(self) -> np.ndarray:
        out = np.empty(self.vocab, dtype=np.int64)
        _check(self.lib.dmtp_vocab_counts(self.v, out.ctypes.data), "dmtp_vocab_counts")
        return out

    def stats(self) -> dict:
        st = dmtp_vocab_stats()
        _check(self.lib.dmtp_vocab_stats_read(self.v, C.byref(st)), "dmtp_vocab_stats_read")
        return {f: getattr(st, f) for f, _ in dmtp_vocab_stats._fields_}

    def close(self):
        if self.v:
            self.lib.dmtp_vocab_free(self.v)
            self.v = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
