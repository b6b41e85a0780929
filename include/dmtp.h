/*
 * dmtp.h - C ABI of the GB300 (sm_103a) DMTP speculative-decoding round.
 *
 * One call of dmtp_round runs one batched DMTP round for all B sequences, as the
 * DMTP blog ("DMTP: A Better First Token for Block Drafting via MTP") states it in
 * §5 "Inference: MTP First, DFlash Second" and §6.1 "Separating Prediction from
 * State Advancement":
 *   a1  T1 = argmax H RMSNorm(h_MTP), h_MTP kept from the previous round;
 *   a2  Delta = W [RMS_e(E(T1)); RMS_m(h_MTP)] (§3, the residual equation) and the
 *       eight drafter slots [E(A), E(T1) + Delta, E(MASK) x 6];
 *   a3  one block-bidirectional drafter forward -> T2..T7 (§2, §6.2);
 *   a4  one target forward over rows [A, T1..T7] -> per-row picks g0..g7;
 *   a5  greedy prefix acceptance: n = longest prefix with T_j == g_{j-1}; commit
 *       T1..Tn and g_n; the KV watermark comes down to the standing rows and a
 *       recurrent layer's per-row snapshot n is swapped in by pointer (colibri
 *       speculative-decoding page, "Undoing rows on a model with recurrent state");
 *   a6  drafter context K/V and MTP state advance over the n+1 committed rows; the
 *       MTP output at the last one is cached as the next h_MTP.
 *
 * Memory ownership. The caller allocates every device buffer (weights, the
 * workspace, round outputs) and keeps it alive while the context lives; the
 * library allocates no device memory. The context owns host bookkeeping and up to
 * two captured CUDA graphs (the round, and the round with forced drafts). All work is
 * enqueued on the stream given to dmtp_init;
 * results are valid once the caller synchronises that stream.
 *
 * Errors. Every int-returning call returns DMTP_OK (0) or a negative DMTP_E* code.
 * Argument errors are detected before any launch and leave the state unchanged.
 * DMTP_EDEVICE means a kernel's own bounds check fired (token id out of range,
 * KV write past max_ctx, a bounded wait that gave up); the context is then
 * poisoned: every later call but dmtp_free returns DMTP_ESTATE.
 *
 * Threading: a context is not thread-safe; distinct contexts are independent.
 */
#ifndef DMTP_H
#define DMTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DMTP_OK 0
#define DMTP_EINVAL (-1)    /* bad shape, pointer or size (nothing launched)           */
#define DMTP_ENOMEM (-2)    /* workspace smaller than dmtp_workspace_size reports      */
#define DMTP_ECAPACITY (-3) /* a sequence would grow past max_ctx (nothing launched)   */
#define DMTP_ECUDA (-4)     /* a CUDA runtime call failed                              */
#define DMTP_EDEVICE (-5)   /* a device-side check fired; context poisoned             */
#define DMTP_ESTATE (-6)    /* context poisoned by an earlier DMTP_EDEVICE             */

#define DMTP_MAX_LAYERS 64
#define DMTP_MAX_DRAFT_LAYERS 8
#define DMTP_MAX_TAPS 8

/* Model and capacity. dtype 0: fp32 weights/KV (CUDA-core path), 1: bf16 weights/KV
 * (tcgen05 tensor-core path). layer_kind[l]: 0 attention, 1 Gated DeltaNet.
 * Attention layers, the MTP block and the drafter share n_heads/n_kv_heads/head_dim.
 * tap_layers: target layers whose residual stream feeds the drafter's context
 * projection (DFlash "KV injection", DFlash vs MTP page). mask_id: the MASK token.
 * draft_window: the drafter sees context positions max(0, a - window) .. a-1 (DMTP
 * §6.2). max_ctx: KV capacity per sequence (prompt + 8 per round + 8 slack).
 * temperature: 0 = greedy verification (the target's picks g_0..g_7 are argmax picks);
 * > 0 (at least 1e-4, finite) = target-only sampled verification (DMTP §5: drafts are
 * checked against the target's samples): the pick for position p of sequence b is
 * argmax_v (l_v / temperature + G_v), an exact draw from softmax(l / temperature),
 * with Gumbel noise G_v = -log(-log u_v), u_v = ((w >> 8) + 1/2) 2^-24 and w word v % 4
 * of the Philox4x32-10 block (Salmon et al., SC 2011) of counter (v / 4, p, b, 0) and key
 * (low, high 32 bits of sample_seed). The noise depends on the position only, so the
 * committed stream equals plain one-token sampled decoding with the same noise. A (the
 * prefill's first token) and the drafts T1..T7 stay argmax picks.
 * draft_head_fp8 (bf16 models only): the heads that only draft (T1 and the drafter's
 * T2..T7; DMTP §6.5 drafting-side head quantisation) read an E4M3 copy of the head, made
 * in the workspace by dmtp_init: per row a power-of-two scale s = 2^e, e the smallest
 * integer with max|row| <= 448 s, and q = round-to-nearest-even(row / s); each head input
 * row (the normalised hidden) is quantised the same way, and the draft logits are
 * s_x s_v (q_x . q_v). The verify head stays bf16, so the committed tokens do not
 * change; only the drafts (and so the acceptance) can.
 * draft_list_cap (bf16 models only; 0: off): capacity, in tokens, of the draft heads'
 * token list (dmtp_set_draft_list); the workspace then holds a compact copy of that many
 * head rows (bf16, or E4M3 with draft_head_fp8) and their ids.
 * variable_depth (0 or 1): 1 also builds the GEMM plans of verifies that carry fewer
 * drafts (dmtp_round_depth with depth 0..6; more work at dmtp_init, no more memory).
 * draft_confidence (0 or 1; bf16 models): 1 makes the T1 and drafter heads also compute
 * each draft's confidence, the probability the head gives its own pick over the scores
 * within 20 of its best, 1 / sum exp(l_v - l_max) over those (the colibri page's
 * per-step estimate for the draft-depth gate; dmtp_round_out.draft_conf).
 * deterministic (0 or 1; bf16 models): 1 makes every round bitwise reproducible: the
 * GEMMs whose K range is split over several CTAs sum the parts in a fixed order (each part
 * writes its tile to workspace scratch, waits, bounded, for the tile's other parts, all
 * resident in one wave, and adds the parts in order into one slice of the output) instead
 * of adding them into the output in arrival order. Costs ~9% of a B32 round and ~40 MB of
 * workspace; two contexts with the same inputs then produce identical bits. */
typedef struct {
  int vocab, d_model, n_layers, n_heads, n_kv_heads, head_dim, ffn;
  int gdn_heads, gdn_dk, gdn_dv;
  uint8_t layer_kind[DMTP_MAX_LAYERS];
  int draft_layers, draft_window;
  int n_taps;
  int tap_layers[DMTP_MAX_TAPS];
  int mask_id;
  float rms_eps, rope_theta;
  int max_ctx, max_batch;
  int dtype;
  float temperature;
  uint64_t sample_seed;
  int draft_head_fp8;
  int draft_list_cap;
  int variable_depth;
  int draft_confidence;
  int deterministic;
} dmtp_config;

/* One decoder layer, row-major [out, in] device matrices of the config's dtype.
 * Attention: wqkv [(hq + 2 hkv) hd, d] (q rows, k rows, v rows), wo [d, hq hd].
 * Gated DeltaNet: gdn_wqkv [H (2 dk + dv), d], gdn_wa/gdn_wb [H, d], gdn_wo [d, H dv].
 * MLP: wgu [2F, d] (gate rows then up rows), wdown [d, F]. Norm gains [d]. */
typedef struct {
  const void *attn_norm, *wqkv, *wo;
  const void *gdn_wqkv, *gdn_wa, *gdn_wb, *gdn_wo;
  const void *mlp_norm, *wgu, *wdown;
} dmtp_layer_weights;

/* All weights (device pointers, caller-owned, alive for the context's lifetime).
 * emb/head [V, d] are shared by target, MTP and drafter (untied). mtp_proj [d, 2d]
 * is M of h' = M [RMSNorm(h); RMSNorm(Emb(t))] (DFlash vs MTP page, "MTP: Sequential
 * Prediction Heads"); fuse_w [d, 2d] is the DMTP residual matrix W; dft_fc
 * [d, n_taps d] the drafter's target-context projection. */
typedef struct {
  const void *emb, *head, *final_norm;
  dmtp_layer_weights layers[DMTP_MAX_LAYERS];
  const void *mtp_norm_h, *mtp_norm_e, *mtp_proj;
  dmtp_layer_weights mtp;
  const void* mtp_final_norm;
  const void *fuse_norm_e, *fuse_norm_m, *fuse_w;
  const void *dft_fc, *dft_norm_c;
  dmtp_layer_weights dft[DMTP_MAX_DRAFT_LAYERS];
  const void* dft_final_norm;
} dmtp_weights;

/* Per-round outputs: device pointers (caller-allocated), each optional (NULL: not
 * written). Integer fields: committed [B][8] (T1..Tn, g_n, then -1), n_accepted [B],
 * drafts [B][7] (T1..T7 as verified), picks [B][8] (g0..g7), kv_len [B] (target
 * watermark after the round), mtp_len [B] (next MTP position = kv_len + 1), snap_slot
 * [B] (installed snapshot row, -1 for attention-only targets). Float debug fields
 * (fp32): t1_logits [B][V], draft_logits [B][6][V], verify_logits [B][8][V], delta
 * [B][d] (Delta of this round), h_mtp [B][d] (the h_MTP this round started from).
 * Requesting a float debug field runs the round uncaptured (same kernels). draft_conf
 * [B][7] (fp32; a context made with draft_confidence = 1, else DMTP_EINVAL): the
 * confidence of the heads' own picks for T1..T7 (of the list's tokens when a draft list
 * is set; forced drafts do not change it); it does not stop the graph. */
typedef struct {
  int32_t *committed, *n_accepted, *drafts, *picks, *kv_len, *mtp_len, *snap_slot;
  float *t1_logits, *draft_logits, *verify_logits, *delta, *h_mtp;
  float* draft_conf;
} dmtp_round_out;

typedef struct dmtp_ctx dmtp_ctx;

/* Bytes of device workspace needed for `batch` sequences (batch <= max_batch,
 * batch * 8 <= 256). Returns DMTP_EINVAL for an unsupported config. */
int dmtp_workspace_size(const dmtp_config* cfg, int batch, size_t* bytes);

/* Create a context and run the prefill, which sets up the state of the target, the MTP
 * module and the drafter (DMTP §6.1): target over each prompt (KV, taps), A = the
 * target's greedy token after it, drafter context K/V, and MTP rows 1..P giving h_MTP.
 * workspace: device buffer of >= dmtp_workspace_size bytes, 256-byte aligned.
 * prompt_ids: host int32, the B prompts concatenated; prompt_lens: host int32 [B],
 * each >= 1. stream: a cudaStream_t (NULL: the default stream). Synchronises the
 * stream before returning. *out receives the context (NULL on error). */
int dmtp_init(const dmtp_config* cfg, const dmtp_weights* w, void* workspace, size_t ws_bytes,
              const int32_t* prompt_ids, const int32_t* prompt_lens, int batch, void* stream,
              dmtp_ctx** out);

/* Enqueue one round (steps a1-a6) for all sequences. out: see dmtp_round_out (may be
 * NULL). forced_drafts: NULL, or device int32 [B][7] replacing T1..T7 (T1 right after
 * the MTP head, so the fusion and drafter see it; T2..T7 after the drafter) - the
 * forced-draft test mode of the colibri page; they are copied into the context and
 * the round runs as its own captured graph. Requesting debug logits in `out` runs the
 * round eagerly instead. Returns DMTP_ECAPACITY if a sequence might pass
 * max_ctx - 8 (checked on the host before launch). Asynchronous. */
int dmtp_round(dmtp_ctx* ctx, const dmtp_round_out* out, const int32_t* forced_drafts);

/* A round whose verify carries only the first `depth` drafts (0..7; 7 is dmtp_round):
 * the colibri speculative-decoding page's draft-depth gate picks how many drafts the
 * next verify carries, and a verify of k drafts is one forward of the pending token and
 * its k drafts. The MTP head and the drafter still propose T1..T7 (drafts [B][7]); the
 * target verifies rows [A, T1..T_depth] only, as B (depth + 1) rows (its GEMMs, attention
 * and recurrence do that much work); at most `depth` drafts are accepted (n <= depth) and
 * a recurrent layer keeps the state after row `depth` live, swapping snapshot n in when
 * n < depth. Outputs as dmtp_round, except picks [B][8] holds g_0..g_depth (-1 after)
 * and verify_logits holds B (depth + 1) rows of V, sequence-major ([B][depth + 1][V]).
 * Depths below 7 need a context made with variable_depth = 1 (DMTP_EINVAL otherwise, or
 * for a depth outside 0..7). Each depth (and forced mode) is captured as its own graph
 * on first use. */
int dmtp_round_depth(dmtp_ctx* ctx, const dmtp_round_out* out, const int32_t* forced_drafts,
                     int depth);

/* One round with host outputs: enqueue the round, copy committed [B][8] and
 * n_accepted [B] (either may be NULL) into host memory and synchronise. */
int dmtp_round_host(dmtp_ctx* ctx, int32_t* committed_host, int32_t* n_accepted_host);

/* Draft heads over a token list (the colibri speculative-decoding page's frequent-token
 * list: the draft heads may score a list of tokens in place of the vocabulary, while the
 * verification scores every token; DMTP blog §6.5 names the LM head as the cost to cut).
 * From the next round on, T1 and the drafter's T2..T7 are the argmax of their logits over
 * the listed tokens only (the lowest id on exact ties); the verify head, and so every
 * committed token, is unchanged. ids: host int32, n strictly increasing token ids in
 * [0, vocab), 1 <= n <= draft_list_cap; n = 0 turns the list off (full heads again).
 * The call copies ids to the device and gathers the listed head rows into the
 * workspace's compact copy, enqueued on the context's stream (the ids array may be reused
 * on return). Upkeep of the list (counts, halvings, joined picks) is the caller's, e.g.
 * dmtp_vocab.h. Debug logits of the draft heads are then written at the listed ids only.
 * Returns DMTP_EINVAL (bad ids or n, or a context made with draft_list_cap 0),
 * DMTP_ESTATE on a poisoned context, DMTP_ECUDA if a copy or launch fails. */
int dmtp_set_draft_list(dmtp_ctx* ctx, const int32_t* ids, int n);

/* Synchronise and read the state: kv_len [B], pending token A [B] (host arrays, each
 * may be NULL) and the acceptance histogram hist[k] = rounds that accepted k drafts
 * (host uint64 [8], may be NULL). Also reports DMTP_EDEVICE if a device check fired. */
int dmtp_read_state(dmtp_ctx* ctx, int32_t* kv_len, int32_t* pending, uint64_t* hist);

/* Number of kernel launches one round enqueues (for launch accounting). */
int dmtp_round_launches(const dmtp_ctx* ctx);

/* Device time of the prefill dmtp_init ran (ms, from CUDA events on its stream around
 * the target, drafter-context and MTP passes over every prompt position and the pick of
 * A; -1 if the events failed) and the prompt tokens it processed. Either pointer may be
 * NULL. The prefill runs the round's kernels 8 positions per sequence at a time. */
int dmtp_prefill_stats(const dmtp_ctx* ctx, double* ms, int64_t* tokens);

/* Kernel classes of dmtp_profile. */
#define DMTP_PROF_GEMM 0   /* tcgen05 (or fp32) projection / MLP GEMMs              */
#define DMTP_PROF_HEAD 1   /* LM-head GEMM with fused argmax (a1, a3, a4)          */
#define DMTP_PROF_ATTN 2   /* split-K attention (partial + merge)                  */
#define DMTP_PROF_GDN 3    /* Gated DeltaNet recurrence with snapshots             */
#define DMTP_PROF_OTHER 4  /* norms, RoPE/KV writes, gathers, accept                */

/* Per-class device time and traffic of one round. ms: summed durations of the class's
 * launches, launch i lasting from the CUDA event recorded before it to the one recorded
 * before the next launch (so the classes add up to round_ms); bytes/flops: what those
 * launches must move/compute by the method (weights once; a projection's input and
 * output rows once in the storage type; visible K/V once per sequence and layer;
 * recurrent state read once and written per snapshot); impl_bytes: what the
 * implementation moves instead (both halves of a split GEMM operand, fp32 accumulator
 * reads and writes); round_ms: the whole profiled round; graph: 1 if the round ran as a
 * captured CUDA graph with the events as graph nodes (launch gaps as in dmtp_round's
 * graph), 0 if it ran eagerly (host launch gaps included). */
typedef struct {
  double ms[8], bytes[8], flops[8], impl_bytes[8];
  int launches[8];
  double round_ms;
  int graph;
} dmtp_profile;

/* Run one real round (state advances as with dmtp_round) as a freshly captured graph with
 * event nodes between its launches (eagerly if the capture fails), synchronise and fill
 * *out. For measurement, not for speed. */
int dmtp_round_profile(dmtp_ctx* ctx, dmtp_profile* out);

/* First-candidate head without any allocation (the pages have no counterpart; this
 * serves embedders that may not call cudaMalloc, e.g. engines that own a fixed memory
 * pool or paths where an allocation's implicit synchronisation is not acceptable).
 * Computes, like step a1 of dmtp_round, ids[r] = argmax_v H[v] . RMSNorm(h[r]) * gain
 * (lowest id on exact ties) and, if logits != NULL, logits[r][v] (fp32).
 * head: device bf16 [vocab][d_model] (16-byte aligned); norm_gain: device bf16
 * [d_model]; h: device fp32 [rows][d_model]; ids: device int32 [rows]; stream: a
 * cudaStream_t or NULL. Limits: 1 <= rows <= DMTP_NOALLOC_MAX_ROWS,
 * 64 <= d_model <= DMTP_NOALLOC_MAX_DMODEL, d_model % 64 == 0; otherwise DMTP_EINVAL.
 * Its scratch is a fixed library-owned device array of DMTP_NOALLOC_MAX_ROWS x
 * DMTP_NOALLOC_MAX_DMODEL bf16 elements plus DMTP_NOALLOC_MAX_ROWS 8-byte keys (262,400
 * bytes, about 0.26 MB), held by every GPU that loads the library until exit. The first
 * call on a device sets that device up (symbol lookup, kernel attribute) and should come
 * before any stream capture; that set-up does not survive cudaDeviceReset. Calls share the
 * array: calls that may overlap on the GPU race and must be serialised by the caller.
 * Returns DMTP_ECUDA, launching nothing, if a CUDA error is already pending on the
 * calling thread (it is not cleared), and DMTP_ECUDA if a launch or the head's tensor-map
 * encoding fails. Asynchronous on `stream`. */
#define DMTP_NOALLOC_MAX_ROWS 32
#define DMTP_NOALLOC_MAX_DMODEL 4096
int dmtp_t1_head_noalloc(const void* head, const void* norm_gain, const float* h, int rows,
                         int vocab, int d_model, float eps, int32_t* ids, float* logits,
                         void* stream);

/* Self-test of the device failure path (the bounded waits and device error word that
 * every pipelined kernel uses; no counterpart on the pages, which describe failure tests
 * of their own engines). Enqueues on the context's stream one kernel that waits, with the
 * kernels' bounded mbarrier wait, on a barrier nothing arrives at; after limit_ns
 * (1e3 .. 1e9 ns) the wait gives up, sets the timeout bit of the context's device error
 * word and the kernel returns: nothing faults, traps or waits longer. The next call that
 * reads the error word (dmtp_read_state) returns DMTP_EDEVICE and poisons the context,
 * exactly as a real timeout inside a round would. Returns DMTP_EINVAL for a limit out of
 * range, DMTP_ESTATE on a poisoned context, DMTP_ECUDA if the launch fails. */
int dmtp_selftest_timeout(dmtp_ctx* ctx, uint64_t limit_ns);

/* The device error word that poisoned the context (0 while it is not poisoned by one):
 * bit 1 a token id outside [0, V), 2 a KV write past max_ctx, 4 a bounded wait that gave
 * up, 8 a snapshot slot outside [0, 8). NULL gives 0. */
uint32_t dmtp_error_word(const dmtp_ctx* ctx);

/* Release the context (host memory and the graph). Never fails; NULL is a no-op.
 * Does not free caller-owned device memory. */
void dmtp_free(dmtp_ctx* ctx);

/* Static description of an error code. */
const char* dmtp_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* DMTP_H */
