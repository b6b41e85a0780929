// Host side of the DMTP round library: the C ABI declared in include/dmtp.h.
//
// Owns no device memory: every buffer is carved out of the caller's workspace.
// dmtp_init lays out the workspace, builds the tcgen05 GEMM plans (TMA tensor maps)
// and runs the prefill; dmtp_round enqueues steps a1-a6 and, when no debug output is
// requested, replays them as one captured CUDA graph (DMTP blog §6.4: the round's inputs are
// staged on the device into buffers whose addresses never change, then the graph runs). All per-sequence metadata
// (positions, accepted lengths, snapshot slots) stays on the device; the host never
// reads a length during normal rounds.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/dmtp.h"
#include "ops.h"

using namespace dmtp;

namespace {

struct Gemm {
  TcPlan tc;            // bf16 path
  HeadPlan hp;          // bf16 path, argmax heads
  const void* W = nullptr;
  const void* X = nullptr;
  int N = 0, K = 0, M = 0;
  bool argmax = false;
  bool split = true;    // X is the [hi; lo] bf16 pair
  bool swiglu = false;  // gate/up with the SwiGLU epilogue (bf16 path); N = 2F
};

struct LayerPlans {
  Gemm qkv, o, gu, down;       // attention (and MLP)
  Gemm gq, ga, gb, go;         // Gated DeltaNet projections
};

// The GEMMs of a verify that carries depth drafts: G = depth + 1 rows per sequence
// (B G token rows) through the target, its head and a6's drafter-context projections.
struct VerifyPlans {
  LayerPlans tgt[DMTP_MAX_LAYERS];
  Gemm head_v, dfc;
  Gemm dkv[DMTP_MAX_DRAFT_LAYERS];
};

}  // namespace

struct dmtp_ctx {
  dmtp_config cfg;
  dmtp_weights w;
  int B, M, dt, nsm;
  cudaStream_t st;
  int d, V, F, hq, hkv, hd, qd, kvd, qkvd, maxc, Ld, L, ntap;
  int gH, gdk, gdv, gld, n_gdn;
  int gdn_index[DMTP_MAX_LAYERS];
  int tap_of_layer[DMTP_MAX_LAYERS];  // tap slot of layer l, or -1
  int pmax;
  int attn_chunk, attn_nchunk;
  int attn_grid;  // CTAs of the persistent tensor-core attention (SM count)
  int mt8, mt6, mt1;  // padded GEMM token rows for 8B, 6B and B operand rows
  size_t ws_bytes;

  // workspace regions
  void* tK[DMTP_MAX_LAYERS];
  void* tV[DMTP_MAX_LAYERS];
  float* gstate[DMTP_MAX_LAYERS];
  void* dK[DMTP_MAX_DRAFT_LAYERS];
  void* dV[DMTP_MAX_DRAFT_LAYERS];
  void *mK, *mV;
  // tcgen05 attention tensor maps: K as [B*hkv*max_ctx, hd], V^T as [B*hkv*hd, max_ctx]
  CUtensorMap tmK[DMTP_MAX_LAYERS], tmV[DMTP_MAX_LAYERS];
  CUtensorMap tmKd[DMTP_MAX_DRAFT_LAYERS], tmVd[DMTP_MAX_DRAFT_LAYERS];
  CUtensorMap tmKm, tmVm;
  CUtensorMap tmQh, tmQl;  // the split query halves as [M][hq][hd], box {64, hq/hkv, 8}
  bool attn_tc;  // bf16 caches and a shape the tcgen05 attention serves
  float2* rope;
  float* x;
  void* xn;
  float* qkv;
  float* q;
  void* qs;  // bf16 [2][M][hq][hd]: split queries for the tensor-core attention
  float *part_o, *part_ml;
  void* att;
  float* gu;
  void* hmid;
  void* taps;
  float* hT32;
  void* hTn;
  void* z;
  void* zf;
  float* xm;
  float* cacc;
  void* cn;
  float* delta;
  float* h_mtp;
  void* t1in;
  void* dn;
  // E4M3 draft heads: the head copy and scales, the T1 and drafter head inputs
  void* h8;
  float* h8s;
  void *t1q, *dnq;
  float *t1qs, *dnqs;
  bool fp8;
  // draft heads over a token list: compact head rows (bf16, or E4M3 with scales), their
  // token ids, and the listed count on the device
  int list_cap;
  void* hc;
  float* hcs;
  int* hc_ids;
  int* hc_n;
  int list_n;  // listed tokens as last set (0: the list is off)
  // the draft heads' confidence: per-thread partials of the T1 and drafter heads, and the
  // combined confidence of T1..T7 [B][7]
  bool conf_on;
  float2 *conf_t1, *conf_d;
  float* dconf;
  float* hlast;
  // fixed-order K-part sums of the split GEMMs: one partial tile per CTA of a wave, and a
  // counter per output tile
  float* gpart;
  int* gcnt;
  size_t gpart_floats;
  int* prompts;
  int2* psched;  // prefill schedule: (sequence, chunk) of each row group of each step
  int* plen;
  int* forced;
  RoundState rs;
  unsigned* err;

  // GEMM plans
  LayerPlans tgt[DMTP_MAX_LAYERS];
  LayerPlans dft[DMTP_MAX_DRAFT_LAYERS];
  LayerPlans mtp;
  Gemm dkv[DMTP_MAX_DRAFT_LAYERS];
  Gemm fuse, head_t1, head_d, head_v, dfc, mproj;
  Gemm head_a;  // A after the prompt: the target's own (bf16) head on the T1 input rows
  Gemm head_t1l, head_dl;  // the T1 and drafter heads over the token list

  cudaGraphExec_t graph[8];         // the round, per verify depth (7: the DMTP round)
  cudaGraphExec_t graph_forced[8];  // the round with drafts read from `forced`
  bool depths;                      // plans for verifies of 0..6 drafts were built
  VerifyPlans* vp[8];               // [G] for G = 1..7 rows per sequence (G = 8: tgt etc.)
  cudaStream_t cap_st;  // private stream the round is captured on (the caller's may be NULL)
  bool poisoned;
  unsigned err_word;  // the device error word that poisoned it
  long kv_bound;
  int launches;
  int round_launches;
  double prefill_ms;     // device time of dmtp_init's prefill (CUDA events), -1 if unknown
  long prefill_tokens;   // prompt tokens it processed
  // per-launch event profiling (dmtp_round_profile only)
  bool prof;
  bool prof_external;  // the events are recorded inside a stream capture (graph nodes)
  std::vector<cudaEvent_t> pev;
  std::vector<int> pcls;
  std::vector<double> pbytes, pflops, pimpl;
  std::vector<int> kv_host;  // kv_len at the start of the profiled round

  ~dmtp_ctx() {
    for (VerifyPlans* v : vp) delete v;
  }
  void drop_graphs() {
    for (int k = 0; k < 8; ++k) {
      if (graph[k]) cudaGraphExecDestroy(graph[k]);
      if (graph_forced[k]) cudaGraphExecDestroy(graph_forced[k]);
      graph[k] = graph_forced[k] = nullptr;
    }
  }
};

// ---------------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------------
namespace {

struct Bump {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t bytes) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? (T*)(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

int derive(dmtp_ctx* c, const dmtp_config* cfg, int B) {
  const dmtp_config& f = *cfg;
  if (f.vocab < 2 || f.d_model < 32 || f.n_layers < 1 || f.n_layers > DMTP_MAX_LAYERS ||
      f.draft_layers < 1 || f.draft_layers > DMTP_MAX_DRAFT_LAYERS || f.n_taps < 1 ||
      f.n_taps > DMTP_MAX_TAPS || f.n_heads < 1 || f.n_kv_heads < 1 ||
      f.n_heads % f.n_kv_heads || f.head_dim < 8 || f.head_dim > 128 || f.head_dim % 2 ||
      f.ffn < 1 || f.max_ctx < 16 || B < 1 || B > f.max_batch || B * 8 > 256 ||
      (f.dtype != 0 && f.dtype != 1) || f.mask_id < 0 || f.mask_id >= f.vocab ||
      f.draft_window < 0 || !(f.temperature == 0.f || (f.temperature >= 1e-4f &&
                                                        f.temperature <= 3.0e38f)) ||
      (f.draft_head_fp8 != 0 && f.draft_head_fp8 != 1) ||
      (f.draft_head_fp8 && (f.dtype != 1 || f.d_model % 128)) || f.draft_list_cap < 0 ||
      f.draft_list_cap > f.vocab || (f.draft_list_cap > 0 && f.dtype != 1) ||
      (f.variable_depth != 0 && f.variable_depth != 1) ||
      (f.draft_confidence != 0 && f.draft_confidence != 1) ||
      (f.draft_confidence && f.dtype != 1) || (f.deterministic != 0 && f.deterministic != 1))
    return DMTP_EINVAL;
  const int grp = f.n_heads / f.n_kv_heads;
  const int QN = 8 * grp;
  if (QN > 256 || 256 % QN || (f.head_dim * QN) % 256 || f.head_dim / (256 / QN) > 32 ||
      (256 / QN) > 32)
    return DMTP_EINVAL;
  c->cfg = f;
  c->B = B;
  c->M = 8 * B;
  c->dt = f.dtype;
  c->fp8 = f.draft_head_fp8 != 0;
  c->list_cap = f.draft_list_cap;
  c->conf_on = f.draft_confidence != 0;
  c->d = f.d_model;
  c->V = f.vocab;
  c->F = f.ffn;
  c->hq = f.n_heads;
  c->hkv = f.n_kv_heads;
  c->hd = f.head_dim;
  c->qd = c->hq * c->hd;
  c->kvd = c->hkv * c->hd;
  c->qkvd = c->qd + 2 * c->kvd;
  c->maxc = (f.max_ctx + 63) / 64 * 64;  // K/V row strides stay 16-byte aligned for TMA
  c->L = f.n_layers;
  c->Ld = f.draft_layers;
  c->ntap = f.n_taps;
  c->gH = f.gdn_heads;
  c->gdk = f.gdn_dk;
  c->gdv = f.gdn_dv;
  c->n_gdn = 0;
  for (int l = 0; l < c->L; ++l) {
    c->tap_of_layer[l] = -1;
    if (f.layer_kind[l] > 1) return DMTP_EINVAL;
    c->gdn_index[l] = f.layer_kind[l] ? c->n_gdn++ : -1;
  }
  for (int i = 0; i < c->ntap; ++i) {
    if (f.tap_layers[i] < 0 || f.tap_layers[i] >= c->L) return DMTP_EINVAL;
    c->tap_of_layer[f.tap_layers[i]] = i;
  }
  if (c->n_gdn) {
    if (c->gH < 1 || c->gdv < 8 || c->gdv > 256 || (c->gdv & (c->gdv - 1)) || c->gdk > 256 ||
        c->gdk % (256 / c->gdv) || c->gdk / (256 / c->gdv) > 64)
      return DMTP_EINVAL;
  }
  c->gld = c->n_gdn ? c->gH * (2 * c->gdk + c->gdv) + 2 * c->gH : 0;
  if (c->dt == 1) {
    // every GEMM reduction length must be a multiple of the 64-wide k block
    const int ks[] = {c->d, c->qd, c->F, 2 * c->d, c->ntap * c->d, c->gH * c->gdv};
    for (int k : ks)
      if (k % 64) return DMTP_EINVAL;
  }
  c->mt8 = tc_mt(c->M);
  c->mt6 = tc_mt(6 * B);
  c->mt1 = tc_mt(B);
  c->attn_tc = c->dt == 1 && (c->hd == 64 || c->hd == 128) && QN <= 64 && B <= kAttnMaxB;
  {  // the persistent tensor-core attention runs one CTA per SM
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        nsm < 1)
      nsm = 256;
    c->attn_grid = nsm;
  }
  c->attn_chunk = 1024;  // keys per attention partial; a multiple of the 64-key tile
  c->attn_nchunk = (c->maxc + 8 + c->attn_chunk - 1) / c->attn_chunk;
  return DMTP_OK;
}

size_t layout(dmtp_ctx* c, char* base) {
  Bump b{base};
  const size_t es = c->dt ? 2 : 4;
  const size_t kvsz = (size_t)c->B * c->hkv * c->maxc * c->hd * es;
  for (int l = 0; l < c->L; ++l) {
    c->tK[l] = c->tV[l] = nullptr;
    c->gstate[l] = nullptr;
    if (c->cfg.layer_kind[l] == 0) {
      c->tK[l] = b.take<char>(kvsz);
      c->tV[l] = b.take<char>(kvsz);
    } else {
      c->gstate[l] = b.take<float>((size_t)c->B * 8 * c->gH * c->gdv * c->gdk * 4);
    }
  }
  for (int j = 0; j < c->Ld; ++j) {
    c->dK[j] = b.take<char>(kvsz);
    c->dV[j] = b.take<char>(kvsz);
  }
  c->mK = b.take<char>(kvsz);
  c->mV = b.take<char>(kvsz);
  c->rope = b.take<float2>((size_t)(c->maxc + 16) * (c->hd / 2) * sizeof(float2));
  const size_t M = c->M, d = c->d, B = c->B;
  const int qkvw = std::max(std::max(c->qkvd, c->gld), 2 * c->kvd);
  // GEMM operand buffers hold [hi; lo] halves of mt rows each on the bf16 path
  const size_t r8 = c->dt ? 2 * (size_t)c->mt8 : M;
  const size_t r6 = c->dt ? 2 * (size_t)c->mt6 : 6 * B;
  const size_t r1 = c->dt ? 2 * (size_t)c->mt1 : B;
  c->x = b.take<float>(M * d * 4);
  c->xn = b.take<char>(r8 * d * es);
  c->qkv = b.take<float>(M * qkvw * 4);
  c->q = b.take<float>(M * c->qd * 4);
  c->qs = b.take<char>(2 * M * c->qd * 2);
  const int QN = 8 * (c->hq / c->hkv);
  // partials: per (sequence, kv head, chunk) for the chunked path, per (CTA, segment)
  // slot for the persistent one
  const size_t slots = std::max((size_t)B * c->hkv * c->attn_nchunk,
                                (size_t)c->attn_grid + (size_t)B * c->hkv);
  c->part_o = b.take<float>(slots * QN * c->hd * 4);
  c->part_ml = b.take<float>(slots * QN * 2 * 4);
  c->att = b.take<char>(r8 * std::max(c->qd, c->gH * c->gdv) * es);
  c->gu = b.take<float>(M * 2 * c->F * 4);
  c->hmid = b.take<char>(r8 * c->F * es);
  c->taps = b.take<char>(r8 * c->ntap * d * es);
  c->hT32 = b.take<float>(M * d * 4);
  c->hTn = b.take<char>(r8 * d * es);
  c->z = b.take<char>(r8 * 2 * d * es);
  c->zf = b.take<char>(r1 * 2 * d * es);
  c->xm = b.take<float>(M * d * 4);
  c->cacc = b.take<float>(M * d * 4);
  c->cn = b.take<char>(r8 * d * es);
  c->delta = b.take<float>(B * d * 4);
  c->h_mtp = b.take<float>(B * d * 4);
  c->t1in = b.take<char>(r1 * d * es);
  c->dn = b.take<char>(r6 * d * es);
  if (c->fp8) {
    const size_t vpad = ((size_t)c->V + 255) / 256 * 256;  // scales read tile-wide
    c->h8 = b.take<char>((size_t)c->V * d);
    c->h8s = b.take<float>(vpad * 4);
    c->t1q = b.take<char>((size_t)B * d);
    c->t1qs = b.take<float>((size_t)B * 4);
    c->dnq = b.take<char>((size_t)6 * B * d);
    c->dnqs = b.take<float>((size_t)6 * B * 4);
  }
  c->hc = nullptr;
  c->hcs = nullptr;
  c->hc_ids = c->hc_n = nullptr;
  if (c->list_cap) {
    const size_t cpad = ((size_t)c->list_cap + 255) / 256 * 256;  // scales read tile-wide
    c->hc = b.take<char>(cpad * d * (c->fp8 ? 1 : 2));
    if (c->fp8) c->hcs = b.take<float>(cpad * 4);
    c->hc_ids = b.take<int>(cpad * 4);
    c->hc_n = b.take<int>(4);
  }
  c->conf_t1 = c->conf_d = nullptr;
  c->dconf = nullptr;
  if (c->conf_on) {  // at most two partials per CTA (8 epilogue warps), one CTA per SM
    c->conf_t1 = b.take<float2>((size_t)2 * c->attn_grid * B * 8);
    c->conf_d = b.take<float2>((size_t)2 * c->attn_grid * 6 * B * 8);
    c->dconf = b.take<float>(B * 7 * 4);
  }
  c->hlast = b.take<float>(B * d * 4);
  if (c->dt == 1 && c->cfg.deterministic) {  // a tile: at most 256 weight x 256 token rows
    c->gpart_floats = (size_t)c->attn_grid * 256 * 256;
    c->gpart = b.take<float>(c->gpart_floats * 4);
    c->gcnt = b.take<int>((size_t)c->attn_grid * 4);
  } else {
    c->gpart_floats = 0;
    c->gpart = nullptr;
    c->gcnt = nullptr;
  }
  c->forced = b.take<int>(B * 7 * 4);
  RoundState& s = c->rs;
  s.kv_len = b.take<int>(B * 4);
  s.pos0 = b.take<int>(B * 4);
  s.A = b.take<int>(B * 4);
  s.drafts = b.take<int>(B * 7 * 4);
  s.g = b.take<int>(B * 8 * 4);
  s.n_acc = b.take<int>(B * 4);
  s.committed = b.take<int>(B * 8 * 4);
  s.tok = b.take<int>(M * 4);
  s.mtp_tok = b.take<int>(M * 4);
  s.mtp_base = b.take<int>(B * 4);
  s.mtp_cnt = b.take<int>(B * 4);
  s.rows_valid = b.take<int>(B * 4);
  s.cseq = b.take<int>(B * 4);
  s.snap_slot = b.take<int>(B * 4);
  s.mtp_len = b.take<int>(B * 4);
  s.hist = b.take<unsigned long long>(8 * 8);
  s.keys = b.take<unsigned long long>(B * 16 * 8);
  s.gdn_live = b.take<int>((size_t)std::max(1, c->n_gdn) * B * 4);
  s.gdn_slot = b.take<int>((size_t)std::max(1, c->n_gdn) * B * 8 * 4);
  s.n_gdn = c->n_gdn;
  s.B = c->B;
  c->err = b.take<unsigned>(256);
  s.err = c->err;
  c->plen = b.take<int>(B * 4);
  return (b.off + 255) & ~(size_t)255;  // the staged prompts start 256-byte aligned
}

// After the fixed layout: the prompts [B][max_ctx] int32, then (256-byte aligned, for its
// 8-byte entries) the prefill schedule of at most B (max_ctx/8 + 2) (sequence, chunk) pairs.
size_t sched_offset(int B, int max_ctx) { return ((size_t)B * max_ctx * 4 + 255) & ~(size_t)255; }
size_t prompt_bytes(int B, int max_ctx) {
  return sched_offset(B, max_ctx) + (size_t)B * (max_ctx / 8 + 2) * 8;
}

// split: X holds [hi; lo] bf16 halves (all GEMMs but the LM head, whose single bf16
// operand keeps the logit error near 1e-3 at half the tensor-core work)
int plan(dmtp_ctx* c, Gemm& g, const void* W, int N, int K, const void* X, int M, bool argmax,
         bool split = true) {
  g.W = W;
  g.X = X;
  g.N = N;
  g.K = K;
  g.M = M;
  g.argmax = argmax;
  g.split = split;
  if (!W) return DMTP_EINVAL;
  if (c->dt == 1 && argmax)  // LM heads: one bf16 operand, token-major argmax kernel
    return split || head_plan(&g.hp, W, N, K, X, M, c->nsm, 256, 8) ? DMTP_EINVAL : DMTP_OK;
  if (c->dt == 1)
    return tc_plan(&g.tc, W, N, K, X, M, c->nsm, split) ? DMTP_EINVAL : DMTP_OK;
  return DMTP_OK;
}

// Gate/up GEMM: on the bf16 path with the SwiGLU epilogue (writes the down GEMM's
// operand directly), on the fp32 path a plain GEMM followed by op_swiglu.
int plan_gu(dmtp_ctx* c, Gemm& g, const void* W, int M) {
  const int r = plan(c, g, W, 2 * c->F, c->d, c->xn, M, false);
  if (r || c->dt != 1) return r;
  g.swiglu = true;
  const int mt = tc_mt(M);
  const int ms = (mt > 128 && mt % 32 == 0) ? 2 : 1;
  return tc_plan_swiglu(&g.tc, W, c->F, c->d, c->xn, M, c->nsm, true, ms) ? DMTP_EINVAL
                                                                          : DMTP_OK;
}

int plan_layer(dmtp_ctx* c, LayerPlans& p, const dmtp_layer_weights& w, int kind, int M) {
  int r = 0;
  if (!w.attn_norm || !w.mlp_norm) return DMTP_EINVAL;
  if (kind == 0) {
    r |= plan(c, p.qkv, w.wqkv, c->qkvd, c->d, c->xn, M, false);
    r |= plan(c, p.o, w.wo, c->d, c->qd, c->att, M, false);
  } else {
    r |= plan(c, p.gq, w.gdn_wqkv, c->gH * (2 * c->gdk + c->gdv), c->d, c->xn, M, false);
    r |= plan(c, p.ga, w.gdn_wa, c->gH, c->d, c->xn, M, false);
    r |= plan(c, p.gb, w.gdn_wb, c->gH, c->d, c->xn, M, false);
    r |= plan(c, p.go, w.gdn_wo, c->d, c->gH * c->gdv, c->att, M, false);
  }
  r |= plan_gu(c, p.gu, w.wgu, M);
  r |= plan(c, p.down, w.wdown, c->d, c->F, c->hmid, M, false);
  return r ? DMTP_EINVAL : DMTP_OK;
}

// ---------------------------------------------------------------------------------
// enqueue helpers
// ---------------------------------------------------------------------------------
enum { P_GEMM = 0, P_HEAD = 1, P_ATTN = 2, P_GDN = 3, P_OTHER = 4 };

// Profiling events: one before every launch and one after the last, so launch i takes
// the time between event i and event i + 1 and the launches' times add up to the round.
// Inside a stream capture they become event-record nodes of the graph.
inline void prof_event(dmtp_ctx* c, size_t i) {
  if (c->prof_external)
    cudaEventRecordWithFlags(c->pev[i], c->st, cudaEventRecordExternal);
  else
    cudaEventRecord(c->pev[i], c->st);
  pdl_fence();
}

// Wraps one launch: counts it and, when profiling, records the event before it, its
// class, its algorithmic (method) bytes and flops, and the bytes the implementation moves
// (impl: e.g. the second bf16 half of a split operand and fp32 accumulator traffic).
template <typename F>
inline void launch(dmtp_ctx* c, int cls, double bytes, double flops, F&& f,
                   double impl = -1.0) {
  if (c->prof && c->pcls.size() + 1 < c->pev.size()) {
    prof_event(c, c->pcls.size());
    f();
    c->pcls.push_back(cls);
    c->pbytes.push_back(bytes);
    c->pflops.push_back(flops);
    c->pimpl.push_back(impl < 0 ? bytes : impl);
  } else {
    f();
  }
  c->launches += 1;
}

inline double esz(const dmtp_ctx* c) { return c->dt ? 2.0 : 4.0; }

// out[M,N] (+)= X[M,K] W[N,K]^T. Method bytes: the weights, the input rows and the output
// rows once each in the storage type. Implementation bytes: the weights, both halves of
// a split operand, and the fp32 output read and written.
void gemm_acc(dmtp_ctx* c, const Gemm& g, float* out, int ldo) {
  const double bytes = ((double)g.N * g.K + (double)g.M * g.K + (double)g.M * g.N) * esz(c);
  const double impl = ((double)g.N * g.K + (double)g.M * g.K * (g.split && c->dt ? 2 : 1)) *
                          esz(c) + 8.0 * g.M * g.N;
  launch(c, P_GEMM, bytes, 2.0 * g.M * g.N * g.K, [&] {
    if (c->dt == 1)
      op_gemm_tc_acc(g.tc, out, ldo, c->err, c->st);
    else
      op_gemm_simt_acc((const float*)g.W, (const float*)g.X, g.N, g.K, g.M, out, ldo, c->st);
  }, impl);
}

// The verify head's sampling: row m = b*G + j of sequence b at position pos0[b] + j (G
// verify rows per sequence).
SampleArgs verify_sampling(const dmtp_ctx* c, int G = 8) {
  return SampleArgs{1.4426950408889634f / c->cfg.temperature, (uint32_t)c->cfg.sample_seed,
                    (uint32_t)(c->cfg.sample_seed >> 32), c->rs.pos0, G};
}

// smp: the verify head's sampled picks (nullptr: argmax picks); conf: the head's
// confidence partials (bf16 path, greedy heads), or null
void gemm_argmax(dmtp_ctx* c, const Gemm& g, unsigned long long* keys, float* logits,
                 const SampleArgs* smp = nullptr, float2* conf = nullptr) {
  const double ew = (c->dt == 1 && g.hp.fp8) ? 1.0 : esz(c);  // bytes per operand element
  const double bytes = ((double)g.N * g.K + (double)g.M * g.K) * ew + 8.0 * g.M;
  launch(c, P_HEAD, bytes, 2.0 * g.M * g.N * g.K, [&] {
    if (c->dt == 1)
      op_head_tc(g.hp, keys, logits, c->V, smp, c->err, c->st, conf);
    else
      op_gemm_simt_argmax((const float*)g.W, (const float*)g.X, g.N, g.K, g.M, keys, logits,
                          c->V, smp, c->st);
  });
}

// Gate/up GEMM with the SwiGLU epilogue: method bytes are the weights, the input rows and
// the F-wide output rows once; the implementation reads both input halves and writes both
// output halves.
void gemm_swiglu(dmtp_ctx* c, const Gemm& g, void* h, long h_lo) {
  const double bytes = ((double)g.N * g.K + (double)g.M * g.K + (double)g.M * (g.N / 2)) *
                       esz(c);
  const double impl = ((double)g.N * g.K + (double)g.M * g.K * 2) * esz(c) +
                      (double)g.M * (g.N / 2) * esz(c) * 2;
  launch(c, P_GEMM, bytes, 2.0 * g.M * g.N * g.K,
         [&] { op_gemm_tc_swiglu(g.tc, h, h_lo, c->err, c->st); }, impl);
}

void zero(dmtp_ctx* c, void* p, size_t bytes) {
  cudaMemsetAsync(p, 0, bytes, c->st);
  pdl_fence();
}

// element offset of the remainder half of an operand with `mt` padded rows of `ld`
inline long lo_of(const dmtp_ctx* c, int mt, int ld) { return c->dt ? (long)mt * ld : 0; }
inline int mt_of_rows(const dmtp_ctx*, int rows) { return tc_mt(rows); }

// zero / nz: also clears the first nz floats of each of the `rows` rows of zero (the
// accumulator of the GEMM that reads y), instead of a separate memset.
void norm(dmtp_ctx* c, const float* x, const void* g, void* y, float* y32, void* tap, int rows,
          RowMap map = RowMap(), bool split = true, float* zero = nullptr, int nz = 0) {
  launch(c, P_OTHER, 0, 0, [&] {
    const int mt = mt_of_rows(c, rows);
    op_rmsnorm(c->dt, x, c->d, g, y, c->d, split ? lo_of(c, mt, c->d) : 0, y32, c->d, tap,
               c->ntap * c->d, lo_of(c, mt, c->ntap * c->d), rows, c->d, c->cfg.rms_eps,
               map, c->st, zero, nz, nz);
  });
}

void* tap_ptr(dmtp_ctx* c, int slot) {
  if (slot < 0) return nullptr;
  return (char*)c->taps + (size_t)slot * c->d * (c->dt ? 2 : 4);
}

struct AttnSpec {
  void *Kc, *Vc;
  const CUtensorMap *tmK, *tmV;
  const int* base;
  int causal, lo_fixed, window;
  int mode_base;  // 1: base = kv_len at round start (target, drafter); 2: kv_len + 1 (MTP)
};

// MLP block over M rows: x += down(SwiGLU(gate/up(RMS(x)))).
void mlp(dmtp_ctx* c, const LayerPlans& p, const dmtp_layer_weights& w, float* xr, int M) {
  const int mt = mt_of_rows(c, M);
  if (p.gu.swiglu) {
    norm(c, xr, w.mlp_norm, c->xn, nullptr, nullptr, M);
    gemm_swiglu(c, p.gu, c->hmid, lo_of(c, mt, c->F));
  } else {
    norm(c, xr, w.mlp_norm, c->xn, nullptr, nullptr, M, RowMap(), true, c->gu, 2 * c->F);
    gemm_acc(c, p.gu, c->gu, 2 * c->F);
    launch(c, P_OTHER, 0, 0, [&] { op_swiglu(c->dt, c->gu, c->hmid, lo_of(c, mt, c->F), M, c->F, c->st); });
  }
  gemm_acc(c, p.down, xr, c->d);
}

// Attention layer over rg rows per sequence (M = B rg rows; 8 but in a shorter verify).
void attn_layer(dmtp_ctx* c, const LayerPlans& p, const dmtp_layer_weights& w, float* xr,
                const AttnSpec& a, void* tap_in, int rg = 8) {
  const int M = c->B * rg;
  norm(c, xr, w.attn_norm, c->xn, nullptr, tap_in, M, RowMap(), true, c->qkv, c->qkvd);
  gemm_acc(c, p.qkv, c->qkv, c->qkvd);
  launch(c, P_OTHER, 0, 0, [&] { op_rope_kv(c->dt, c->qkv, c->qkvd, 0, c->qd, c->qd + c->kvd, c->q, c->attn_tc ? c->qs : nullptr, (long)M * c->qd, a.Kc, a.Vc, a.base, c->rs.cseq, c->rope,
             M, c->hq, c->hkv, c->hd, c->maxc, c->err, c->st, rg); });
  AttnArgs aa;
  aa.Kc = a.Kc;
  aa.Vc = a.Vc;
  aa.q = c->q;
  aa.part_o = c->part_o;
  aa.part_ml = c->part_ml;
  aa.out = c->att;
  aa.out_lo = lo_of(c, mt_of_rows(c, M), c->qd);
  aa.base = a.base;
  aa.cseq = c->rs.cseq;
  aa.causal = a.causal;
  aa.lo_fixed = a.lo_fixed;
  aa.window = a.window;
  aa.B = c->B;
  aa.hq = c->hq;
  aa.hkv = c->hkv;
  aa.hd = c->hd;
  aa.max_ctx = c->maxc;
  aa.chunk = c->attn_chunk;
  aa.nchunk = c->attn_nchunk;
  aa.qs = c->qs;
  aa.qs_lo = (long)M * c->qd;
  aa.rows = rg;
  aa.pgrid = c->attn_grid;
  aa.ptk = kAttnTile;
  double kv_bytes = 0;
  if (c->prof) {
    // keys each sequence's rows can see: lo .. base+7, K and V, all kv heads
    for (int b = 0; b < c->B; ++b) {
      const int a0 = c->kv_host[b];
      const int base = a.mode_base == 2 ? a0 + 1 : a0;
      int lo = a.lo_fixed;
      if (a.window > 0) lo = std::max(lo, base - a.window);
      kv_bytes += (double)(base + rg - lo) * c->kvd * esz(c) * 2;
    }
    kv_bytes += (double)M * c->qd * esz(c) * 2;  // q in, o out
  }
  launch(c, P_ATTN, kv_bytes, 0, [&] {
    if (c->attn_tc)
      op_attention_tc(aa, *a.tmK, *a.tmV, c->tmQh, c->tmQl, c->err, c->st);
    else
      op_attention(c->dt, aa, c->st);
  });
  c->launches += 1;  // partial + merge
  gemm_acc(c, p.o, xr, c->d);
  mlp(c, p, w, xr, M);
}

void gdn_layer(dmtp_ctx* c, const LayerPlans& p, int l, float* xr, void* tap_in, bool snapshots,
               int rg) {
  const dmtp_layer_weights& w = c->w.layers[l];
  const int M = c->B * rg, gi = c->gdn_index[l];
  const int nqkv = c->gH * (2 * c->gdk + c->gdv);
  norm(c, xr, w.attn_norm, c->xn, nullptr, tap_in, M, RowMap(), true, c->qkv, c->gld);
  gemm_acc(c, p.gq, c->qkv, c->gld);
  gemm_acc(c, p.ga, c->qkv + nqkv, c->gld);
  gemm_acc(c, p.gb, c->qkv + nqkv + c->gH, c->gld);
  GdnArgs ga;
  ga.qkvab = c->qkv;
  ga.ld = c->gld;
  ga.states = c->gstate[l];
  ga.live = c->rs.gdn_live + (size_t)gi * c->B;
  ga.slot = c->rs.gdn_slot + (size_t)gi * c->B * 8;
  ga.rows_valid = c->rs.rows_valid;
  ga.snapshots = snapshots ? 1 : 0;
  ga.out = c->att;
  ga.out_lo = lo_of(c, mt_of_rows(c, M), c->gH * c->gdv);
  ga.rows = rg;
  ga.B = c->B;
  ga.H = c->gH;
  ga.dk = c->gdk;
  ga.dv = c->gdv;
  ga.err = c->err;
  const double st_bytes = (double)c->B * c->gH * c->gdv * c->gdk * 4 * (snapshots ? 9 : 2);
  launch(c, P_GDN, st_bytes, 0, [&] { op_gdn(c->dt, ga, c->st); });
  gemm_acc(c, p.go, xr, c->d);
  mlp(c, p, w, xr, M);
}

// target forward over rg rows of every sequence (8; fewer in a verify of fewer drafts):
// tokens in rs.tok, row m = b rg + s at position pos0[b] + s; leaves the final-normed
// hidden in hT32 (fp32) and hTn (operand type), taps filled. tgt: the layers' GEMM plans
// for B rg rows.
void target_forward(dmtp_ctx* c, bool snapshots, int rg, const LayerPlans* tgt) {
  const int M = c->B * rg;
  launch(c, P_OTHER, 0, 0, [&] { op_embed(c->dt, c->w.emb, c->rs.tok, c->V, c->x, M, c->d, c->err, c->st); });
  for (int l = 0; l < c->L; ++l) {
    void* tap_in = l > 0 ? tap_ptr(c, c->tap_of_layer[l - 1]) : nullptr;
    if (c->cfg.layer_kind[l] == 0) {
      AttnSpec a{c->tK[l], c->tV[l], &c->tmK[l], &c->tmV[l], c->rs.pos0, 1, 0, 0, 1};
      attn_layer(c, tgt[l], c->w.layers[l], c->x, a, tap_in, rg);
    } else {
      gdn_layer(c, tgt[l], l, c->x, tap_in, snapshots, rg);
    }
  }
  norm(c, c->x, c->w.final_norm, c->hTn, c->hT32, tap_ptr(c, c->tap_of_layer[c->L - 1]), M,
       RowMap(), false);
}

// a6 (and each prefill chunk): drafter context K/V at positions pos0+s from the taps of
// the rg rows per sequence (dfc / dkv: their GEMM plans for B rg rows), then the MTP rows
// (token mtp_tok, hidden hT32 row) at positions mtp_base+s.
void drafter_ctx(dmtp_ctx* c, int rg, const Gemm& dfc, const Gemm* dkv) {
  const int M = c->B * rg;
  zero(c, c->cacc, (size_t)M * c->d * 4);
  gemm_acc(c, dfc, c->cacc, c->d);
  norm(c, c->cacc, c->w.dft_norm_c, c->cn, nullptr, nullptr, M, RowMap(), true, c->qkv,
       2 * c->kvd);
  for (int j = 0; j < c->Ld; ++j) {
    if (j > 0) zero(c, c->qkv, (size_t)M * 2 * c->kvd * 4);
    gemm_acc(c, dkv[j], c->qkv, 2 * c->kvd);
    launch(c, P_OTHER, 0, 0, [&] { op_rope_kv(c->dt, c->qkv, 2 * c->kvd, -1, 0, c->kvd, nullptr, nullptr, 0, c->dK[j], c->dV[j],
               c->rs.pos0, c->rs.cseq, c->rope, M, c->hq, c->hkv, c->hd, c->maxc, c->err, c->st, rg); });
  }
}

// The MTP advance always runs 8 rows per sequence; its target hidden rows come from a
// step of rg rows per sequence (hT32 row b rg + s; rows past the step's are never
// committed and land in the MTP cache's stale tail).
void mtp_advance(dmtp_ctx* c, int rg = 8) {
  const int M = c->M;
  ConcatPart ph, pe;
  ph.src32 = c->hT32;
  ph.ld = c->d;
  ph.map.out_group = 8;
  ph.map.in_group = rg;
  ph.g = c->w.mtp_norm_h;
  pe.tok = c->rs.mtp_tok;
  pe.g = c->w.mtp_norm_e;
  launch(c, P_OTHER, 0, 0, [&] { op_concat_rms2(c->dt, c->w.emb, c->V, ph, pe, c->z, lo_of(c, c->mt8, 2 * c->d), M, c->d, c->cfg.rms_eps, c->err, c->st); });
  zero(c, c->xm, (size_t)M * c->d * 4);
  gemm_acc(c, c->mproj, c->xm, c->d);
  AttnSpec a{c->mK, c->mV, &c->tmKm, &c->tmVm, c->rs.mtp_base, 1, 1, 0, 2};
  attn_layer(c, c->mtp, c->w.mtp, c->xm, a, nullptr);
  launch(c, P_OTHER, 0, 0, [&] { op_gather_hmtp(c->xm, c->rs.mtp_cnt, c->h_mtp, c->B, c->d, c->st); });
}

struct Dbg {
  float *t1, *dl, *vl;
};

// One round whose verify carries `depth` drafts (0..7; 7: the DMTP round): rows
// [A, T1..T_depth] at G = depth + 1 rows per sequence (colibri page: a verify of k drafts
// is one forward of the token and its k drafts).
void enqueue_round(dmtp_ctx* c, const Dbg& dbg, const int* forced, int depth = 7) {
  const int G = depth + 1;
  const VerifyPlans* vp = G < 8 ? c->vp[G] : nullptr;
  RoundState& s = c->rs;
  const int B = c->B;
  pdl_fence();  // the round's first launch follows host copies: no programmatic overlap
  launch(c, P_OTHER, 0, 0, [&] { op_round_begin(s, c->st); });
  // a1: T1 from h_MTP as the previous round left it
  if (c->fp8)
    launch(c, P_OTHER, 0, 0, [&] { op_rmsnorm_e4m3(c->h_mtp, c->d, c->w.mtp_final_norm, c->t1q, c->d, c->t1qs, B, c->d, c->cfg.rms_eps, RowMap(), c->st); });
  else
    norm(c, c->h_mtp, c->w.mtp_final_norm, c->t1in, nullptr, nullptr, B, RowMap(), false);
  // the draft heads score the token list when one is set (dmtp_set_draft_list)
  const bool listed = c->list_n > 0;
  const int* lmap = listed ? c->hc_ids : nullptr;
  const Gemm& ht1 = listed ? c->head_t1l : c->head_t1;
  gemm_argmax(c, ht1, s.keys, dbg.t1, nullptr, c->conf_t1);
  launch(c, P_OTHER, 0, 0, [&] { op_keys_to_ids(s.keys, B, 1, s.drafts, 7, 0, forced, 7, 0, c->st, lmap); });
  if (c->conf_on)  // the T1 head's probability of its own pick (colibri per-step gate)
    launch(c, P_OTHER, 0, 0, [&] { op_conf_combine(ht1.hp, c->conf_t1, 1, c->dconf, 7, 0, c->st); });
  // a2: Delta = W [RMS_e(E(T1)); RMS_m(h_MTP)]; slots [E(A), E(T1)+Delta, E(MASK) x 6]
  ConcatPart pe, pm;
  pe.tok = s.drafts;  // T1 of sequence b is drafts[b*7]
  pe.tok_stride = 7;
  pe.g = c->w.fuse_norm_e;
  pm.src32 = c->h_mtp;
  pm.ld = c->d;
  pm.g = c->w.fuse_norm_m;
  launch(c, P_OTHER, 0, 0, [&] { op_concat_rms2(c->dt, c->w.emb, c->V, pe, pm, c->zf, lo_of(c, c->mt1, 2 * c->d), B, c->d, c->cfg.rms_eps, c->err, c->st); });
  zero(c, c->delta, (size_t)B * c->d * 4);
  gemm_acc(c, c->fuse, c->delta, c->d);
  launch(c, P_OTHER, 0, 0, [&] { op_build_slots(c->dt, c->w.emb, c->V, s.A, s.drafts, c->delta, c->cfg.mask_id, c->x, B, c->d,
                 c->err, c->st); });
  // a3: block drafter over the 8 slots
  for (int j = 0; j < c->Ld; ++j) {
    AttnSpec a{c->dK[j], c->dV[j], &c->tmKd[j], &c->tmVd[j], s.pos0, 0, 0, c->cfg.draft_window,
               1};
    attn_layer(c, c->dft[j], c->w.dft[j], c->x, a, nullptr);
  }
  RowMap m6;
  m6.out_group = 6;
  m6.in_group = 8;
  m6.in_offset = 2;
  if (c->fp8)
    launch(c, P_OTHER, 0, 0, [&] { op_rmsnorm_e4m3(c->x, c->d, c->w.dft_final_norm, c->dnq, c->d, c->dnqs, 6 * B, c->d, c->cfg.rms_eps, m6, c->st); });
  else
    norm(c, c->x, c->w.dft_final_norm, c->dn, nullptr, nullptr, 6 * B, m6, false);
  const Gemm& hd = listed ? c->head_dl : c->head_d;
  gemm_argmax(c, hd, s.keys + B, dbg.dl, nullptr, c->conf_d);
  launch(c, P_OTHER, 0, 0, [&] { op_keys_to_ids(s.keys + B, B, 6, s.drafts, 7, 1, forced, 7, 1, c->st, lmap); });
  if (c->conf_on)
    launch(c, P_OTHER, 0, 0, [&] { op_conf_combine(hd.hp, c->conf_d, 6, c->dconf, 7, 1, c->st); });
  // a4: target verify of [A, T1..T_depth]
  launch(c, P_OTHER, 0, 0, [&] { op_verify_tokens(s, depth, c->st); });
  target_forward(c, true, G, vp ? vp->tgt : c->tgt);
  const Gemm& hv = vp ? vp->head_v : c->head_v;
  if (c->cfg.temperature > 0.f) {  // target-only sampled verification (DMTP §5)
    const SampleArgs smp = verify_sampling(c, G);
    gemm_argmax(c, hv, s.keys + 7 * B, dbg.vl, &smp);
  } else {
    gemm_argmax(c, hv, s.keys + 7 * B, dbg.vl);
  }
  launch(c, P_OTHER, 0, 0, [&] { op_keys_to_ids(s.keys + 7 * B, B, G, s.g, 8, 0, nullptr, 0, 0, c->st); });
  // a5: prefix acceptance, commit, watermarks, snapshot swap
  launch(c, P_OTHER, 0, 0, [&] { op_accept(s, depth, c->st); });
  // a6: drafter context and MTP advance over the committed rows
  drafter_ctx(c, G, vp ? vp->dfc : c->dfc, vp ? vp->dkv : c->dkv);
  mtp_advance(c, G);
}

int check_err(dmtp_ctx* c) {
  unsigned e = 0;
  if (cudaMemcpyAsync(&e, c->err, 4, cudaMemcpyDeviceToHost, c->st) != cudaSuccess)
    return DMTP_ECUDA;
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return DMTP_ECUDA;
  if (e) {
    c->poisoned = true;
    c->err_word = e;
    if (getenv("DMTP_VERBOSE"))
      fprintf(stderr, "dmtp: device error word 0x%x (1 token id, 2 KV position, 4 wait timed "
              "out, 8 snapshot slot)\n", e);
    return DMTP_EDEVICE;
  }
  return DMTP_OK;
}

}  // namespace

// ---------------------------------------------------------------------------------
// C ABI
// ---- GEMM tile selection by measurement ----
// Every distinct GEMM shape (N, K, M, operand, epilogue) is timed on the device with
// each tile shape (128 or 256 weight rows per CTA, one to four token parts, K splits
// around the wave-count choice), cold: the L2 is flushed by a 256 MB read before each
// run, as in the round, where each weight matrix is streamed once. The fastest shape
// serves every GEMM of that shape. The LM heads are timed the same way over their tile
// (128 or 256 vocabulary rows) and epilogue width (4 or 8 warps), the verify head with
// its sampling epilogue when the context samples. Outputs go to scratch (the gate/up
// accumulator and the argmax keys), which the round clears before use.
namespace {
struct TuneKey {
  int dev, N, K, M;
  bool split, argmax, swiglu, sample, fp8;
  bool operator==(const TuneKey& o) const {
    return dev == o.dev && N == o.N && K == o.K && M == o.M && split == o.split &&
           argmax == o.argmax && swiglu == o.swiglu && sample == o.sample && fp8 == o.fp8;
  }
};
struct TuneChoice {
  int wide, msplit, splits;  // projection GEMMs
  int nv, ew;                // LM heads: vocabulary rows per tile, epilogue warps
  int pair;                  // projection GEMMs: CTA pairs (M = 256 MMAs over two SMs)
};
// Choices are kept for the life of the process: a later context on the same device
// reuses them (same kernels, same reduction order, no second timing pass).
std::mutex g_tune_mu;
std::vector<std::pair<TuneKey, TuneChoice>> g_tune;

void collect(LayerPlans& p, std::vector<Gemm*>& v) {
  for (Gemm* g : {&p.qkv, &p.o, &p.gu, &p.down, &p.gq, &p.ga, &p.gb, &p.go}) v.push_back(g);
}

// the plan with the fixed-order K-part scratch of the context (deterministic contexts)
TcPlan with_parts(const dmtp_ctx* c, TcPlan p) {
  if (!c->gpart) return p;
  p.part = c->gpart;
  p.tile_cnt = c->gcnt;
  p.part_floats = c->gpart_floats;
  return p;
}

float time_plan(dmtp_ctx* c, const TcPlan& p0, const void* flush, size_t flush_bytes,
                cudaEvent_t e0, cudaEvent_t e1) {
  const TcPlan p = with_parts(c, p0);
  float best = 1e30f;
  for (int rep = 0; rep < 3; ++rep) {
    op_l2_flush(flush, flush_bytes, c->err, c->st);
    cudaEventRecord(e0, c->st);
    pdl_fence();
    op_gemm_tc_acc(p, c->gu, p.N, c->err, c->st);
    cudaEventRecord(e1, c->st);
    float ms = 1e30f;
    if (cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      return 1e30f;
    best = std::min(best, ms);
  }
  return best;
}

float time_head(dmtp_ctx* c, const HeadPlan& p, const SampleArgs* smp, const void* flush,
                size_t flush_bytes, cudaEvent_t e0, cudaEvent_t e1) {
  float best = 1e30f;
  for (int rep = 0; rep < 3; ++rep) {
    op_l2_flush(flush, flush_bytes, c->err, c->st);
    cudaEventRecord(e0, c->st);
    pdl_fence();
    op_head_tc(p, c->rs.keys, nullptr, 0, smp, c->err, c->st);
    cudaEventRecord(e1, c->st);
    float ms = 1e30f;
    if (cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      return 1e30f;
    best = std::min(best, ms);
  }
  return best;
}

float time_swiglu(dmtp_ctx* c, const TcPlan& p, const void* flush, size_t flush_bytes,
                  cudaEvent_t e0, cudaEvent_t e1) {
  float best = 1e30f;
  for (int rep = 0; rep < 3; ++rep) {
    op_l2_flush(flush, flush_bytes, c->err, c->st);
    cudaEventRecord(e0, c->st);
    pdl_fence();
    op_gemm_tc_swiglu(p, c->hmid, (long)p.MT * c->F, c->err, c->st);
    cudaEventRecord(e1, c->st);
    float ms = 1e30f;
    if (cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      return 1e30f;
    best = std::min(best, ms);
  }
  return best;
}

int autotune(dmtp_ctx* c, const void* flush, size_t flush_bytes) {
  if (c->dt != 1) return DMTP_OK;
  std::vector<Gemm*> all;
  for (int l = 0; l < c->L; ++l) collect(c->tgt[l], all);
  for (int j = 0; j < c->Ld; ++j) {
    collect(c->dft[j], all);
    all.push_back(&c->dkv[j]);
  }
  collect(c->mtp, all);
  for (Gemm* g : {&c->fuse, &c->head_t1, &c->head_d, &c->head_v, &c->head_a, &c->dfc,
                  &c->mproj, &c->head_t1l, &c->head_dl})
    all.push_back(g);
  for (int G = 1; G < 8; ++G) {
    VerifyPlans* v = c->vp[G];
    if (!v) continue;
    for (int l = 0; l < c->L; ++l) collect(v->tgt[l], all);
    all.push_back(&v->head_v);
    all.push_back(&v->dfc);
    for (int j = 0; j < c->Ld; ++j) all.push_back(&v->dkv[j]);
  }
  const size_t scratch = (size_t)c->M * 2 * c->F;  // floats of the gate/up accumulator
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return DMTP_ECUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return DMTP_ECUDA;
  }
  const bool verbose = getenv("DMTP_VERBOSE") != nullptr;
  // DMTP_GEMM_PAIRS=1 / 0: projection GEMMs with split operands always / never run as CTA
  // pairs where the shape allows (a test of either kernel form); unset: the faster one
  const char* pairs_env = getenv("DMTP_GEMM_PAIRS");
  const int force_pair = pairs_env ? (pairs_env[0] == '1' ? 1 : 0) : -1;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_tune_mu);
  int rc = DMTP_OK;
  for (Gemm* g : all) {
    if (!g->W) continue;
    if (!g->swiglu && !g->argmax && (size_t)g->M * g->N > scratch) continue;  // default shape
    // the verify head under sampled verification runs the sampling epilogue
    bool vhead = g == &c->head_v;
    for (int G = 1; G < 8; ++G) vhead = vhead || (c->vp[G] && g == &c->vp[G]->head_v);
    const bool sample = vhead && c->cfg.temperature > 0.f;
    const SampleArgs smp = sample ? verify_sampling(c, g->M / c->B) : SampleArgs{};
    const bool fp8 = g->argmax && g->hp.fp8;
    const TuneKey key{dev, g->N, g->K, g->M, g->split, g->argmax, g->swiglu, sample, fp8};
    const TuneChoice* hit = nullptr;
    for (auto& e : g_tune)
      if (e.first == key && force_pair < 0) hit = &e.second;
    // a head plan with another tile and warp count, same operands
    auto replan = [&](HeadPlan* p, int nv, int ew) {
      return fp8 ? head_plan_e4m3(p, g->W, g->hp.wscale, g->N, g->K, g->X, g->hp.xscale, g->M,
                                  c->nsm, nv, ew)
                 : head_plan(p, g->W, g->N, g->K, g->X, g->M, c->nsm, nv, ew);
    };
    if (hit && g->argmax) {
      if (replan(&g->hp, hit->nv, hit->ew)) rc = DMTP_EINVAL;
      continue;
    }
    if (hit) {
      const int r = g->swiglu ? tc_plan_swiglu(&g->tc, g->W, c->F, g->K, g->X, g->M, c->nsm,
                                               g->split, hit->msplit, hit->pair)
                              : tc_plan_shape(&g->tc, g->W, g->N, g->K, g->X, g->M, c->nsm,
                                              g->split, hit->wide, hit->msplit,
                                              hit->splits, hit->pair);
      if (r) rc = DMTP_EINVAL;
      continue;
    }
    if (g->swiglu) {  // tile shape: one to four token parts, CTA pairs or not; no K split
      TcPlan best_p = g->tc;
      float best_t = force_pair == 1 ? 1e30f : time_swiglu(c, g->tc, flush, flush_bytes, e0, e1);
      for (int pair = 0; pair <= (g->split ? 1 : 0); ++pair)
        for (int ms = 1; ms <= 4; ++ms) {
          TcPlan p;
          if ((force_pair >= 0 && pair != force_pair) ||
              (ms == g->tc.msplit && pair == g->tc.pair) ||
              tc_plan_swiglu(&p, g->W, c->F, g->K, g->X, g->M, c->nsm, g->split, ms, pair))
            continue;
          const float t = time_swiglu(c, p, flush, flush_bytes, e0, e1);
          if (t < best_t) {
            best_t = t;
            best_p = p;
          }
        }
      g->tc = best_p;
      if (force_pair < 0) g_tune.push_back({key, TuneChoice{2, best_p.msplit, 1, 0, 0, best_p.pair}});
      if (verbose)
        fprintf(stderr, "dmtp: gate/up F=%d K=%d M=%d: %d token part(s)%s, %.1f us\n", c->F,
                g->K, g->M, best_p.msplit, best_p.pair ? ", CTA pairs" : "", best_t * 1e3f);
      continue;
    }
    if (g->argmax) {  // LM head: vocabulary tile of 128 or 256 rows, 4 or 8 epilogue warps
      HeadPlan best_p = g->hp;
      float best_t = 1e30f;
      for (int nv = 128; nv <= 256; nv *= 2)
        for (int ew = 4; ew <= 8; ew *= 2) {
          HeadPlan p;
          if (replan(&p, nv, ew)) continue;
          const float t = time_head(c, p, sample ? &smp : nullptr, flush, flush_bytes, e0, e1);
          if (t < best_t) {
            best_t = t;
            best_p = p;
          }
        }
      g->hp = best_p;
      g_tune.push_back({key, TuneChoice{0, 0, 0, best_p.NV, best_p.ew, 0}});
      if (verbose)
        fprintf(stderr, "dmtp: head V=%d K=%d M=%d%s%s: %d vocabulary rows per tile, %d "
                "epilogue warps, %.1f us\n", g->N, g->K, g->M, sample ? " sampled" : "",
                fp8 ? " e4m3" : "", best_p.NV, best_p.ew, best_t * 1e3f);
      continue;
    }
    TuneChoice best{g->tc.wide, g->tc.msplit, g->tc.splits, 0, 0, g->tc.pair};
    float best_ms = force_pair == 1 ? 1e30f : time_plan(c, g->tc, flush, flush_bytes, e0, e1);
    for (int pair = 0; pair <= (g->split ? 1 : 0); ++pair)
      for (int wide = 1; wide <= 2; ++wide)
        for (int ms = 1; ms <= 4; ++ms) {
          TcPlan p0;
          if ((force_pair >= 0 && pair != force_pair) ||
              tc_plan_shape(&p0, g->W, g->N, g->K, g->X, g->M, c->nsm, g->split, wide, ms, 0,
                            pair))
            continue;
          const int cand[3] = {p0.splits, std::max(1, p0.splits / 2),
                               std::min(32, 2 * p0.splits)};
          for (int i = 0; i < 3; ++i) {
            if (i > 0 && (cand[i] == cand[0] || (i == 2 && cand[2] == cand[1]))) continue;
            TcPlan p;
            if (tc_plan_shape(&p, g->W, g->N, g->K, g->X, g->M, c->nsm, g->split, wide, ms,
                              cand[i], pair))
              continue;
            const float t = time_plan(c, p, flush, flush_bytes, e0, e1);
            if (t < best_ms) {
              best_ms = t;
              best = TuneChoice{wide, ms, p.splits, 0, 0, pair};
            }
          }
        }
    if (best_ms >= 1e30f) {  // forced pairs, none of this shape: the plan from planning
      best = TuneChoice{g->tc.wide, g->tc.msplit, g->tc.splits, 0, 0, g->tc.pair};
      best_ms = 0.f;
    }
    if (tc_plan_shape(&g->tc, g->W, g->N, g->K, g->X, g->M, c->nsm, g->split, best.wide,
                      best.msplit, best.splits, best.pair))
      rc = DMTP_EINVAL;
    if (force_pair < 0) g_tune.push_back({key, best});
    if (verbose)
      fprintf(stderr, "dmtp: gemm N=%d K=%d M=%d%s: %d x 128 weight rows%s, %d token part(s), "
              "%d K split(s), %.1f us\n", g->N, g->K, g->M, g->split ? " split" : "",
              best.wide, best.pair ? " (CTA pairs)" : "", best.msplit, best.splits,
              best_ms * 1e3f);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  for (Gemm* g : all)  // every projection GEMM sums its K parts in a fixed order
    if (!g->argmax) g->tc = with_parts(c, g->tc);
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return DMTP_ECUDA;
  return rc;
}
}  // namespace

// ---------------------------------------------------------------------------------
extern "C" {

int dmtp_workspace_size(const dmtp_config* cfg, int batch, size_t* bytes) {
  if (!cfg || !bytes) return DMTP_EINVAL;
  dmtp_ctx* c = new dmtp_ctx();
  int r = derive(c, cfg, batch);
  if (r == DMTP_OK) *bytes = layout(c, nullptr) + prompt_bytes(batch, c->maxc);
  delete c;
  return r;
}

int dmtp_init(const dmtp_config* cfg, const dmtp_weights* w, void* workspace, size_t ws_bytes,
              const int32_t* prompt_ids, const int32_t* prompt_lens, int batch, void* stream,
              dmtp_ctx** out) {
  if (!out) return DMTP_EINVAL;
  *out = nullptr;
  if (!cfg || !w || !workspace || !prompt_ids || !prompt_lens) return DMTP_EINVAL;
  if ((uintptr_t)workspace & 255) return DMTP_EINVAL;
  dmtp_ctx* c = new dmtp_ctx();
  int r = derive(c, cfg, batch);
  if (r) {
    delete c;
    return r;
  }
  c->w = *w;
  c->st = (cudaStream_t)stream;
  for (int k = 0; k < 8; ++k) c->graph[k] = c->graph_forced[k] = nullptr;
  c->poisoned = false;
  c->err_word = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&c->nsm, cudaDevAttrMultiProcessorCount, dev);
  int pmax = 0;
  long total = 0;
  for (int b = 0; b < batch; ++b) {
    if (prompt_lens[b] < 1) {
      delete c;
      return DMTP_EINVAL;
    }
    pmax = std::max(pmax, (int)prompt_lens[b]);
    total += prompt_lens[b];
  }
  if (pmax + 24 > c->maxc) {
    delete c;
    return DMTP_ECAPACITY;
  }
  c->pmax = pmax;
  const size_t need = layout(c, nullptr) + prompt_bytes(batch, c->maxc);
  if (ws_bytes < need) {
    delete c;
    return DMTP_ENOMEM;
  }
  c->ws_bytes = need;
  const size_t fixed = layout(c, (char*)workspace);
  c->prompts = (int*)((char*)workspace + fixed);
  c->psched = (int2*)((char*)c->prompts + sched_offset(batch, c->maxc));
  if (((uintptr_t)c->prompts | (uintptr_t)c->psched) & 255) {  // 8-byte schedule loads
    delete c;
    return DMTP_EINVAL;
  }
  if (!w->emb || !w->head || !w->final_norm || !w->mtp_norm_h || !w->mtp_norm_e ||
      !w->mtp_final_norm || !w->fuse_norm_e || !w->fuse_norm_m || !w->dft_norm_c ||
      !w->dft_final_norm) {
    delete c;
    return DMTP_EINVAL;
  }
  // GEMM plans
  int pr = 0;
  const int M = c->M, B = c->B;
  for (int l = 0; l < c->L; ++l) pr |= plan_layer(c, c->tgt[l], w->layers[l], cfg->layer_kind[l], M);
  for (int j = 0; j < c->Ld; ++j) {
    pr |= plan_layer(c, c->dft[j], w->dft[j], 0, M);
    const char* wk = (const char*)w->dft[j].wqkv;
    pr |= plan(c, c->dkv[j], wk ? wk + (size_t)c->qd * c->d * (c->dt ? 2 : 4) : nullptr,
               2 * c->kvd, c->d, c->cn, M, false);
  }
  pr |= plan_layer(c, c->mtp, w->mtp, 0, M);
  pr |= plan(c, c->fuse, w->fuse_w, c->d, 2 * c->d, c->zf, B, false);
  if (c->fp8) {  // draft heads on the E4M3 head copy (DMTP §6.5)
    c->head_t1.argmax = c->head_d.argmax = true;
    c->head_t1.W = c->head_d.W = c->h8;
    c->head_t1.N = c->head_d.N = c->V;
    c->head_t1.K = c->head_d.K = c->d;
    c->head_t1.X = c->t1q;
    c->head_t1.M = B;
    c->head_d.X = c->dnq;
    c->head_d.M = 6 * B;
    c->head_t1.split = c->head_d.split = false;
    pr |= head_plan_e4m3(&c->head_t1.hp, c->h8, c->h8s, c->V, c->d, c->t1q, c->t1qs, B,
                         c->nsm, 256, 8) ? DMTP_EINVAL : 0;
    pr |= head_plan_e4m3(&c->head_d.hp, c->h8, c->h8s, c->V, c->d, c->dnq, c->dnqs, 6 * B,
                         c->nsm, 256, 8) ? DMTP_EINVAL : 0;
  } else {
    pr |= plan(c, c->head_t1, w->head, c->V, c->d, c->t1in, B, true, false);
    pr |= plan(c, c->head_d, w->head, c->V, c->d, c->dn, 6 * B, true, false);
  }
  if (c->list_cap) {  // the same heads over the compact rows of the token list
    for (Gemm* g : {&c->head_t1l, &c->head_dl}) {
      const bool t1 = g == &c->head_t1l;
      g->argmax = true;
      g->split = false;
      g->W = c->hc;
      g->N = c->list_cap;
      g->K = c->d;
      g->M = t1 ? B : 6 * B;
      if (c->fp8) {
        g->X = t1 ? c->t1q : c->dnq;
        pr |= head_plan_e4m3(&g->hp, c->hc, c->hcs, c->list_cap, c->d, g->X,
                             t1 ? c->t1qs : c->dnqs, g->M, c->nsm, 256, 8) ? DMTP_EINVAL : 0;
      } else {
        g->X = t1 ? c->t1in : c->dn;
        pr |= head_plan(&g->hp, c->hc, c->list_cap, c->d, g->X, g->M, c->nsm, 256, 8)
                  ? DMTP_EINVAL : 0;
      }
    }
  }
  pr |= plan(c, c->head_a, w->head, c->V, c->d, c->t1in, B, true, false);
  pr |= plan(c, c->head_v, w->head, c->V, c->d, c->hTn, M, true, false);
  pr |= plan(c, c->dfc, w->dft_fc, c->d, c->ntap * c->d, c->taps, M, false);
  pr |= plan(c, c->mproj, w->mtp_proj, c->d, 2 * c->d, c->z, M, false);
  c->depths = cfg->variable_depth != 0;
  if (c->depths) {  // verifies of 0..6 drafts: G = 1..7 rows per sequence
    for (int G = 1; G < 8; ++G) {
      VerifyPlans* v = new (std::nothrow) VerifyPlans();
      if (!v) {
        delete c;
        return DMTP_ENOMEM;
      }
      c->vp[G] = v;
      const int MG = B * G;
      for (int l = 0; l < c->L; ++l)
        pr |= plan_layer(c, v->tgt[l], w->layers[l], cfg->layer_kind[l], MG);
      pr |= plan(c, v->head_v, w->head, c->V, c->d, c->hTn, MG, true, false);
      pr |= plan(c, v->dfc, w->dft_fc, c->d, c->ntap * c->d, c->taps, MG, false);
      for (int j = 0; j < c->Ld; ++j) {
        const char* wk = (const char*)w->dft[j].wqkv;
        pr |= plan(c, v->dkv[j], wk ? wk + (size_t)c->qd * c->d * (c->dt ? 2 : 4) : nullptr,
                   2 * c->kvd, c->d, c->cn, MG, false);
      }
    }
  }
  if (pr) {
    delete c;
    return DMTP_EINVAL;
  }
  if (c->dt == 1 && (tc_init_attributes() || attn_tc_init_attributes() ||
                     head_init_attributes())) {
    delete c;
    return DMTP_ECUDA;
  }
  if (c->attn_tc) {
    // K: [B*hkv*max_ctx][hd]; V^T blocked by 64 keys: [B*hkv*(max_ctx/64)][hd][64]; each
    // key tile of either is one TMA request (a 3-D box over its 64-wide slabs)
    const uint64_t krows = (uint64_t)B * c->hkv * c->maxc;
    const uint64_t vblocks = (uint64_t)B * c->hkv * (c->maxc / 64);
    const uint64_t hd = c->hd;
    int e = 0;
    auto maps = [&](CUtensorMap* mk, CUtensorMap* mv, void* K, void* V) {
      e |= tc_make_tmap3s(mk, K, 64, krows, hd / 64, hd * 2, 128, kAttnTile, (uint32_t)(hd / 64));
      e |= tc_make_tmap3s(mv, V, 64, hd, vblocks, 128, hd * 128, (uint32_t)hd, kAttnTile / 64);
    };
    for (int l = 0; l < c->L; ++l)
      if (c->tK[l]) maps(&c->tmK[l], &c->tmV[l], c->tK[l], c->tV[l]);
    for (int j = 0; j < c->Ld; ++j) maps(&c->tmKd[j], &c->tmVd[j], c->dK[j], c->dV[j]);
    maps(&c->tmKm, &c->tmVm, c->mK, c->mV);
    const int grp = c->hq / c->hkv;
    e |= tc_make_tmap3(&c->tmQh, c->qs, c->hd, c->hq, c->M, grp, 8);
    e |= tc_make_tmap3(&c->tmQl, (char*)c->qs + (size_t)c->M * c->qd * 2, c->hd, c->hq, c->M,
                       grp, 8);
    if (e) {
      delete c;
      return DMTP_EINVAL;
    }
  }
  // ---- initial device state ----
  cudaStream_t st = c->st;
  RoundState& s = c->rs;
  // padding rows of the GEMM operands are read (and ignored): start from zeros
  zero(c, workspace, need);
  if (c->fp8) op_quant_rows_e4m3(w->head, c->V, c->d, c->h8, c->h8s, st);
  {
    const int r = autotune(c, workspace, std::min(need, (size_t)256 << 20));
    if (r) {
      delete c;
      return r;
    }
  }
  // the list heads score the first *hc_n compact rows and map rows to ids (after the
  // tile choice above, which re-plans without them)
  for (Gemm* g : {&c->head_t1l, &c->head_dl}) {
    g->hp.vdev = c->hc_n;
    g->hp.vmap = c->hc_ids;
  }
  c->list_n = 0;
  zero(c, c->err, 4);
  zero(c, s.hist, 64);
  zero(c, s.keys, (size_t)B * 16 * 8);
  for (int l = 0; l < c->L; ++l)
    if (c->gstate[l]) zero(c, c->gstate[l], (size_t)B * 8 * c->gH * c->gdv * c->gdk * 4);
  if (c->n_gdn) {
    std::vector<int> live((size_t)c->n_gdn * B, 0), slot((size_t)c->n_gdn * B * 8);
    // buffer 0 is live, buffers 1..7 hold the snapshots after rows 0..6 (slot 7 unused)
    for (size_t i = 0; i < slot.size(); ++i) slot[i] = (i % 8) < 7 ? (int)(i % 8) + 1 : 0;
    cudaMemcpyAsync(s.gdn_live, live.data(), live.size() * 4, cudaMemcpyHostToDevice, st);
    cudaMemcpyAsync(s.gdn_slot, slot.data(), slot.size() * 4, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
  }
  op_rope_table(c->rope, c->maxc + 16, c->hd, cfg->rope_theta, st);
  {
    std::vector<int> pp((size_t)B * c->maxc, 0);
    long off = 0;
    for (int b = 0; b < B; ++b) {
      memcpy(&pp[(size_t)b * c->maxc], prompt_ids + off, (size_t)prompt_lens[b] * 4);
      off += prompt_lens[b];
    }
    cudaMemcpyAsync(c->prompts, pp.data(), pp.size() * 4, cudaMemcpyHostToDevice, st);
    cudaMemcpyAsync(c->plen, prompt_lens, (size_t)B * 4, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
  }
  // ---- prefill: steps of B row groups, each 8 positions of one prompt ----
  // Row group pb of a step takes chunk (sequence, index) of the schedule. Attention-only
  // targets take every prompt's chunks in order, several chunks of one prompt in a step
  // where they fit: all of the step's K/V rows are written before its attention reads
  // them, so each chunk sees the chunks before it. Groups past the last chunk repeat the
  // chunk just past the last prompt's end (their K/V rows land in its unused tail). A
  // Gated DeltaNet state advances one chunk per step, so hybrid targets take chunk t of
  // every prompt in step t.
  std::vector<int2> sched;
  if (c->n_gdn == 0) {
    for (int b = 0; b < B; ++b)
      for (int ch = 0; ch < (prompt_lens[b] + 7) / 8; ++ch) sched.push_back(make_int2(b, ch));
    const int2 pad = make_int2(B - 1, (prompt_lens[B - 1] + 7) / 8);
    while (sched.size() % B) sched.push_back(pad);
  } else {
    for (int ch = 0; ch < (pmax + 7) / 8; ++ch)
      for (int b = 0; b < B; ++b) sched.push_back(make_int2(b, ch));
  }
  const int nsteps = (int)(sched.size() / B);
  cudaEvent_t pe0 = nullptr, pe1 = nullptr;
  if (cudaEventCreate(&pe0) == cudaSuccess && cudaEventCreate(&pe1) == cudaSuccess)
    cudaEventRecord(pe0, st);
  auto fail_prefill = [&]() {
    if (pe0) cudaEventDestroy(pe0);
    if (pe1) cudaEventDestroy(pe1);
    delete c;
    return DMTP_ECUDA;
  };
  if (cudaMemcpyAsync(c->psched, sched.data(), sched.size() * sizeof(int2),
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return fail_prefill();
  pdl_fence();
  for (int t = 0; t < nsteps; ++t) {
    op_prefill_chunk(s, c->prompts, c->plen, c->maxc, c->psched + (size_t)t * B, st);
    target_forward(c, false, 8, c->tgt);
    op_prefill_save_last(c->hT32, c->plen, c->psched + (size_t)t * B, c->hlast, B, c->d, st);
    drafter_ctx(c, 8, c->dfc, c->dkv);
    mtp_advance(c);
    if ((t & 63) == 63 && cudaStreamSynchronize(st) != cudaSuccess) return fail_prefill();
  }
  // A = the target's greedy token after the prompt; MTP consumes (h^T_{P-1}, A) at P
  op_cast_rows(c->dt, c->hlast, c->d, c->t1in, c->d, 0, B, c->d, RowMap(), st);
  zero(c, s.keys, (size_t)B * 8);
  gemm_argmax(c, c->head_a, s.keys, nullptr);
  op_keys_to_ids(s.keys, B, 1, s.A, 1, 0, nullptr, 0, 0, st);
  op_prefill_final(s, c->plen, c->hlast, c->hT32, c->d, st);
  mtp_advance(c);
  op_prefill_done(s, c->plen, st);
  if (pe1) cudaEventRecord(pe1, st);
  // a launch that failed (e.g. for its resources) leaves no device error word: ask for it
  cudaError_t ce = cudaGetLastError();
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  c->prefill_ms = -1.0;
  c->prefill_tokens = total;
  if (pe1) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, pe0, pe1) == cudaSuccess) c->prefill_ms = ms;
  }
  if (pe0) cudaEventDestroy(pe0);
  if (pe1) cudaEventDestroy(pe1);
  if (ce != cudaSuccess) {
    fprintf(stderr, "dmtp_init: %s\n", cudaGetErrorString(ce));
    delete c;
    return DMTP_ECUDA;
  }
  r = check_err(c);
  if (r) {
    delete c;
    return r;
  }
  c->kv_bound = pmax;
  c->round_launches = 0;
  *out = c;
  return DMTP_OK;
}

static int copy_out(dmtp_ctx* c, void* dst, const void* src, size_t bytes) {
  if (!dst) return 0;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, c->st) != cudaSuccess;
}

int dmtp_round(dmtp_ctx* c, const dmtp_round_out* out, const int32_t* forced) {
  return dmtp_round_depth(c, out, forced, 7);
}

int dmtp_round_depth(dmtp_ctx* c, const dmtp_round_out* out, const int32_t* forced, int depth) {
  if (!c || depth < 0 || depth > 7 || (depth < 7 && !c->depths)) return DMTP_EINVAL;
  if (out && out->draft_conf && !c->conf_on) return DMTP_EINVAL;
  if (c->poisoned) return DMTP_ESTATE;
  const int B = c->B;
  if (c->kv_bound + 16 >= c->maxc) {
    std::vector<int> kv(B);
    if (cudaMemcpyAsync(kv.data(), c->rs.kv_len, B * 4, cudaMemcpyDeviceToHost, c->st) !=
            cudaSuccess ||
        cudaStreamSynchronize(c->st) != cudaSuccess)
      return DMTP_ECUDA;
    c->kv_bound = *std::max_element(kv.begin(), kv.end());
    if (c->kv_bound + 16 >= c->maxc) return DMTP_ECAPACITY;
  }
  Dbg dbg{nullptr, nullptr, nullptr};
  if (out) {
    dbg.t1 = out->t1_logits;
    dbg.dl = out->draft_logits;
    dbg.vl = out->verify_logits;
    if (out->h_mtp && copy_out(c, out->h_mtp, c->h_mtp, (size_t)B * c->d * 4)) return DMTP_ECUDA;
  }
  const bool eager = dbg.t1 || dbg.dl || dbg.vl;
  if (forced) {
    if (cudaMemcpyAsync(c->forced, forced, (size_t)B * 7 * 4, cudaMemcpyDeviceToDevice, c->st) !=
        cudaSuccess)
      return DMTP_ECUDA;
  }
  if (eager) {
    c->launches = 0;
    enqueue_round(c, dbg, forced ? c->forced : nullptr, depth);
    c->round_launches = c->launches;
  } else {
    // one graph per mode and depth; forced drafts are read from the context's own buffer,
    // which the copy above fills before the replay
    cudaGraphExec_t& graph = forced ? c->graph_forced[depth] : c->graph[depth];
    if (!graph) {
      // capture records work without running it, on a private stream (the legacy
      // default stream cannot be captured); the graph is then replayed on c->st
      if (!c->cap_st && cudaStreamCreateWithFlags(&c->cap_st, cudaStreamNonBlocking) != cudaSuccess)
        return DMTP_ECUDA;
      cudaGraph_t g;
      cudaStream_t user = c->st;
      c->st = c->cap_st;
      if (cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        c->st = user;
        return DMTP_ECUDA;
      }
      c->launches = 0;
      enqueue_round(c, dbg, forced ? c->forced : nullptr, depth);
      c->round_launches = c->launches;
      const cudaError_t ce = cudaStreamEndCapture(c->st, &g);
      c->st = user;
      if (ce != cudaSuccess) return DMTP_ECUDA;
      if (cudaGraphInstantiate(&graph, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        graph = nullptr;
        return DMTP_ECUDA;
      }
      cudaGraphDestroy(g);
    }
    if (cudaGraphLaunch(graph, c->st) != cudaSuccess) return DMTP_ECUDA;
  }
  if (cudaPeekAtLastError() != cudaSuccess) return DMTP_ECUDA;
  c->kv_bound += 8;
  if (out) {
    const RoundState& s = c->rs;
    int e = 0;
    e |= copy_out(c, out->committed, s.committed, (size_t)B * 8 * 4);
    e |= copy_out(c, out->n_accepted, s.n_acc, (size_t)B * 4);
    e |= copy_out(c, out->drafts, s.drafts, (size_t)B * 7 * 4);
    e |= copy_out(c, out->picks, s.g, (size_t)B * 8 * 4);
    e |= copy_out(c, out->kv_len, s.kv_len, (size_t)B * 4);
    e |= copy_out(c, out->snap_slot, s.snap_slot, (size_t)B * 4);
    e |= copy_out(c, out->delta, c->delta, (size_t)B * c->d * 4);
    e |= copy_out(c, out->mtp_len, s.mtp_len, (size_t)B * 4);
    if (out->draft_conf) e |= copy_out(c, out->draft_conf, c->dconf, (size_t)B * 7 * 4);
    if (e) return DMTP_ECUDA;
  }
  return DMTP_OK;
}

int dmtp_round_host(dmtp_ctx* c, int32_t* committed_host, int32_t* n_host) {
  if (!c) return DMTP_EINVAL;
  int r = dmtp_round(c, nullptr, nullptr);
  if (r) return r;
  if (committed_host &&
      cudaMemcpyAsync(committed_host, c->rs.committed, (size_t)c->B * 8 * 4,
                      cudaMemcpyDeviceToHost, c->st) != cudaSuccess)
    return DMTP_ECUDA;
  if (n_host && cudaMemcpyAsync(n_host, c->rs.n_acc, (size_t)c->B * 4, cudaMemcpyDeviceToHost,
                                c->st) != cudaSuccess)
    return DMTP_ECUDA;
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return DMTP_ECUDA;
  return DMTP_OK;
}

int dmtp_read_state(dmtp_ctx* c, int32_t* kv_len, int32_t* pending, uint64_t* hist) {
  if (!c) return DMTP_EINVAL;
  if (c->poisoned) return DMTP_ESTATE;
  const int B = c->B;
  if (kv_len && cudaMemcpyAsync(kv_len, c->rs.kv_len, B * 4, cudaMemcpyDeviceToHost, c->st))
    return DMTP_ECUDA;
  if (pending && cudaMemcpyAsync(pending, c->rs.A, B * 4, cudaMemcpyDeviceToHost, c->st))
    return DMTP_ECUDA;
  if (hist && cudaMemcpyAsync(hist, c->rs.hist, 64, cudaMemcpyDeviceToHost, c->st))
    return DMTP_ECUDA;
  return check_err(c);
}

int dmtp_round_launches(const dmtp_ctx* c) { return c ? c->round_launches : 0; }

int dmtp_prefill_stats(const dmtp_ctx* c, double* ms, int64_t* tokens) {
  if (!c) return DMTP_EINVAL;
  if (ms) *ms = c->prefill_ms;
  if (tokens) *tokens = c->prefill_tokens;
  return DMTP_OK;
}

int dmtp_round_profile(dmtp_ctx* c, dmtp_profile* out) {
  if (!c || !out) return DMTP_EINVAL;
  if (c->poisoned) return DMTP_ESTATE;
  const int B = c->B;
  c->kv_host.assign(B, 0);
  if (cudaMemcpyAsync(c->kv_host.data(), c->rs.kv_len, B * 4, cudaMemcpyDeviceToHost, c->st) !=
          cudaSuccess ||
      cudaStreamSynchronize(c->st) != cudaSuccess)
    return DMTP_ECUDA;
  const int mx = *std::max_element(c->kv_host.begin(), c->kv_host.end());
  if (mx + 16 >= c->maxc) return DMTP_ECAPACITY;
  while (c->pev.size() < 2048) {  // more than one round's launches, made before any capture
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return DMTP_ECUDA;
    c->pev.push_back(e);
  }
  auto record = [&]() {
    c->prof = true;
    c->pcls.clear();
    c->pbytes.clear();
    c->pflops.clear();
    c->pimpl.clear();
    c->launches = 0;
    enqueue_round(c, Dbg{nullptr, nullptr, nullptr}, nullptr);
    prof_event(c, c->pcls.size());  // after the last launch
    c->prof = false;
  };
  // The round as a CUDA graph with event-record nodes between its launches, replayed once
  // on the context's stream: launch times as in the timed graph, without host launch gaps.
  // If the capture fails, the round runs eagerly with the same events.
  bool graph_ok = false;
  if (c->cap_st || cudaStreamCreateWithFlags(&c->cap_st, cudaStreamNonBlocking) == cudaSuccess) {
    cudaStream_t user = c->st;
    c->st = c->cap_st;
    c->prof_external = true;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    if (cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
      record();
      const cudaError_t ce = cudaStreamEndCapture(c->st, &g);
      if (ce == cudaSuccess && cudaGraphInstantiate(&ge, g, 0) == cudaSuccess) graph_ok = true;
    }
    c->st = user;
    c->prof_external = false;
    if (g) cudaGraphDestroy(g);
    if (graph_ok) {
      graph_ok = cudaGraphLaunch(ge, c->st) == cudaSuccess;
      if (!graph_ok) return DMTP_ECUDA;  // nothing of the round ran twice: report and stop
    }
    if (ge) cudaGraphExecDestroy(ge);
    cudaGetLastError();  // a failed capture leaves no sticky error; clear its record
  }
  if (!graph_ok) record();
  c->kv_bound = std::max<long>(c->kv_bound, mx) + 8;
  if (cudaStreamSynchronize(c->st) != cudaSuccess) return DMTP_ECUDA;
  memset(out, 0, sizeof(*out));
  const size_t n = c->pcls.size();
  for (size_t i = 0; i < n; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, c->pev[i], c->pev[i + 1]) != cudaSuccess) return DMTP_ECUDA;
    const int k = c->pcls[i];
    out->ms[k] += ms;
    out->bytes[k] += c->pbytes[i];
    out->impl_bytes[k] += c->pimpl[i];
    out->flops[k] += c->pflops[i];
    out->launches[k] += 1;
  }
  float tot = 0.f;
  if (n && cudaEventElapsedTime(&tot, c->pev[0], c->pev[n]) != cudaSuccess) return DMTP_ECUDA;
  out->round_ms = tot;
  out->graph = graph_ok ? 1 : 0;
  return check_err(c);
}

int dmtp_set_draft_list(dmtp_ctx* c, const int32_t* ids, int n) {
  if (!c) return DMTP_EINVAL;
  if (c->poisoned) return DMTP_ESTATE;
  if (!c->list_cap || n < 0 || n > c->list_cap || (n > 0 && !ids)) return DMTP_EINVAL;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= c->V || (i > 0 && ids[i] <= ids[i - 1])) return DMTP_EINVAL;
  if ((n > 0) != (c->list_n > 0)) c->drop_graphs();  // the heads change: capture again
  c->list_n = n;
  if (n == 0) return DMTP_OK;
  // pageable host sources: each copy has left the caller's memory when the call returns
  if (cudaMemcpyAsync(c->hc_ids, ids, (size_t)n * 4, cudaMemcpyHostToDevice, c->st) !=
          cudaSuccess ||
      cudaMemcpyAsync(c->hc_n, &c->list_n, 4, cudaMemcpyHostToDevice, c->st) != cudaSuccess)
    return DMTP_ECUDA;
  if (c->fp8)
    op_gather_rows(c->h8, c->hc, (size_t)c->d, c->hc_ids, n, c->h8s, c->hcs, c->st);
  else
    op_gather_rows(c->w.head, c->hc, (size_t)c->d * 2, c->hc_ids, n, nullptr, nullptr, c->st);
  return cudaGetLastError() == cudaSuccess ? DMTP_OK : DMTP_ECUDA;
}

uint32_t dmtp_error_word(const dmtp_ctx* c) { return c ? c->err_word : 0u; }

int dmtp_selftest_timeout(dmtp_ctx* c, uint64_t limit_ns) {
  if (!c) return DMTP_EINVAL;
  if (c->poisoned) return DMTP_ESTATE;
  if (limit_ns < 1000ull || limit_ns > 1000000000ull) return DMTP_EINVAL;
  op_wait_selftest(c->err, (unsigned long long)limit_ns, c->st);
  return cudaGetLastError() == cudaSuccess ? DMTP_OK : DMTP_ECUDA;
}

void dmtp_free(dmtp_ctx* c) {
  if (!c) return;
  c->drop_graphs();
  if (c->cap_st) cudaStreamDestroy(c->cap_st);
  for (cudaEvent_t e : c->pev) cudaEventDestroy(e);
  delete c;
}

const char* dmtp_strerror(int code) {
  switch (code) {
    case DMTP_OK: return "ok";
    case DMTP_EINVAL: return "invalid argument or unsupported configuration";
    case DMTP_ENOMEM: return "workspace too small";
    case DMTP_ECAPACITY: return "KV capacity (max_ctx) exceeded";
    case DMTP_ECUDA: return "CUDA runtime error";
    case DMTP_EDEVICE: return "device-side check failed (bad token id, position or timeout)";
    case DMTP_ESTATE: return "context poisoned by an earlier device error";
    default: return "unknown error";
  }
}

}  // extern "C"
