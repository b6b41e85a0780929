// Host-side launchers for the DMTP round kernels. `dt` selects the storage type of
// weights, KV caches and GEMM operands: 0 = fp32, 1 = bf16. The residual stream,
// GEMM outputs, softmax and the GDN state are always fp32.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dmtp {

// Programmatic dependent launch bookkeeping (launch_pdl in common.cuh): whether the
// previous operation this host thread enqueued was a kernel launch, since a programmatic
// edge needs a kernel on both sides. Memsets, copies and event records in a stream that
// also gets launch_pdl() launches call pdl_fence() after themselves.
extern thread_local bool g_pdl_prev;
bool pdl_enabled();  // process-wide: the environment variable DMTP_PDL=0 turns it off
inline void pdl_fence() { g_pdl_prev = false; }

// Row mapping shared by the row-wise kernels: output row r reads input row
//   (r / out_group) * in_group + in_offset + (r % out_group).
struct RowMap {
  int out_group = 1, in_group = 1, in_offset = 0;
};

// ---- elementwise.cu --------------------------------------------------------------
// y[r] = RMSNorm(x[map(r)]) * g, stored as dt (y) and optionally as fp32 (y32);
// tap (optional, dt): raw copy of x[map(r)] into column block of a tap buffer.
// *_lo arguments: element offset of the bf16 remainder half of a split operand (0: none).
// zero (optional): rows [rows][ldz] of which the first nz floats are set to 0.
void op_rmsnorm(int dt, const float* x, int ldx, const void* g, void* y, int ldy, long y_lo,
                float* y32, int ld32, void* tap, int ldtap, long tap_lo, int rows, int d,
                float eps, RowMap map, cudaStream_t st, float* zero = nullptr, int ldz = 0,
                int nz = 0);
// Draft-head quantisation to E4M3 rows with power-of-two scales (common.cuh):
// q [rows][d] bytes and qs [rows] scales of the bf16 matrix W [rows][d] (d % 4 == 0) ...
void op_quant_rows_e4m3(const void* W, int rows, int d, void* q, float* qs, cudaStream_t st);
// ... and of RMSNorm(x[map(r)]) * g (bf16 gain; d % 4 == 0, d <= 4096), row pitch ldq.
void op_rmsnorm_e4m3(const float* x, int ldx, const void* g, void* q, int ldq, float* qs,
                     int rows, int d, float eps, RowMap map, cudaStream_t st);
// x[m] = E[tok[m]] (fp32 rows)
void op_embed(int dt, const void* E, const int* tok, int vocab, float* x, int rows, int d,
              unsigned* err, cudaStream_t st);
// z[r] = [RMS(partA[r]) * gA ; RMS(partB[r]) * gB] as dt; each part is an fp32 row
// (src32 != null, row map) or an embedding row E[tok[r]] (tok != null).
struct ConcatPart {
  const float* src32 = nullptr;
  int ld = 0;
  RowMap map;
  const int* tok = nullptr;
  int tok_stride = 1;
  const void* g = nullptr;
};
void op_concat_rms2(int dt, const void* E, int vocab, ConcatPart a, ConcatPart b, void* z,
                    long z_lo, int rows, int d, float eps, unsigned* err, cudaStream_t st);
// Drafter slots: x[b*8+s] = E[A_b] (s=0), E[T1_b] + delta_b (s=1), E[mask] (s>=2)
void op_build_slots(int dt, const void* E, int vocab, const int* A, const int* drafts,
                    const float* delta, int mask_id, float* x, int B, int d, unsigned* err,
                    cudaStream_t st);
// h = silu(gu[:, :F]) * gu[:, F:] as dt
// Read `bytes` (multiple of 16, 16-byte aligned) of buf to evict the L2; sink[1] is a
// write target that is never written in practice.
void op_l2_flush(const void* buf, size_t bytes, unsigned* sink, cudaStream_t st);
void op_swiglu(int dt, const float* gu, void* h, long h_lo, int rows, int F, cudaStream_t st);
// RoPE (table) + cache write. src rows m = b*rg + s at position base[b] + s (rg rows per
// sequence: 8, or fewer in a verify of fewer drafts).
// q_off < 0: no q. q_out fp32 [rows][hq][hd], or, when q_split != null (bf16 models),
// q as a bf16 pair: hi at q_split, remainder at q_split + q_lo (elements).
void op_rope_kv(int dt, const float* src, int ld, int q_off, int k_off, int v_off, float* q_out,
                void* q_split, long q_lo, void* Kc, void* Vc, const int* base, const int* cseq,
                const float2* tab, int rows, int hq, int hkv, int hd, int max_ctx, unsigned* err,
                cudaStream_t st, int rg = 8);
// fp32 -> dt copy of rows (with row map)
void op_cast_rows(int dt, const float* x, int ldx, void* y, int ldy, long y_lo, int rows, int d,
                  RowMap map, cudaStream_t st);
void op_rope_table(float2* tab, int npos, int hd, float theta, cudaStream_t st);

// ---- round control (elementwise.cu) -------------------------------------------------
struct RoundState {
  int* kv_len;        // [B]
  int* pos0;          // [B] position of row 0 in the current step
  int* A;             // [B] pending token
  int* drafts;        // [B][7]
  int* g;             // [B][8]
  int* n_acc;         // [B]
  int* committed;     // [B][8]
  int* tok;           // [B*8] tokens of the target rows
  int* mtp_tok;       // [B*8] tokens of the MTP rows
  int* mtp_base;      // [B] position of MTP row 0
  int* mtp_cnt;       // [B] valid MTP rows
  int* rows_valid;    // [B] valid target rows (GDN state advance)
  int* cseq;          // [B] cache sequence of each row group (the group itself in rounds;
                      // a prefill step may give several groups one sequence)
  int* snap_slot;     // [B]
  int* mtp_len;       // [B] next MTP position (= kv_len + 1)
  unsigned long long* hist;  // [8]
  unsigned long long* keys;  // [B*16] argmax keys (T1 | drafter | verify)
  int* gdn_live;      // [n_gdn][B] index of the live state buffer (0..8)
  int* gdn_slot;      // [n_gdn][B][8] buffer index of each snapshot slot
  int n_gdn;
  int B;
  unsigned* err;
};
void op_round_begin(const RoundState& s, cudaStream_t st);
// keys -> ids: dst[b*dst_stride + dst_off + j] = id(keys[b*per + j]) (or forced value);
// map (optional): the key's index is a row of a token list, whose id is map[index]
void op_keys_to_ids(const unsigned long long* keys, int B, int per, int* dst, int dst_stride,
                    int dst_off, const int* forced, int forced_stride, int forced_off,
                    cudaStream_t st, const int* map = nullptr);
// Token list of the draft heads: dst row i = src row ids[i] (row_bytes each, a multiple of
// 16, 16-byte aligned rows) for i < n; with scale arrays, dst_s[i] = src_s[ids[i]].
void op_gather_rows(const void* src, void* dst, size_t row_bytes, const int* ids, int n,
                    const float* src_s, float* dst_s, cudaStream_t st);
// Verify rows of a round that carries `depth` drafts (0..7): rows [A, T1..T_depth] of each
// sequence, row m = b*(depth+1) + r; picks past the depth cleared to -1; rows_valid set.
void op_verify_tokens(const RoundState& s, int depth, cudaStream_t st);
// Prefix acceptance over the first `depth` drafts (n <= depth); the live recurrent state
// is the one after row depth, so slot n is swapped in when n < depth.
void op_accept(const RoundState& s, int depth, cudaStream_t st);
// h_mtp[b] = x[b*8 + cnt[b]-1]
void op_gather_hmtp(const float* x, const int* cnt, float* h_mtp, int B, int d, cudaStream_t st);
// Prefill step: row group pb takes chunk sched[pb] = (sequence, chunk of 8 positions);
// sets tokens, positions, MTP rows and the cache-sequence map of every row group.
void op_prefill_chunk(const RoundState& s, const int* prompts, const int* plen, int pmax,
                      const int2* sched, cudaStream_t st);
void op_prefill_save_last(const float* hT, const int* plen, const int2* sched, float* hlast,
                          int B, int d, cudaStream_t st);
void op_prefill_final(const RoundState& s, const int* plen, const float* hlast, float* hT, int d,
                      cudaStream_t st);
void op_prefill_done(const RoundState& s, const int* plen, cudaStream_t st);
// Failure-path self-test: one bounded mbarrier wait that nothing satisfies gives up after
// limit_ns and sets DMTP_ERR_TIMEOUT in err.
void op_wait_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t st);

// ---- attention.cu ------------------------------------------------------------------
struct AttnArgs {
  const void* Kc;      // [B][hkv][max_ctx][hd] dt
  const void* Vc;      // [B][hkv][max_ctx/64][hd][64] dt (transposed, blocked by 64 keys)
  const float* q;      // [B*8][hq][hd] fp32
  float* part_o;       // [B][hkv][nchunk][QN][hd]
  float* part_ml;      // [B][hkv][nchunk][QN][2]
  void* out;           // [B*8][hq*hd] dt
  long out_lo;         // element offset of the remainder half (0: none)
  const int* base;     // [B] position of row 0
  const int* cseq;     // [B] cache sequence of each row group (nullptr: the group itself)
  int causal;          // 1: row s sees keys <= base+s; 0: keys <= base+7
  int lo_fixed;        // lowest key index
  int window;          // > 0: lo = max(lo_fixed, base - window)
  int B, hq, hkv, hd, max_ctx, chunk, nchunk;  // chunk: keys per partial (absolute grid)
  const void* qs;      // tensor-core path: queries as bf16 hi [B*8][hq][hd] ...
  long qs_lo;          // ... and remainder at qs + qs_lo
  int pgrid;           // tensor-core path: persistent CTAs; partials [pgrid + B*hkv]
  int ptk;             // tensor-core path: keys per tile (kAttnTile)
  int rows = 8;        // rows per sequence (a verify of fewer drafts has fewer): row m of
                       // q / out is sequence m / rows at position base + m % rows
};
void op_attention(int dt, const AttnArgs& a, cudaStream_t st);
void op_attention_merge(int dt, const AttnArgs& a, cudaStream_t st);
constexpr int kAttnTile = 128;  // keys per tile of the tensor-core attention
constexpr int kAttnMaxB = 1024; // sequences its in-kernel schedule handles
// tcgen05 attention (bf16 caches, head_dim 64 or 128, 8 x GQA-group <= 64 queries);
// tmK: K cache as 3-D {64 dims, B*hkv*max_ctx keys (stride hd*2 B), hd/64 blocks (stride
// 128 B)}, box {64, kAttnTile, hd/64}; tmV: transposed V cache blocked by 64 keys as 3-D
// {64 keys, hd rows (stride 128 B), B*hkv*max_ctx/64 blocks (stride hd*128 B)}, box
// {64, hd, kAttnTile/64}: one request per tile for each; tmQh / tmQl: the bf16 query halves as 3-D
// [B*8][hq][hd] maps, box {64, hq/hkv, 8}. Persistent: a.pgrid CTAs split the visible key
// tiles of all (sequence, kv head) pairs evenly; partial (CTA i, pair seg) goes to slot
// i + seg of part_o / part_ml (pgrid + B*hkv slots); then merges into out.
void op_attention_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     const CUtensorMap& tmQh, const CUtensorMap& tmQl, unsigned* err,
                     cudaStream_t st);
int attn_tc_init_attributes();

// Target-only sampled verification in the verify head's argmax epilogue: row m is
// sequence m / group at position pos0[m / group] + m % group, and its pick is the
// sample argmax_v (l_v / T + G_v) for the next position (Philox4x32-10 Gumbel noise
// keyed by (seed_lo, seed_hi), common.cuh), compared as l_v * scale2 + G2_v with
// scale2 = log2(e) / T. nullptr / scale2 0: greedy argmax.
struct SampleArgs {
  float scale2;
  uint32_t seed_lo, seed_hi;
  const int* pos0;
  int group;
};

// ---- gemm_simt.cu (fp32 storage) ------------------------------------------------------
// out[m*ldo + n] += sum_k X[m*K + k] * W[n*K + k]   (fp32 W and X)
void op_gemm_simt_acc(const float* W, const float* X, int N, int K, int M, float* out, int ldo,
                      cudaStream_t st);
// argmax over n of sum_k X[m,k] W[n,k] -> atomicMax into keys[m]; logits optional
// smp: sampled picks (nullptr: argmax of the logits)
void op_gemm_simt_argmax(const float* W, const float* X, int N, int K, int M,
                         unsigned long long* keys, float* logits, long ldl,
                         const SampleArgs* smp, cudaStream_t st);

// ---- gemm_tc.cu (bf16, tcgen05) -------------------------------------------------------
struct TcPlan {
  CUtensorMap tmW, tmX;
  int N, K, M, MT, splits, stages;
  int wide;       // 128-row weight halves per CTA (1 or 2)
  int msplit;     // token parts: CTAs per weight tile (1..4; the last part may be short)
  int mct;        // token rows per CTA
  int split;      // X is the [hi; lo] bf16 pair
  int xbox, nx;   // X rows per box, boxes per stage
  int x3d;        // the two halves' boxes as one 3-D request
  int merged;     // hi and lo in one MMA of 2*mct columns
  int pair;       // CTA pairs along the weight tiles: one M = 256 MMA over two SMs, each
                  // CTA loading its weight rows and one half (hi or lo) of the tokens
  int acc_cols;   // TMEM columns per accumulator
  int swiglu, F;  // SwiGLU epilogue: W = [gate; up] of F rows each
  size_t smem;
  size_t stage_area;  // bytes of the stage ring (reused to stage output tiles)
  int nsm;            // SMs of the device (one CTA per SM)
  // Fixed-order K-part sums (K split within one wave): partial-tile scratch of
  // part_floats floats and a counter per output tile (zeroed once, left zero by every
  // launch); null: the parts add into the output in arrival order.
  float* part;
  int* tile_cnt;
  size_t part_floats;
};
// Padded token rows of an M-row operand (multiple of 16, >= 16).
int tc_mt(int M);
// Tensor map of a row-major bf16 [rows, cols] matrix, box {64, box_rows}, 128-B swizzle.
int tc_make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
// Tensor map of a row-major fp32 matrix [rows, cols] with row pitch ld elements, box
// {box_cols, box_rows}, no swizzle.
int tc_make_tmap_f32(CUtensorMap* tm, void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_cols, uint32_t box_rows);
// 3-D bf16 view [d2][d1][d0] with byte strides s1, s2, unswizzled box {b0, b1, b2}.
int tc_make_tmap3s_box(CUtensorMap* tm, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);
// Tensor map of a row-major byte matrix [rows, cols] (E4M3), box {128, box_rows}, 128-B
// swizzle.
int tc_make_tmap_u8(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);
// 3-D bf16 tensor [d2][d1][d0] (d0 innermost), box {64, b1, b2}, 128-B swizzle.
int tc_make_tmap3(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint32_t b1, uint32_t b2);
// 3-D bf16 view with explicit byte strides s1 (dim 1) and s2 (dim 2), box {64, b1, b2},
// 128-B swizzle: one TMA request moves b2 slabs of b1 rows x 128 B.
int tc_make_tmap3s(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b1, uint32_t b2);
// Builds the tensor maps and launch shape for out[M,N] = X[M,K] . W[N,K]^T. split: X
// holds 2*tc_mt(M) rows, the bf16 high halves then the low halves (X = hi + lo).
int tc_plan(TcPlan* p, const void* W, int N, int K, const void* X, int M, int nsm, bool split);
// Gate/up GEMM with the SwiGLU epilogue: W = [gate; up] ([2F, K]), each CTA pairs gate
// rows n0.. with up rows F + n0.. (two accumulators) and writes h = silu(g) * u, a bf16
// pair [M][F] (remainder at h + h_lo), so no fp32 output or separate SwiGLU pass.
int tc_plan_swiglu(TcPlan* p, const void* W, int F, int K, const void* X, int M, int nsm,
                   bool split, int msplit, int pair = 0);
void op_gemm_tc_swiglu(const TcPlan& p, void* h, long h_lo, unsigned* err, cudaStream_t st);
// tc_plan with the tile shape given: wide (1, 2), msplit (1..4), splits (<= 0: chosen) and
// pair (1: CTA pairs, split operands whose token part fits one MMA, 2 mct <= 256).
int tc_plan_shape(TcPlan* p, const void* W, int N, int K, const void* X, int M, int nsm,
                  bool split, int wide, int msplit, int splits, int pair = 0);
// out[m*ldo + n] += (X W^T)[m][n] for the plan's M x N (out fp32, zeroed or holding the
// residual; K parts and CTAs add element-wise atomically).
void op_gemm_tc_acc(const TcPlan& p, float* out, int ldo, unsigned* err, cudaStream_t st);
int tc_init_attributes();

// ---- head_tc.cu (bf16 LM head with fused argmax, tcgen05) -------------------------------
// keys[m] = max over v of argmax_key(l[m][v], v) with l = X[m] . W[v] (X [M, K] bf16, one
// operand; W [V, K] bf16), or of the sampled scores l * scale2 + G2 under smp. Token-major
// persistent kernel: tokens are the MMA's M side (TH halves of 128 rows), NV (128 or
// 256) vocabulary rows per tile, one CTA per SM.
struct HeadPlan {
  CUtensorMap tmW, tmX;
  int V, K, M, MT, TH, NV, ew, tiles, grid, stages;
  int fp8;                       // E4M3 operands (draft heads)
  const float *wscale, *xscale;  // E4M3 row scales of W (padded past V) and of X
  size_t smem;
  // A token list in place of the vocabulary (draft heads): W holds V rows of capacity,
  // of which the first *vdev (read on the device at launch) are scored; vmap[i] is the
  // token id of row i, where the debug logits go. Both null: the full vocabulary.
  const int* vdev;
  const int* vmap;
};
// ew: epilogue warps (4 or 8)
int head_plan(HeadPlan* p, const void* W, int V, int K, const void* X, int M, int nsm, int nv,
              int ew);
// Draft head on E4M3 operands (op_quant_rows_e4m3 / op_rmsnorm_e4m3): W8 [V][K] bytes with
// scales wscale (readable up to the vocabulary rounded up to 256 rows), X8 [M][K] bytes
// with xscale [M]; K % 128 == 0. The argmax ranks acc * wscale[v] (xscale[m] is common to
// the row); debug logits are acc * wscale[v] * xscale[m].
int head_plan_e4m3(HeadPlan* p, const void* W8, const float* wscale, int V, int K,
                   const void* X8, const float* xscale, int M, int nsm, int nv, int ew);
// logits (optional, fp32 [M][ldl]) receives the raw logits; smp: sampled picks (nullptr:
// argmax of the logits). keys must hold zeros (or earlier keys to combine with).
// conf (optional, greedy heads only): per-thread partials of the head's confidence, the
// probability it gives its own pick over the scores within 20 of the best (max and
// windowed sum; head_conf_parts(p) x M float2), combined by op_conf_combine.
void op_head_tc(const HeadPlan& p, unsigned long long* keys, float* logits, long ldl,
                const SampleArgs* smp, unsigned* err, cudaStream_t st, float2* conf = nullptr);
int head_conf_parts(const HeadPlan& p);
// dst[(m / per) * stride + off + m % per] = 1 / sum over the scores within 20 of the best
// of exp(score - best), row m of the head's M rows.
void op_conf_combine(const HeadPlan& p, const float2* parts, int per, float* dst, int stride,
                     int off, cudaStream_t st);
int head_init_attributes();

// ---- gdn.cu ----------------------------------------------------------------------------
struct GdnArgs {
  const float* qkvab;    // [B*8][ld] fp32: q | k | v | alpha-logit | beta-logit
  int ld;
  float* states;         // [B][8][H][dv][dk] fp32 for this layer
  const int* live;       // [B]
  const int* slot;       // [B][8]
  const int* rows_valid; // [B]
  int snapshots;         // 1: write the state after each row r < rows-1 to slot[b][r]
  int rows = 8;          // rows per sequence (row m of qkvab / out: sequence m / rows)
  void* out;             // [B*8][H*dv] dt
  long out_lo;           // element offset of the remainder half (0: none)
  int B, H, dk, dv;
  unsigned* err;
};
void op_gdn(int dt, const GdnArgs& a, cudaStream_t st);

}  // namespace dmtp
