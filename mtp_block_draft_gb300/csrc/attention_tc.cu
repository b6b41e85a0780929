// Decode attention on the 5th-generation tensor cores (sm_103a), persistent and
// evenly split over the SMs.
//
// Work: for every (sequence, kv head) segment, the 128-key tiles its 8 rows can see.
// All segments' tiles are laid end to end and the grid (one CTA per SM) takes equal
// contiguous ranges of that list, so every CTA streams the same number of tiles
// whatever the context lengths; a CTA's range covers pieces of one or more segments.
// Each piece serves all 8 rows x the GQA group of query heads of its kv head (QN <= 64
// queries), so each cached K/V byte is read from HBM once per sequence and layer, and
// leaves a partial (m, l, O) for the merge kernel. Keys stream through shared memory
// in tiles of TK keys (TMA, 128-byte swizzle, NST stages) continuously across pieces.
// Per tile:
//   S = Q K^T  : tcgen05 M=128, N=TK keys, K = hd, A from TMEM: the fp32 queries enter
//                as a bf16 pair, Q_hi in operand rows 0..63 and Q_lo in rows 64..127, so
//                TMEM lanes r and r+64 hold Q_hi K^T and Q_lo K^T of query row r; the
//                softmax threads of the two lanes swap a quarter of the tile through
//                shared memory and each sums its own quarter, which keeps the queries'
//                fp32 precision at half the MMA work of a pair along K. S is
//                double-buffered in TMEM: the next tile's scores are computed during this
//                tile's softmax.
//   softmax    : warps 0-7, four threads per query row, each a quarter of the
//                tile's keys: mask (causal rows / anchor window / segment bounds; skipped
//                on interior tiles), exponentiate against a per-row reference max, and
//                write P as a bf16 pair, P_hi in operand rows 0..63, P_lo in 64..127.
//   O += P V   : tcgen05 M=128, N=hd, K=TK keys, B = the transposed V tile (K-major);
//                O stays in TMEM for the whole piece: lanes 0..63 accumulate P_hi V,
//                lanes 64..127 P_lo V; they are summed once at the end of the piece.
// The reference max only moves when a row's scores exceed it by more than 2^11; then
// that row's O (both halves) is rescaled in TMEM. Keeping a stale reference is exact:
// the same factor multiplies O and the running sum l.
// The queries, already split into bf16 halves by the RoPE kernel, live in TMEM as the
// A operand of S (written by the softmax warps at the start of each piece), which
// leaves the shared memory to the K/V ring: three 64 KB stages.
// Warp 8 lane 0 issues the K/V loads, warp 9 lane 0 the MMAs.
//
// Visibility follows the DMTP blog §6.2: target and MTP rows are causal over their
// cache; the drafter sees its anchor-relative window and the whole 8-slot block.
// Every mbarrier wait is bounded; on a timeout the error word is set, in-flight copies
// and MMAs are drained and TMEM is freed before the CTA returns.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

namespace {

constexpr int kBlk = 128 * 128;  // one 128-row x 64-element bf16 operand block (16 KB)

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// byte offset of the 16-byte chunk c (0..7) of row r inside a 128-B-swizzled block
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulate (kind::f16). A holds
// row m in TMEM lane m, two consecutive k elements per 32-bit column (even k low).
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers (no wait).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// scale `n` TMEM columns of this warp's 32 lanes by a per-lane factor f
__device__ __forceinline__ void tmem_scale(uint32_t taddr, int n, float f) {
  for (int cc = 0; cc < n; cc += 16) {
    float v[16];
    tmem_ld16(taddr + cc, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] *= f;
    tmem_st16(taddr + cc, v);
  }
}


// First visible key of a sequence whose block rows start at `base`; the last is
// base + rows - 1.
__device__ __forceinline__ int vis_lo(const AttnArgs& a, int base) {
  int lo = a.lo_fixed;
  if (a.window > 0) lo = max(lo, base - a.window);
  return lo;
}
// Visible key tiles of a sequence (tile size tk).
__device__ __forceinline__ int vis_tiles(const AttnArgs& a, int base, int tk) {
  return (base + a.rows - 1) / tk - vis_lo(a, base) / tk + 1;
}
// Work units of a (sequence, kv head) segment in the even split over the CTAs: its key
// tiles plus kPieceCost units standing for the fixed cost of a piece (writing the
// queries, reading out O and writing a partial: about three to four tiles' time), so
// that a CTA whose range crosses more segment starts is given fewer key tiles. The
// overhead units come first in each segment and carry no keys. Five units gave the
// shortest B32 launches (2: 45.9, 3: 44.3, 5: 42.7, 7: 43.9, 10: 47.8 us).
constexpr int kPieceCost = 5;
__device__ __forceinline__ int seg_units(const AttnArgs& a, int base, int tk) {
  return vis_tiles(a, base, tk) + kPieceCost;
}

// Shared-memory plan (TK keys per tile, NST stages). P (128 rows x TK keys) of tile t is
// written into the K area of its stage when that is large enough (K(t) is dead once S(t)
// is computed), else into a double buffer of its own.
template <int HD, int TK, int NST>
struct Smem {
  static constexpr int kDB = HD / 64;                 // 64-wide head-dim blocks
  static constexpr uint32_t kKBox = TK * 128;         // TK keys x 64 head dims
  static constexpr uint32_t kKTile = kDB * kKBox;
  static constexpr uint32_t kVBox = HD * 128;         // HD rows x 64 keys
  static constexpr uint32_t kVTile = (TK / 64) * kVBox;
  static constexpr uint32_t kStage = kKTile + kVTile;
  static constexpr uint32_t kPTile = (TK / 64) * kBlk;  // 128 rows x TK keys
  static constexpr bool kPinK = kKTile >= kPTile;
  static constexpr uint32_t kP = kPinK ? 0 : 2 * kPTile;
  static constexpr uint32_t kX = 64 * (HD / 2 + 4) * 4;  // P_lo V half rows, final sum
  // barriers, tile maxima [2][4][64], running sums [4][64], tile-count prefix [B + 1]
  static constexpr uint32_t kSmall = 256 + 2048 + 1024 + 4 * (kAttnMaxB + 1);
  static constexpr uint32_t kBig = NST * kStage + kP + kX;  // 1024-aligned region
  // the big region starts at the first 1024-byte boundary past kSmall: room for any base
  // address (a CTA sharing its SM with another kernel's CTAs, under programmatic launch,
  // gets a dynamic shared memory base that is not 1024-aligned)
  static constexpr uint32_t kBytes = (kSmall + 1024 + kBig + 127) / 128 * 128;
  static_assert(kBytes <= 232448, "shared memory plan exceeds 227 KB");
};

}  // namespace

template <int HD, int TK, int NST>
__global__ void __launch_bounds__(320, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmQl,
              AttnArgs a, unsigned* err) {
  using L = Smem<HD, TK, NST>;
  constexpr int HALF = HD / 2;
  constexpr int KQ = TK / 4;  // keys per softmax thread (a quarter of the tile)
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  const int grp = a.hq / a.hkv, QN = a.rows * grp, B = a.B, hkv = a.hkv;
  uint64_t* bars = (uint64_t*)smem_raw;
  float* sMax = (float*)(bars + 32);  // [2 tiles][4 quarters][64] tile maxima (log2)
  float* sL = sMax + 512;             // [4][64] running sums at the end of a piece
  int* s_pref = (int*)(sL + 256);     // [B + 1] prefix sums of per-sequence tile counts

  // ---- schedule: this CTA's range [x0, x1) of the global tile list ----
  if (threadIdx.x < 32) {  // warp 0: inclusive scan of the tile counts, 32 at a time
    const int ln = threadIdx.x;
    int carry = 0;
    if (ln == 0) s_pref[0] = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      int v = b0 + ln < B ? seg_units(a, a.base[b0 + ln], TK) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (ln >= o) v += u;
      }
      if (b0 + ln < B) s_pref[b0 + ln + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const long T = (long)hkv * s_pref[B];
  const long x0 = T * blockIdx.x / gridDim.x, x1 = T * (blockIdx.x + 1) / gridDim.x;
  if (x0 >= x1) return;
  // The piece that starts at unit x: sequence b, kv head g, first key tile kt0 (absolute),
  // key tile count nt (0 when the piece holds only a segment's overhead units), the
  // sequence's base position, and the units it spans (adv).
  struct Pc {
    int b, g, kt0, nt, base;
    long adv;
  };
  auto piece_at = [&](long x) -> Pc {
    Pc q;
    int lo_b = 0, hi_b = B;  // largest b with hkv * s_pref[b] <= x
    while (hi_b - lo_b > 1) {
      const int mid = (lo_b + hi_b) >> 1;
      if ((long)hkv * s_pref[mid] <= x) lo_b = mid; else hi_b = mid;
    }
    q.b = lo_b;
    const int nu = s_pref[q.b + 1] - s_pref[q.b];  // units of one segment of sequence b
    const long r = x - (long)hkv * s_pref[q.b];
    q.g = (int)(r / nu);
    const int off = (int)(r % nu);
    q.adv = min((long)(nu - off), x1 - x);
    const int first = max(off, kPieceCost);  // first unit that is a key tile
    q.nt = (int)max(0L, off + q.adv - first);
    q.base = a.base[q.b];
    q.kt0 = vis_lo(a, q.base) / TK + (first - kPieceCost);
    return q;
  };
  // the first piece at or after unit x that has key tiles (x1 if none)
  auto first_piece = [&](long x, Pc& q) -> long {
    while (x < x1) {
      q = piece_at(x);
      if (q.nt > 0) return x;
      x += q.adv;
    }
    return x1;
  };
  {
    Pc q;
    if (first_piece(x0, q) >= x1) return;  // only overhead units: nothing to do
  }

  uint8_t* sm = smem_raw + L::kSmall;
  sm += (1024 - (smem_u32(sm) & 1023)) & 1023;
  if (sm + L::kBig > smem_raw + L::kBytes) {  // dynamic shared memory base not aligned enough
    if (threadIdx.x == 0) set_err(err, DMTP_ERR_TIMEOUT);
    return;
  }
  uint8_t* sKV = sm;
  uint8_t* sPsep = sKV + NST * L::kStage;
  float* xo = (float*)(sPsep + L::kP);  // [64][HALF + 4]
  auto stage = [&](int t) -> uint8_t* { return sKV + (t % NST) * L::kStage; };
  auto p_buf = [&](int t) -> uint8_t* {
    return L::kPinK ? stage(t) : sPsep + (t & 1) * L::kPTile;
  };
  uint64_t* kv_full = bars;             // [NST]
  uint64_t* kv_empty = bars + NST;      // [NST]
  uint64_t* s_full = bars + 2 * NST;    // [2] (S is double-buffered in TMEM)
  uint64_t* q_full = s_full + 2;        // the 256 softmax threads wrote a piece's queries
  uint64_t* p_full = q_full + 1;        // the 256 softmax threads wrote this tile's P
  uint64_t* o_full = p_full + 1;        // one commit per tile's P V
  uint64_t* pfin = o_full + 1;          // a piece's last P V completed
  uint64_t* o_drained = pfin + 1;       // the 256 softmax threads read a piece's O
  uint64_t* fin = o_drained + 1;
  uint32_t* tmem_slot = (uint32_t*)(fin + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(smem_u32(&kv_full[i]), 1);
      mbar_init(smem_u32(&kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&s_full[0]), 1);
    mbar_init(smem_u32(&s_full[1]), 1);
    mbar_init(smem_u32(q_full), 256);
    mbar_init(smem_u32(p_full), 256);
    mbar_init(smem_u32(o_full), 1);
    mbar_init(smem_u32(pfin), 1);
    mbar_init(smem_u32(o_drained), 256);
    mbar_init(smem_u32(fin), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // S buffers at columns 0 and TK, O (HD columns) after them, then two Q buffers (one per
  // piece parity): HD bf16 per lane = HD/2 columns each
  constexpr uint32_t kTmemCols = 2 * TK + 2 * HD <= 256 ? 256 : 512;
  static_assert(2 * TK + 2 * HD <= 512, "TMEM plan exceeds 512 columns");
  if (warp == 8) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Up to here the CTA read only the sequences' base positions, which the launch before
  // this one (the RoPE / KV-row writer) does not write and lets this launch begin only
  // after its own wait; the queries and the K/V tiles come after the wait.
  pdl_trigger();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 2 * TK;
  auto tQb = [&](int buf) -> uint32_t { return tO + HD + (uint32_t)buf * (HD / 2); };

  if (warp == 8) {
    if (lane == 0) {
      // ---------------- K/V producer: every tile of the range, in order ----------------
      const uint64_t pol = policy_evict_first();
      int gt = 0;
      bool ok = true;
      Pc pc;
      for (long x = first_piece(x0, pc); x < x1 && ok; x = first_piece(x + pc.adv, pc)) {
        const int b = pc.b, g = pc.g, kt0 = pc.kt0, nt = pc.nt;
        const int cb = a.cseq ? a.cseq[b] : b;  // cache sequence of the row group
        const long krow0 = ((long)cb * hkv + g) * a.max_ctx;
        const long vblk0 = ((long)cb * hkv + g) * (a.max_ctx / 64);  // 64-key V^T blocks
        for (int t = 0; t < nt; ++t, ++gt) {
          const int s = gt % NST;
          if (!mbar_wait(smem_u32(&kv_empty[s]), ((gt / NST) & 1) ^ 1, err)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&kv_full[s]);
          mbar_expect_tx(full, L::kStage);
          const int key0 = (kt0 + t) * TK;
          uint8_t* st = stage(gt);
          // K: the tile's keys x all head-dim slabs; V^T: its 64-key blocks; one request each
          tma_load_3d(smem_u32(st), &tmK, 0, (int)(krow0 + key0), 0, full, pol);
          tma_load_3d(smem_u32(st + L::kKTile), &tmV, 0, 0, (int)(vblk0 + key0 / 64), full, pol);
        }
      }
      for (int j = (gt > NST ? gt - NST : 0); j < gt; ++j)
        mbar_wait(smem_u32(&kv_full[j % NST]), (j / NST) & 1, err);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t id_qk = umma_idesc_bf16(128, TK);
      const uint32_t id_pv = umma_idesc_bf16(128, HD);
      auto issue_qk = [&](int xg, uint32_t tQ) -> bool {
        const int s = xg % NST;
        if (!mbar_wait(smem_u32(&kv_full[s]), (xg / NST) & 1, err)) return false;
        tc_fence_after();
        uint8_t* st = stage(xg);
#pragma unroll
        for (int kb = 0; kb < L::kDB; ++kb) {  // [Q_hi; Q_lo] rows against K
          const uint64_t dk = umma_desc_sw128(smem_u32(st + kb * L::kKBox));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 k = 8 TMEM columns of Q per MMA
            umma_bf16_ta(tmem + (xg & 1) * TK, tQ + kb * 32 + kk * 8, dk + 2 * kk, id_qk,
                         (kb | kk) ? 1u : 0u);
        }
        umma_commit(smem_u32(&s_full[xg & 1]));
        return true;
      };
      int gt = 0, p = 0;
      bool ok = true;
      Pc pc;
      for (long x = first_piece(x0, pc); x < x1 && ok; x = first_piece(x + pc.adv, pc), ++p) {
        const int nt = pc.nt;
        ok = mbar_wait(smem_u32(q_full), p & 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tQ = tQb(p & 1);
        // S of the piece's first tile (its buffer was released by the p_full of the
        // tile before, waited for in the previous iteration)
        ok = issue_qk(gt, tQ);
        for (int t = 0; t < nt && ok; ++t) {
          const int xg = gt + t;
          // the next tile's scores overlap this tile's softmax
          if (t + 1 < nt) {
            if (!issue_qk(xg + 1, tQ)) {
              ok = false;
              break;
            }
          }
          if (!mbar_wait(smem_u32(p_full), xg & 1, err)) {
            ok = false;
            break;
          }
          // the first P V of a piece overwrites O: the previous piece's O has been read
          if (t == 0 && p > 0 && !mbar_wait(smem_u32(o_drained), (p - 1) & 1, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* st = stage(xg);
          uint8_t* sP = p_buf(xg);
#pragma unroll
          for (int kb = 0; kb < TK / 64; ++kb) {
            const uint64_t dp = umma_desc_sw128(smem_u32(sP + kb * kBlk));
            const uint64_t dv = umma_desc_sw128(smem_u32(st + L::kKTile + kb * L::kVBox));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tO, dp + 2 * kk, dv + 2 * kk, id_pv, (t | kb | kk) ? 1u : 0u);
          }
          umma_commit(smem_u32(o_full));
          umma_commit(smem_u32(&kv_empty[xg % NST]));
        }
        if (!ok) break;
        umma_commit(smem_u32(pfin));
        gt += nt;
      }
      umma_commit(smem_u32(fin));  // all issued MMAs complete before TMEM is freed
    }
  } else {
    // warps 0-7. Warp w reads TMEM lanes 32*(w%4)..+31; lanes r and r+64 hold the same
    // scores. Thread (lane row lrow, warp w): query row r = lrow % 64, key quarter
    // kq = 2*(w/4) + (lrow >= 64), O row lrow (P_hi V if < 64, P_lo V otherwise) and
    // head-dim half hf = w/4.
    const int hf = warp >> 2;
    const int lrow = (warp & 3) * 32 + lane;
    const int r = lrow & 63;
    const int kq = 2 * hf + (lrow >> 6);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tOw = tO + lane_off + hf * HALF;
    const int srow = r / grp;
    const float scale = rsqrtf((float)HD) * kLog2e;
    // the quarter's keys in P: block (kq*KQ)/64, first 16-byte chunk ((kq*KQ)%64)/8
    const int pblk = (kq * KQ) / 64, pch = ((kq * KQ) % 64) / 8;
    bool ok = true;
    int gt = 0, p = 0;
    // The queries of a piece into TMEM Q buffer `buf` (A operand of S): lane lrow holds
    // query row lrow % 64 (zeros past QN), the hi half in lanes 0..63 and the lo half in
    // lanes 64..127; the warps of head-dim half hf write columns hf*HD/4.. of the lane's
    // HD/2. The buffer was last read by the S of the piece before the previous one, all
    // consumed by then.
    auto write_q = [&](int b, int g, int buf) {
      constexpr int NW = HD / 4;  // 32-bit columns per thread
      uint32_t w[NW];
      if (r < QN) {
        const int s_ = r / grp, hh = r % grp;
        const bf16* src = (const bf16*)a.qs + ((long)(b * a.rows + s_) * a.hq + g * grp + hh) * HD +
                          (lrow >= 64 ? a.qs_lo : 0) + hf * (HD / 2);
#pragma unroll
        for (int i = 0; i < NW; i += 4) {
          const uint4 u = *reinterpret_cast<const uint4*>(src + 2 * i);
          w[i] = u.x;
          w[i + 1] = u.y;
          w[i + 2] = u.z;
          w[i + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = 0u;
      }
#pragma unroll
      for (int c16 = 0; c16 < NW / 16; ++c16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = w[c16 * 16 + i];
        tmem_st16u(tQb(buf) + lane_off + hf * NW + c16 * 16, v);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(smem_u32(q_full));
    };
    Pc pc;
    {
      first_piece(x0, pc);
      write_q(pc.b, pc.g, 0);
    }
    // Every thread runs the same pieces and the same named barriers, whether or not a
    // wait timed out (then the work is skipped), so the barriers always complete.
    for (long x = first_piece(x0, pc); x < x1; x = first_piece(x + pc.adv, pc), ++p) {
      const int b = pc.b, g = pc.g, kt0 = pc.kt0, nt = pc.nt, base = pc.base;
      const int lo = vis_lo(a, base), k_end = base + a.rows;
      const int row_hi = a.causal ? base + srow : base + a.rows - 1;
      float m = -INFINITY, l = 0.f;  // reference max and running sum, log2 units
      // Every iteration runs both named barriers (bar 3: swap posted, bar 4: maxima
      // posted) on every thread, whether or not a wait timed out, so they complete.
      for (int t = 0; t < nt; ++t) {
        const int xg = gt + t;
        if (ok) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[xg & 1]), (xg >> 1) & 1, err));
          tc_fence_after();
        }
        const int kt = (kt0 + t) * TK;
        const int key0 = kt + kq * KQ;
        // interior tiles need no mask: every key of the tile is visible to every row
        const bool interior =
            kt >= lo && kt + TK <= k_end && (!a.causal || kt + TK <= base + 1);
        // The partner thread (lane lrow ^ 64, same warp group) holds the other half
        // (hi or lo) of this row's scores: post its quarter (kq ^ 1) of this lane's half
        // in the tile's P buffer (free until P is written, after barrier 4), take this
        // quarter of the partner's half back.
        float4* xch = (float4*)p_buf(xg);  // [KQ/4][256] float4, thread-minor
        const int tid = threadIdx.x, ptid = (((warp & 4) | ((warp & 3) ^ 2)) << 5) | lane;
        float sv[KQ];
        if (ok) {
          static_assert(KQ == 32, "the swap loads two 16-column blocks per quarter");
          // all four loads in flight before one wait
          uint32_t q0[16], q1[16], o0[16], o1[16];
          const uint32_t ts = tmem + (xg & 1) * TK + lane_off;
          tmem_ld16_raw(ts + (kq ^ 1) * KQ, q0);
          tmem_ld16_raw(ts + (kq ^ 1) * KQ + 16, q1);
          tmem_ld16_raw(ts + kq * KQ, o0);
          tmem_ld16_raw(ts + kq * KQ + 16, o1);
          tmem_wait_ld16(q0);
          reg_fence16(q1);
          reg_fence16(o0);
          reg_fence16(o1);
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            xch[(j / 4) * 256 + tid] =
                make_float4(__uint_as_float(q0[j]), __uint_as_float(q0[j + 1]),
                            __uint_as_float(q0[j + 2]), __uint_as_float(q0[j + 3]));
            xch[(4 + j / 4) * 256 + tid] =
                make_float4(__uint_as_float(q1[j]), __uint_as_float(q1[j + 1]),
                            __uint_as_float(q1[j + 2]), __uint_as_float(q1[j + 3]));
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            sv[j] = __uint_as_float(o0[j]);
            sv[16 + j] = __uint_as_float(o1[j]);
          }
        }
        asm volatile("bar.sync 3, 256;" ::: "memory");
        float* smx = sMax + (xg & 1) * 256;
        if (ok) {
#pragma unroll
          for (int j = 0; j < KQ; j += 4) {
            const float4 o = xch[(j / 4) * 256 + ptid];
            sv[j] = (sv[j] + o.x) * scale;
            sv[j + 1] = (sv[j + 1] + o.y) * scale;
            sv[j + 2] = (sv[j + 2] + o.z) * scale;
            sv[j + 3] = (sv[j + 3] + o.w) * scale;
          }
          if (!interior) {
#pragma unroll
            for (int j = 0; j < KQ; ++j) {
              const int key = key0 + j;
              if (!(key >= lo && key < k_end && key <= row_hi)) sv[j] = -INFINITY;
            }
          }
          float mt = sv[0];
#pragma unroll
          for (int j = 1; j < KQ; ++j) mt = fmaxf(mt, sv[j]);
          smx[kq * 64 + r] = mt;
        }
        asm volatile("bar.sync 4, 256;" ::: "memory");
        if (ok) {
          const float mt = fmaxf(fmaxf(smx[r], smx[64 + r]), fmaxf(smx[128 + r], smx[192 + r]));
          // reference max: set on the first visible scores, moved only past 2^11
          float corr = 1.f;
          if (mt > -INFINITY && (m == -INFINITY || mt > m + 11.f)) {
            corr = (m == -INFINITY) ? 1.f : exp2f(m - mt);
            m = mt;
          }
          // a rescale of O waits for the previous tile's P V (s_full of this tile implies
          // every P V before it has completed, so o_full is at most one phase behind)
          if (t > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_full), (xg - 1) & 1, err));
            if (ok) {
              tc_fence_after();
              tmem_scale(tOw, HALF, corr);
            }
          }
          l *= corr;
          const float mu = (m == -INFINITY) ? 0.f : m;
          uint8_t* pb_ = p_buf(xg) + pblk * kBlk;
#pragma unroll
          for (int cc = 0; cc < KQ / 8; ++cc) {
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
              const float p0 = exp2f(sv[cc * 8 + j] - mu), p1 = exp2f(sv[cc * 8 + j + 1] - mu);
              l += p0 + p1;
              const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
              const __nv_bfloat162 pr =
                  __floats2bfloat162_rn(p0 - __low2float(pb), p1 - __high2float(pb));
              ph[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
              pl[j / 2] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            *(uint4*)(pb_ + sw128(r, pch + cc)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *(uint4*)(pb_ + sw128(r + 64, pch + cc)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          }
          fence_proxy_async();
          tc_fence_before();
        }
        mbar_arrive(smem_u32(p_full));
      }
      // ---- end of the piece ----
      // the next piece's queries into the other Q buffer first, so that its first S is
      // computed while this piece's O is read out and written
      {
        Pc nx;
        if (first_piece(x + pc.adv, nx) < x1) write_q(nx.b, nx.g, (p + 1) & 1);
      }
      // O once its last P V completed
      float O[HALF];
      ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(pfin), p & 1, err));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < HALF / 16; ++cc) {
          float v[16];
          tmem_ld16(tOw + cc * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) O[cc * 16 + j] = v[j];
        }
      }
      sL[kq * 64 + r] = l;
      const long slot = (long)blockIdx.x + (long)b * hkv + g;  // partial of (CTA, segment)
      // the P_lo V rows meet the P_hi V rows in shared memory, one head-dim half at a time
      for (int pass = 0; pass < 2; ++pass) {
        if (hf == pass && lrow >= 64 && ok) {
#pragma unroll
          for (int i = 0; i < HALF; i += 4)
            *(float4*)(xo + r * (HALF + 4) + i) = make_float4(O[i], O[i + 1], O[i + 2], O[i + 3]);
        }
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (hf == pass && lrow < 64 && r < QN && ok) {
          float* po = a.part_o + (slot * QN + r) * HD + hf * HALF;
          const float* lo_row = xo + r * (HALF + 4);
#pragma unroll
          for (int i = 0; i < HALF; i += 4)
            *(float4*)(po + i) = make_float4(O[i] + lo_row[i], O[i + 1] + lo_row[i + 1],
                                             O[i + 2] + lo_row[i + 2], O[i + 3] + lo_row[i + 3]);
          if (hf == 0) {
            constexpr float kLn2 = 0.6931471805599453f;
            a.part_ml[(slot * QN + r) * 2] = m * kLn2;  // natural units for the merge
            a.part_ml[(slot * QN + r) * 2 + 1] = sL[r] + sL[64 + r] + sL[128 + r] + sL[192 + r];
          }
        }
        asm volatile("bar.sync 2, 256;" ::: "memory");
      }
      tc_fence_before();
      mbar_arrive(smem_u32(o_drained));
      gt += nt;
    }
  }
  __syncwarp();
  mbar_wait(smem_u32(fin), 0, err);
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Combine the partials of the persistent kernel: one warp per (row, query head); the
// (CTA, segment) partials of a segment are those of the CTAs whose tile ranges meet it.
template <int DPL>
__global__ void __launch_bounds__(256) k_attn_merge_p(AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + warp;
  if (h >= a.hq) return;
  const int mrow = blockIdx.x, b = mrow / a.rows, s = mrow % a.rows;
  const int grp = a.hq / a.hkv, g = h / grp, hh = h % grp, qi = s * grp + hh, QN = a.rows * grp;
  const int TK = a.ptk, G = a.pgrid;
  int pre = 0, tot = 0;  // units of the sequences before b, of all sequences
  for (int bb = lane; bb < a.B; bb += 32) {
    const int n = seg_units(a, a.base[bb], TK);
    tot += n;
    if (bb < b) pre += n;
  }
  for (int o = 16; o > 0; o >>= 1) {
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
  }
  const long T = (long)a.hkv * tot;
  const int nb = vis_tiles(a, a.base[b], TK);
  // the segment's first and last key-tile units (its overhead units come first)
  const long xf = (long)a.hkv * pre + (long)g * (nb + kPieceCost) + kPieceCost,
             xl = xf + nb - 1;
  // CTA i covers [floor(T i / G), floor(T (i+1) / G)): the owner of x is
  // floor(((x + 1) G - 1) / T)
  const int c0 = (int)(((xf + 1) * G - 1) / T), c1 = (int)(((xl + 1) * G - 1) / T);
  const long seg = (long)b * a.hkv + g;
  // CTAs with an empty range (more CTAs than tiles) wrote nothing
  auto empty = [&](int i) { return T * i / G == T * (i + 1) / G; };
  // online merge over the contributing CTAs, four at a time with all of a batch's loads
  // in flight: running maximum Mx, sum L and output acc, rescaled as the maximum moves
  float Mx = -INFINITY, L = 0.f;
  float acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
  for (int i0 = c0; i0 <= c1; i0 += 4) {
    float mi[4], li[4];
    float2 oi[4][DPL / 2];
    bool vi[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u;
      vi[u] = i <= c1 && !empty(i);
      mi[u] = -INFINITY;
      li[u] = 0.f;
      if (vi[u]) {
        const float* ml = a.part_ml + ((i + seg) * QN + qi) * 2;
        mi[u] = ml[0];
        li[u] = ml[1];
        const float* pc = a.part_o + ((i + seg) * QN + qi) * a.hd + lane * DPL;
#pragma unroll
        for (int j = 0; j < DPL / 2; ++j) oi[u][j] = *reinterpret_cast<const float2*>(pc + 2 * j);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!vi[u] || mi[u] == -INFINITY) continue;  // a partial with no visible key
      const float Mn = fmaxf(Mx, mi[u]);
      const float s0 = __expf(Mx - Mn), s1 = __expf(mi[u] - Mn);  // Mx = -inf: s0 = 0
      L = L * s0 + li[u] * s1;
#pragma unroll
      for (int j = 0; j < DPL / 2; ++j) {
        acc[2 * j] = acc[2 * j] * s0 + oi[u][j].x * s1;
        acc[2 * j + 1] = acc[2 * j + 1] * s0 + oi[u][j].y * s1;
      }
      Mx = Mn;
    }
  }
  const float invL = 1.f / L;
  bf16* out = (bf16*)a.out + (long)mrow * a.hq * a.hd + h * a.hd + lane * DPL;
#pragma unroll
  for (int j = 0; j < DPL; ++j) store_act(out + j, a.out_lo, acc[j] * invL);
}

// tile keys and stage count per head dim
constexpr int kTK128 = kAttnTile, kNST128 = 3;
constexpr int kTK64 = kAttnTile, kNST64 = 4;

int attn_tc_init_attributes() {
  cudaError_t e1 = cudaFuncSetAttribute(k_attn_tc<128, kTK128, kNST128>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Smem<128, kTK128, kNST128>::kBytes);
  cudaError_t e2 = cudaFuncSetAttribute(k_attn_tc<64, kTK64, kNST64>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Smem<64, kTK64, kNST64>::kBytes);
  return (e1 == cudaSuccess && e2 == cudaSuccess) ? 0 : -1;
}

void op_attention_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     const CUtensorMap& tmQh, const CUtensorMap& tmQl, unsigned* err,
                     cudaStream_t st) {
  if (a.B > kAttnMaxB || a.pgrid < 1 || a.ptk != kAttnTile || a.rows < 1 || a.rows > 8)
    return;  // excluded by the caller
  if (a.hd == 128)
    launch_pdl(k_attn_tc<128, kTK128, kNST128>, a.pgrid, 320, Smem<128, kTK128, kNST128>::kBytes,
               st, tmK, tmV, tmQh, tmQl, a, err);
  else
    launch_pdl(k_attn_tc<64, kTK64, kNST64>, a.pgrid, 320, Smem<64, kTK64, kNST64>::kBytes, st,
               tmK, tmV, tmQh, tmQl, a, err);
  dim3 g(a.B * a.rows, (a.hq + 7) / 8);
  if (a.hd == 128)
    launch_pdl(k_attn_merge_p<4>, g, 256, 0, st, a);
  else
    launch_pdl(k_attn_merge_p<2>, g, 256, 0, st, a);
}

}  // namespace dmtp
