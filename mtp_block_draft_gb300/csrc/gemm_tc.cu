// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   out[m, n] (+)= sum_k X[m, k] * W[n, k]        W: [N, K] weights, X: [M, K] tokens
//
// The round multiplies few token rows (M = 8 .. 256) by large weight matrices, so the
// kernel is "swap-AB": 128 weight rows form the MMA's M side (TMEM lanes) and all M
// token rows (padded to MT, a multiple of 16, <= 256) form its N side (TMEM columns).
// CTAs split the weight rows in tiles of 128 (or 256), the token rows in 1..4 parts
// (each part re-reads its weight tile, the second read from L2) and, where that leaves
// SMs idle, the K range (split-K). Each CTA stages its output tile in the idle stage ring
// and adds it into the output with one TMA bulk reduction (element-wise atomic, so the
// split-K parts and the residual add into the residual stream need no other pass);
// outputs a tensor map cannot describe fall back to per-element fp32 atomics. With a K
// split and a partial scratch (and a grid of at most one wave: every CTA resident at
// once), the K parts are summed in a fixed order instead, so the result does not depend
// on which part finishes first: each part writes its tile to the scratch, counts itself
// in at its tile's counter, waits (bounded) for the tile's other parts, and then adds the
// parts 0, 1, ... of one slice of the tile's token rows into `out`.
//
// Pipeline per CTA (256 threads):
//   warp 0 lane 0: TMA producer, weights with L2 evict-first, tokens evict-last;
//   warp 1 lane 0: MMA issuer, 4 x (M=128, N=MT, K=16) per 64-wide k block;
//   warp 2: TMEM allocation; all 8 warps: epilogue (TMEM lane = weight row; warps w and
//   w + 4 read the same lane quarter and take alternate 16-column chunks of the tokens).
// The gate/up GEMM pairs gate and up rows in one CTA and writes silu(g) u as the next
// GEMM's bf16 pair with one TMA store.
// Stages are 64-element (128 B) k slices with 128-byte swizzle.
//
// CTA pairs (a plan option): two CTAs of a cluster, adjacent in x, run one M = 256
// tcgen05.mma.cta_group::2 per k step. Each holds its own 128 (or 256) weight rows and
// one half of the merged [hi; lo] token columns (CTA 0 the hi rows, CTA 1 the
// remainders), so each SM loads and reads half the token bytes; both CTAs' loads complete
// on CTA 0's barriers, CTA 0 issues the MMAs and its commits arrive on both CTAs'
// barriers, and each CTA's epilogue reads its own rows from its own TMEM.
//
// Launched with programmatic serialisation (common.cuh): barrier set-up and the TMEM
// allocation overlap the previous kernel, every load follows the grid dependency.
//
// Split activations: the token operand may come as two bf16 halves, X = X_hi + X_lo
// (X_lo = the rounding remainder of X_hi), stored as 2*MT rows [hi; lo]. Both halves
// are multiplied by the same weight tile (one TMA load of W). Up to 128 token rows the
// halves are one load and one MMA of 2*MT columns, summed in the epilogue; above that
// they are two loads and two MMAs accumulating into the same TMEM columns. Either way
// the activations keep ~16 significant bits while the weights stay bf16 and each
// weight byte is still read once.
//
// The LM heads (GEMM fused with the row argmax) run token-major in head_tc.cu.
//
// Every mbarrier wait is bounded (common.cuh); a timeout sets the error word, the
// producer drains its in-flight copies and the CTA frees its TMEM before returning.
#include <stdio.h>

#include <algorithm>

#include "common.cuh"
#include "ops.h"

namespace dmtp {

static constexpr int kHalfN = 128;  // weight rows per MMA (M) and per accumulator
static constexpr int kBlockK = 64;   // k elements per stage (128 B of bf16)
static constexpr uint32_t kHalfBytes = kHalfN * kBlockK * 2;  // one 128-row weight k slice

struct TcArgs {
  int N, K, M, MT, stages;
  int wide;        // weight halves of 128 rows per CTA (1 or 2), one accumulator each
  int mct;         // token rows per CTA (MT, or MT / 2 with two token halves)
  int split;       // 1: X holds [hi; lo] halves of MT rows each
  int xbox, nx;    // X rows per box, boxes per stage
  int x3d;         // the nx boxes (hi rows, lo rows) come as one 3-D request
  int merged;      // split with hi and lo adjacent in shared memory: one MMA of 2*mct columns
  int acc_cols;    // TMEM columns per accumulator
  float* out;
  int ldo;
  int tma_out;     // EPI 0: add the tile into out with TMA bulk reductions (tmO)
  bf16* h;         // EPI 2: SwiGLU output [M][F] (hi), remainder at h + h_lo
  long h_lo;
  int F;           // EPI 2: gate rows 0..F-1, up rows F..2F-1 of W
  unsigned* err;
  float* part;     // deterministic split-K: per-CTA partial tiles [grid][WIDE][mct][128]
  int* tile_cnt;   // ... and a counter per output tile, zero between launches
  long stage_bytes;  // bytes of the stage ring (the parts' slices are gathered there)
};

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// memory into this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16 accumulator columns of this warp's lanes at taddr, plus (merged) the lo columns
// mct further: both loads in flight before one wait.
template <bool MERGED>
__device__ __forceinline__ void acc_ld16(uint32_t taddr, int mct, float (&v)[16]) {
  uint32_t rv[16], rw[16];
  tmem_ld16_raw(taddr, rv);
  if (MERGED) tmem_ld16_raw(taddr + mct, rw);
  tmem_wait_ld16(rv);
  if (MERGED) reg_fence16(rw);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = MERGED ? __uint_as_float(rv[j]) + __uint_as_float(rw[j]) : __uint_as_float(rv[j]);
}

__host__ __device__ inline uint32_t tmem_cols_for(int cols) {
  uint32_t c = 32;
  while (c < (uint32_t)cols) c <<= 1;
  return c;
}

// EPI 0: atomic add into out, 2: SwiGLU (WIDE = 2, no K
// split: weight half 0 = gate rows n0.., half 1 = the matching up rows F + n0.., and the
// epilogue writes silu(g) * u as the next GEMM's bf16 pair). WIDE, NMMA (MMAs per k
// step and weight half) and MERGED are compile-time copies of a.wide, (merged ? 1 : nx)
// and a.merged, so that the issue loop and the epilogue have no runtime trip counts.
// One GEMM pass of a CTA over its tile (bx, by, bz) of a (gx, *, gz) tile grid: TMA
// producer, MMA issuer and epilogue, on shared memory (stage ring at smem) and barriers
// already initialised, with `tmem` allocated. grid_dep: the pass reads the previous
// launch's outputs, so every thread first waits for the grid dependency (programmatic
// launch).
struct GemmBars {
  uint64_t *full, *empty, *accum, *sumbar;
};

template <int EPI, int WIDE, int NMMA, bool MERGED, bool PAIR>
__device__ __forceinline__ void gemm_pass(const CUtensorMap* tmW, const CUtensorMap* tmX,
                                          const CUtensorMap* tmO, const TcArgs& a,
                                          uint8_t* smem, GemmBars bars, uint32_t tmem,
                                          uint32_t rank, int bx, int by, int bz, int gx, int gz,
                                          bool grid_dep) {
  const int S = a.stages;
  const uint32_t wbytes = (uint32_t)WIDE * kHalfBytes;
  const uint32_t xbytes = (uint32_t)a.xbox * a.nx * kBlockK * 2;
  uint8_t* sW = smem;
  uint8_t* sX = smem + S * wbytes;
  uint64_t* full = bars.full;
  uint64_t* empty = bars.empty;
  uint64_t* accum = bars.accum;
  uint64_t* sumbar = bars.sumbar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // epilogue: TMEM lane quarter of this warp, and its first 16-column token chunk
  const int wq = warp & 3, c_first = (warp >> 2) * 16;
  // grid: (token halves, weight tiles, K splits); CTAs sharing a weight tile are
  // adjacent in launch order, so its second read comes from L2
  // (a pair's two CTAs are adjacent in x, the cluster dimension: x = 2 part + rank, and
  // y counts pairs of weight tiles)
  const int part = PAIR ? (bx >> 1) : bx;
  const int wtile = PAIR ? (by * 2 + (int)rank) : by;
  const int mrow0 = part * a.mct;
  const int n0 = wtile * kHalfN * (EPI == 2 ? 1 : WIDE);
  const int nkb = a.K / kBlockK;
  const int kb0 = (int)((long)bz * nkb / gz);
  const int kb1 = (int)((long)(bz + 1) * nkb / gz);
  if (grid_dep) pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pw = policy_evict_first(), px = policy_evict_last();
    // a pair's loads (this CTA's weight rows and its half of the token columns: the hi
    // rows in CTA 0, the remainder rows in CTA 1) complete on CTA 0's full barrier
    const uint32_t stage_bytes = (PAIR ? 2u : 1u) * (wbytes + xbytes);
    auto full_bar = [&](int s) {
      return PAIR ? smem_in_rank(smem_u32(&full[s]), 0) : smem_u32(&full[s]);
    };
    auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y, int s, uint64_t pol) {
      if (PAIR)
        tma_load_2d_pair(dst, tm, x, y, full_bar(s), pol);
      else
        tma_load_2d(dst, tm, x, y, smem_u32(&full[s]), pol);
    };
    auto load_w = [&](int s, int kb) {
      if (EPI == 2) {  // gate rows n0.. and up rows F + n0.., one 128-row box each
        load(smem_u32(sW + s * wbytes), tmW, kb * kBlockK, n0, s, pw);
        load(smem_u32(sW + s * wbytes + kHalfBytes), tmW, kb * kBlockK, a.F + n0, s, pw);
      } else {
        load(smem_u32(sW + s * wbytes), tmW, kb * kBlockK, n0, s, pw);
      }
    };
    int issued = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++issued) {
      const int s = issued % S;
      const uint32_t ph = (issued / S) & 1;
      if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, a.err)) break;
      if (rank == 0) mbar_expect_tx(smem_u32(&full[s]), stage_bytes);
      load_w(s, kb);
      if (PAIR) {
        load(smem_u32(sX + s * xbytes), tmX, kb * kBlockK, (int)rank * a.MT + mrow0, s, px);
        continue;
      }
      // one box of [hi; lo] rows, or hi rows then (split) remainder rows: one 3-D
      // request over both halves, or a request per half
      if (a.x3d)
        tma_load_3d(smem_u32(sX + s * xbytes), tmX, kb * kBlockK, mrow0, 0, smem_u32(&full[s]),
                    px);
      else
        for (int j = 0; j < a.nx; ++j)
          tma_load_2d(smem_u32(sX + s * xbytes + j * a.xbox * kBlockK * 2), tmX, kb * kBlockK,
                      j * a.MT + mrow0, smem_u32(&full[s]), px);
    }
    // drain: every stage's last issued load has landed before the CTA may exit (a pair's
    // loads all complete on CTA 0's barriers, and CTA 1 exits after CTA 0 has drained)
    if (rank == 0)
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
        mbar_wait(smem_u32(&full[j % S]), (j / S) & 1, a.err);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer ----------------
    // merged: N = 2*mct over [hi; lo] (lo accumulates in columns mct..); otherwise the
    // nx token loads each get an MMA of N = mct into the same accumulator columns
    // a pair: M = 256 (128 weight rows per CTA), N = 2 mct over [hi (CTA 0); lo (CTA 1)]
    const uint32_t idesc = umma_idesc_bf16(PAIR ? 2 * kHalfN : kHalfN, MERGED ? 2 * a.mct : a.mct);
    int it = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      if (!mbar_wait(smem_u32(&full[s]), ph, a.err)) break;
      tc_fence_after();
      uint64_t dw[WIDE], dx[NMMA];
#pragma unroll
      for (int h = 0; h < WIDE; ++h)
        dw[h] = umma_desc_sw128(smem_u32(sW + s * wbytes + h * kHalfBytes));
#pragma unroll
      for (int j = 0; j < NMMA; ++j)
        dx[j] = umma_desc_sw128(smem_u32(sX + s * xbytes + j * a.mct * kBlockK * 2));
#pragma unroll
      for (int k = 0; k < kBlockK / 16; ++k)  // +32 B per K=16 step inside the swizzle atom
#pragma unroll
        for (int h = 0; h < WIDE; ++h)
#pragma unroll
          for (int j = 0; j < NMMA; ++j) {
            const uint32_t acc = (kb > kb0 || k > 0 || j > 0) ? 1u : 0u;
            if (PAIR)
              umma_bf16_pair(tmem + h * a.acc_cols, dw[h] + 2 * k, dx[j] + 2 * k, idesc, acc);
            else
              umma_bf16(tmem + h * a.acc_cols, dw[h] + 2 * k, dx[j] + 2 * k, idesc, acc);
          }
      if (PAIR)
        umma_commit_pair(smem_u32(&empty[s]));
      else
        umma_commit(smem_u32(&empty[s]));
    }
    // always: the epilogues wait on it
    if (PAIR)
      umma_commit_pair(smem_u32(accum));
    else
      umma_commit(smem_u32(accum));
  }
  __syncwarp();

  // ---------------- epilogue ----------------
  bool ok = mbar_wait(smem_u32(accum), 0, a.err);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  if (EPI == 0 && a.part && gz > 1) {
    // ---- K parts summed in a fixed order ----
    const int S = gz, z = bz;
    const long tile = (long)by * gx + bx;
    const long tile_elems = (long)WIDE * kHalfN * a.mct;
    // this part's tile, [half][token][128 rows] (a warp's stores are 128 contiguous bytes)
    float* mine = a.part + (tile * S + z) * tile_elems;
    if (ok) {
#pragma unroll
      for (int h = 0; h < WIDE; ++h) {
        const uint32_t tbase = tmem + h * a.acc_cols + ((uint32_t)(wq * 32) << 16);
        for (int c = c_first; c < a.mct; c += 32) {
          float v[16];
          acc_ld16<MERGED>(tbase + c, a.mct, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            mine[((long)h * a.mct + c + j) * kHalfN + wq * 32 + lane] = v[j];
        }
      }
    }
    __threadfence();
    __syncthreads();
    __shared__ int s_go;
    if (threadIdx.x == 0) {
      int* cnt = a.tile_cnt + tile;
      atomicAdd(cnt, 1);
      bool arrived = true;
      const uint64_t t0 = global_timer();
      while (ld_acquire(cnt) < S) {  // every part of the tile is resident (one wave)
        if (global_timer() - t0 > DMTP_WAIT_NS) {
          set_err(a.err, DMTP_ERR_TIMEOUT);
          arrived = false;
          break;
        }
      }
      s_go = arrived && ok;
    }
    __syncthreads();
    // this part sums token rows [t0, t1) of the tile over the parts 0..S-1, in order; the
    // parts' slices of those rows (one contiguous run per part and weight half) are
    // gathered into the idle stage ring by bulk copies, all in flight at once
    const int t0 = (int)((long)a.mct * z / S), t1 = (int)((long)a.mct * (z + 1) / S);
    const int nt = t1 - t0, per_tok = WIDE * kHalfN;
    const uint32_t slice_b = (uint32_t)nt * kHalfN * 4;
    const float* base = a.part + tile * S * tile_elems;
    float* sl = reinterpret_cast<float*>(smem);
    bool got = s_go && nt > 0 && (long)S * WIDE * slice_b <= a.stage_bytes;
    if (got) {
      if (threadIdx.x == 0) {
        // the other parts' tiles were written by the generic proxy: order them before
        // these async-proxy reads
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_expect_tx(smem_u32(sumbar), (uint32_t)(S * WIDE) * slice_b);
        for (int q = 0; q < S; ++q)
#pragma unroll
          for (int h = 0; h < WIDE; ++h)
            bulk_g2s(smem_u32(sl + (size_t)(q * WIDE + h) * nt * kHalfN),
                     base + q * tile_elems + ((long)h * a.mct + t0) * kHalfN, slice_b,
                     smem_u32(sumbar));
      }
      got = __syncthreads_and(mbar_wait(smem_u32(sumbar), 0, a.err));
    }
    if (got) {
      for (int idx = threadIdx.x; idx < nt * per_tok; idx += blockDim.x) {
        const int tok = idx / per_tok, f = idx % per_tok;
        const int h = f / kHalfN, r = f % kHalfN;
        const int m = mrow0 + t0 + tok, n = n0 + h * kHalfN + r;
        if (m >= a.M || n >= a.N) continue;
        float acc = a.out[(long)m * a.ldo + n];
        for (int q = 0; q < S; ++q) acc += sl[((size_t)(q * WIDE + h) * nt + tok) * kHalfN + r];
        a.out[(long)m * a.ldo + n] = acc;
      }
    } else if (s_go) {  // the slices do not fit the ring: read them from L2 directly
      __threadfence();
      for (int idx = threadIdx.x; idx < nt * per_tok; idx += blockDim.x) {
        const int tok = t0 + idx / per_tok, f = idx % per_tok;
        const int h = f / kHalfN, r = f % kHalfN;
        const int m = mrow0 + tok, n = n0 + h * kHalfN + r;
        if (m >= a.M || n >= a.N) continue;
        float acc = a.out[(long)m * a.ldo + n];
        const float* pp = base + ((long)h * a.mct + tok) * kHalfN + r;
        for (int q = 0; q < S; ++q) acc += __ldcg(pp + q * tile_elems);
        a.out[(long)m * a.ldo + n] = acc;
      }
    }
    __syncthreads();
    // the last part out resets the counter for the next launch
    if (threadIdx.x == 0 && atomicAdd(a.tile_cnt + tile, 1) == 2 * S - 1) a.tile_cnt[tile] = 0;
  } else if (EPI == 0 && a.tma_out) {
    // Each weight half's [mct tokens][128 rows] fp32 tile is staged in the idle stage
    // buffers (rows = TMEM lanes: a warp's stores are contiguous) and added into `out`
    // by one TMA bulk reduction, in place of mct scattered atomics per thread. Where the
    // ring holds both halves' tiles, both reductions are in flight at once.
    const bool okb = __syncthreads_and(ok);
    const bool both = a.stage_bytes >= (long)WIDE * a.mct * kHalfN * 4;
#pragma unroll
    for (int h = 0; h < WIDE; ++h) {
      if (h > 0 && !both) {  // the previous reduction has read the staging tile
        if (threadIdx.x == 0) bulk_wait_read0();
        __syncthreads();
      }
      float* stg = reinterpret_cast<float*>(smem) + (both ? (long)h * a.mct * kHalfN : 0);
      if (okb) {
        const uint32_t tbase = tmem + h * a.acc_cols + ((uint32_t)(wq * 32) << 16);
        for (int c = c_first; c < a.mct; c += 32) {
          float v[16];
          acc_ld16<MERGED>(tbase + c, a.mct, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) stg[(c + j) * kHalfN + wq * 32 + lane] = v[j];
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0 && okb && n0 + h * kHalfN < a.N && mrow0 < a.M) {
        tma_reduce_add_2d(tmO, n0 + h * kHalfN, mrow0, smem_u32(stg));
        bulk_commit();
      }
    }
    if (threadIdx.x == 0) bulk_wait_read0();  // the staging tile is read before exit
  } else if (EPI == 0) {
    if (ok) {
#pragma unroll
      for (int h = 0; h < WIDE; ++h) {
        const int n = n0 + h * kHalfN + wq * 32 + lane;
        const uint32_t tbase = tmem + h * a.acc_cols + ((uint32_t)(wq * 32) << 16);
        for (int c = c_first; c < a.mct; c += 32) {
          float v[16];
          acc_ld16<MERGED>(tbase + c, a.mct, v);
          if (n < a.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int m = mrow0 + c + j;
              if (m < a.M) atomicAdd(&a.out[(long)m * a.ldo + n], v[j]);
            }
          }
        }
      }
    }
  } else if (EPI == 2 && a.tma_out) {
    // silu(g) u as the down GEMM's bf16 pair, staged as [hi | lo][mct tokens][128
    // features] in the idle stage ring and written by one 3-D TMA store
    const bool okb = __syncthreads_and(ok);
    bf16* sh = reinterpret_cast<bf16*>(smem);
    const int row = wq * 32 + lane;
    if (okb) {
      const uint32_t tg = tmem + ((uint32_t)(wq * 32) << 16);
      const uint32_t tu = tg + a.acc_cols;
      for (int c = c_first; c < a.mct; c += 32) {
        uint32_t rg[16], ru[16], rgl[16], rul[16];
        tmem_ld16_raw(tg + c, rg);
        tmem_ld16_raw(tu + c, ru);
        if (MERGED) {
          tmem_ld16_raw(tg + a.mct + c, rgl);
          tmem_ld16_raw(tu + a.mct + c, rul);
        }
        tmem_wait_ld16(rg);
        reg_fence16(ru);
        if (MERGED) {
          reg_fence16(rgl);
          reg_fence16(rul);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float g = __uint_as_float(rg[j]), u = __uint_as_float(ru[j]);
          if (MERGED) {
            g += __uint_as_float(rgl[j]);
            u += __uint_as_float(rul[j]);
          }
          // silu(g) u = g sigmoid(g) u
          const float v = __fdividef(g, 1.f + __expf(-g)) * u;
          const bf16 hi = __float2bfloat16_rn(v);
          sh[(c + j) * kHalfN + row] = hi;
          sh[(a.mct + c + j) * kHalfN + row] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0 && okb && n0 < a.F && mrow0 < a.M) {
      tma_store_3d(tmO, n0, mrow0, 0, smem_u32(sh));
      bulk_commit();
      bulk_wait_read0();
    }
  } else if (EPI == 2) {
    if (ok) {
      const int n = n0 + wq * 32 + lane;  // feature
      const uint32_t tg = tmem + ((uint32_t)(wq * 32) << 16);
      const uint32_t tu = tg + a.acc_cols;
      for (int c = c_first; c < a.mct; c += 32) {
        uint32_t rg[16], ru[16], rgl[16], rul[16];
        tmem_ld16_raw(tg + c, rg);
        tmem_ld16_raw(tu + c, ru);
        if (MERGED) {
          tmem_ld16_raw(tg + a.mct + c, rgl);
          tmem_ld16_raw(tu + a.mct + c, rul);
        }
        tmem_wait_ld16(rg);
        reg_fence16(ru);
        if (MERGED) {
          reg_fence16(rgl);
          reg_fence16(rul);
        }
        if (n < a.F) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = mrow0 + c + j;
            float g = __uint_as_float(rg[j]), u = __uint_as_float(ru[j]);
            if (MERGED) {
              g += __uint_as_float(rgl[j]);
              u += __uint_as_float(rul[j]);
            }
            // silu(g) u = g sigmoid(g) u
            if (m < a.M)
              store_act(a.h + (long)m * a.F + n, a.h_lo, __fdividef(g, 1.f + __expf(-g)) * u);
          }
        }
      }
    }
  }
}

template <int EPI, int WIDE, int NMMA, bool MERGED, bool PAIR>
__global__ void __launch_bounds__(256, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmO, TcArgs a) {
  static_assert(!PAIR || (MERGED && NMMA == 1), "CTA pairs take the merged [hi; lo] operand");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // 1024-B aligned tiles
  const int S = a.stages;
  const uint32_t wbytes = (uint32_t)WIDE * kHalfBytes;
  const uint32_t xbytes = (uint32_t)a.xbox * a.nx * kBlockK * 2;
  uint64_t* full = (uint64_t*)(smem + S * (wbytes + xbytes));
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  uint64_t* sumbar = accum + 2;  // the K parts' slices landed (fixed-order sum)
  const int warp = threadIdx.x >> 5;
  // CTA pair: rank 0 issues the MMAs of both; its full barriers count both CTAs' loads
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const uint32_t ncols = tmem_cols_for(WIDE * a.acc_cols);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    mbar_init(smem_u32(sumbar), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) {
    if (PAIR)
      tmem_alloc_pair(smem_u32(tmem_slot), ncols);
    else
      tmem_alloc(smem_u32(tmem_slot), ncols);
  }
  tc_fence_before();
  __syncthreads();
  // a pair's barriers are initialised before either CTA signals the other's
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next launch may begin (this CTA holds its TMEM)
  pdl_trigger();
  gemm_pass<EPI, WIDE, NMMA, MERGED, PAIR>(&tmW, &tmX, &tmO, a, smem,
                                           GemmBars{full, empty, accum, sumbar}, tmem, rank,
                                           blockIdx.x, blockIdx.y, blockIdx.z, gridDim.x,
                                           gridDim.z, true);
  tc_fence_before();
  __syncthreads();
  // neither CTA of a pair frees its TMEM or exits while the other may still signal its
  // barriers or read its shared memory
  if (PAIR) cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem, ncols);
    else
      tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t get_encode() {
  static PFN_encodeTiled_t fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_encodeTiled_t)p;
  }
  return fn;
}

// [rows, cols] row-major bf16, box {64, box_rows}, 128-byte swizzle, zero fill.
int tc_make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || (cols * 2) % 16) return -2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBlockK, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

// [rows, cols] fp32 with a row pitch of ld elements, box {box_cols, box_rows}, no swizzle
// (the plain row-major layout of a staged output tile).
int tc_make_tmap_f32(CUtensorMap* tm, void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_cols, uint32_t box_rows) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || (ld * 4) % 16 || box_cols * 4 % 16) return -2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

// 3-D bf16 view [d2][d1][d0] with byte strides s1, s2 and an unswizzled box {b0, b1, b2}
// (a plain row-major staging layout; used for output tiles).
int tc_make_tmap3s_box(CUtensorMap* tm, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || s1 % 16 || s2 % 16 || (b0 * 2) % 16) return -2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

// [rows, cols] row-major bytes (E4M3), box {128, box_rows}, 128-byte swizzle: the same
// shared-memory layout as a bf16 box of 64 columns.
int tc_make_tmap_u8(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || cols % 16) return -2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

int tc_make_tmap3(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint32_t b1, uint32_t b2) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || (d0 * 2) % 16) return -2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {(cuuint32_t)kBlockK, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

int tc_make_tmap3s(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b1, uint32_t b2) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return -1;
  if (((uintptr_t)base & 15) || (d0 * 2) % 16 || s1 % 16 || s2 % 16) return -2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {(cuuint32_t)kBlockK, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

static size_t smem_bytes(int wide, int xrows, int stages) {
  size_t b = 1024 + (size_t)stages * (wide * kHalfBytes + (size_t)xrows * kBlockK * 2);
  b += (2 * stages + 3) * 8;
  return b;
}

static constexpr size_t kSmemBudget = 200 * 1024;

int tc_mt(int M) { return std::max(16, (M + 15) / 16 * 16); }

int tc_plan_shape(TcPlan* p, const void* W, int N, int K, const void* X, int M, int nsm,
                  bool split, int wide, int msplit, int splits, int pair) {
  if (M < 1 || M > 256 || K % kBlockK || N < 1 || (wide != 1 && wide != 2) || msplit < 1 ||
      msplit > 4 || (pair && !split))
    return -10;
  p->N = N;
  p->K = K;
  p->M = M;
  p->swiglu = 0;
  p->F = 0;
  p->MT = tc_mt(M);
  p->split = split ? 1 : 0;
  p->wide = wide;
  p->msplit = msplit;
  // token parts of mct rows (a multiple of 16); the last part may be short: its rows past
  // MT read as zeros (tensor-map bounds) and are not written
  p->mct = (p->MT / msplit + 15) / 16 * 16;
  if (p->mct * msplit < p->MT) p->mct += 16;
  if (p->mct * (msplit - 1) >= p->MT) return -10;  // every part has rows
  if (split && msplit == 1 && 2 * p->MT <= 256) {  // [hi; lo] rows adjacent: one load
    p->xbox = 2 * p->MT;
    p->nx = 1;
  } else {
    p->xbox = p->mct;
    p->nx = split ? 2 : 1;
  }
  p->merged = split && 2 * p->mct <= 256;
  p->pair = pair ? 1 : 0;
  if (pair) {  // each CTA of a pair loads one half of its token part: one box of mct rows
    if (!p->merged) return -10;
    p->xbox = p->mct;
    p->nx = 1;
  }
  p->acc_cols = p->merged ? 2 * p->mct : p->mct;
  if (wide * p->acc_cols > 512) return -10;
  const int xrows = p->xbox * p->nx;
  int st = 8;
  while (st > 2 && smem_bytes(wide, xrows, st) > kSmemBudget) --st;
  p->stages = st;
  p->smem = smem_bytes(wide, xrows, st);
  p->stage_area = (size_t)st * (wide * kHalfBytes + (size_t)xrows * kBlockK * 2);
  if (p->smem > kSmemBudget) return -10;
  int ytiles = (N + kHalfN * wide - 1) / (kHalfN * wide);
  if (pair) ytiles += ytiles & 1;  // whole pairs (a last odd tile reads zeros, writes nothing)
  const int tiles = ytiles * msplit;
  const int nkb = K / kBlockK;
  int best = splits > 0 ? std::min(splits, nkb) : 1;
  if (splits <= 0) {
    // minimise waves(tiles * s) * (k blocks per CTA + fixed cost of ~3 k blocks)
    double best_cost = 1e30;
    for (int s = 1; s <= std::min(nkb, 32); ++s) {
      const int waves = (tiles * s + nsm - 1) / nsm;
      const double cost = waves * ((double)nkb / s + 3.0);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = s;
      }
    }
  }
  // a K split stays within one wave of CTAs (its parts are summed in a fixed order by
  // parts that must all be resident at once)
  if (best > 1) best = std::max(1, std::min(best, nsm / tiles));
  p->splits = best;
  p->nsm = nsm;
  p->part = nullptr;
  p->tile_cnt = nullptr;
  p->part_floats = 0;
  int r = tc_make_tmap(&p->tmW, W, (uint64_t)N, (uint64_t)K, (uint32_t)(kHalfN * wide));
  if (r) return r;
  // split: the tensor spans both halves (rows >= M of each half are ignored columns);
  // two boxes per stage become one 3-D request over {k, row, half}
  p->x3d = split && p->nx == 2;
  if (pair)  // the [hi; lo] rows as one 2-D tensor: CTA r of a pair reads rows r MT + ..
    return tc_make_tmap(&p->tmX, X, (uint64_t)2 * p->MT, (uint64_t)K, (uint32_t)p->mct);
  if (p->x3d)
    return tc_make_tmap3s(&p->tmX, X, (uint64_t)K, (uint64_t)p->MT, 2, (uint64_t)K * 2,
                          (uint64_t)p->MT * K * 2, (uint32_t)p->xbox, 2);
  r = tc_make_tmap(&p->tmX, X, (uint64_t)(split ? 2 * p->MT : M), (uint64_t)K,
                   (uint32_t)p->xbox);
  return r;
}

int tc_plan_swiglu(TcPlan* p, const void* W, int F, int K, const void* X, int M, int nsm,
                   bool split, int msplit, int pair) {
  int r = tc_plan_shape(p, W, 2 * F, K, X, M, nsm, split, 2, msplit, 1, pair);
  if (r) return r;
  p->swiglu = 1;
  p->F = F;
  // one 128-row box per weight half (gate and up rows are F apart)
  return tc_make_tmap(&p->tmW, W, (uint64_t)2 * F, (uint64_t)K, (uint32_t)kHalfN);
}

int tc_plan(TcPlan* p, const void* W, int N, int K, const void* X, int M, int nsm, bool split) {
  return tc_plan_shape(p, W, N, K, X, M, nsm, split, 1, 1, 0);
}

// The kernel instantiation for a plan: (wide, MMAs per k step, merged).
template <int EPI>
static void (*kernel_for(const TcPlan& p))(const CUtensorMap, const CUtensorMap,
                                             const CUtensorMap, TcArgs) {
  const int nmma = p.merged ? 1 : p.nx;
  if (EPI == 2) {
    if (p.pair) return k_gemm_tc<2, 2, 1, true, true>;
    if (p.merged) return k_gemm_tc<2, 2, 1, true, false>;
    return nmma == 1 ? k_gemm_tc<2, 2, 1, false, false> : k_gemm_tc<2, 2, 2, false, false>;
  }
  if (p.wide == 1) {
    if (p.pair) return k_gemm_tc<EPI, 1, 1, true, true>;
    if (p.merged) return k_gemm_tc<EPI, 1, 1, true, false>;
    return nmma == 1 ? k_gemm_tc<EPI, 1, 1, false, false> : k_gemm_tc<EPI, 1, 2, false, false>;
  }
  if (p.pair) return k_gemm_tc<EPI, 2, 1, true, true>;
  if (p.merged) return k_gemm_tc<EPI, 2, 1, true, false>;
  return nmma == 1 ? k_gemm_tc<EPI, 2, 1, false, false> : k_gemm_tc<EPI, 2, 2, false, false>;
}

int tc_init_attributes() {
  const int bytes = (int)(kSmemBudget + 8 * 1024);
  void (*ks[])(const CUtensorMap, const CUtensorMap, const CUtensorMap, TcArgs) = {
      k_gemm_tc<0, 1, 1, true, false>,  k_gemm_tc<0, 1, 1, false, false>,
      k_gemm_tc<0, 1, 2, false, false>, k_gemm_tc<0, 2, 1, true, false>,
      k_gemm_tc<0, 2, 1, false, false>, k_gemm_tc<0, 2, 2, false, false>,
      k_gemm_tc<2, 2, 1, true, false>,  k_gemm_tc<2, 2, 1, false, false>,
      k_gemm_tc<2, 2, 2, false, false>, k_gemm_tc<0, 1, 1, true, true>,
      k_gemm_tc<0, 2, 1, true, true>,   k_gemm_tc<2, 2, 1, true, true>};
  for (auto k : ks)
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
      return -1;
  return 0;
}

// Kernel arguments, output tensor map and grid of the SwiGLU (gate/up) GEMM.
static void swiglu_args(const TcPlan& p, void* h, long h_lo, unsigned* err, TcArgs* a,
                        CUtensorMap* tmO, dim3* grid) {
  // the TMA-store epilogue when the [hi | lo] tile fits the stage buffers
  *tmO = p.tmW;
  int tma = 0;
  if (p.stage_area >= (size_t)p.mct * kHalfN * 4 && h_lo > 0 && aligned_to(h, 16) &&
      (p.F * 2) % 16 == 0 && (h_lo * 2) % 16 == 0)
    tma = tc_make_tmap3s_box(tmO, h, (uint64_t)p.F, (uint64_t)p.M, 2, (uint64_t)p.F * 2,
                             (uint64_t)h_lo * 2, kHalfN, (uint32_t)p.mct, 2) == 0;
  *a = TcArgs{p.N,     p.K,     p.M,     p.MT,     p.stages, p.wide, p.mct,
              p.split, p.xbox,  p.nx,    p.x3d,    p.merged, p.acc_cols, nullptr,
              0,       tma,     (bf16*)h, h_lo,    p.F,      err,      nullptr, nullptr, 0};
  const int gy = (p.F + kHalfN - 1) / kHalfN;
  // CTA pairs: clusters of two along x (x = 2 token part + rank, y = pairs of weight tiles)
  *grid = p.pair ? dim3(2 * p.msplit, (gy + 1) / 2, 1) : dim3(p.msplit, gy, 1);
}

// The same for a GEMM adding into an fp32 output (part: the fixed-order K-part sums).
static void acc_args(const TcPlan& p, float* out, int ldo, unsigned* err, TcArgs* a,
                     CUtensorMap* tmO, dim3* grid) {
  // the TMA bulk-reduction epilogue when a weight half's tile fits the stage buffers and
  // out can be described by a tensor map; else per-element atomics
  *tmO = p.tmW;
  int tma = 0;
  if (p.stage_area >= (size_t)p.mct * kHalfN * 4 && ldo % 4 == 0 && aligned_to(out, 16))
    tma = tc_make_tmap_f32(tmO, out, (uint64_t)p.M, (uint64_t)p.N, (uint64_t)ldo, kHalfN,
                           (uint32_t)p.mct) == 0;
  const int gy = (p.N + kHalfN * p.wide - 1) / (kHalfN * p.wide);
  *grid = p.pair ? dim3(2 * p.msplit, (gy + 1) / 2, p.splits) : dim3(p.msplit, gy, p.splits);
  // the fixed-order K-part sum needs every CTA resident at once: one wave, one CTA per SM
  const long ctas = (long)grid->x * grid->y * grid->z;
  const bool det = p.part && p.tile_cnt && p.splits > 1 && ctas <= p.nsm &&
                   (size_t)ctas * p.wide * kHalfN * p.mct <= p.part_floats;
  *a = TcArgs{p.N,     p.K,     p.M,     p.MT,     p.stages, p.wide, p.mct,
              p.split, p.xbox,  p.nx,    p.x3d,    p.merged, p.acc_cols, out,
              ldo,     tma,     nullptr, 0,        0,        err,
              det ? p.part : nullptr, det ? p.tile_cnt : nullptr, (long)p.stage_area};
}

void op_gemm_tc_swiglu(const TcPlan& p, void* h, long h_lo, unsigned* err, cudaStream_t st) {
  TcArgs a;
  CUtensorMap tmO;
  dim3 grid;
  swiglu_args(p, h, h_lo, err, &a, &tmO, &grid);
  launch_pdl_cluster(kernel_for<2>(p), grid, 256, p.smem, st, dim3(p.pair ? 2 : 1, 1, 1), p.tmW,
                     p.tmX, tmO, a);
}

void op_gemm_tc_acc(const TcPlan& p, float* out, int ldo, unsigned* err, cudaStream_t st) {
  TcArgs a;
  CUtensorMap tmO;
  dim3 grid;
  acc_args(p, out, ldo, err, &a, &tmO, &grid);
  launch_pdl_cluster(kernel_for<0>(p), grid, 256, p.smem, st, dim3(p.pair ? 2 : 1, 1, 1), p.tmW,
                     p.tmX, tmO, a);
}

}  // namespace dmtp
