// Split-K decode attention on the 5th-generation tensor cores (sm_103a).
//
// One CTA per (512-key chunk, kv head, sequence) serves all 8 rows x the GQA group of
// query heads that share the kv head (QN <= 64 queries), so each cached K/V byte is read
// from HBM once per sequence and layer. Keys stream through shared memory in tiles of
// 128 (TMA, 128-byte swizzle, two stages); per tile:
//   S = Q K^T  : tcgen05 M=128, N=128 keys, K = 2*hd. The fp32 queries enter as a bf16
//                pair [Q_hi | Q_lo] along K against [K | K], so S carries the fp32
//                queries' precision; rows 0..QN-1 of the 128-row operand are queries.
//   softmax    : warps 0,1,4,5 (TMEM lanes 0..63, one query row per warp pair, each
//                thread half of the tile's keys) read S, apply the
//                visibility mask (causal rows / anchor window / chunk bounds), update the
//                running max m and sum l, and write P as a bf16 pair: P_hi in operand
//                rows 0..63, P_lo (the rounding remainder) in rows 64..127;
//   O_t = P V  : tcgen05 M=128, N=hd, K=128 keys, B = the transposed V tile (K-major);
//                TMEM lanes 0..63 hold P_hi V, lanes 64..127 P_lo V. Warps 0,1,4,5 and
//                2,3,6,7 add them (half the head dims per thread) into fp32 registers
//                rescaled by exp(m_old - m_new); the two are summed once at the end.
// S is double-buffered in TMEM, so the next tile's Q K^T overlaps this tile's softmax.
// Warp 8 lane 0 issues the TMA loads, warp 9 lane 0 the MMAs. The partial (m, l, O) of
// each chunk goes to global memory and a merge kernel combines the chunks (attention.cu).
//
// Visibility follows the DMTP blog §6.2: target and MTP rows are causal over their
// cache; the drafter sees its anchor-relative window and the whole 8-slot block.
// Every mbarrier wait is bounded; on a timeout the error word is set, in-flight copies
// and MMAs are drained and TMEM is freed before the CTA returns.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

namespace {

constexpr int kTileKeys = 128;
constexpr int kBlk = 128 * 128;  // one 128-row x 64-element bf16 block (16 KB)

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
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int HD>
struct Smem {
  static constexpr int kQBlocks = 2 * HD / 64;            // [hi | lo] along K
  static constexpr int kKBlocks = HD / 64;                // K tile: 128 keys x HD
  static constexpr uint32_t kQ = kQBlocks * kBlk;
  static constexpr uint32_t kKTile = kKBlocks * kBlk;
  static constexpr uint32_t kVTile = 2 * HD * 128;        // V^T tile: HD rows x 128 keys
  static constexpr uint32_t kStage = kKTile + kVTile;
  static constexpr uint32_t kP = 2 * kBlk;                // 128 rows x 128 keys
  static constexpr uint32_t kBytes = 1024 + kQ + 2 * kStage + kP + 2048;
};

}  // namespace

template <int HD>
__global__ void __launch_bounds__(320, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              AttnArgs a, unsigned* err) {
  using L = Smem<HD>;
  constexpr int HALF = HD / 2;  // head dims (and keys) per thread of a row pair
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int grp = a.hq / a.hkv, QN = 8 * grp;
  const int base = a.base[b];
  int lo = a.lo_fixed;
  if (a.window > 0) lo = max(lo, base - a.window);
  const int hi_max = base + 7;
  const int k_begin = max(lo, c * a.chunk);
  const int k_end = min((c + 1) * a.chunk, hi_max + 1);
  if (k_begin >= k_end) return;  // chunk outside this sequence's visible keys
  const int t0 = k_begin / kTileKeys;
  const int ntiles = (k_end + kTileKeys - 1) / kTileKeys - t0;

  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = sm;
  uint8_t* sKV = sQ + L::kQ;
  uint8_t* sP = sKV + 2 * L::kStage;
  uint64_t* bars = (uint64_t*)(sP + L::kP);
  uint64_t* kv_full = bars;       // [2]
  uint64_t* kv_empty = bars + 2;  // [2]
  uint64_t* s_full = bars + 4;    // [2] (S is double-buffered in TMEM)
  uint64_t* p_full = bars + 6;
  uint64_t* o_full = bars + 7;
  uint64_t* o_free = bars + 8;
  uint64_t* fin = bars + 9;
  uint64_t* mx = bars + 10;       // the two halves of a row have posted their tile maxima
  uint32_t* tmem_slot = (uint32_t*)(bars + 11);
  float* sCorr = (float*)(bars + 12);  // [64] per-query rescale factor of the current tile
  float* sMax = sCorr + 64;            // [2 tiles][2 halves][64] tile maxima
  float* sL = sMax + 256;              // [2][64] per-half running sums (at the end)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&kv_full[i]), 1);
      mbar_init(smem_u32(&kv_empty[i]), 1);
      mbar_init(smem_u32(&s_full[i]), 1);
    }
    mbar_init(smem_u32(p_full), 128);
    mbar_init(smem_u32(o_full), 1);
    mbar_init(smem_u32(o_free), 256);
    mbar_init(smem_u32(fin), 1);
    mbar_init(smem_u32(mx), 128);
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 8) tmem_alloc(smem_u32(tmem_slot), 512);

  // queries: fp32 -> bf16 [hi | lo] into the swizzled A operand (rows >= QN unused)
  {
    const int groups = QN * HD / 8;
    for (int idx = threadIdx.x; idx < groups; idx += blockDim.x) {
      const int r = idx / (HD / 8), k0 = (idx % (HD / 8)) * 8;
      const int s = r / grp, h = g * grp + (r % grp);
      const float* q = a.q + ((long)(b * 8 + s) * a.hq + h) * HD + k0;
      const float4 x0 = *(const float4*)q, x1 = *(const float4*)(q + 4);
      const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t hi[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * i + 1]);
        hi[i] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
        lw[i] = pack_bf16x2(v[2 * i] - __bfloat162float(h0), v[2 * i + 1] - __bfloat162float(h1));
      }
      const int blk = k0 / 64, ch = (k0 % 64) / 8;
      *(uint4*)(sQ + blk * kBlk + sw128(r, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *(uint4*)(sQ + (HD / 64 + blk) * kBlk + sw128(r, ch)) =
          make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 256;  // S buffers at columns 0 and 128, O at 256

  if (warp == 8) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol = policy_evict_first();
      const long krow0 = ((long)b * a.hkv + g) * a.max_ctx;
      const int vrow0 = (b * a.hkv + g) * HD;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t, ++issued) {
        const int s = t & 1;
        if (!mbar_wait(smem_u32(&kv_empty[s]), ((t >> 1) & 1) ^ 1, err)) break;
        const uint32_t full = smem_u32(&kv_full[s]);
        mbar_expect_tx(full, L::kStage);
        const int key0 = (t0 + t) * kTileKeys;
        uint8_t* st = sKV + s * L::kStage;
        for (int hb = 0; hb < HD / 64; ++hb)
          tma_load_2d(smem_u32(st + hb * kBlk), &tmK, hb * 64, (int)(krow0 + key0), full, pol);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(smem_u32(st + L::kKTile + kb * HD * 128), &tmV, key0 + kb * 64, vrow0,
                      full, pol);
      }
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
        mbar_wait(smem_u32(&kv_full[j & 1]), (j >> 1) & 1, err);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t id_qk = umma_idesc_bf16(128, kTileKeys);
      const uint32_t id_pv = umma_idesc_bf16(128, HD);
      auto issue_qk = [&](int t) -> bool {
        const int s = t & 1;
        if (!mbar_wait(smem_u32(&kv_full[s]), (t >> 1) & 1, err)) return false;
        tc_fence_after();
        uint8_t* st = sKV + s * L::kStage;
#pragma unroll
        for (int kb = 0; kb < L::kQBlocks; ++kb) {
          const uint64_t dq = umma_desc_sw128(smem_u32(sQ + kb * kBlk));
          const uint64_t dk = umma_desc_sw128(smem_u32(st + (kb % (HD / 64)) * kBlk));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + s * 128, dq + 2 * kk, dk + 2 * kk, id_qk, (kb | kk) ? 1u : 0u);
        }
        umma_commit(smem_u32(&s_full[s]));
        return true;
      };
      bool ok = issue_qk(0);
      for (int t = 0; t < ntiles && ok; ++t) {
        const int s = t & 1;
        // next tile's scores while the softmax of this one runs (its S buffer was
        // released when the softmax of tile t-1 arrived on p_full)
        if (t + 1 < ntiles && !issue_qk(t + 1)) break;
        if (!mbar_wait(smem_u32(p_full), t & 1, err)) break;
        if (t > 0 && !mbar_wait(smem_u32(o_free), (t - 1) & 1, err)) break;
        tc_fence_after();
        uint8_t* st = sKV + s * L::kStage;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t dp = umma_desc_sw128(smem_u32(sP + kb * kBlk));
          const uint64_t dv = umma_desc_sw128(smem_u32(st + L::kKTile + kb * HD * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tO, dp + 2 * kk, dv + 2 * kk, id_pv, (kb | kk) ? 1u : 0u);
        }
        umma_commit(smem_u32(o_full));
        umma_commit(smem_u32(&kv_empty[s]));
      }
      umma_commit(smem_u32(fin));  // all issued MMAs complete before TMEM is freed
    }
  } else {
    // warps 0-7. Warp w reads TMEM lanes 32*(w%4)..+31: warps 0,1,4,5 own the query rows
    // (lanes 0..63, softmax + P_hi.V), warps 2,3,6,7 the P_lo.V rows (lanes 64..127).
    // Warps w and w+4 share a row; w/4 picks the half of the keys / head dims.
    const int hf = warp >> 2;
    const int lrow = (warp & 3) * 32 + lane;  // TMEM lane
    const bool qrow = lrow < 64;
    const int r = qrow ? lrow : lrow - 64;     // query row 0..63
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float O[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) O[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int srow = r / grp;
    const int row_hi = a.causal ? base + srow : hi_max;
    const float scale = rsqrtf((float)HD);
    for (int t = 0; t < ntiles && ok; ++t) {
      float corr;
      if (qrow) {
        const int s = t & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[s]), (t >> 1) & 1, err));
        if (!ok) break;
        tc_fence_after();
        const int key0 = (t0 + t) * kTileKeys + hf * 64;
        const uint32_t tS = tmem + s * 128 + hf * 64 + lane_off;
        float mt = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float v[16];
          tmem_ld16(tS + cc * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int key = key0 + cc * 16 + j;
            if (key >= k_begin && key < k_end && key <= row_hi) mt = fmaxf(mt, v[j] * scale);
          }
        }
        float* smx = sMax + (t & 1) * 128;
        smx[hf * 64 + r] = mt;
        mbar_arrive(smem_u32(mx));
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(mx), t & 1, err));
        if (!ok) break;
        mt = fmaxf(mt, smx[(1 - hf) * 64 + r]);
        const float m_new = fmaxf(m, mt);
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
        corr = (m == -INFINITY) ? 0.f : __expf(m - mu);
        float lsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float v[16];
          tmem_ld16(tS + cc * 16, v);
          uint32_t ph[8], pl[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const int key = key0 + cc * 16 + j;
            const bool v0 = key >= k_begin && key < k_end && key <= row_hi;
            const bool v1 = key + 1 >= k_begin && key + 1 < k_end && key + 1 <= row_hi;
            const float p0 = v0 ? __expf(v[j] * scale - mu) : 0.f;
            const float p1 = v1 ? __expf(v[j + 1] * scale - mu) : 0.f;
            lsum += p0 + p1;
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            const __nv_bfloat162 pr =
                __floats2bfloat162_rn(p0 - __low2float(pb), p1 - __high2float(pb));
            ph[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
            pl[j / 2] = *reinterpret_cast<const uint32_t*>(&pr);
          }
          const int ch = cc * 2;  // block hf holds keys hf*64 .. hf*64+63
          uint8_t* pblk = sP + hf * kBlk;
          *(uint4*)(pblk + sw128(r, ch)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *(uint4*)(pblk + sw128(r, ch + 1)) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
          *(uint4*)(pblk + sw128(r + 64, ch)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          *(uint4*)(pblk + sw128(r + 64, ch + 1)) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
        }
        l = l * corr + lsum;
        m = m_new;
        if (hf == 0) sCorr[r] = corr;
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(smem_u32(p_full));
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(p_full), t & 1, err));
        if (!ok) break;
        corr = sCorr[r];
      }
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_full), t & 1, err));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < HALF / 16; ++cc) {
        float v[16];
        tmem_ld16(tO + lane_off + hf * HALF + cc * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) O[cc * 16 + j] = O[cc * 16 + j] * corr + v[j];
      }
      tc_fence_before();
      mbar_arrive(smem_u32(o_free));
    }
    // combine: P_lo.V rows and the second half's running sum arrive through shared memory
    // (the Q operand area is free once every MMA has completed)
    mbar_wait(smem_u32(fin), 0, err);
    float* xo = (float*)sQ;  // [64][HD + 4]
    if (!qrow) {
#pragma unroll
      for (int i = 0; i < HALF; i += 4)
        *(float4*)(xo + r * (HD + 4) + hf * HALF + i) = make_float4(O[i], O[i + 1], O[i + 2], O[i + 3]);
    } else {
      sL[hf * 64 + r] = l;
    }
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (qrow && r < QN) {
      const long pidx = ((long)b * a.hkv + g) * a.nchunk + c;
      float* po = a.part_o + (pidx * QN + r) * HD + hf * HALF;
      const float* lo_row = xo + r * (HD + 4) + hf * HALF;
#pragma unroll
      for (int i = 0; i < HALF; i += 4)
        *(float4*)(po + i) = make_float4(O[i] + lo_row[i], O[i + 1] + lo_row[i + 1],
                                         O[i + 2] + lo_row[i + 2], O[i + 3] + lo_row[i + 3]);
      if (hf == 0) {
        a.part_ml[(pidx * QN + r) * 2] = m;
        a.part_ml[(pidx * QN + r) * 2 + 1] = l + sL[64 + r];
      }
    }
  }
  __syncwarp();
  mbar_wait(smem_u32(fin), 0, err);
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int attn_tc_init_attributes() {
  cudaError_t e1 = cudaFuncSetAttribute(k_attn_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Smem<128>::kBytes);
  cudaError_t e2 = cudaFuncSetAttribute(k_attn_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Smem<64>::kBytes);
  return (e1 == cudaSuccess && e2 == cudaSuccess) ? 0 : -1;
}

void op_attention_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     unsigned* err, cudaStream_t st) {
  dim3 grid(a.nchunk, a.hkv, a.B);
  if (a.hd == 128)
    k_attn_tc<128><<<grid, 320, Smem<128>::kBytes, st>>>(tmK, tmV, a, err);
  else
    k_attn_tc<64><<<grid, 320, Smem<64>::kBytes, st>>>(tmK, tmV, a, err);
  op_attention_merge(1, a, st);
}

}  // namespace dmtp
