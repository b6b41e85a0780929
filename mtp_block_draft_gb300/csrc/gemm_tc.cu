// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   out[m, n] (+)= sum_k X[m, k] * W[n, k]        W: [N, K] weights, X: [M, K] tokens
//
// The round multiplies few token rows (M = 8 .. 256) by large weight matrices, so the
// kernel is "swap-AB": 128 weight rows form the MMA's M side (TMEM lanes) and all M
// token rows (padded to MT, a multiple of 16, <= 256) form its N side (TMEM columns).
// Each weight byte is loaded by exactly one CTA. CTAs split the weight rows in tiles
// of 128 and, where that leaves SMs idle, the K range (split-K); partial sums are
// reduced with fp32 atomic adds into the output (which may be the residual stream,
// so the residual add is fused).
//
// Pipeline per CTA (128 threads):
//   warp 0 lane 0: TMA producer, weights with L2 evict-first, tokens evict-last;
//   warp 1 lane 0: MMA issuer, 4 x (M=128, N=MT, K=16) per 64-wide k block;
//   warp 2: TMEM allocation; all 4 warps: epilogue (TMEM lane = weight row).
// Stages are 64-element (128 B) k slices with 128-byte swizzle.
//
// Split activations: the token operand may come as two bf16 halves, X = X_hi + X_lo
// (X_lo = the rounding remainder of X_hi), stored as 2*MT rows [hi; lo]. Both halves
// are multiplied by the same weight tile (one TMA load of W). Up to 128 token rows the
// halves are one load and one MMA of 2*MT columns, summed in the epilogue; above that
// they are two loads and two MMAs accumulating into the same TMEM columns. Either way
// the activations keep ~16 significant bits while the weights stay bf16 and each
// weight byte is still read once.
//
// The LM-head variant fuses the row argmax (DMTP blog §6.5: the vocabulary output
// layer scores every token): per column the CTA reduces its 128 vocabulary rows to a
// packed (value, index) key and merges it with one 64-bit atomicMax per column.
//
// Every mbarrier wait is bounded (common.cuh); a timeout sets the error word, the
// producer drains its in-flight copies and the CTA frees its TMEM before returning.
#include <stdio.h>

#include <algorithm>

#include "common.cuh"
#include "ops.h"

namespace dmtp {

static constexpr int kTileN = 128;   // weight rows per CTA (MMA M)
static constexpr int kBlockK = 64;   // k elements per stage (128 B of bf16)
static constexpr uint32_t kWBytes = kTileN * kBlockK * 2;

struct TcArgs {
  int N, K, M, MT, stages;
  int split;       // 1: X holds [hi; lo] halves of MT rows each
  int xbox, nx;    // X rows per TMA load / MMA, loads per stage
  float* out;
  int ldo;
  unsigned long long* keys;
  float* logits;
  long ldl;
  unsigned* err;
};

__host__ __device__ inline uint32_t tmem_cols_for(int MT) {
  uint32_t c = 32;
  while (c < (uint32_t)MT) c <<= 1;
  return c;
}

template <int EPI>  // 0: atomic add into out, 1: argmax keys (+ logits)
__global__ void __launch_bounds__(128, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // 1024-B aligned tiles
  const int S = a.stages;
  const uint32_t xbytes = (uint32_t)a.xbox * a.nx * kBlockK * 2;
  uint8_t* sW = smem;
  uint8_t* sX = smem + S * kWBytes;
  uint64_t* full = (uint64_t*)(sX + S * xbytes);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  unsigned long long* red = (unsigned long long*)(accum + 2);  // [4][MT] (argmax)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN;
  const int nkb = a.K / kBlockK;
  const int kb0 = (int)((long)blockIdx.y * nkb / gridDim.y);
  const int kb1 = (int)((long)(blockIdx.y + 1) * nkb / gridDim.y);
  // one accumulator of xbox columns; with two loads per stage (nx = 2: the hi and lo
  // halves of more than 128 token rows) both products accumulate into it
  const uint32_t ncols = tmem_cols_for(a.xbox);
  const bool lo_cols = a.split && a.nx == 1;  // hi and lo in one load: lo in columns MT..

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) tmem_alloc(smem_u32(tmem_slot), ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pw = policy_evict_first(), px = policy_evict_last();
    int issued = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++issued) {
      const int s = issued % S;
      const uint32_t ph = (issued / S) & 1;
      if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, a.err)) break;
      mbar_expect_tx(smem_u32(&full[s]), kWBytes + xbytes);
      tma_load_2d(smem_u32(sW + s * kWBytes), &tmW, kb * kBlockK, n0, smem_u32(&full[s]), pw);
      for (int j = 0; j < a.nx; ++j)
        tma_load_2d(smem_u32(sX + s * xbytes + j * a.xbox * kBlockK * 2), &tmX, kb * kBlockK,
                    j * a.xbox, smem_u32(&full[s]), px);
    }
    // drain: every stage's last issued load has landed before the CTA may exit
    for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
      mbar_wait(smem_u32(&full[j % S]), (j / S) & 1, a.err);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = umma_idesc_bf16(kTileN, a.xbox);
    int it = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      if (!mbar_wait(smem_u32(&full[s]), ph, a.err)) break;
      tc_fence_after();
      const uint64_t dw = umma_desc_sw128(smem_u32(sW + s * kWBytes));
#pragma unroll
      for (int k = 0; k < kBlockK / 16; ++k) {  // +32 B per K=16 step inside the swizzle atom
        for (int j = 0; j < a.nx; ++j) {
          const uint64_t dx =
              umma_desc_sw128(smem_u32(sX + s * xbytes + j * a.xbox * kBlockK * 2));
          umma_bf16(tmem, dw + 2 * k, dx + 2 * k, idesc, (kb > kb0 || k > 0 || j > 0) ? 1u : 0u);
        }
      }
      umma_commit(smem_u32(&empty[s]));
    }
    umma_commit(smem_u32(accum));  // always: the epilogue waits on it
  }
  __syncwarp();

  // ---------------- epilogue ----------------
  bool ok = mbar_wait(smem_u32(accum), 0, a.err);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  const int row = warp * 32 + lane;
  const int n = n0 + row;
  const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
  if (EPI == 0) {
    if (ok) {
      for (int c = 0; c < a.MT; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        if (lo_cols) {
          float w[16];
          tmem_ld16(tbase + a.MT + c, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += w[j];
        }
        if (n < a.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = c + j;
            if (m < a.M) atomicAdd(&a.out[(long)m * a.ldo + n], v[j]);
          }
        }
      }
    }
  } else {
    const bool okb = __syncthreads_and(ok);
    if (okb) {
      for (int c = 0; c < a.MT; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        if (lo_cols) {
          float w[16];
          tmem_ld16(tbase + a.MT + c, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += w[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = c + j;
          unsigned long long key = (n < a.N) ? argmax_key(v[j], n) : 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
            key = other > key ? other : key;
          }
          if (lane == 0) red[warp * a.MT + m] = key;
          if (a.logits && n < a.N && m < a.M) a.logits[(long)m * a.ldl + n] = v[j];
        }
      }
      __syncthreads();
      for (int m = threadIdx.x; m < a.M; m += blockDim.x) {
        unsigned long long k = red[m];
        for (int w = 1; w < 4; ++w) k = red[w * a.MT + m] > k ? red[w * a.MT + m] : k;
        atomicMax(&a.keys[m], k);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
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

static size_t smem_bytes(int MT, int xrows, int stages, bool argmax) {
  size_t b = 1024 + (size_t)stages * (kWBytes + (size_t)xrows * kBlockK * 2);
  b += (2 * stages + 2) * 8;
  if (argmax) b += 4 * (size_t)MT * 8;
  return b;
}

static constexpr size_t kSmemBudget = 200 * 1024;

int tc_mt(int M) { return std::max(16, (M + 15) / 16 * 16); }

int tc_plan(TcPlan* p, const void* W, int N, int K, const void* X, int M, int nsm, bool argmax,
            bool split) {
  if (M < 1 || M > 256 || K % kBlockK || N < 1) return -10;
  p->N = N;
  p->K = K;
  p->M = M;
  p->MT = tc_mt(M);
  p->split = split ? 1 : 0;
  const int xrows = split ? 2 * p->MT : p->MT;
  p->xbox = xrows <= 256 ? xrows : p->MT;
  p->nx = xrows / p->xbox;
  int st = 8;
  while (st > 2 && smem_bytes(p->MT, xrows, st, argmax) > kSmemBudget) --st;
  p->stages = st;
  p->smem = smem_bytes(p->MT, xrows, st, argmax);
  const int tiles = (N + kTileN - 1) / kTileN;
  const int nkb = K / kBlockK;
  int best = 1;
  if (!argmax) {
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
  p->splits = best;
  int r = tc_make_tmap(&p->tmW, W, (uint64_t)N, (uint64_t)K, kTileN);
  if (r) return r;
  // split: the tensor spans both halves (rows >= M of each half are ignored columns)
  r = tc_make_tmap(&p->tmX, X, (uint64_t)(split ? xrows : M), (uint64_t)K, (uint32_t)p->xbox);
  return r;
}

int tc_init_attributes() {
  cudaError_t e1 = cudaFuncSetAttribute(k_gemm_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(kSmemBudget + 8 * 1024));
  cudaError_t e2 = cudaFuncSetAttribute(k_gemm_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(kSmemBudget + 8 * 1024));
  return (e1 == cudaSuccess && e2 == cudaSuccess) ? 0 : -1;
}

void op_gemm_tc_acc(const TcPlan& p, float* out, int ldo, unsigned* err, cudaStream_t st) {
  TcArgs a{p.N, p.K, p.M, p.MT, p.stages, p.split, p.xbox, p.nx, out, ldo, nullptr, nullptr, 0,
           err};
  dim3 grid((p.N + kTileN - 1) / kTileN, p.splits);
  k_gemm_tc<0><<<grid, 128, p.smem, st>>>(p.tmW, p.tmX, a);
}

void op_gemm_tc_argmax(const TcPlan& p, unsigned long long* keys, float* logits, long ldl,
                       unsigned* err, cudaStream_t st) {
  TcArgs a{p.N, p.K, p.M, p.MT, p.stages, p.split, p.xbox, p.nx, nullptr, 0, keys, logits, ldl,
           err};
  dim3 grid((p.N + kTileN - 1) / kTileN, 1);
  k_gemm_tc<1><<<grid, 128, p.smem, st>>>(p.tmW, p.tmX, a);
}

}  // namespace dmtp
