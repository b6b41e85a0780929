// fp32 GEMM for fp32-storage models (the tiny correctness configuration):
// out[m, n] (+)= sum_k X[m, k] W[n, k], with an accumulate epilogue or a fused
// row-argmax epilogue for the LM head. CUDA-core FMA; the bf16 models use the
// tcgen05 kernels in gemm_tc.cu instead.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

static constexpr int BN = 64, BM = 32, BK = 16;

// MODE 0: out += acc, 1: argmax keys (+ logits); with smp.scale2 > 0 the keys rank
// the sampled scores l * scale2 + G2 (common.cuh) instead of the logits.
template <int MODE>
__global__ void __launch_bounds__(256) k_gemm_simt(const float* __restrict__ W,
                                                   const float* __restrict__ X, int N, int K,
                                                   int M, float* out, int ldo,
                                                   unsigned long long* keys, float* logits,
                                                   long ldl, SampleArgs smp) {
  __shared__ float Ws[BK][BN + 1];
  __shared__ float Xs[BK][BM + 1];
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int tn = threadIdx.x % BN, tm = threadIdx.x / BN;  // tm in 0..3, 8 rows each
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int e = threadIdx.x; e < BK * BN; e += 256) {
      const int nn = e / BK, kk = e % BK;
      const int n = n0 + nn, k = k0 + kk;
      Ws[kk][nn] = (n < N && k < K) ? W[(long)n * K + k] : 0.f;
    }
    for (int e = threadIdx.x; e < BK * BM; e += 256) {
      const int mm = e / BK, kk = e % BK;
      const int m = m0 + mm, k = k0 + kk;
      Xs[kk][mm] = (m < M && k < K) ? X[(long)m * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float w = Ws[kk][tn];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += w * Xs[kk][tm * 8 + j];
    }
    __syncthreads();
  }
  const int n = n0 + tn;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int m = m0 + tm * 8 + j;
    if (MODE == 0) {
      if (n < N && m < M) out[(long)m * ldo + n] += acc[j];
    } else {
      float score = acc[j];
      if (smp.scale2 > 0.f && n < N && m < M) {
        const uint4 blk = sample_block(n >> 2, m, smp.pos0, smp.group, smp.seed_lo, smp.seed_hi);
        score = fmaf(acc[j], smp.scale2, gumbel2_of_word(word4(blk, n & 3)));
      }
      unsigned long long key = (n < N && m < M) ? argmax_key(score, n) : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other > key ? other : key;
      }
      if ((threadIdx.x & 31) == 0 && m < M && key) atomicMax(&keys[m], key);
      if (logits && n < N && m < M) logits[(long)m * ldl + n] = acc[j];
    }
  }
}

void op_gemm_simt_acc(const float* W, const float* X, int N, int K, int M, float* out, int ldo,
                      cudaStream_t st) {
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  k_gemm_simt<0><<<grid, 256, 0, st>>>(W, X, N, K, M, out, ldo, nullptr, nullptr, 0,
                                       SampleArgs{});
}

void op_gemm_simt_argmax(const float* W, const float* X, int N, int K, int M,
                         unsigned long long* keys, float* logits, long ldl,
                         const SampleArgs* smp, cudaStream_t st) {
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  k_gemm_simt<1><<<grid, 256, 0, st>>>(W, X, N, K, M, nullptr, 0, keys, logits, ldl,
                                       smp ? *smp : SampleArgs{});
}

}  // namespace dmtp
