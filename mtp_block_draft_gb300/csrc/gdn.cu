// Gated DeltaNet recurrence over the 8 verify rows with per-row state snapshots.
//
// Per head: q, k L2-normalised; alpha = sigmoid(a), beta = sigmoid(b);
//   S <- alpha * S (I - beta k k^T) + beta v k^T  =  alpha * S + u k^T,
//   u = beta * v - alpha * beta * (S k);   o = S q.
// Snapshots and the pointer swap follow the colibri speculative-decoding page,
// "Undoing rows on a model with recurrent state": the verify keeps a copy of the state
// as it stands after every row except the final one (slot r holds the state after row
// r), and when row r is the last accepted, slot r becomes the live state by an index
// swap, with no recomputation.
//
// One CTA per (sequence, head) keeps the fp32 state [dv][dk] in registers (256 / dv
// threads per state row), reads it once, writes the snapshots after rows 0..6 into the slot
// buffers and the state after the last row back into the live buffer. Buffers are
// [B][8][H][dv][dk]; live[b] and slot[b][r] index them.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

template <typename T>
__global__ void __launch_bounds__(256) k_gdn(GdnArgs a) {
  __shared__ float qs[256], ks[256], red[32];
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int dk = a.dk, dv = a.dv;
  const int TPR = 256 / dv;      // threads per state row (host checks 8 <= dv <= 256)
  const int cpt = dk / TPR;      // state columns per thread (host checks <= 64)
  const int i = threadIdx.x / TPR, sub = threadIdx.x % TPR;
  const int j0 = sub * cpt;
  const long hstride = (long)dv * dk;
  const int live = a.live[b];
  float* Sbuf = a.states + ((long)b * 8 * a.H) * hstride;
  const float* Sl = Sbuf + ((long)live * a.H + h) * hstride + (long)i * dk + j0;
  float S[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) S[c] = (c < cpt) ? Sl[c] : 0.f;
  const int nv = a.rows_valid[b];
  for (int r = 0; r < 8; ++r) {
    const float* row = a.qkvab + (long)(b * 8 + r) * a.ld;
    const float qv = threadIdx.x < dk ? row[h * dk + threadIdx.x] : 0.f;
    const float kv = threadIdx.x < dk ? row[a.H * dk + h * dk + threadIdx.x] : 0.f;
    const float qn = block_sum(qv * qv, red);
    const float kn = block_sum(kv * kv, red);
    if (threadIdx.x < dk) {
      qs[threadIdx.x] = qv * rsqrtf(fmaxf(qn, 1e-30f));
      ks[threadIdx.x] = kv * rsqrtf(fmaxf(kn, 1e-30f));
    }
    __syncthreads();
    const float al = 1.f / (1.f + __expf(-row[2 * a.H * dk + a.H * dv + h]));
    const float be = 1.f / (1.f + __expf(-row[2 * a.H * dk + a.H * dv + a.H + h]));
    float sk = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < cpt) sk += S[c] * ks[j0 + c];
    for (int o = TPR >> 1; o > 0; o >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
    const float u = be * row[2 * a.H * dk + h * dv + i] - al * be * sk;
    if (r < nv) {
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c < cpt) S[c] = al * S[c] + u * ks[j0 + c];
    }
    float o = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < cpt) o += S[c] * qs[j0 + c];
    for (int w = TPR >> 1; w > 0; w >>= 1) o += __shfl_xor_sync(0xffffffffu, o, w);
    if (sub == 0) store_act((T*)a.out + (long)(b * 8 + r) * a.H * dv + h * dv + i, a.out_lo, o);
    if (a.snapshots && r < 7) {
      float* Sd = Sbuf + ((long)a.slot[b * 8 + r] * a.H + h) * hstride + (long)i * dk + j0;
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c < cpt) Sd[c] = S[c];
    }
    __syncthreads();
  }
  float* Sd = Sbuf + ((long)live * a.H + h) * hstride + (long)i * dk + j0;
#pragma unroll
  for (int c = 0; c < 64; ++c)
    if (c < cpt) Sd[c] = S[c];
}

void op_gdn(int dt, const GdnArgs& a, cudaStream_t st) {
  if (dt)
    k_gdn<bf16><<<a.B * a.H, 256, 0, st>>>(a);
  else
    k_gdn<float><<<a.B * a.H, 256, 0, st>>>(a);
}

}  // namespace dmtp
