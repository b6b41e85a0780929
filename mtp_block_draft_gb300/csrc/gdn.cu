// Gated DeltaNet recurrence over the verify rows (8, or fewer in a verify of fewer
// drafts) with per-row state snapshots.
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
// The fp32 state [dv][dk] of a (sequence, head) is read once into registers; the snapshots
// after rows 0..6 go to the slot buffers and the state after the last row back to the live
// buffer. Buffers are [B][8][H][dv][dk]; live[b] and slot[b][r] index them.
//
// k_gdn_cols (dk = 64 or 128, dv a multiple of 64): a CTA of 4 warps takes 64 state rows of
// one (sequence, head); lane l holds columns CW l .. CW l + CW - 1 (CW = dk / 32) of 16
// rows, so each warp's state loads and snapshot stores are contiguous runs of one row.
// The row products S k and S q of a warp's 16 rows (32 sums) reduce across its lanes by a
// reduce-scatter butterfly that leaves sum l on lane l (31 shuffles). The 8 rows'
// normalised q and k, v, the gates and k.q are prepared once in shared memory, so the row
// loop needs no block barrier; the output is taken as S_new q = alpha (S q) + u (k.q).
// k_gdn (other shapes): one CTA per (sequence, head), 256 / dv threads per state row.
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
  for (int r = 0; r < a.rows; ++r) {
    const float* row = a.qkvab + (long)(b * a.rows + r) * a.ld;
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
    if (sub == 0) store_act((T*)a.out + (long)(b * a.rows + r) * a.H * dv + h * dv + i, a.out_lo, o);
    if (a.snapshots && r < a.rows - 1) {
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

template <int CW>
__device__ __forceinline__ void load_cw(const float* p, float (&x)[CW]) {
  if constexpr (CW == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x, x[1] = v.y;
  }
}

template <int CW>
__device__ __forceinline__ void store_cw(float* p, const float (&x)[CW]) {
  if constexpr (CW == 4)
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}

// v[0..31] of each lane -> the sum over the warp of v[lane] (returned on lane `lane`).
// Level n pairs lanes l and l ^ n: the lane with bit n set keeps entries n..2n-1, the
// other entries 0..n-1, and each adds the partner's copy of the entries it keeps.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int n = 16; n >= 1; n >>= 1) {
    const bool up = lane & n;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = up ? v[k] : v[k + n];
      const float keep = up ? v[k + n] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, n);
    }
  }
  return v[0];
}

template <typename T, int CW>
__global__ void __launch_bounds__(128, 4) k_gdn_cols(GdnArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int DK = 32 * CW;
  __shared__ __align__(16) float qs[8][DK], ks[8][DK];
  __shared__ float vs[8][64], als[8], bes[8], kqs[8];
  const int H = a.H, dv = a.dv;
  const int nparts = dv / 64;
  const int bh = blockIdx.x / nparts, part = blockIdx.x % nparts;
  const int b = bh / H, h = bh % H;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // warp w prepares rows w and w + 4
  for (int r = w; r < a.rows; r += 4) {
    const float* row = a.qkvab + (long)(b * a.rows + r) * a.ld;
    float q[CW], k[CW];
    load_cw<CW>(row + h * DK + CW * lane, q);
    load_cw<CW>(row + H * DK + h * DK + CW * lane, k);
    float qn = 0.f, kn = 0.f, kq = 0.f;
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      qn += q[c] * q[c];
      kn += k[c] * k[c];
      kq += q[c] * k[c];
    }
    qn = warp_sum(qn);
    kn = warp_sum(kn);
    kq = warp_sum(kq);
    const float rq = rsqrtf(fmaxf(qn, 1e-30f)), rk = rsqrtf(fmaxf(kn, 1e-30f));
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      qs[r][CW * lane + c] = q[c] * rq;
      ks[r][CW * lane + c] = k[c] * rk;
    }
    const float* vrow = row + 2 * H * DK + h * dv + part * 64;
    vs[r][lane] = vrow[lane];
    vs[r][lane + 32] = vrow[lane + 32];
    if (lane == 0) {
      als[r] = 1.f / (1.f + __expf(-row[2 * H * DK + H * dv + h]));
      bes[r] = 1.f / (1.f + __expf(-row[2 * H * DK + H * dv + H + h]));
      kqs[r] = kq * rq * rk;
    }
  }
  __syncthreads();
  const long hs = (long)dv * DK;
  const int i0 = part * 64 + w * 16;  // this warp's first state row
  const int live = a.live[b];
  float* Sbuf = a.states + (long)b * 8 * H * hs;
  const long off = (long)h * hs + (long)i0 * DK + CW * lane;  // within one buffer
  float S[16][CW];
#pragma unroll
  for (int t = 0; t < 16; ++t) load_cw<CW>(Sbuf + (long)live * H * hs + off + t * DK, S[t]);
  const int nv = a.rows_valid[b];
  const int t_own = lane & 15;
  for (int r = 0; r < a.rows; ++r) {
    float k[CW], q[CW];
    load_cw<CW>(&ks[r][CW * lane], k);
    load_cw<CW>(&qs[r][CW * lane], q);
    float v[32];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int c = 0; c < CW; ++c) {
        sk += S[t][c] * k[c];
        sq += S[t][c] * q[c];
      }
      v[t] = sk;
      v[16 + t] = sq;
    }
    // lanes 0..15: (S k) of row i0 + lane; lanes 16..31: (S q) of row i0 + lane - 16
    const float x = reduce_scatter32(v, lane);
    const float al = als[r], be = bes[r];
    const float u = be * vs[r][w * 16 + t_own] - al * be * x;  // valid on lanes 0..15
    const float u_own = __shfl_sync(0xffffffffu, u, t_own);
    const bool upd = r < nv;
    if (lane >= 16)
      store_act((T*)a.out + (long)(b * a.rows + r) * H * dv + h * dv + i0 + t_own, a.out_lo,
                upd ? al * x + u_own * kqs[r] : x);
    if (upd) {
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float ut = __shfl_sync(0xffffffffu, u, t);
#pragma unroll
        for (int c = 0; c < CW; ++c) S[t][c] = al * S[t][c] + ut * k[c];
      }
    }
    if (a.snapshots && r < a.rows - 1) {
      float* Sd = Sbuf + (long)a.slot[b * 8 + r] * H * hs + off;
#pragma unroll
      for (int t = 0; t < 16; ++t) store_cw<CW>(Sd + t * DK, S[t]);
    }
  }
  float* Sd = Sbuf + (long)live * H * hs + off;
#pragma unroll
  for (int t = 0; t < 16; ++t) store_cw<CW>(Sd + t * DK, S[t]);
}

void op_gdn(int dt, const GdnArgs& a, cudaStream_t st) {
  if (a.rows < 1 || a.rows > 8) return;  // the host passes 1..8 rows per sequence
  const bool cols = (a.dk == 64 || a.dk == 128) && a.dv % 64 == 0 && a.ld % 4 == 0 &&
                    aligned_to(a.qkvab, 16) && aligned_to(a.states, 16);
  if (cols) {
    const int grid = a.B * a.H * (a.dv / 64);
    if (a.dk == 128) {
      if (dt)
        launch_pdl(k_gdn_cols<bf16, 4>, grid, 128, 0, st, a);
      else
        launch_pdl(k_gdn_cols<float, 4>, grid, 128, 0, st, a);
    } else {
      if (dt)
        launch_pdl(k_gdn_cols<bf16, 2>, grid, 128, 0, st, a);
      else
        launch_pdl(k_gdn_cols<float, 2>, grid, 128, 0, st, a);
    }
    return;
  }
  if (dt)
    k_gdn<bf16><<<a.B * a.H, 256, 0, st>>>(a);
  else
    k_gdn<float><<<a.B * a.H, 256, 0, st>>>(a);
}

}  // namespace dmtp
