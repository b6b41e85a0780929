// Split-K decode attention for the 8 rows of a round against a per-sequence KV cache.
//
// One CTA per (KV chunk, kv head, sequence) computes, for all 8 rows x the GQA group of
// query heads that share the kv head, a partial softmax (running max m, sum l and the
// unnormalised P.V) over its chunk of keys, so each cached K/V byte is read once per
// sequence and layer. A merge kernel combines the chunks.
//
// Visibility (DMTP blog §6.2 "Attention: One Backend, Different Visibility Rules"):
//   target verify and MTP rows are causal: row s sees keys lo..base+s;
//   the block drafter sees the anchor-relative window max(0, base-4096)..base-1 plus all
//   8 block keys (no mask inside the block: DFlash's block-diagonal mask).
// Caches: K [B][hkv][max_ctx][hd], V transposed and blocked by 64 keys
// [B][hkv][max_ctx/64][hd][64]. Chunks lie on
// an absolute grid of `chunk` keys (chunk c covers keys [c*chunk, (c+1)*chunk)), so
// tiles start at aligned key indices. Scores scaled by 1/sqrt(hd); softmax in fp32.
// This file holds the CUDA-core version (fp32 models); attention_tc.cu the tcgen05 one.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

static constexpr int kTK = 32;      // keys per shared-memory tile
static constexpr int kMaxDPT = 32;  // max head dims per thread

template <typename T>
__global__ void __launch_bounds__(256) k_attn_partial(AttnArgs a) {
  __shared__ float Ks[kTK][128];
  __shared__ float Vs[kTK][128];
  const int chunk_id = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int grp = a.hq / a.hkv, QN = 8 * grp, hd = a.hd;
  const int base = a.base[b];
  int lo = a.lo_fixed;
  if (a.window > 0) lo = max(lo, base - a.window);
  const int hi_max = base + a.rows - 1;
  const int k_begin = max(lo, chunk_id * a.chunk);
  const int k_end = min((chunk_id + 1) * a.chunk, hi_max + 1);
  const long pidx = ((long)b * a.hkv + g) * a.nchunk + chunk_id;
  float* pml = a.part_ml + pidx * QN * 2;
  float* po = a.part_o + pidx * QN * hd;
  if (k_begin >= k_end) return;  // the merge reads only chunks that hold keys

  const int TPQ = 256 / QN;  // threads per query
  const int DPT = hd / TPQ;  // head dims per thread, interleaved: dim = sub + TPQ * i
  const int qi = threadIdx.x / TPQ, sub = threadIdx.x % TPQ;
  const int s = qi / grp, hh = qi % grp, h = g * grp + hh;
  const int row_hi = a.causal ? base + s : hi_max;
  const float scale = rsqrtf((float)hd);

  float qr[kMaxDPT], acc[kMaxDPT];
  // query rows past the sequence's rows (a verify of fewer drafts) compute on zeros and
  // are never merged
  const bool live = s < a.rows;
  const float* qp = a.q + ((long)(b * a.rows + (live ? s : 0)) * a.hq + h) * hd;
#pragma unroll
  for (int i = 0; i < kMaxDPT; ++i) {
    qr[i] = (i < DPT && live) ? qp[sub + TPQ * i] * scale : 0.f;
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int cb = a.cseq ? a.cseq[b] : b;  // cache sequence of the row group
  const T* Kb = (const T*)a.Kc + ((long)cb * a.hkv + g) * a.max_ctx * hd;
  const T* Vb = (const T*)a.Vc + ((long)cb * a.hkv + g) * hd * a.max_ctx;  // [max_ctx/64][hd][64]

  for (int kt = k_begin; kt < k_end; kt += kTK) {
    const int nk = min(kTK, k_end - kt);
    __syncthreads();
    for (int e = threadIdx.x; e < kTK * hd; e += blockDim.x) {
      const int j = e / hd, dd = e % hd;
      Ks[j][dd] = (j < nk) ? to_f32(Kb[(long)(kt + j) * hd + dd]) : 0.f;
    }
    for (int e = threadIdx.x; e < kTK * hd; e += blockDim.x) {
      const int j = e % kTK, dd = e / kTK;  // keys contiguous in the transposed V
      const int key = kt + j;
      Vs[j][dd] = (j < nk) ? to_f32(Vb[((long)(key / 64) * hd + dd) * 64 + key % 64]) : 0.f;
    }
    __syncthreads();
    float sc[kTK];
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTK; ++j) {
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxDPT; ++i)
        if (i < DPT) p += qr[i] * Ks[j][sub + TPQ * i];
      for (int o = TPQ >> 1; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      const bool vis = (j < nk) && (kt + j <= row_hi);
      sc[j] = vis ? p : -INFINITY;
      mt = fmaxf(mt, sc[j]);
    }
    const float m_new = fmaxf(m, mt);
    if (m_new == -INFINITY) continue;
    const float corr = __expf(m - m_new);
    l *= corr;
#pragma unroll
    for (int i = 0; i < kMaxDPT; ++i) acc[i] *= corr;
#pragma unroll
    for (int j = 0; j < kTK; ++j) {
      const float p = __expf(sc[j] - m_new);
      l += p;
#pragma unroll
      for (int i = 0; i < kMaxDPT; ++i)
        if (i < DPT) acc[i] += p * Vs[j][sub + TPQ * i];
    }
    m = m_new;
  }
#pragma unroll
  for (int i = 0; i < kMaxDPT; ++i)
    if (i < DPT) po[(long)qi * hd + sub + TPQ * i] = acc[i];
  if (sub == 0) {
    pml[qi * 2] = m;
    pml[qi * 2 + 1] = l;
  }
}

template <typename T>
__global__ void k_attn_merge(AttnArgs a) {
  const int mrow = blockIdx.x, h = blockIdx.y;
  const int b = mrow / a.rows, s = mrow % a.rows;
  const int grp = a.hq / a.hkv, g = h / grp, hh = h % grp, qi = s * grp + hh, QN = 8 * grp;
  const int base = a.base[b];
  int lo = a.lo_fixed;
  if (a.window > 0) lo = max(lo, base - a.window);
  const int c0 = lo / a.chunk, c1 = min(a.nchunk - 1, (base + a.rows - 1) / a.chunk);
  const long p0 = ((long)b * a.hkv + g) * a.nchunk;
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c) M = fmaxf(M, a.part_ml[((p0 + c) * QN + qi) * 2]);
  float L = 0.f;
  for (int c = c0; c <= c1; ++c) {
    const float mc = a.part_ml[((p0 + c) * QN + qi) * 2];
    L += a.part_ml[((p0 + c) * QN + qi) * 2 + 1] * __expf(mc - M);
  }
  const float invL = 1.f / L;
  for (int dd = threadIdx.x; dd < a.hd; dd += blockDim.x) {
    float o = 0.f;
    for (int c = c0; c <= c1; ++c) {
      const float mc = a.part_ml[((p0 + c) * QN + qi) * 2];
      o += a.part_o[((p0 + c) * QN + qi) * a.hd + dd] * __expf(mc - M);
    }
    store_act((T*)a.out + (long)mrow * a.hq * a.hd + h * a.hd + dd, a.out_lo, o * invL);
  }
}

// Warp form: one warp per (row, query head), hd / 32 dimensions per lane; the lanes
// stride over the chunks for the maxima and sums.
template <typename T, int DPL>
__global__ void __launch_bounds__(256) k_attn_merge_w(AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + warp;
  if (h >= a.hq) return;
  const int mrow = blockIdx.x;
  const int b = mrow / a.rows, s = mrow % a.rows;
  const int grp = a.hq / a.hkv, g = h / grp, hh = h % grp, qi = s * grp + hh, QN = 8 * grp;
  const int base = a.base[b];
  int lo = a.lo_fixed;
  if (a.window > 0) lo = max(lo, base - a.window);
  const int c0 = lo / a.chunk, c1 = min(a.nchunk - 1, (base + a.rows - 1) / a.chunk);
  const long p0 = ((long)b * a.hkv + g) * a.nchunk;
  const float* ml = a.part_ml + (p0 * QN + qi) * 2;  // chunk c at ml[c * QN * 2]
  float M = -INFINITY;
  for (int c = c0 + lane; c <= c1; c += 32) M = fmaxf(M, ml[(long)c * QN * 2]);
  M = warp_max(M);
  float L = 0.f;
  for (int c = c0 + lane; c <= c1; c += 32)
    L += ml[(long)c * QN * 2 + 1] * __expf(ml[(long)c * QN * 2] - M);
  L = warp_sum(L);
  const float invL = 1.f / L;
  float acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
  const float* po = a.part_o + (p0 * QN + qi) * a.hd + lane * DPL;
  for (int c = c0; c <= c1; ++c) {
    const float w = __expf(ml[(long)c * QN * 2] - M);
    const float* pc = po + (long)c * QN * a.hd;
    if (DPL % 4 == 0) {
#pragma unroll
      for (int j = 0; j < DPL; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(pc + j);
        acc[j] += v.x * w;
        acc[j + 1] += v.y * w;
        acc[j + 2] += v.z * w;
        acc[j + 3] += v.w * w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[j] += pc[j] * w;
    }
  }
  T* out = (T*)a.out + (long)mrow * a.hq * a.hd + h * a.hd + lane * DPL;
  if (DPL % 4 == 0) {
#pragma unroll
    for (int j = 0; j < DPL; j += 4)
      store_act4(out + j, a.out_lo,
                 make_float4(acc[j] * invL, acc[j + 1] * invL, acc[j + 2] * invL,
                             acc[j + 3] * invL));
  } else {
#pragma unroll
    for (int j = 0; j < DPL; ++j) store_act(out + j, a.out_lo, acc[j] * invL);
  }
}

template <typename T>
static bool merge_w(const AttnArgs& a, cudaStream_t st) {
  const unsigned eo = sizeof(T) * 4;
  if (a.hd % 32 || !aligned_to(a.part_o, 16) || !aligned_to(a.out, eo) || a.out_lo % 4)
    return false;
  dim3 g(a.B * a.rows, (a.hq + 7) / 8);
  switch (a.hd / 32) {
    case 1: k_attn_merge_w<T, 1><<<g, 256, 0, st>>>(a); return true;
    case 2: k_attn_merge_w<T, 2><<<g, 256, 0, st>>>(a); return true;
    case 4: k_attn_merge_w<T, 4><<<g, 256, 0, st>>>(a); return true;
    case 8: k_attn_merge_w<T, 8><<<g, 256, 0, st>>>(a); return true;
    default: return false;
  }
}

void op_attention(int dt, const AttnArgs& a, cudaStream_t st) {
  dim3 g1(a.nchunk, a.hkv, a.B);
  if (dt)
    k_attn_partial<bf16><<<g1, 256, 0, st>>>(a);
  else
    k_attn_partial<float><<<g1, 256, 0, st>>>(a);
  op_attention_merge(dt, a, st);
}

void op_attention_merge(int dt, const AttnArgs& a, cudaStream_t st) {
  if (dt ? merge_w<bf16>(a, st) : merge_w<float>(a, st)) return;
  dim3 g2(a.B * a.rows, a.hq);
  if (dt)
    k_attn_merge<bf16><<<g2, 128, 0, st>>>(a);
  else
    k_attn_merge<float><<<g2, 128, 0, st>>>(a);
}

}  // namespace dmtp
