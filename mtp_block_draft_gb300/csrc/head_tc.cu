// LM head with the row argmax fused (steps a1, a3 and a4 of the round): for every token
// row m, argmax_v of l[m][v] = X[m] . W[v] over the whole vocabulary, or under sampled
// verification argmax_v of l[m][v] / temperature + G(m, v) (Gumbel-max sampling; the
// noise and its base-2 comparison form come from common.cuh).
//
// Token-major tcgen05 GEMM. Tokens are the MMA's M side (one or two 128-row halves,
// TH), vocabulary rows its N side (NV = 128 or 256 per tile), so each epilogue lane owns
// one token row and walks consecutive vocabulary columns: the argmax is a running
// compare in registers, with no cross-lane reduction, and a sampled pick's Philox block
// serves four adjacent columns of the same lane. One CTA per SM loops over the vocabulary
// tiles; with two TMEM accumulator buffers (when 2 * TH * NV <= 512 columns) the
// epilogue of tile i overlaps the MMAs of tile i + 1.
//
// Warps: 0 TMA producer (W tile and the token rows, every k block), 1 MMA issuer (and
// TMEM owner), 2.. epilogue (4 or 8 warps; TMEM lane quarter = warp % 4). Each CTA folds its running
// maxima into the global keys with one atomicMax per token row at the end.
//
// Every mbarrier wait is bounded (common.cuh): a timeout sets the error word and the
// role stops; the producer drains its in-flight copies and TMEM is freed before exit.
#include "common.cuh"
#include "ops.h"

namespace dmtp {

namespace {

constexpr int kRowB = 128;  // bytes of one operand row per stage: 64 bf16 or 128 E4M3 k
constexpr size_t kHeadSmemBudget = 200 * 1024;

__device__ __forceinline__ void arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

struct HeadArgs {
  int V, K, M, MT, stages, tiles;
  unsigned long long* keys;
  float* logits;
  long ldl;
  SampleArgs smp;
  unsigned* err;
  const float* wscale;  // E4M3 operands: per vocabulary row scale (padded past V)
  const float* xscale;  // E4M3 operands: per token row scale
  const int* vdev;      // token list: rows scored (device, read at launch), else null
  const int* vmap;      // token list: token id of each row (debug logits), else null
  float2* conf;         // confidence partials [grid * EW/4][M] (max, windowed sum), or null
};

// Window of the head confidence: scores more than this far below the best are left out
// of the normalising sum (the colibri page's per-step estimate for MTP-style heads).
constexpr float kConfWindow = 20.f;

// Running (max, sum of exp(l - max) over l >= max - window) of one token row over 16
// columns: lim valid columns; FP8: the accumulators times the column scales and the row's
// own scale xs give the logits.
template <bool FP8>
__device__ __forceinline__ void conf16(const uint32_t (&r)[16], int n0, int lim, float xs,
                                       const float* wscale, float& cm, float& cs) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= lim) break;
    const float x = __uint_as_float(r[j]) * (FP8 ? wscale[n0 + j] * xs : 1.f);
    if (x > cm) {
      cs = cs * __expf(cm - x) + 1.f;  // cm = -inf: cs = 0 * 0 + 1
      cm = x;
    } else if (x >= cm - kConfWindow) {
      cs += __expf(x - cm);
    }
  }
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 inputs, fp32 accumulate (kind::f8f6f4).
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor: D fp32, A and B E4M3 (format code 0), both K-major, M x N.
constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Running (best value, first index) of one token row over 16 columns n0 + j; FULL: all
// 16 columns are inside the vocabulary (else only j < lim). FP8: the accumulators are
// scaled by the columns' power-of-two scales (exact; the row's own scale is common to
// the row and left out of the comparison).
template <bool SAMPLE, bool FULL, bool FP8>
__device__ __forceinline__ void scan16(const uint32_t (&r)[16], int n0, int lim, float& best,
                                       int& bidx, const SampleArgs& s, int pos, int seq,
                                       const float* wscale) {
  float sc[16];
  if (FP8) {
    const float4* ws = reinterpret_cast<const float4*>(wscale + n0);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float4 w4 = __ldg(ws + g);
      sc[4 * g + 0] = __uint_as_float(r[4 * g + 0]) * w4.x;
      sc[4 * g + 1] = __uint_as_float(r[4 * g + 1]) * w4.y;
      sc[4 * g + 2] = __uint_as_float(r[4 * g + 2]) * w4.z;
      sc[4 * g + 3] = __uint_as_float(r[4 * g + 3]) * w4.w;
    }
  } else if (SAMPLE) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 blk = philox4x32_10(
          make_uint4((uint32_t)((n0 >> 2) + g), (uint32_t)pos, (uint32_t)seq, 0u), s.seed_lo,
          s.seed_hi);
      sc[4 * g + 0] = fmaf(__uint_as_float(r[4 * g + 0]), s.scale2, gumbel2_of_word(blk.x));
      sc[4 * g + 1] = fmaf(__uint_as_float(r[4 * g + 1]), s.scale2, gumbel2_of_word(blk.y));
      sc[4 * g + 2] = fmaf(__uint_as_float(r[4 * g + 2]), s.scale2, gumbel2_of_word(blk.z));
      sc[4 * g + 3] = fmaf(__uint_as_float(r[4 * g + 3]), s.scale2, gumbel2_of_word(blk.w));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) sc[j] = __uint_as_float(r[j]);
  }
  // strict '>' in increasing column order keeps the first index of equal maxima
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool take = sc[j] > best && (FULL || j < lim);
    best = take ? sc[j] : best;
    bidx = take ? n0 + j : bidx;
  }
}

// EW epilogue warps (4 or 8): with 8, two warps share each TMEM lane quarter and take
// alternate 32-column chunks of every accumulator. FP8: E4M3 operands (draft heads).
template <int NV, int TH, bool SAMPLE, int EW, bool FP8>
__global__ void __launch_bounds__(64 + 32 * EW, 1)
    k_head_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              HeadArgs a) {
  constexpr int NB = (2 * TH * NV <= 512) ? 2 : 1;  // accumulator buffers
  constexpr int ACC = TH * NV;                       // TMEM columns per buffer
  constexpr uint32_t kCols = NB * ACC;               // 256 or 512
  constexpr int kBK = FP8 ? 128 : 64;               // k elements per stage
  constexpr uint32_t kWBytes = NV * kRowB;
  constexpr uint32_t kXSlot = TH * 128 * kRowB;      // smem per stage for token rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int S = a.stages;
  uint8_t* sW = smem;
  uint8_t* sX = smem + (size_t)S * kWBytes;
  uint64_t* full = (uint64_t*)(sX + (size_t)S * kXSlot);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + NB;
  uint64_t* mma_done = acc_empty + NB;
  uint32_t* tmem_slot = (uint32_t*)(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = a.K / kBK;
  const uint32_t xbytes = (uint32_t)a.MT * kRowB;
  // rows scored: the vocabulary, or the first *vdev rows of a token list (same value for
  // every thread, so every role walks the same tiles)
  const int V = a.vdev ? max(0, min(a.V, __ldg(a.vdev))) : a.V;
  const int tiles = a.vdev ? (V + NV - 1) / NV : a.tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(smem_u32(&acc_full[i]), 1);
      mbar_init(smem_u32(&acc_empty[i]), EW);
    }
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next launch may begin (this CTA holds its TMEM); then the grid dependency (the
  // token list's length, read above, is set before a round starts)
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pw = policy_evict_first(), px = policy_evict_last();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(smem_u32(&empty[s]), ((it / S) & 1) ^ 1, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(smem_u32(&full[s]), kWBytes + xbytes);
          tma_load_2d(smem_u32(sW + (size_t)s * kWBytes), &tmW, kb * kBK, t * NV,
                      smem_u32(&full[s]), pw);
          tma_load_2d(smem_u32(sX + (size_t)s * kXSlot), &tmX, kb * kBK, 0, smem_u32(&full[s]),
                      px);
        }
      }
      // drain: every stage's last issued load has landed before the CTA may exit
      for (int j = (it > S ? it - S : 0); j < it; ++j)
        mbar_wait(smem_u32(&full[j % S]), (j / S) & 1, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = FP8 ? umma_idesc_e4m3(128, NV) : umma_idesc_bf16(128, NV);
      int it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
        const int buf = tl % NB;
        // the epilogue has drained this buffer's previous tile
        if (!mbar_wait(smem_u32(&acc_empty[buf]), ((tl / NB) & 1) ^ 1, a.err)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + buf * ACC;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw = umma_desc_sw128(smem_u32(sW + (size_t)s * kWBytes));
          uint64_t dx[TH];
#pragma unroll
          for (int h = 0; h < TH; ++h)
            dx[h] = umma_desc_sw128(smem_u32(sX + (size_t)s * kXSlot + h * 128 * kRowB));
#pragma unroll
          for (int k = 0; k < 4; ++k)  // +32 B per MMA step (16 bf16 or 32 E4M3 k)
#pragma unroll
            for (int h = 0; h < TH; ++h) {
              if (FP8)
                umma_e4m3(dacc + h * NV, dx[h] + 2 * k, dw + 2 * k, idesc,
                          (kb > 0 || k > 0) ? 1u : 0u);
              else
                umma_bf16(dacc + h * NV, dx[h] + 2 * k, dw + 2 * k, idesc,
                          (kb > 0 || k > 0) ? 1u : 0u);
            }
          umma_commit(smem_u32(&empty[s]));
        }
        if (ok) umma_commit(smem_u32(&acc_full[buf]));
      }
      // every MMA issued here has completed before TMEM may be freed
      umma_commit(smem_u32(mma_done));
      mbar_wait(smem_u32(mma_done), 0, a.err);
    }
  } else {
    // ---------------- epilogue: one token row per lane and token half ----------------
    const int q = warp & 3;           // TMEM lane quarter this warp may read
    const int grp = (warp - 2) >> 2;  // which of the quarter's EW / 4 warps
    int m[TH], pos[TH], seq[TH], bidx[TH];
    float best[TH], cm[TH], cs[TH];
#pragma unroll
    for (int h = 0; h < TH; ++h) {
      m[h] = h * 128 + q * 32 + lane;
      best[h] = -__int_as_float(0x7f800000);  // -inf
      cm[h] = best[h];
      cs[h] = 0.f;
      bidx[h] = -1;
      pos[h] = seq[h] = 0;
      if (SAMPLE) {
        const int mc = min(m[h], a.M - 1);
        seq[h] = mc / a.smp.group;
        pos[h] = __ldg(a.smp.pos0 + seq[h]) + (mc - seq[h] * a.smp.group) + 1;
      }
    }
    int tl = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
      const int buf = tl % NB;
      if (!mbar_wait(smem_u32(&acc_full[buf]), (tl / NB) & 1, a.err)) break;
      tc_fence_after();
      const int n0 = t * NV;
      const int lim = V - n0;  // valid columns of this tile
#pragma unroll
      for (int h = 0; h < TH; ++h) {
        const uint32_t tb = tmem + buf * ACC + h * NV + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
        for (int c = grp * 32; c < NV; c += 32 * (EW / 4)) {
          uint32_t r0[16], r1[16];
          tmem_ld16_raw(tb + c, r0);
          tmem_ld16_raw(tb + c + 16, r1);
          tmem_wait_ld16(r0);
          reg_fence16(r1);
          if (a.logits && m[h] < a.M) {  // debug copy of the logits
            float* lr = a.logits + (long)m[h] * a.ldl;
            const float xs = FP8 ? a.xscale[m[h]] : 1.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int v0 = n0 + c + j, v1 = n0 + c + 16 + j;
              const float w0 = FP8 ? a.wscale[v0] * xs : 1.f;
              const float w1 = FP8 ? a.wscale[v1] * xs : 1.f;
              if (c + j < lim) lr[a.vmap ? a.vmap[v0] : v0] = __uint_as_float(r0[j]) * w0;
              if (c + 16 + j < lim) lr[a.vmap ? a.vmap[v1] : v1] = __uint_as_float(r1[j]) * w1;
            }
          }
          if (a.conf && m[h] < a.M) {  // the head's confidence (greedy draft heads)
            const float xs = FP8 ? a.xscale[m[h]] : 1.f;
            conf16<FP8>(r0, n0 + c, lim - c, xs, a.wscale, cm[h], cs[h]);
            conf16<FP8>(r1, n0 + c + 16, lim - c - 16, xs, a.wscale, cm[h], cs[h]);
          }
          if (c + 32 <= lim) {
            scan16<SAMPLE, true, FP8>(r0, n0 + c, 0, best[h], bidx[h], a.smp, pos[h], seq[h],
                                      a.wscale);
            scan16<SAMPLE, true, FP8>(r1, n0 + c + 16, 0, best[h], bidx[h], a.smp, pos[h],
                                      seq[h], a.wscale);
          } else {  // the vocabulary's ragged end
            scan16<SAMPLE, false, FP8>(r0, n0 + c, lim - c, best[h], bidx[h], a.smp, pos[h],
                                       seq[h], a.wscale);
            scan16<SAMPLE, false, FP8>(r1, n0 + c + 16, lim - c - 16, best[h], bidx[h], a.smp,
                                       pos[h], seq[h], a.wscale);
          }
        }
      }
      // this warp has read the buffer: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive(smem_u32(&acc_empty[buf]));
    }
#pragma unroll
    for (int h = 0; h < TH; ++h)
      if (m[h] < a.M && bidx[h] >= 0) atomicMax(&a.keys[m[h]], argmax_key(best[h], bidx[h]));
    if (a.conf) {  // this thread's partial of its rows, combined by op_conf_combine
      const long part = (long)blockIdx.x * (EW / 4) + grp;
#pragma unroll
      for (int h = 0; h < TH; ++h)
        if (m[h] < a.M) a.conf[part * a.M + m[h]] = make_float2(cm[h], cs[h]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

template <int NV, int TH, bool SAMPLE, int EW, bool FP8>
int set_attr(size_t smem) {
  return cudaFuncSetAttribute(k_head_tc<NV, TH, SAMPLE, EW, FP8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
         cudaSuccess;
}
// instances: greedy and sampled bf16 heads, greedy E4M3 draft heads
template <int NV, int TH>
int set_attrs(size_t smem) {
  return set_attr<NV, TH, false, 4, false>(smem) | set_attr<NV, TH, true, 4, false>(smem) |
         set_attr<NV, TH, false, 8, false>(smem) | set_attr<NV, TH, true, 8, false>(smem) |
         set_attr<NV, TH, false, 4, true>(smem) | set_attr<NV, TH, false, 8, true>(smem);
}

size_t head_smem(int nv, int th, int stages) {
  return 1024 + (size_t)stages * ((size_t)nv * kRowB + (size_t)th * 128 * kRowB) +
         (size_t)(2 * stages + 5) * 8 + 16;
}

int plan_common(HeadPlan* p, const void* W, int V, int K, const void* X, int M, int nsm, int nv,
                int ew, int kbk) {
  if (!W || !X || V < 1 || K < kbk || K % kbk || M < 1 || M > 256 || nsm < 1 ||
      (nv != 128 && nv != 256) || (ew != 4 && ew != 8) || ((uintptr_t)W & 15) ||
      ((uintptr_t)X & 15))
    return -10;
  p->ew = ew;
  p->V = V;
  p->K = K;
  p->M = M;
  p->MT = tc_mt(M);
  p->TH = p->MT > 128 ? 2 : 1;
  p->NV = nv;
  p->tiles = (V + nv - 1) / nv;
  p->grid = p->tiles < nsm ? p->tiles : nsm;
  int st = 8;
  while (st > 2 && head_smem(nv, p->TH, st) > kHeadSmemBudget) --st;
  p->stages = st;
  p->smem = head_smem(nv, p->TH, st);
  p->fp8 = 0;
  p->wscale = p->xscale = nullptr;
  p->vdev = p->vmap = nullptr;
  return p->smem > kHeadSmemBudget ? -10 : 0;
}

}  // namespace

int head_plan(HeadPlan* p, const void* W, int V, int K, const void* X, int M, int nsm, int nv,
              int ew) {
  int r = plan_common(p, W, V, K, X, M, nsm, nv, ew, 64);
  if (r) return r;
  r = tc_make_tmap(&p->tmW, W, (uint64_t)V, (uint64_t)K, (uint32_t)nv);
  if (r) return r;
  return tc_make_tmap(&p->tmX, X, (uint64_t)M, (uint64_t)K, (uint32_t)p->MT);
}

int head_plan_e4m3(HeadPlan* p, const void* W8, const float* wscale, int V, int K,
                   const void* X8, const float* xscale, int M, int nsm, int nv, int ew) {
  if (!wscale || !xscale || ((uintptr_t)wscale & 15)) return -10;
  int r = plan_common(p, W8, V, K, X8, M, nsm, nv, ew, 128);
  if (r) return r;
  p->fp8 = 1;
  p->wscale = wscale;
  p->xscale = xscale;
  r = tc_make_tmap_u8(&p->tmW, W8, (uint64_t)V, (uint64_t)K, (uint32_t)nv);
  if (r) return r;
  return tc_make_tmap_u8(&p->tmX, X8, (uint64_t)M, (uint64_t)K, (uint32_t)p->MT);
}

int head_init_attributes() {
  const size_t s = kHeadSmemBudget;
  return set_attrs<128, 1>(s) | set_attrs<128, 2>(s) | set_attrs<256, 1>(s) |
         set_attrs<256, 2>(s);
}

template <int NV, int TH, int EW>
void launch_ew(const HeadPlan& p, const HeadArgs& a, bool sample, cudaStream_t st) {
  const int threads = 64 + 32 * EW;
  if (p.fp8)
    launch_pdl(k_head_tc<NV, TH, false, EW, true>, p.grid, threads, p.smem, st, p.tmW, p.tmX, a);
  else if (sample)
    launch_pdl(k_head_tc<NV, TH, true, EW, false>, p.grid, threads, p.smem, st, p.tmW, p.tmX, a);
  else
    launch_pdl(k_head_tc<NV, TH, false, EW, false>, p.grid, threads, p.smem, st, p.tmW, p.tmX,
               a);
}
template <int NV, int TH>
void launch(const HeadPlan& p, const HeadArgs& a, bool sample, cudaStream_t st) {
  if (p.ew == 8)
    launch_ew<NV, TH, 8>(p, a, sample, st);
  else
    launch_ew<NV, TH, 4>(p, a, sample, st);
}

void op_head_tc(const HeadPlan& p, unsigned long long* keys, float* logits, long ldl,
                const SampleArgs* smp, unsigned* err, cudaStream_t st, float2* conf) {
  // the E4M3 draft heads never sample (only the verify head does)
  const bool sample = !p.fp8 && smp && smp->scale2 > 0.f;
  const HeadArgs a{p.V,  p.K,    p.M,   p.MT, p.stages, p.tiles,
                   keys, logits, ldl,   sample ? *smp : SampleArgs{}, err, p.wscale, p.xscale,
                   p.vdev, p.vmap, sample ? nullptr : conf};
  if (p.NV == 128)
    p.TH == 1 ? launch<128, 1>(p, a, sample, st) : launch<128, 2>(p, a, sample, st);
  else
    p.TH == 1 ? launch<256, 1>(p, a, sample, st) : launch<256, 2>(p, a, sample, st);
}

}  // namespace dmtp

namespace dmtp {

// Confidence of each head row from the partials: M* = the largest partial maximum, S =
// sum over partials within the window of M* of sum_i exp(max_i - M*), conf = 1 / S.
// Row m goes to dst[(m / per) * stride + off + m % per].
__global__ void k_conf_combine(const float2* __restrict__ parts, int nparts, int M, int per,
                               float* dst, int stride, int off) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float mx = -__int_as_float(0x7f800000);
  for (int i = 0; i < nparts; ++i) mx = fmaxf(mx, parts[(long)i * M + m].x);
  float S = 0.f;
  for (int i = 0; i < nparts; ++i) {
    const float2 p = parts[(long)i * M + m];
    if (p.y > 0.f && p.x >= mx - kConfWindow) S += p.y * __expf(p.x - mx);
  }
  dst[(m / per) * stride + off + m % per] = S > 0.f ? 1.f / S : 0.f;
}

int head_conf_parts(const HeadPlan& p) { return p.grid * (p.ew / 4); }

void op_conf_combine(const HeadPlan& p, const float2* parts, int per, float* dst, int stride,
                     int off, cudaStream_t st) {
  launch_pdl(k_conf_combine, (p.M + 127) / 128, 128, 0, st, parts, head_conf_parts(p), p.M, per,
             dst, stride, off);
}

}  // namespace dmtp
