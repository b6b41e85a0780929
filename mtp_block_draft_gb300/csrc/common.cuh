// Shared device helpers for the DMTP round kernels (sm_103a).
//
// Inline PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the 5th-generation
// tensor cores (tcgen05: TMEM alloc, MMA, commit, TMEM loads), bf16 conversions, and
// the device error word. Every spin-wait is bounded by the global timer: after
// DMTP_WAIT_NS nanoseconds it sets an error bit and returns false, so a broken
// pipeline ends the kernel instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#define DMTP_WAIT_NS 2000000000ull

// bits of the device error word
#define DMTP_ERR_TOKEN 1u      // a token id outside [0, V)
#define DMTP_ERR_POS 2u        // a KV write at a position >= max_ctx
#define DMTP_ERR_TIMEOUT 4u    // a bounded mbarrier wait gave up
#define DMTP_ERR_SLOT 8u       // a snapshot slot index outside [0, 8)

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------------
// Programmatic dependent launch (griddepcontrol). A kernel launched with launch_pdl()
// may begin while the kernel before it in the stream is still running: its CTAs set up
// shared memory, barriers and TMEM, but read nothing that an earlier launch writes until
// pdl_wait() returns (the previous grid has completed and its writes are visible). pdl_trigger() lets the next launch begin; a CTA that
// allocates TMEM calls it only after its allocation, so that a successor's CTA never
// holds the columns a running CTA is still waiting for. Both are no-ops in a kernel
// launched without the attribute.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

namespace dmtp {
extern thread_local bool g_pdl_prev;  // ops.h
bool pdl_enabled();

// Launch `k` (a kernel that calls pdl_wait() before touching memory that earlier
// launches write) allowing programmatic overlap with the previous kernel of `st`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = (g_pdl_prev && pdl_enabled()) ? 1 : 0;
  g_pdl_prev = true;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}
// The same, launched in clusters of `cluster` CTAs (1: no clusters).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (cluster.x * cluster.y * cluster.z > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster.x;
    at[n].val.clusterDim.y = cluster.y;
    at[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  if (g_pdl_prev && pdl_enabled()) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  g_pdl_prev = true;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
  if (e != cudaSuccess && getenv("DMTP_VERBOSE"))
    fprintf(stderr, "dmtp: launch of grid (%u, %u, %u) x %u threads, %zu B shared, cluster "
            "(%u, %u, %u), %u attribute(s): %s\n", grid.x, grid.y, grid.z, block.x, smem,
            cluster.x, cluster.y, cluster.z, n, cudaGetErrorString(e));
  return e;
}
}  // namespace dmtp

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Store one element of a GEMM operand. bf16 storage writes the rounded value at p[0]
// and, when lo_off != 0, the bf16 rounding remainder v - hi at p[lo_off] (the "lo"
// half: hi + lo carries ~16 significant bits). fp32 storage keeps v itself.
__device__ __forceinline__ void store_act(float* p, long lo_off, float v) {
  (void)lo_off;
  p[0] = v;
}
__device__ __forceinline__ void store_act(bf16* p, long lo_off, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  p[0] = h;
  if (lo_off) p[lo_off] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// Four consecutive elements: p 16-byte aligned (fp32) or 8-byte aligned (bf16), and,
// for bf16, p + lo_off 8-byte aligned. Same rounding as four store_act calls.
__device__ __forceinline__ void store_act4(float* p, long lo_off, float4 v) {
  (void)lo_off;
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void store_act4(bf16* p, long lo_off, float4 v) {
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
  uint2 hv;
  hv.x = *reinterpret_cast<const uint32_t*>(&h01);
  hv.y = *reinterpret_cast<const uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(p) = hv;
  if (lo_off) {
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
    uint2 lv;
    lv.x = *reinterpret_cast<const uint32_t*>(&l01);
    lv.y = *reinterpret_cast<const uint32_t*>(&l23);
    *reinterpret_cast<uint2*>(p + lo_off) = lv;
  }
}
__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__host__ __device__ inline bool aligned_to(const void* p, unsigned bytes) {
  return ((uintptr_t)p % bytes) == 0;
}

__device__ __forceinline__ void set_err(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Maximum over a block of up to 1024 threads; `red` is >= 32 floats of shared memory.
__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : -INFINITY;
  return warp_max(t);
}

// E4M3 rows (draft-head quantisation): a row with largest magnitude amax gets the scale
// 2^e, e the smallest integer with amax <= 448 * 2^e (0 for an all-zero row), and its
// values are stored as round-to-nearest-even E4M3 of value * 2^-e (exact scaling).
__device__ __forceinline__ int e4m3_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  frexpf(amax * (1.f / 448.f), &e);  // a guess within one step; made exact below
  while (amax > ldexpf(448.f, e)) ++e;
  while (amax <= ldexpf(448.f, e - 1)) --e;
  return e;
}
// Four values (already scaled into [-448, 448]) as four E4M3 bytes, x at the lowest address.
__device__ __forceinline__ uint32_t e4m3x4(float4 v) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Sum over a block of up to 1024 threads; `red` is >= 32 floats of shared memory.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// Argmax key: orderable float bits in the high word, (0xffffffff - index) in the low
// word, so that an unsigned max picks the largest value and, among equal values,
// the lowest index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  unsigned u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - (unsigned)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xffffffffu - (unsigned)(k & 0xffffffffull));
}
__device__ __forceinline__ float argmax_key_value(unsigned long long k) {
  unsigned u = (unsigned)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
  return __uint_as_float(u);
}

// ---------------------------------------------------------------------------------
// Sampling noise for target-only sampled verification
// ---------------------------------------------------------------------------------
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011): each round multiplies counter words 0 and 2 by the
// two round constants and forms (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
// lo(M0 c0)); the key then takes one Weyl step.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}
__device__ __forceinline__ uint32_t word4(const uint4& b, int i) {
  return i == 0 ? b.x : i == 1 ? b.y : i == 2 ? b.z : b.w;
}
// Gumbel(0, 1) noise of one generator word, in base-2 units: G = -ln(-ln u) with
// u = ((w >> 8) + 1/2) 2^-24 in (0, 1) equals ln2 * G2 - ln(ln 2) for the returned
// G2 = -log2(e2), e2 = -log2(u). So argmax_v (l_v / T + G_v) = argmax_v (l_v log2(e) / T
// + G2_v): the sampled scores compare in this scaled form (one exact monotone map).
// e2 is formed without cancellation: for t = 1 - u < 2^-6 (exact in fp32 there) from
// the series -ln(1 - t) = t + t^2/2 + t^3/3 + ... (three terms: relative error below
// t^3/4 < 1e-6), elsewhere (e2 > 0.022) from the fp32 base-2 logarithm of u. G2's
// absolute error stays near 1e-5.
__device__ __forceinline__ float gumbel2_of_word(uint32_t w) {
  const float k = (float)(w >> 8);
  const float u = fmaf(k, 5.9604644775390625e-8f, 2.98023223876953125e-8f);
  const float t = fmaf(-k, 5.9604644775390625e-8f, 1.f) - 2.98023223876953125e-8f;
  const float series =  // log2(e) (t + t^2/2 + t^3/3)
      t * fmaf(t, fmaf(t, 0.48089834696298783f, 0.72134752044448170f), 1.4426950408889634f);
  const float e2 = t < 0.015625f ? series : -__log2f(u);
  return -__log2f(e2);
}
// Sampled verification: row m of the verify head is sequence b = m / group at position
// p = pos0[b] + m % group; its sample for position p + 1 is argmax_v (l_v / tau + G_v),
// G_v from the Philox block of counter (v / 4, p + 1, b, 0) and key (k0, k1), word v % 4.
__device__ __forceinline__ uint4 sample_block(int v4, int m, const int* pos0, int group,
                                              uint32_t k0, uint32_t k1) {
  const int b = m / group;
  const int p = __ldg(pos0 + b) + (m - b * group) + 1;
  return philox4x32_10(make_uint4((uint32_t)v4, (uint32_t)p, (uint32_t)b, 0u), k0, k1);
}

// ---------------------------------------------------------------------------------
// mbarrier / TMA / tcgen05 (inline PTX)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity; gives up after limit_ns nanoseconds of the
// global timer, sets the timeout bit of the error word and returns false.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned* err,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer() - t0 > limit_ns) {
      set_err(err, DMTP_ERR_TIMEOUT);
      return false;
    }
  }
}
// The kernels' wait: gives up after DMTP_WAIT_NS.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err) {
  return mbar_wait_for(bar, parity, err, DMTP_WAIT_NS);
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}
// 2-D tiled TMA load global -> shared, completing on an mbarrier (x = inner coordinate).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"((uint64_t)tm), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load (x = inner coordinate).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk tensor reduction: add the shared-memory tile at smem (the box of the tensor map)
// into global memory at coordinates (x, y), element-wise atomically; completion of the
// shared-memory read is tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* tm, int x, int y,
                                                  uint32_t smem) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];"
      ::"l"((uint64_t)tm), "r"(x), "r"(y), "r"(smem)
      : "memory");
}
// Bulk tensor store of the shared-memory tile at smem to global coordinates (x, y, z).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, int x, int y, int z,
                                             uint32_t smem) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
      ::"l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(smem)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk operation of this thread has read its shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Make this thread's shared-memory writes visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Whole warp: allocate ncols TMEM columns (power of two >= 32); address goes to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate (kind::f16).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// ---- CTA pairs (cta_group::2): one MMA of M = 256 rows over the two SMs of a cluster
// of two; each CTA holds 128 rows of A and half of B's columns in its shared memory and
// gets its 128 rows of D in its own TMEM. Every tcgen05 allocation, MMA and commit of a
// pair kernel is of the cta_group::2 form.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t smem_in_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// All threads of both CTAs: release this CTA's prior shared-memory writes (barrier
// initialisation) to the cluster and wait for the other CTA to arrive.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// One warp of each CTA of the pair, collectively.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Issued by one thread of the even CTA: descriptors and TMEM address name the same
// offsets in both CTAs.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at this offset in both CTAs once the issued MMAs complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(both)
      : "memory");
}
// Tiled load into this CTA's shared memory completing on an mbarrier of either CTA of
// the pair (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int x,
                                                 int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx"
      "::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"((uint64_t)tm), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait: issue several, then tmem_wait_ld16 on the first set
// and reg_fence16 on the others, so no use of the registers moves above the wait.
__device__ __forceinline__ void tmem_ld16_raw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 64 elements (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                    // swizzle mode: 128 B
  return d;
}
// Instruction descriptor: D fp32, A and B bf16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
